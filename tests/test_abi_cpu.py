"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol,
and rejects bad arguments on the host before anything is launched."""
import ctypes
import os
import re

import pytest

from block_sparse_long_pool_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_pool.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"SPARSE_API\s+[\w\s\*]+?\b(sparse_\w+)\s*\(", text)


def test_header_declares_the_five_calls():
    names = set(declared_symbols())
    assert {"sparse_pool_append", "sparse_select_topk", "sparse_decode_attn", "sparse_verify_attn_grouped",
            "sparse_gather_offloaded"} <= names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(raw, name), f"{name} is declared but not exported"
        assert name in binding.SIGNATURES, f"{name} has no binding signature"


def test_only_declared_symbols_are_exported():
    out = os.popen(f"nm -D --defined-only {binding.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("sparse_")}
    assert ours == set(declared_symbols())


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    for code in range(-6, 0):
        assert binding.status_string(code) not in ("", "unknown status")
    assert lib.sparse_version() >= 100


FAKE = ctypes.c_void_p(0x10000)      # aligned, never dereferenced: validation fails first
ODD = ctypes.c_void_p(0x10002)


def test_append_rejects_bad_arguments(lib):
    f = lib.sparse_pool_append
    assert f(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 2, 0, 1, None) == binding.SPARSE_ERR_INVALID_ARG
    assert f(ODD, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 2, 0, 1, None) == binding.SPARSE_ERR_INVALID_ARG
    # 100 + 40 tokens do not fit T_cap = 128
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 3, 100, 40, None) == binding.SPARSE_ERR_INVALID_ARG
    assert "T_cap" in lib.sparse_last_error().decode()
    # 129 tokens need 3 compressed rows
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 2, 128, 1, None) == binding.SPARSE_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 4, 0, 0, None) == binding.SPARSE_ERR_INVALID_ARG


def test_select_rejects_bad_arguments(lib):
    f = lib.sparse_select_topk
    # k_tot smaller than n_init + n_local + k
    assert f(FAKE, FAKE, FAKE, 1, 2, 64, 1, 2, 8, FAKE, FAKE, 10, None, None) == binding.SPARSE_ERR_INVALID_ARG
    assert f(None, FAKE, FAKE, 1, 2, 64, 1, 2, 8, FAKE, FAKE, 11, None, None) == binding.SPARSE_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 1, 2, 64, -1, 2, 8, FAKE, FAKE, 11, None, None) == binding.SPARSE_ERR_INVALID_ARG


def test_select_ex_rejects_unknown_flags(lib):
    f = lib.sparse_select_topk_ex
    ok_flags = binding.SPARSE_SELECT_KEYS_READY
    assert f(FAKE, FAKE, FAKE, 1, 2, 64, 1, 2, 8, FAKE, FAKE, 11, 0x10, None, None) == binding.SPARSE_ERR_INVALID_ARG
    assert "flags" in lib.sparse_last_error().decode()
    # the flag itself is accepted: the call fails later, on the null F
    assert f(None, FAKE, FAKE, 1, 2, 64, 1, 2, 8, FAKE, FAKE, 11, ok_flags, None, None) == \
        binding.SPARSE_ERR_INVALID_ARG
    assert "null" in lib.sparse_last_error().decode()


def test_decode_rejects_bad_arguments(lib):
    f = lib.sparse_decode_attn
    args = [FAKE, FAKE, FAKE, 4096, None, FAKE, FAKE, 11, FAKE, 1, 8, 2, 0.0, FAKE, None, 0, 0, None, 0, None, None]
    bad = list(args)
    bad[10] = 7                                   # H_q not a multiple of H_kv
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    bad = list(args)
    bad[10], bad[11] = 34, 2                      # G = 17 > 16
    assert f(*bad) == binding.SPARSE_ERR_UNSUPPORTED
    bad = list(args)
    bad[0] = ODD
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    bad = list(args)
    bad[12] = float("nan")
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    ex = lib.sparse_decode_attn_ex
    assert ex(*args[:19], None, 1, 0, None, None) == binding.SPARSE_ERR_INVALID_ARG
    bad = list(args)
    bad[16], bad[17], bad[18] = binding.SPARSE_ATTN_TENSOR_MEMORY, FAKE, 1 << 20   # tensor memory + workspace
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    bad = list(args)
    bad[16] = 64                                  # an unknown flag bit
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    na = lib.sparse_decode_attn_noalloc
    assert na(*args[:16], binding.SPARSE_ATTN_TENSOR_MEMORY, None, None) == binding.SPARSE_ERR_INVALID_ARG


def test_verify_rejects_bad_arguments(lib):
    f = lib.sparse_verify_attn_grouped
    args = [FAKE, FAKE, FAKE, 65536, FAKE, 16, 8, 4, 8, FAKE, 4, 32, 8, 0.0, FAKE, None, 0, 0, None, None]
    bad = list(args)
    bad[7] = 5                                    # C*G = 20 rows > 16
    assert f(*bad) == binding.SPARSE_ERR_UNSUPPORTED
    bad = list(args)
    bad[5], bad[7] = 200, 3                       # union bound 3*200+8 > 512
    bad[11], bad[12] = 8, 8
    assert f(*bad) == binding.SPARSE_ERR_UNSUPPORTED
    bad = list(args)
    bad[4] = None
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    bad = list(args)
    bad[17] = 8                                   # an unknown flag bit
    assert f(*bad) == binding.SPARSE_ERR_INVALID_ARG
    assert lib.sparse_verify_attn_shared(*bad) == binding.SPARSE_ERR_INVALID_ARG


def test_gather_rejects_bad_arguments(lib):
    f = lib.sparse_gather_offloaded
    assert f(FAKE, FAKE, 4096, FAKE, FAKE, 11, 1, 2, FAKE, FAKE, None, 2000, None, None) == \
        binding.SPARSE_ERR_INVALID_ARG
    assert f(FAKE, ODD, 4096, FAKE, FAKE, 11, 1, 2, FAKE, FAKE, None, 8, None, None) == \
        binding.SPARSE_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        binding.sparse_select_topk(torch.zeros(1, 2, 128, dtype=torch.bfloat16),
                                   torch.zeros(1, 2, 64, 128), torch.zeros(1, dtype=torch.int32), 1, 2, 8,
                                   torch.zeros(1, 2, 11, dtype=torch.int32), torch.zeros(1, 2, dtype=torch.int32))


def test_decode_attn_forecast_rejects_bad_arguments(lib):
    f = lib.sparse_decode_attn_forecast
    #       Q     K     V     T_cap idx   cnt   k_tot seq   B  H_q H_kv scale O     lse
    args = [FAKE, FAKE, FAKE, 4096, FAKE, FAKE, 11, FAKE, 1, 8, 2, 0.0, FAKE, None,
            # F   ktil  N_cap n_init n_local k idx_next cnt_next k_tot_next n_split flags status stream
            FAKE, FAKE, 64, 1, 2, 8, FAKE, FAKE, 11, 0, 0, None, None]
    assert len(args) == len(binding.SIGNATURES["sparse_decode_attn_forecast"][1])

    def call(**kw):
        a = list(args)
        names = ["Q", "K", "V", "T_cap", "idx", "cnt", "k_tot", "seq", "B", "H_q", "H_kv", "scale", "O", "lse",
                 "F", "ktil", "N_cap", "n_init", "n_local", "k", "idx_next", "cnt_next", "k_tot_next", "n_split",
                 "flags", "status", "stream"]
        for k_, v in kw.items():
            a[names.index(k_)] = v
        return f(*a)

    assert call(Q=None) == binding.SPARSE_ERR_INVALID_ARG
    assert call(O=ODD) == binding.SPARSE_ERR_INVALID_ARG
    assert call(H_q=12, H_kv=8) == binding.SPARSE_ERR_INVALID_ARG              # H_q not a multiple of H_kv
    assert call(H_q=64, H_kv=2) == binding.SPARSE_ERR_UNSUPPORTED              # G = 32 > 16
    assert call(flags=binding.SPARSE_ATTN_STREAM_K) == binding.SPARSE_ERR_INVALID_ARG
    assert call(ktil=None) == binding.SPARSE_ERR_INVALID_ARG                   # F without compressed keys
    assert "ktil_next" in lib.sparse_last_error().decode()
    assert call(k_tot_next=10) == binding.SPARSE_ERR_INVALID_ARG               # < n_init + n_local + k
    assert call(ktil=ODD) == binding.SPARSE_ERR_INVALID_ARG
    assert call(n_local=-1) == binding.SPARSE_ERR_INVALID_ARG
    assert call(scale=float("inf")) == binding.SPARSE_ERR_INVALID_ARG


def test_select_heads_rejects_bad_arguments(lib):
    f = lib.sparse_select_topk_heads
    #        Q     ktil  seq   B  H_q H_kv N_cap scale init local k  idx   cnt   k_tot status stream
    args = [FAKE, FAKE, FAKE, 1, 8, 2, 64, 0.0, 1, 2, 8, FAKE, FAKE, 11, None, None]
    assert len(args) == len(binding.SIGNATURES["sparse_select_topk_heads"][1])

    def call(i, v):
        a = list(args)
        a[i] = v
        return f(*a)

    assert call(0, None) == binding.SPARSE_ERR_INVALID_ARG                 # no Q
    assert call(1, ODD) == binding.SPARSE_ERR_INVALID_ARG                  # misaligned keys
    assert call(4, 9) == binding.SPARSE_ERR_INVALID_ARG                    # H_q not a multiple of H_kv
    assert call(4, 64) == binding.SPARSE_ERR_UNSUPPORTED                   # G = 32 > 16
    assert call(7, -1.0) == binding.SPARSE_ERR_INVALID_ARG                 # negative scale
    assert call(13, 10) == binding.SPARSE_ERR_INVALID_ARG                  # k_tot < n_init + n_local + k


def test_append_kv_rejects_bad_arguments(lib):
    f = lib.sparse_pool_append_kv
    ok = (FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1, 1, 128, 2, 0, 1, None)
    bad_vtil = ok[:3] + (None,) + ok[4:]
    assert f(*bad_vtil) == binding.SPARSE_ERR_INVALID_ARG
    odd_khat = ok[:4] + (ODD,) + ok[5:]
    assert f(*odd_khat) == binding.SPARSE_ERR_INVALID_ARG
    too_long = ok[:12] + (100, 40) + ok[14:]   # 140 tokens do not fit T_cap = 128
    assert f(*too_long) == binding.SPARSE_ERR_INVALID_ARG


def test_nsa_rejects_bad_arguments(lib):
    f = lib.sparse_decode_attn_nsa
    # Q, K, V, T_cap, khat, vhat, N_cap, cmp_len, cmp_stride, idx, count, k_tot, seq_len, B, H_q, H_kv, w,
    # gates, scale, O, ws, ws_bytes, n_split, flags, status, stream
    ok = [FAKE, FAKE, FAKE, 4096, FAKE, FAKE, 64, 0, 0, FAKE, FAKE, 8, FAKE, 1, 8, 1, 512, FAKE, 0.0, FAKE, FAKE,
          1 << 20, 0, 0, None, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a4=None) == binding.SPARSE_ERR_INVALID_ARG            # no khat
    assert call(a20=None, a23=binding.SPARSE_NSA_BRANCH_GRID) == binding.SPARSE_ERR_INVALID_ARG  # no workspace
    assert call(a20=None, a14=16) == binding.SPARSE_ERR_INVALID_ARG   # G = 16 needs the workspace
    assert call(a5=ODD) == binding.SPARSE_ERR_INVALID_ARG             # misaligned vhat
    assert call(a14=12, a15=8) == binding.SPARSE_ERR_INVALID_ARG      # H_q not a multiple of H_kv
    assert call(a16=-1) == binding.SPARSE_ERR_INVALID_ARG             # negative window
    assert call(a16=5000) == binding.SPARSE_ERR_UNSUPPORTED           # window beyond T_cap
    assert call(a14=32, a15=1) == binding.SPARSE_ERR_UNSUPPORTED      # G = 32
    assert call(a21=16, a14=16) == binding.SPARSE_ERR_INVALID_ARG     # workspace too small
    assert call(a23=8) == binding.SPARSE_ERR_INVALID_ARG              # unknown flag
    assert call(a18=float("nan")) == binding.SPARSE_ERR_INVALID_ARG   # scale
    assert call(a7=16, a8=32) == binding.SPARSE_ERR_INVALID_ARG       # stride above the kernel
    assert call(a7=32, a8=0) == binding.SPARSE_ERR_INVALID_ARG        # zero stride
    assert lib.sparse_decode_attn_nsa_workspace_size(0, 8, 1) == 0
    assert lib.sparse_decode_attn_nsa_workspace_size(8, 64, 8) == 256 + 3 * 8 * 64 * 128 * 4


def test_nsa_compress_and_select_reject_bad_arguments(lib):
    f = lib.sparse_nsa_compress
    # k_cache, v_cache, T_cap, B, H_kv, len_before, n_new, l, s, khat, vhat, n_rows_cap, stream
    ok = [FAKE, FAKE, 1024, 1, 1, 0, 100, 32, 16, FAKE, FAKE, 64, None]

    def call_c(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call_c(a9=None) == binding.SPARSE_ERR_INVALID_ARG          # no khat
    assert call_c(a10=ODD) == binding.SPARSE_ERR_INVALID_ARG          # misaligned vhat
    assert call_c(a7=8) == binding.SPARSE_ERR_INVALID_ARG             # kernel below the stride
    assert call_c(a6=2000) == binding.SPARSE_ERR_INVALID_ARG          # beyond T_cap
    assert call_c(a11=3) == binding.SPARSE_ERR_INVALID_ARG            # more windows than rows
    assert call_c(a5=0, a6=20) == binding.SPARSE_OK                   # no window completes: nothing to do
    g = lib.sparse_nsa_select
    # Q, khat, n_rows_cap, l, s, seq_len, B, N_q, H_q, H_kv, scale, n_init, n_local, k, idx, count, k_tot,
    # status, stream
    ok2 = [FAKE, FAKE, 64, 32, 16, FAKE, 1, 1, 8, 1, 0.0, 1, 2, 4, FAKE, FAKE, 7, None, None]

    def call_s(**kw):
        a = list(ok2)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return g(*a)

    assert call_s(a1=None) == binding.SPARSE_ERR_INVALID_ARG          # no khat
    assert call_s(a16=6) == binding.SPARSE_ERR_INVALID_ARG            # k_tot too small
    assert call_s(a3=16, a4=32) == binding.SPARSE_ERR_INVALID_ARG     # stride above the kernel
    assert call_s(a8=64, a9=2) == binding.SPARSE_ERR_UNSUPPORTED      # G = 32
    assert call_s(a10=-1.0) == binding.SPARSE_ERR_INVALID_ARG         # negative scale
    assert call_s(a7=0) == binding.SPARSE_ERR_INVALID_ARG             # no query
    assert call_s(a6=4096, a7=16) == binding.SPARSE_ERR_UNSUPPORTED   # too many (pair, query) units


def test_prefill_select_rejects_bad_arguments(lib):
    f = lib.sparse_prefill_select
    # F, T_cap, ktil, N_cap, seq_len, B, H_kv, n_init, n_local, k, idx, count, k_tot, status, stream
    ok = [FAKE, 4096, FAKE, 64, FAKE, 1, 2, 1, 2, 8, FAKE, FAKE, 11, None, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a0=None) == binding.SPARSE_ERR_INVALID_ARG        # no F
    assert call(a2=ODD) == binding.SPARSE_ERR_INVALID_ARG         # misaligned keys
    assert call(a8=0) == binding.SPARSE_ERR_INVALID_ARG           # n_local = 0: the own block must be local
    assert call(a12=10) == binding.SPARSE_ERR_INVALID_ARG         # k_tot too small
    assert call(a3=4096) == binding.SPARSE_ERR_UNSUPPORTED        # more than 2048 compressed keys
