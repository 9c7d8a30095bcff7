"""GPU parity: every entry point of the C ABI against the fp64 oracle on seeded inputs.

Oracle inputs come only from the seeded generators (never from the CUDA path); the
CUDA path is called through the ctypes binding of libsparsepool.so.  Tolerances are
stated in parity_utils.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl
from parity_utils import (BLK, D, GpuLayer, assert_attn_close, assert_selection_matches, bits,
                          oracle_attn_on_taken_lists, oracle_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _lens_pair(lens_b, H_kv):
    return np.repeat(np.asarray(lens_b, dtype=np.int64), H_kv)


def _seq(lens_b):
    return torch.tensor(lens_b, dtype=torch.int32, device="cuda")


def _check_lse(lse_gpu, lse_ref, mask=None):
    g = lse_gpu.cpu().double().numpy().reshape(lse_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.allclose(g[fin], lse_ref[fin], rtol=0, atol=2e-3)


# ----------------------------------------------------------------------------- append / pooling


def test_append_bulk_then_incremental_matches_oracle():
    B, H_kv, T_cap = 2, 3, 10 * BLK
    N_cap = T_cap // BLK
    K = wl.randn_bf16((B, H_kv, T_cap, D), 501, "cuda")
    V = wl.randn_bf16((B, H_kv, T_cap, D), 502, "cuda")
    L = GpuLayer(B, 4 * H_kv, H_kv, T_cap, N_cap, 1, 2, 4)
    steps = [(0, 5 * BLK + 17), (5 * BLK + 17, 1), (5 * BLK + 18, 100), (5 * BLK + 118, 2 * BLK)]
    for start, n in steps:
        L.append(K[:, :, start:start + n], V[:, :, start:start + n], start)
        torch.cuda.synchronize()
        end = start + n
        assert torch.equal(L.k_cache[:, :, :end], K[:, :, :end])
        assert torch.equal(L.v_cache[:, :, :end], V[:, :, :end])
        assert not L.k_cache[:, :, end:].any()
        ref = oracle.pool(bits(K).reshape(B * H_kv, T_cap, D), [end] * (B * H_kv), N_cap)
        nb = (end + BLK - 1) // BLK
        got = L.ktil.cpu().double().numpy().reshape(B * H_kv, N_cap, D)
        assert np.allclose(got[:, :nb], ref[:, :nb], rtol=1e-5, atol=1e-6), f"after append to {end}"


def test_append_one_token_per_call_steady_decode():
    """Steady decode on the 32K append workload's shape (B=8, H_kv=8, G=4, k=32): from
    32672 tokens (mid block 510), 160 appends of ONE token each, so blocks 511 and 512
    are filled one token per call from empty (64 updates of their running mean each)
    and two block boundaries are crossed.  Every 16 appends the compressed keys are
    compared with the oracle's block means (1e-5 relative), the Forecast selection with
    the oracle's (near-tie rule), and at the end the attention over the oracle's lists."""
    sh = wl.LLAMA8B_32K
    B, H_kv, G, P = sh.B, sh.H_kv, sh.G, sh.pairs
    start, n_steps = 32768 - 96, 160
    T_end = start + n_steps
    N_cap = (T_end + BLK - 1) // BLK
    planted = wl.planted_sets(sh, 1)[0]
    K = torch.empty((B, H_kv, T_end, D), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    for p in range(P):
        b, h = divmod(p, H_kv)
        K[b, h], V[b, h] = wl.kv_pair(sh, 0, p, planted[p], "cuda", tokens=T_end)
    Kb, Vb = bits(K).reshape(P, T_end, D), bits(V).reshape(P, T_end, D)
    F = wl.forecast(sh, 0, 0, "cuda")
    Fb = bits(F).reshape(P, D)
    L = GpuLayer(B, sh.H_q, H_kv, T_end, N_cap, sh.n_init, sh.n_local, sh.k)
    L.append(K[:, :, :start], V[:, :, :start], 0)
    checked = 0
    for i in range(n_steps):
        pos = start + i
        L.append(K[:, :, pos:pos + 1], V[:, :, pos:pos + 1], pos)
        if (i + 1) % 16:
            continue
        end = pos + 1
        lens_p = [end] * P
        seq = _seq([end] * B)
        L.select(F, seq)
        torch.cuda.synchronize()
        assert L.status.item() == 0
        ref = oracle.pool(Kb, lens_p, N_cap)
        nb = (end + BLK - 1) // BLK
        got = L.ktil.cpu().double().numpy().reshape(P, N_cap, D)
        assert np.allclose(got[:, :nb], ref[:, :nb], rtol=1e-5, atol=1e-6), f"compressed keys after append to {end}"
        ridx, rcnt, rs = oracle.select(Fb, ref, lens_p, sh.n_init, sh.n_local, sh.k)
        assert_selection_matches(L.idx, L.count, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
        checked += 1
    assert checked == n_steps // 16
    assert torch.equal(L.k_cache, K) and torch.equal(L.v_cache, V)
    Q = wl.queries(sh, 0, "cuda")
    O = torch.zeros((B, sh.H_q, D), dtype=torch.bfloat16, device="cuda")
    binding.sparse_decode_attn(Q, L.k_cache, L.v_cache, torch.from_numpy(ridx).cuda().view(B, H_kv, -1),
                               torch.from_numpy(rcnt).cuda().view(B, H_kv), _seq([T_end] * B), O)
    torch.cuda.synchronize()
    Oref, _ = oracle.attn(bits(Q).reshape(P, G, D), Kb, Vb, ridx, rcnt, [T_end] * P)
    assert_attn_close(O, Oref.reshape(B, sh.H_q, D))


# ----------------------------------------------------------------------------- selection


def _select_case(lens_b, H_kv, N_cap, n_init, n_local, k, ktil_np, F):
    B = len(lens_b)
    P = B * H_kv
    k_cap = n_init + n_local + k
    ktil = torch.from_numpy(ktil_np.astype(np.float32)).cuda().view(B, H_kv, N_cap, D)
    idx = torch.full((B, H_kv, k_cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_select_topk(F, ktil, _seq(lens_b), n_init, n_local, k, idx, cnt, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    lens_p = _lens_pair(lens_b, H_kv)
    ref = oracle.select(bits(F).reshape(P, D), ktil_np.astype(np.float32).astype(np.float64), lens_p, n_init,
                        n_local, k, k_cap)
    return idx, cnt, ref, lens_p


@pytest.mark.parametrize("N_cap,lens_b,k", [(64, [4096, 3001, 65, 0], 8), (513, [32769, 32768], 32),
                                            (2048, [131072, 100000], 64), (16384, [1 << 20], 64),
                                            (5000, [320000, 319937, 1], 200)])
def test_select_matches_oracle_random_scores(N_cap, lens_b, k):
    H_kv = 3
    P = len(lens_b) * H_kv
    rng = np.random.default_rng(N_cap)
    ktil_np = rng.standard_normal((P, N_cap, D)).astype(np.float32)
    F = wl.randn_bf16((len(lens_b), H_kv, D), N_cap + 1, "cuda")
    idx, cnt, (ridx, rcnt, rs), lens_p = _select_case(lens_b, H_kv, N_cap, 1, 2, k, ktil_np, F)
    assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, 1, 2, k)


def test_select_keys_ready_overlaps_the_decode_append():
    """A decode step's append followed on the same stream by sparse_select_topk_ex with
    SPARSE_SELECT_KEYS_READY (the append writes only the new token's block, a local
    block, so the selection streams the candidates' keys while the append runs): over
    40 appends crossing a block boundary the lists equal those of a plain selection
    issued after the append completed, and the last ones equal the oracle's."""
    sh = wl.DecodeShape("keys_ready", B=2, H_q=16, H_kv=4, T=40 * BLK - 20, n_init=1, n_local=2, k=12,
                        n_planted=10, seed=91)
    B, H_kv, P = sh.B, sh.H_kv, sh.pairs
    T_end = sh.T + 40
    N_cap = (T_end + BLK - 1) // BLK
    planted = wl.planted_sets(sh, 1)[0]
    K = torch.empty((B, H_kv, T_end, D), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    for p in range(P):
        b, h = divmod(p, H_kv)
        K[b, h], V[b, h] = wl.kv_pair(sh, 0, p, planted[p], "cuda", tokens=T_end)
    F = wl.forecast(sh, 0, 0, "cuda")
    L = GpuLayer(B, sh.H_q, H_kv, T_end, N_cap, sh.n_init, sh.n_local, sh.k)
    L.append(K[:, :, :sh.T], V[:, :, :sh.T], 0)
    idx_b, cnt_b = torch.empty_like(L.idx), torch.empty_like(L.count)
    for i in range(40):
        pos = sh.T + i
        seq = _seq([pos + 1] * B)
        L.append(K[:, :, pos:pos + 1], V[:, :, pos:pos + 1], pos)
        binding.sparse_select_topk(F, L.ktil, seq, sh.n_init, sh.n_local, sh.k, L.idx, L.count, status=L.status,
                                   flags=binding.SPARSE_SELECT_KEYS_READY)
        torch.cuda.synchronize()
        binding.sparse_select_topk(F, L.ktil, seq, sh.n_init, sh.n_local, sh.k, idx_b, cnt_b, status=L.status)
        torch.cuda.synchronize()
        assert L.status.item() == 0
        assert torch.equal(L.idx, idx_b) and torch.equal(L.count, cnt_b), f"after append {i}"
    lens_p = [T_end] * P
    ref = oracle.pool(bits(K).reshape(P, T_end, D), lens_p, N_cap)
    ridx, rcnt, rs = oracle.select(bits(F).reshape(P, D), ref, lens_p, sh.n_init, sh.n_local, sh.k)
    assert_selection_matches(L.idx, L.count, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)


def test_select_ties_go_to_the_lower_index_exactly():
    # integer scores: fp32 and fp64 agree exactly, so the tie rule alone decides
    lens_b, H_kv, N_cap, k = [300 * BLK, 77 * BLK + 5], 2, 300, 16
    P = len(lens_b) * H_kv
    rng = np.random.default_rng(7)
    ktil_np = np.zeros((P, N_cap, D), np.float32)
    ktil_np[:, :, 5] = rng.integers(-4, 5, size=(P, N_cap))
    F = torch.zeros((len(lens_b), H_kv, D), dtype=torch.bfloat16, device="cuda")
    F[..., 5] = 1.0
    idx, cnt, (ridx, rcnt, _), _ = _select_case(lens_b, H_kv, N_cap, 1, 2, k, ktil_np, F)
    assert np.array_equal(idx.cpu().numpy().reshape(ridx.shape), ridx)
    assert np.array_equal(cnt.cpu().numpy().reshape(rcnt.shape), rcnt)
    # all-equal scores: the lowest candidate indices
    idx, cnt, (ridx, rcnt, _), _ = _select_case(lens_b, H_kv, N_cap, 1, 2, k, np.zeros_like(ktil_np), F)
    assert np.array_equal(idx.cpu().numpy().reshape(ridx.shape), ridx)
    assert list(ridx[0, :rcnt[0]]) == list(range(0, k + 1)) + [298, 299]


def test_select_k_zero_keeps_only_init_and_local():
    lens_b, H_kv, N_cap = [40 * BLK, 3 * BLK + 1, 65], 2, 40
    P = len(lens_b) * H_kv
    ktil_np = np.random.default_rng(9).standard_normal((P, N_cap, D)).astype(np.float32)
    F = wl.randn_bf16((len(lens_b), H_kv, D), 10, "cuda")
    idx, cnt, (ridx, rcnt, _), _ = _select_case(lens_b, H_kv, N_cap, 1, 2, 0, ktil_np, F)
    assert np.array_equal(idx.cpu().numpy().reshape(ridx.shape), ridx)
    assert np.array_equal(cnt.cpu().numpy().reshape(rcnt.shape), rcnt)
    assert list(ridx[0]) == [0, 38, 39]


@pytest.mark.parametrize("lens_b", [[7 * BLK, 2 * BLK, 65, 1, 0]])
def test_select_few_blocks_takes_all(lens_b):
    H_kv, N_cap = 2, 8
    P = len(lens_b) * H_kv
    ktil_np = np.random.default_rng(3).standard_normal((P, N_cap, D)).astype(np.float32)
    F = wl.randn_bf16((len(lens_b), H_kv, D), 4, "cuda")
    idx, cnt, (ridx, rcnt, _), _ = _select_case(lens_b, H_kv, N_cap, 1, 2, 8, ktil_np, F)
    assert np.array_equal(idx.cpu().numpy().reshape(ridx.shape), ridx)
    assert list(rcnt.reshape(-1, H_kv)[:, 0]) == [7, 2, 2, 1, 0]


# ----------------------------------------------------------------------------- decode attention


# "tmem": the cluster path with SPARSE_ATTN_TENSOR_MEMORY (tcgen05.mma, tensor-memory
# accumulators) instead of mma.sync
PATHS = ("cluster", "split", "stream_k", "tmem")


def _decode_direct(B, H_q, H_kv, T_cap, lens_b, k_cap, seed, n_split=0, idx_np=None, cnt_np=None,
                   path="cluster"):
    """sparse_decode_attn on given (or random distinct) block lists vs oracle.attn.
    ``path``: "cluster" (no workspace), "split" (workspace: per-pair slices merged by the
    last CTA), "stream_k" (workspace and SPARSE_ATTN_STREAM_K) or "tmem" (no workspace,
    SPARSE_ATTN_TENSOR_MEMORY); with a workspace the arrival counters must end at zero."""
    G = H_q // H_kv
    P = B * H_kv
    rng = np.random.default_rng(seed)
    K = wl.randn_bf16((B, H_kv, T_cap, D), seed + 1, "cuda")
    V = wl.randn_bf16((B, H_kv, T_cap, D), seed + 2, "cuda")
    Q = wl.randn_bf16((B, H_q, D), seed + 3, "cuda")
    lens_p = _lens_pair(lens_b, H_kv)
    if idx_np is None:
        idx_np = np.full((P, k_cap), -1, np.int32)
        cnt_np = np.zeros(P, np.int32)
        for p in range(P):
            nb = (int(lens_p[p]) + BLK - 1) // BLK
            c = min(nb, k_cap)
            idx_np[p, :c] = rng.permutation(nb)[:c]          # distinct, unsorted
            cnt_np[p] = c
    O = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H_q), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert path in PATHS
    ws = binding.decode_workspace(B, H_q, H_kv, k_cap, n_split) if path in ("split", "stream_k") else None
    flags = {"stream_k": binding.SPARSE_ATTN_STREAM_K, "tmem": binding.SPARSE_ATTN_TENSOR_MEMORY}.get(path, 0)
    binding.sparse_decode_attn(Q, K, V, torch.from_numpy(idx_np).cuda().view(B, H_kv, k_cap),
                               torch.from_numpy(cnt_np).cuda().view(B, H_kv), _seq(lens_b), O, lse,
                               n_split=n_split, workspace=ws, status=status, flags=flags)
    torch.cuda.synchronize()
    assert status.item() == 0
    if ws is not None:
        assert not ws[:4 * P].any(), "arrival counters not back to zero"
    Oref, lref = oracle.attn(bits(Q).reshape(P, G, D), bits(K).reshape(P, T_cap, D), bits(V).reshape(P, T_cap, D),
                             idx_np, cnt_np, lens_p)
    return O, lse, Oref, lref


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (64, 8), (16, 16), (32, 2), (24, 4)])
def test_decode_attn_matches_oracle_group_sizes(H_q, H_kv, path):
    # (stream-K serves G <= 8; G = 16 with that flag runs the cluster path)
    O, lse, Oref, lref = _decode_direct(2, H_q, H_kv, 40 * BLK, [40 * BLK, 25 * BLK + 11], 19, seed=H_q * 7 + H_kv,
                                        path=path)
    assert_attn_close(O, Oref.reshape(2, H_q, D))
    _check_lse(lse, lref.reshape(2, H_q))


@pytest.mark.parametrize("path,splits", [("cluster", (1, 2, 4, 8)), ("split", (1, 2, 3, 4, 8, 17, 64)),
                                         ("tmem", (1, 2, 4, 8))])
def test_decode_attn_split_invariance(path, splits):
    outs = {}
    for n_split in splits:
        O, lse, Oref, lref = _decode_direct(2, 32, 8, 80 * BLK, [80 * BLK, 79 * BLK + 1], 67, seed=99,
                                            n_split=n_split, path=path)
        assert_attn_close(O, Oref.reshape(2, 32, D), f"{path} n_split={n_split}")
        _check_lse(lse, lref.reshape(2, 32))
        outs[n_split] = O
    for n_split in splits[1:]:
        diff = (outs[n_split].float() - outs[1].float()).abs().max().item()
        assert diff <= 2 ** -7, f"{path}: split {n_split} changes the output by {diff}"


@pytest.mark.parametrize("n_split", [1, 2, 5, 16, 0])
@pytest.mark.parametrize("H_q", [24, 48])
def test_decode_attn_split_path_ragged_and_empty_pairs(n_split, H_q):
    """The split path with ragged, short and empty pairs (count < k_tot: trailing
    slices empty), for G = 8 and G = 16 (two n-tiles)."""
    B, H_kv, T_cap, k_cap = 3, 3, 48 * BLK, 21
    P = B * H_kv
    lens_b = [48 * BLK, 30 * BLK + 5, 7 * BLK]
    lens_p = _lens_pair(lens_b, H_kv)
    rng = np.random.default_rng(13)
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    for p in range(P):
        nb = (int(lens_p[p]) + BLK - 1) // BLK
        c = min([k_cap, 5, 0, 1][p % 4], nb)
        idx_np[p, :c] = rng.permutation(nb)[:c]
        cnt_np[p] = c
    O, lse, Oref, lref = _decode_direct(B, H_q, H_kv, T_cap, lens_b, k_cap, 17, n_split=n_split, idx_np=idx_np,
                                        cnt_np=cnt_np, path="split")
    assert_attn_close(O, Oref.reshape(B, H_q, D), f"n_split={n_split}")
    _check_lse(lse, lref.reshape(B, H_q))


@pytest.mark.parametrize("n_ctas", [1, 2, 3, 7, 13, 64, 0])
def test_decode_attn_stream_k_partitions(n_ctas):
    """Equal ranges of the flattened (pair, block) list: pairs split across 1..many
    CTAs, ragged and empty pairs, every CTA count gives the oracle's result."""
    B, H_q, H_kv, T_cap, k_cap = 3, 24, 3, 48 * BLK, 21
    P = B * H_kv
    lens_b = [48 * BLK, 30 * BLK + 5, 7 * BLK]
    lens_p = _lens_pair(lens_b, H_kv)
    rng = np.random.default_rng(11)
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    for p in range(P):
        nb = (int(lens_p[p]) + BLK - 1) // BLK
        c = [k_cap, 5, 0, min(nb, k_cap)][p % 4]
        c = min(c, nb)
        idx_np[p, :c] = rng.permutation(nb)[:c]
        cnt_np[p] = c
    O, lse, Oref, lref = _decode_direct(B, H_q, H_kv, T_cap, lens_b, k_cap, 7, n_split=n_ctas, idx_np=idx_np,
                                        cnt_np=cnt_np, path="stream_k")
    assert_attn_close(O, Oref.reshape(B, H_q, D), f"n_ctas={n_ctas}")
    _check_lse(lse, lref.reshape(B, H_q))


def test_decode_attn_paths_agree_and_are_deterministic():
    a = _decode_direct(2, 64, 8, 80 * BLK, [80 * BLK, 79 * BLK + 1], 67, seed=5)[0]
    for path in ("split", "stream_k"):
        b = _decode_direct(2, 64, 8, 80 * BLK, [80 * BLK, 79 * BLK + 1], 67, seed=5, path=path)[0]
        c = _decode_direct(2, 64, 8, 80 * BLK, [80 * BLK, 79 * BLK + 1], 67, seed=5, path=path)[0]
        assert (a.float() - b.float()).abs().max().item() <= 2 ** -7, path
        assert torch.equal(b, c), f"{path} is not deterministic"


@pytest.mark.parametrize("path", ["cluster", "tmem"])
def test_decode_attn_empty_and_tiny_sets(path):
    B, H_q, H_kv, T_cap, k_cap = 3, 8, 2, 4 * BLK, 5
    P = B * H_kv
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    idx_np[1, 0], cnt_np[1] = 0, 1          # one block, length 1 -> one token
    idx_np[2, :2], cnt_np[2] = [3, 1], 2
    idx_np[3, :4], cnt_np[3] = [0, 1, 2, 3], 4
    O, lse, Oref, lref = _decode_direct(B, H_q, H_kv, T_cap, [4 * BLK, 1, 3 * BLK + 7], k_cap, 5,
                                        idx_np=idx_np, cnt_np=cnt_np, path=path)
    assert_attn_close(O, Oref.reshape(B, H_q, D))
    assert not O[0, :4].any()                            # pair 0: empty set -> zeros
    assert torch.isneginf(lse[0, :4]).all()
    _check_lse(lse, lref.reshape(B, H_q))


def test_decode_attn_is_deterministic():
    a = _decode_direct(2, 32, 8, 64 * BLK, [64 * BLK, 64 * BLK], 35, seed=3)[0]
    b = _decode_direct(2, 32, 8, 64 * BLK, [64 * BLK, 64 * BLK], 35, seed=3)[0]
    assert torch.equal(a, b)


@pytest.mark.parametrize("order", ["rising", "falling", "mixed"])
@pytest.mark.parametrize("n_split", [1, 2])
def test_decode_attn_tensor_memory_rescales_when_the_max_jumps(order, n_split):
    """Blocks whose keys are scaled by 1, 3, 9, 27: block maxima differ by far more than
    the 2^8 the tensor-memory path lets a row's running max lag, so it must rescale O
    in tensor memory (rising order), never rescale (falling), or both (mixed); the
    output equals the oracle and the mma.sync path."""
    B, H_q, H_kv, nb = 1, 8, 1, 8
    T_cap = nb * BLK
    K = wl.randn_bf16((B, H_kv, T_cap, D), 71, "cuda").float()
    scale_of = {"rising": [1, 1, 3, 3, 9, 9, 27, 27], "falling": [27, 27, 9, 9, 3, 3, 1, 1],
                "mixed": [1, 27, 1, 9, 3, 27, 1, 3]}[order]
    for j, f in enumerate(scale_of):
        K[:, :, j * BLK:(j + 1) * BLK] *= f
    K = K.to(torch.bfloat16)
    V = wl.randn_bf16((B, H_kv, T_cap, D), 72, "cuda")
    Q = wl.randn_bf16((B, H_q, D), 73, "cuda")
    idx_np = np.arange(nb, dtype=np.int32).reshape(1, nb)
    cnt_np = np.array([nb], np.int32)
    idx = torch.from_numpy(idx_np).cuda().view(B, H_kv, nb)
    cnt = torch.from_numpy(cnt_np).cuda().view(B, H_kv)
    outs = {}
    for path, flags in (("cluster", 0), ("tmem", binding.SPARSE_ATTN_TENSOR_MEMORY)):
        O = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros((B, H_q), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.sparse_decode_attn(Q, K, V, idx, cnt, _seq([T_cap]), O, lse, n_split=n_split, flags=flags,
                                   status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        outs[path] = (O, lse)
    Oref, lref = oracle.attn(bits(Q).reshape(1, H_q, D), bits(K).reshape(1, T_cap, D), bits(V).reshape(1, T_cap, D),
                             idx_np, cnt_np, np.array([T_cap]))
    for path, (O, lse) in outs.items():
        assert_attn_close(O, Oref.reshape(B, H_q, D), f"{order} {path}")
        _check_lse(lse, lref.reshape(B, H_q))
    assert (outs["tmem"][0].float() - outs["cluster"][0].float()).abs().max().item() <= 2 ** -6


@pytest.mark.parametrize("path", ["cluster", "split", "tmem"])
def test_decode_attn_reports_bad_block_ids_without_faulting(path):
    B, H_q, H_kv, T_cap, k_cap = 1, 8, 2, 8 * BLK, 3
    ws = binding.decode_workspace(B, H_q, H_kv, k_cap, 2) if path == "split" else None
    flags = binding.SPARSE_ATTN_TENSOR_MEMORY if path == "tmem" else 0
    K = wl.randn_bf16((B, H_kv, T_cap, D), 1, "cuda")
    Q = wl.randn_bf16((B, H_q, D), 2, "cuda")
    idx = torch.tensor([[[0, 1 << 20, 2], [3, -5, 4]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[3, 3]], dtype=torch.int32, device="cuda")
    O = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn(Q, K, K, idx, cnt, _seq([T_cap]), O, status=status, workspace=ws,
                               n_split=2 if ws is not None else 0, flags=flags)
    torch.cuda.synchronize()
    assert status.item() == binding.SPARSE_ERR_BAD_INDEX
    good_idx = torch.tensor([[[0, 2, 2], [3, 4, 4]]], dtype=torch.int32, device="cuda")
    good_cnt = torch.tensor([[2, 2]], dtype=torch.int32, device="cuda")
    O2 = torch.zeros_like(O)
    binding.sparse_decode_attn(Q, K, K, good_idx, good_cnt, _seq([T_cap]), O2)
    torch.cuda.synchronize()
    assert (O.float() - O2.float()).abs().max().item() <= 2 ** -8


def test_decode_attn_ex_ready_word():
    B, H_q, H_kv, T_cap, k_cap = 1, 8, 2, 8 * BLK, 3
    K = wl.randn_bf16((B, H_kv, T_cap, D), 11, "cuda")
    Q = wl.randn_bf16((B, H_q, D), 12, "cuda")
    idx = torch.tensor([[[0, 1, 2], [3, 4, 5]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[3, 3]], dtype=torch.int32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sentinel = torch.full((B, H_q, D), 7.0, dtype=torch.bfloat16, device="cuda")
    # a word that nothing sets: the bounded wait gives up and leaves O untouched
    O = sentinel.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn_ex(Q, K, K, idx, cnt, _seq([T_cap]), O, flag, 1, 50_000_000, status=status)
    torch.cuda.synchronize()
    assert status.item() == binding.SPARSE_ERR_TIMEOUT
    assert torch.equal(O, sentinel)
    # the same through the stream-K path (pairs split across CTAs): untouched, counters zero
    ws = binding.decode_workspace(B, H_q, H_kv, k_cap, 4)
    status.zero_()
    binding.sparse_decode_attn_ex(Q, K, K, idx, cnt, _seq([T_cap]), O, flag, 1, 20_000_000, n_split=4,
                                  workspace=ws, flags=binding.SPARSE_ATTN_STREAM_K, status=status)
    torch.cuda.synchronize()
    assert status.item() == binding.SPARSE_ERR_TIMEOUT
    assert torch.equal(O, sentinel) and not ws[:8].any()
    # and through the split path
    status.zero_()
    binding.sparse_decode_attn_ex(Q, K, K, idx, cnt, _seq([T_cap]), O, flag, 1, 20_000_000, n_split=2,
                                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == binding.SPARSE_ERR_TIMEOUT
    assert torch.equal(O, sentinel) and not ws[:8].any()
    status.zero_()
    binding.sparse_decode_attn_ex(Q, K, K, idx, cnt, _seq([T_cap]), O, flag, 1, 0, status=status)
    torch.cuda.synchronize()
    assert status.item() == binding.SPARSE_ERR_NOT_READY
    # once the word reaches the target the call computes the plain result
    flag.fill_(1)
    status.zero_()
    binding.sparse_decode_attn_ex(Q, K, K, idx, cnt, _seq([T_cap]), O, flag, 1, 1_000_000, status=status)
    ref = torch.zeros_like(O)
    binding.sparse_decode_attn(Q, K, K, idx, cnt, _seq([T_cap]), ref)
    torch.cuda.synchronize()
    assert status.item() == 0 and torch.equal(O, ref)


# ----------------------------------------------------------------------------- whole single-layer workloads


def _pipeline(sh, lens_b=None):
    """append -> select -> attend on the GPU; pool -> select -> attend in the oracle."""
    inp = wl.single_layer(sh, device="cuda")
    B, H_kv, G, P = sh.B, sh.H_kv, sh.G, sh.pairs
    L = GpuLayer(B, sh.H_q, H_kv, sh.T_cap, sh.N_b, sh.n_init, sh.n_local, sh.k)
    K_all, V_all = inp["K"].clone(), inp["V"].clone()
    if lens_b is None:
        L.append(inp["K"][:, :, :sh.T], inp["V"][:, :, :sh.T], 0)
    else:
        # a ragged batch: element b holds lens_b[b] tokens
        assert sh.n_new == 0
        for b, n in enumerate(lens_b):
            binding.sparse_pool_append(L.k_cache[b:b + 1], L.v_cache[b:b + 1], L.ktil[b:b + 1],
                                       inp["K"][b:b + 1, :, :n].contiguous(), inp["V"][b:b + 1, :, :n].contiguous(), 0)
            K_all[b, :, n:] = 0
            V_all[b, :, n:] = 0
    if sh.n_new:
        L.append(inp["k_new"], inp["v_new"], sh.T)
        K_all[:, :, sh.T:sh.len_after] = inp["k_new"]
        V_all[:, :, sh.T:sh.len_after] = inp["v_new"]
    if lens_b is None:
        lens_b = [sh.len_after] * B
    seq = _seq(lens_b)
    L.select(inp["F"], seq)
    L.attend(inp["Q"], seq)
    torch.cuda.synchronize()
    assert L.status.item() == 0
    assert torch.equal(L.k_cache, K_all) and torch.equal(L.v_cache, V_all)
    lens_p = _lens_pair(lens_b, H_kv)
    Kb, Vb = bits(K_all).reshape(P, sh.T_cap, D), bits(V_all).reshape(P, sh.T_cap, D)
    Qb = bits(inp["Q"])
    ktil, ridx, rcnt, rs, Oref, lref = oracle_layer(Kb, Vb, Qb, bits(inp["F"]), lens_p, sh.N_b, sh.n_init,
                                                     sh.n_local, sh.k, G)
    got = L.ktil.cpu().double().numpy().reshape(P, sh.N_b, D)
    assert np.allclose(got, ktil, rtol=1e-5, atol=1e-6)
    exempt = assert_selection_matches(L.idx, L.count, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
    # end-to-end: the GPU's own chain against the oracle over the lists the GPU took
    # (the oracle's own, except where a near tie, validated above, allowed another)
    same = (L.idx.cpu().numpy().reshape(ridx.shape) == ridx).all(axis=1)
    Oown, _ = oracle_attn_on_taken_lists(L.idx, L.count, ridx, rcnt, Oref, Qb.reshape(P, G, D), Kb, Vb, lens_p)
    assert_attn_close(L.O, Oown.reshape(B, sh.H_q, D), "chain")
    _check_lse(L.lse.view(P, G)[torch.from_numpy(same)], lref[same])
    # attention alone over the oracle's selection, all pairs
    O_gpu_on_ref = torch.zeros_like(L.O)
    binding.sparse_decode_attn(inp["Q"], L.k_cache, L.v_cache, torch.from_numpy(ridx).cuda().view(B, H_kv, -1),
                               torch.from_numpy(rcnt).cuda().view(B, H_kv), seq, O_gpu_on_ref)
    torch.cuda.synchronize()
    stats = assert_attn_close(O_gpu_on_ref, Oref.reshape(B, sh.H_q, D))
    return exempt, stats


def test_single_layer_4k_workload():
    _pipeline(wl.SINGLE_4K)


def test_llama8b_32k_append_workload():
    exempt, _ = _pipeline(wl.LLAMA8B_32K)
    assert exempt <= 2


def test_ragged_batch_lengths():
    sh = wl.DecodeShape("ragged", B=3, H_q=16, H_kv=4, T=8192, n_init=1, n_local=2, k=16, n_planted=12,
                        seed=77)
    _pipeline(sh, lens_b=[8192, 5000, 129])


def test_decode_128k_layer_all_pairs_at_full_size():
    """One physical layer of the 128K, B=8, G=8 workload at full size: append all
    131072 tokens, select with two Forecast vectors, attend.  Every one of the 64 pairs
    is checked against the oracle: compressed keys, selection (near-tie rule), the
    GPU's attention over the oracle's lists, and the GPU chain's own output.  Where a
    near tie let the GPU take a different (valid) list, that output is checked against
    the oracle's attention over the list the GPU took."""
    sh = wl.DECODE_128K
    B, H_kv, G, P = sh.B, sh.H_kv, sh.G, sh.pairs
    planted = wl.planted_sets(sh, 2)
    L = GpuLayer(B, sh.H_q, H_kv, sh.T, sh.N_b, sh.n_init, sh.n_local, sh.k)
    Kh = np.empty((P, sh.T, D), np.uint16)
    Vh = np.empty((P, sh.T, D), np.uint16)
    for b in range(B):
        Kb = torch.empty((1, H_kv, sh.T, D), dtype=torch.bfloat16, device="cuda")
        Vb = torch.empty_like(Kb)
        for h in range(H_kv):
            p = b * H_kv + h
            Kb[0, h], Vb[0, h] = wl.kv_pair(sh, 1, p, planted[1, p], "cuda")
        Kh[b * H_kv:(b + 1) * H_kv] = bits(Kb[0])
        Vh[b * H_kv:(b + 1) * H_kv] = bits(Vb[0])
        binding.sparse_pool_append(L.k_cache[b:b + 1], L.v_cache[b:b + 1], L.ktil[b:b + 1], Kb, Vb, 0)
    torch.cuda.synchronize()
    del Kb, Vb
    lens_p = [sh.T] * P
    ktil = oracle.pool(Kh, lens_p, sh.N_b)
    got = L.ktil.view(P, sh.N_b, D).cpu().double().numpy()
    assert np.allclose(got, ktil, rtol=1e-5, atol=1e-6)
    seq = _seq([sh.T] * B)
    for logical in (0, 10):            # F_0 and F_10 both target physical layer 1
        F = wl.forecast(sh, 1, logical, "cuda")
        Q = wl.queries(sh, logical + 1, "cuda")
        L.select(F, seq)
        L.attend(Q, seq)
        torch.cuda.synchronize()
        assert L.status.item() == 0
        Fb, Qb = bits(F).reshape(P, D), bits(Q).reshape(P, G, D)
        ridx, rcnt, rs = oracle.select(Fb, ktil, lens_p, sh.n_init, sh.n_local, sh.k)
        assert_selection_matches(L.idx, L.count, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
        for p in range(P):   # generator sanity: the planted blocks are the ones selected
            assert len(set(planted[1, p].tolist()) & set(ridx[p].tolist())) >= 40
        Oref, _ = oracle.attn(Qb, Kh, Vh, ridx, rcnt, lens_p)
        # the attention alone over the oracle's lists, every pair
        O_on_ref = torch.zeros_like(L.O)
        binding.sparse_decode_attn(Q, L.k_cache, L.v_cache, torch.from_numpy(ridx).cuda().view(B, H_kv, -1),
                                   torch.from_numpy(rcnt).cuda().view(B, H_kv), seq, O_on_ref)
        torch.cuda.synchronize()
        assert_attn_close(O_on_ref, Oref.reshape(B, sh.H_q, D), f"logical layer {logical}")
        # the GPU chain's output: where the GPU's list differs (a near tie, validated
        # above) the oracle attends over the list the GPU took
        Oown, _ = oracle_attn_on_taken_lists(L.idx, L.count, ridx, rcnt, Oref, Qb, Kh, Vh, lens_p)
        assert_attn_close(L.O, Oown.reshape(B, sh.H_q, D), f"chain, logical layer {logical}")


# ----------------------------------------------------------------------------- grouped verification


def _verify(sh, n_split=0, shared=False, flags=0):
    inp = wl.verify_inputs(sh, device="cuda")
    O = torch.zeros((sh.B, sh.N_q, sh.H_q, D), dtype=torch.bfloat16, device="cuda")
    loaded = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_verify_attn_grouped(inp["Q"], inp["K"], inp["V"], inp["I"], sh.C, sh.window_blocks,
                                       inp["seq_len"], O, blocks_loaded=loaded, n_split=n_split, status=status,
                                       shared=shared, flags=flags)
    torch.cuda.synchronize()
    assert status.item() == 0
    return inp, O, int(loaded.item())


TM = binding.SPARSE_ATTN_TENSOR_MEMORY


@pytest.mark.parametrize("flags", [0, TM])
def test_verify_64k_workload_matches_oracle_and_saves_loads(flags):
    sh = wl.VERIFY_64K
    inp, O, loaded = _verify(sh, flags=flags)
    Oref, union, per_query = oracle.verify(bits(inp["Q"]), bits(inp["K"]), bits(inp["V"]), inp["I"].cpu().numpy(),
                                           sh.C, sh.window_blocks, [sh.T] * sh.B)
    assert_attn_close(O, Oref)
    assert loaded == union
    bound = (1 + (sh.C - 1) * (1 - sh.gamma)) / sh.C
    assert loaded / per_query <= bound
    assert loaded / per_query == pytest.approx(36 / 96)


def test_verify_equals_per_query_decode():
    sh = wl.VerifyShape("small", B=2, H_q=8, H_kv=2, T=3000, N_q=6, n_sel=5, gamma=0.6, window_tokens=3 * BLK, C=3,
                        seed=31)
    inp, O, _ = _verify(sh)
    nb = (sh.T + BLK - 1) // BLK
    W = list(range(nb - sh.window_blocks, nb))
    k_cap = sh.n_sel + sh.window_blocks
    for q in range(sh.N_q):
        idx = torch.full((sh.B, sh.H_kv, k_cap), -1, dtype=torch.int32)
        for b in range(sh.B):
            for h in range(sh.H_kv):
                s = sorted(set(inp["I"][b, h, q].tolist()) | set(W))
                idx[b, h, :len(s)] = torch.tensor(s)
        cnt = (idx >= 0).sum(-1).to(torch.int32)
        Od = torch.zeros((sh.B, sh.H_q, D), dtype=torch.bfloat16, device="cuda")
        binding.sparse_decode_attn(inp["Q"][:, q].contiguous(), inp["K"], inp["V"], idx.cuda(), cnt.cuda(),
                                   inp["seq_len"], Od)
        torch.cuda.synchronize()
        assert (Od.float() - O[:, q].float()).abs().max().item() <= 2 ** -7


@pytest.mark.parametrize("flags", [0, TM])
@pytest.mark.parametrize("n_split", [1, 2, 8])
def test_verify_split_invariance(n_split, flags):
    sh = wl.VerifyShape("split", B=1, H_q=16, H_kv=4, T=64 * BLK, N_q=8, n_sel=16, gamma=0.75,
                        window_tokens=8 * BLK, C=4, seed=33)
    inp, O, loaded = _verify(sh, n_split=n_split, flags=flags)
    Oref, union, _ = oracle.verify(bits(inp["Q"]), bits(inp["K"]), bits(inp["V"]), inp["I"].cpu().numpy(), sh.C,
                                   sh.window_blocks, [sh.T] * sh.B)
    assert_attn_close(O, Oref)
    assert loaded == union


@pytest.mark.parametrize("flags", [0, TM])
def test_verify_shared_layout_64k_workload_matches_oracle(flags):
    """SSV mode B on the 64K verification workload: every query over its group's first
    query's layout; each group loads n_sel + window blocks."""
    sh = wl.VERIFY_64K
    inp, O, loaded = _verify(sh, shared=True, flags=flags)
    Oref, union, per_query = oracle.verify(bits(inp["Q"]), bits(inp["K"]), bits(inp["V"]), inp["I"].cpu().numpy(),
                                           sh.C, sh.window_blocks, [sh.T] * sh.B, shared=True)
    assert_attn_close(O, Oref)
    assert loaded == union == sh.B * sh.H_kv * (sh.N_q // sh.C) * (sh.n_sel + sh.window_blocks)


@pytest.mark.parametrize("flags", [0, TM])
@pytest.mark.parametrize("n_split,C", [(1, 4), (2, 3), (8, 4), (0, 1)])
def test_verify_shared_layout_ragged_groups(n_split, C, flags):
    sh = wl.VerifyShape("shared", B=2, H_q=8, H_kv=2, T=40 * BLK + 17, N_q=7, n_sel=6, gamma=0.5,
                        window_tokens=2 * BLK, C=C, seed=35)
    inp, O, loaded = _verify(sh, n_split=n_split, shared=True, flags=flags)
    Oref, union, _ = oracle.verify(bits(inp["Q"]), bits(inp["K"]), bits(inp["V"]), inp["I"].cpu().numpy(), sh.C,
                                   sh.window_blocks, [sh.T] * sh.B, shared=True)
    assert_attn_close(O, Oref)
    assert loaded == union


@pytest.mark.parametrize("tm", [0, TM])
@pytest.mark.parametrize("shared", [False, True])
def test_verify_chain_with_blocks_ready(shared, tm):
    """A chain of verification launches on one stream where each launch's Q is the
    previous launch's O: with SPARSE_ATTN_BLOCKS_READY the union and the K/V stream start
    early but Q still waits, so the chain equals the one without the flag bit for bit,
    and its first link equals the oracle."""
    sh = wl.VerifyShape("chain", B=2, H_q=16, H_kv=4, T=48 * BLK + 5, N_q=8, n_sel=12, gamma=0.6,
                        window_tokens=4 * BLK, C=4, seed=37)
    inp = wl.verify_inputs(sh, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def chain(flags):
        outs = [inp["Q"]]
        for _ in range(4):
            O = torch.full_like(inp["Q"], 3.0)
            outs.append(O)
        for l in range(4):
            binding.sparse_verify_attn_grouped(outs[l], inp["K"], inp["V"], inp["I"], sh.C, sh.window_blocks,
                                               inp["seq_len"], outs[l + 1], status=status, shared=shared,
                                               flags=flags | tm)
        torch.cuda.synchronize()
        return outs[1:]

    plain = chain(0)
    early = chain(binding.SPARSE_ATTN_BLOCKS_READY)
    assert status.item() == 0
    for a, b in zip(plain, early):
        assert torch.equal(a, b)
    Oref, _, _ = oracle.verify(bits(inp["Q"]), bits(inp["K"]), bits(inp["V"]), inp["I"].cpu().numpy(), sh.C,
                               sh.window_blocks, [sh.T] * sh.B, shared=shared)
    assert_attn_close(early[0], Oref)


# ----------------------------------------------------------------------------- offloaded gather


def test_gather_from_pinned_host_and_attend_over_the_ring():
    B, H_q, H_kv, T = 2, 16, 4, 96 * BLK + 10
    P, k_cap = B * H_kv, 15
    lens_b = [T, T - 700]
    lens_p = _lens_pair(lens_b, H_kv)
    K = wl.randn_bf16((B, H_kv, T, D), 61).pin_memory()
    V = wl.randn_bf16((B, H_kv, T, D), 62).pin_memory()
    # staged block lists from the generator: ascending, distinct, the last (partial) block included
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    for p in range(P):
        nb = (int(lens_p[p]) + BLK - 1) // BLK
        c = k_cap if p % 3 else k_cap - 4
        blocks = wl.draw_blocks(c - 1, 0, nb - 1, seed=900 + p).tolist() + [nb - 1]
        idx_np[p, :c], cnt_np[p] = blocks, c
    idx = torch.from_numpy(idx_np).cuda().view(B, H_kv, k_cap)
    cnt = torch.from_numpy(cnt_np).cuda().view(B, H_kv)
    seq = _seq(lens_b)
    k_ring = torch.full((B, H_kv, k_cap, BLK, D), 3.0, dtype=torch.bfloat16, device="cuda")
    v_ring = torch.full_like(k_ring, 3.0)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy = torch.cuda.Stream()
    copy.wait_stream(torch.cuda.current_stream())
    binding.sparse_gather_offloaded(K, V, idx, cnt, k_ring, v_ring, ready_flag=flag, n_ctas=24, stream=copy)
    torch.cuda.current_stream().wait_stream(copy)
    torch.cuda.synchronize()
    assert flag.item() == 24
    ring_ref = np.full((P, k_cap, BLK, D), bits(torch.tensor(3.0, dtype=torch.bfloat16)), np.uint16)
    oracle.gather(bits(K).reshape(P, T, D), idx_np, cnt_np, ring_ref)
    assert np.array_equal(bits(k_ring).reshape(ring_ref.shape), ring_ref)
    oracle.gather(bits(V).reshape(P, T, D), idx_np, cnt_np, ring_ref)
    assert np.array_equal(bits(v_ring).reshape(ring_ref.shape), ring_ref)
    # attention over the ring (slot = list position) equals attention over the resident cache
    Kd, Vd = K.cuda(), V.cuda()
    Q = wl.randn_bf16((B, H_q, D), 64, "cuda")
    O_ring = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda")
    O_res = torch.zeros_like(O_ring)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.arange(k_cap, dtype=torch.int32, device="cuda").repeat(B, H_kv, 1).contiguous()
    binding.sparse_decode_attn_ex(Q, k_ring, v_ring, idx, cnt, seq, O_ring, flag, 24, 1_000_000, blk_slot=slots,
                                  status=status)
    binding.sparse_decode_attn(Q, Kd, Vd, idx, cnt, seq, O_res)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(O_ring, O_res)
    Oref, _ = oracle.attn(bits(Q).reshape(P, H_q // H_kv, D), bits(K).reshape(P, T, D), bits(V).reshape(P, T, D),
                          idx_np, cnt_np, lens_p)
    assert_attn_close(O_ring, Oref.reshape(B, H_q, D))


def test_offload_128k_layer_sampled_at_full_size():
    """One layer of the offloaded 128K workload at full size (B=4, H_kv=8, T=131072:
    2 GiB of pinned host K/V), in the bench's launch configuration: select from the
    resident compressed keys, gather the selected blocks into the HBM ring with the
    default CTA count, attend over the ring.  Every one of the 32 pairs is checked: the
    selection (near-tie rule), the ring bit-exactly against the oracle's staging copy of
    the list the GPU selected (the oracle's own list unless a near tie, validated first,
    let the GPU take another), and the attention over the ring against the oracle's
    attention over that same list."""
    sh = wl.OFFLOAD_128K
    B, H_kv, H_q, T, G, P = sh.B, sh.H_kv, sh.H_q, sh.T, sh.G, sh.pairs
    planted = wl.planted_sets(sh, 1)
    kc = torch.empty((B, H_kv, T, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    for p in range(P):
        b, h = divmod(p, H_kv)
        kc[b, h], vc[b, h] = wl.kv_pair(sh, 0, p, planted[0, p], "cuda")
    kd, vd = torch.zeros_like(kc), torch.zeros_like(vc)
    ktil = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device="cuda")
    binding.sparse_pool_append(kd, vd, ktil, kc, vc, 0)
    del kd, vd
    kh = torch.empty(kc.shape, dtype=torch.bfloat16, pin_memory=True)
    vh = torch.empty(kc.shape, dtype=torch.bfloat16, pin_memory=True)
    kh.copy_(kc)
    vh.copy_(vc)
    del kc, vc
    Kh, Vh = bits(kh).reshape(P, T, D), bits(vh).reshape(P, T, D)   # views of the pinned host cache
    seq = _seq([T] * B)
    F = wl.forecast(sh, 0, 0, "cuda")
    Q = wl.queries(sh, 0, "cuda")
    idx = torch.full((B, H_kv, sh.k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_select_topk(F, ktil, seq, sh.n_init, sh.n_local, sh.k, idx, cnt, status=status)
    k_ring = torch.full((B, H_kv, sh.k_tot, BLK, D), 5.0, dtype=torch.bfloat16, device="cuda")
    v_ring = torch.full_like(k_ring, 5.0)
    binding.sparse_gather_offloaded(kh, vh, idx, cnt, k_ring, v_ring, status=status)
    slots = torch.arange(sh.k_tot, dtype=torch.int32, device="cuda").repeat(B, H_kv, 1).contiguous()
    O = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda")
    binding.sparse_decode_attn(Q, k_ring, v_ring, idx, cnt, seq, O, blk_slot=slots, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Fb, Qb = bits(F).reshape(P, D), bits(Q).reshape(P, G, D)
    ring_k = bits(k_ring).reshape(P, sh.k_tot, BLK, D)
    ring_v = bits(v_ring).reshape(P, sh.k_tot, BLK, D)
    lens_p = [T] * P
    _, ridx, rcnt, rs, _, _ = oracle_layer(Kh, Vh, Qb, Fb, lens_p, sh.N_b, sh.n_init, sh.n_local, sh.k, G)
    assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
    # staging is a plain copy of the listed blocks; the lists are the oracle's, except
    # where a near tie (validated just above) let the GPU take another valid one
    gidx = idx.view(P, -1).cpu().numpy()
    gcnt = cnt.view(P).cpu().numpy()
    lists = ridx.copy()
    for p in range(P):
        if not np.array_equal(gidx[p], ridx[p]):
            lists[p] = gidx[p]
    fill = bits(torch.tensor(5.0, dtype=torch.bfloat16))
    ref = np.full((P, sh.k_tot, BLK, D), fill, np.uint16)
    oracle.gather(Kh, lists, rcnt, ref)
    assert np.array_equal(ring_k, ref)
    ref.fill(fill)
    oracle.gather(Vh, lists, rcnt, ref)
    assert np.array_equal(ring_v, ref)
    del ref
    assert np.array_equal(gcnt, rcnt)
    Oref, _ = oracle.attn(Qb, Kh, Vh, lists, rcnt, lens_p)
    assert_attn_close(O, Oref.reshape(B, H_q, D))
