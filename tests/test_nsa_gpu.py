"""GPU parity of NSA's gated three-branch decode (SSV notes, "NSA three-branch math"
steps 3-6) and of the pooled-value append that feeds its compressed branch.

sparse_decode_attn_nsa is checked against oracle.nsa:
  * with the compressed rows given to both sides as the same bf16 values (the bf16
    rounding of the oracle's fp64 pooling), so only the kernel's arithmetic differs;
  * through the whole chain (sparse_pool_append_kv builds the caches and the bf16
    compressed rows on the GPU; the oracle pools in fp64), which adds the bf16
    rounding of the compressed rows (relative 2^-9) to the error budget;
  * branch by branch (gates (1,0,0), (0,1,0), (0,0,1)) and with random gates.
Tolerances: those of parity_utils (max abs 2e-2, mean abs 2e-3).  Every input comes
from the seeded generators or from the oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl
from parity_utils import BLK, D, assert_attn_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 (round to nearest even, through torch) as uint16 bit patterns."""
    return wl.bf16_bits(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16))


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed, gates_kind="random"):
    P = B * H_kv
    G = H_q // H_kv
    rng = np.random.default_rng(seed)
    K = wl.randn_bf16((B, H_kv, T_cap, D), seed + 1, "cuda")
    V = wl.randn_bf16((B, H_kv, T_cap, D), seed + 2, "cuda")
    Q = wl.randn_bf16((B, H_q, D), seed + 3, "cuda")
    lens_p = np.repeat(np.asarray(lens_b, dtype=np.int64), H_kv)
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    for p in range(P):
        nb = (int(lens_p[p]) + BLK - 1) // BLK
        c = min(nb, k_cap) if p % 3 else min(nb, max(0, k_cap - 3))
        idx_np[p, :c] = np.sort(rng.permutation(nb)[:c])
        cnt_np[p] = c
    if gates_kind == "random":
        gates = rng.uniform(0.0, 1.0, (B, H_q, 3))
    else:
        gates = np.zeros((B, H_q, 3))
        gates[..., gates_kind] = 1.0
    Kb = bits(K).reshape(P, T_cap, D)
    Vb = bits(V).reshape(P, T_cap, D)
    return dict(K=K, V=V, Q=Q, Kb=Kb, Vb=Vb, Qb=bits(Q).reshape(P, G, D), lens_p=lens_p, idx_np=idx_np,
                cnt_np=cnt_np, gates_np=gates,
                idx=torch.from_numpy(idx_np).cuda().view(B, H_kv, k_cap),
                cnt=torch.from_numpy(cnt_np).cuda().view(B, H_kv),
                gates=torch.from_numpy(gates.astype(np.float32)).cuda(),
                seq=torch.tensor(lens_b, dtype=torch.int32, device="cuda"))


def _rows_from_oracle(c, N_cap, B, H_kv):
    """Compressed rows: the oracle's fp64 means, rounded to bf16 (both sides use these)."""
    kh = _to_bf16_bits(oracle.pool(c["Kb"], c["lens_p"], N_cap))
    vh = _to_bf16_bits(oracle.pool(c["Vb"], c["lens_p"], N_cap))
    to_dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda().view(B, H_kv, N_cap, D)
    return kh, vh, to_dev(kh), to_dev(vh)


def _gpu_nsa(c, khat, vhat, window, B, H_q, n_split=0, ws=None, status=None, flags=0):
    """The fused form for G <= 8 (no workspace), the branch grid for G > 8 or when asked."""
    H_kv = c["K"].shape[1]
    O = torch.full((B, H_q, D), 7.0, dtype=torch.bfloat16, device="cuda")
    grid = H_q // H_kv > 8 or flags & binding.SPARSE_NSA_BRANCH_GRID
    if ws is None and grid:
        ws = binding.nsa_workspace(B, H_q, H_kv)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn_nsa(c["Q"], c["K"], c["V"], khat, vhat, c["idx"], c["cnt"], c["seq"], window,
                                   c["gates"], O, ws, n_split=n_split, flags=flags, status=status)
    torch.cuda.synchronize()
    return O, ws, status


def _oracle_nsa(c, kh_bits, vh_bits, window):
    return oracle.nsa(c["Qb"], c["Kb"], c["Vb"], _bits_to_f64(kh_bits), _bits_to_f64(vh_bits), c["idx_np"],
                      c["cnt_np"], c["lens_p"], window, c["gates_np"].reshape(len(c["lens_p"]), -1, 3))


@pytest.mark.parametrize("flags", [0, binding.SPARSE_NSA_BRANCH_GRID])
@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (64, 8), (32, 2), (6, 6)])
@pytest.mark.parametrize("n_split", [0, 1, 2, 4, 8])
def test_nsa_matches_oracle(H_q, H_kv, n_split, flags):
    B, T_cap, k_cap, N_cap = 2, 40 * BLK, 9, 40
    lens_b = [40 * BLK, 27 * BLK + 13]
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=11 + n_split + H_q)
    kh, vh, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O, ws, status = _gpu_nsa(c, khat, vhat, 200, B, H_q, n_split, flags=flags)
    assert status.item() == 0
    ref = _oracle_nsa(c, kh, vh, 200)
    assert_attn_close(O, ref, "nsa")
    if ws is not None:   # the arrival counters are back at zero
        n_cnt = B * H_kv
        assert int(ws[: 4 * n_cnt].view(torch.int32).abs().sum().item()) == 0


@pytest.mark.parametrize("n_split", [1, 2, 4, 8])
def test_nsa_fused_and_branch_grid_agree(n_split):
    """The two forms merge the same per-CTA partial states in different places
    (DSMEM vs the workspace): equal up to fp32 rounding of the gated sum."""
    B, H_q, H_kv, T_cap, k_cap, N_cap = 3, 64, 8, 50 * BLK, 12, 50
    c = _case(B, H_q, H_kv, T_cap, [50 * BLK, 31 * BLK + 7, 2 * BLK], k_cap, N_cap, seed=3 + n_split)
    _, _, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O1, _, s1 = _gpu_nsa(c, khat, vhat, 300, B, H_q, n_split)
    O2, _, s2 = _gpu_nsa(c, khat, vhat, 300, B, H_q, n_split, flags=binding.SPARSE_NSA_BRANCH_GRID)
    assert s1.item() == 0 and s2.item() == 0
    assert (O1.float() - O2.float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("branch", [0, 1, 2])
@pytest.mark.parametrize("window", [0, 1, 64, 100, 513])
def test_nsa_each_branch(branch, window):
    """Gates (1,0,0) / (0,1,0) / (0,0,1): the compressed, selected and window branch alone."""
    B, H_q, H_kv, T_cap, k_cap, N_cap = 3, 16, 2, 30 * BLK, 7, 100
    lens_b = [30 * BLK, 11 * BLK + 1, 5]
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=40 + branch + window, gates_kind=branch)
    kh, vh, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O, _, status = _gpu_nsa(c, khat, vhat, window, B, H_q)
    assert status.item() == 0
    ref = _oracle_nsa(c, kh, vh, window)
    assert_attn_close(O, ref, f"nsa branch {branch} w={window}")
    if branch == 2 and window == 0:   # an empty window contributes zero
        assert float(O.float().abs().max()) == 0.0


def test_nsa_degenerate_lengths_and_counts():
    """Empty sequences, single tokens, empty selections, a window longer than the
    sequence, G = 16 (two n-tiles)."""
    B, H_q, H_kv, T_cap, k_cap, N_cap = 4, 32, 2, 20 * BLK, 5, 20
    lens_b = [0, 1, 65, 20 * BLK]
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=77)
    c["cnt_np"][2] = 0
    c["cnt"] = torch.from_numpy(c["cnt_np"]).cuda().view(B, H_kv)
    kh, vh, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O, _, status = _gpu_nsa(c, khat, vhat, T_cap, B, H_q)
    assert status.item() == 0
    ref = _oracle_nsa(c, kh, vh, T_cap)
    assert_attn_close(O, ref, "nsa degenerate")
    assert float(O[0].float().abs().max()) == 0.0   # no token: every branch is empty


@pytest.mark.parametrize("flags", [0, binding.SPARSE_NSA_BRANCH_GRID])
def test_nsa_repeat_calls_are_deterministic(flags):
    B, H_q, H_kv, T_cap, k_cap, N_cap = 2, 64, 8, 33 * BLK, 6, 33
    c = _case(B, H_q, H_kv, T_cap, [33 * BLK, 17 * BLK + 30], k_cap, N_cap, seed=5)
    _, _, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O1, ws, _ = _gpu_nsa(c, khat, vhat, 256, B, H_q, flags=flags)
    O2, _, _ = _gpu_nsa(c, khat, vhat, 256, B, H_q, ws=ws, flags=flags)
    O3, _, _ = _gpu_nsa(c, khat, vhat, 256, B, H_q, ws=ws, flags=flags)
    assert torch.equal(O1, O2) and torch.equal(O2, O3)


def test_nsa_bad_block_ids_are_reported():
    B, H_q, H_kv, T_cap, k_cap, N_cap = 1, 8, 1, 10 * BLK, 4, 10
    c = _case(B, H_q, H_kv, T_cap, [10 * BLK], k_cap, N_cap, seed=9)
    c["idx"][0, 0, 0] = 1 << 20   # far outside the cache: skipped, reported
    _, _, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O, _, status = _gpu_nsa(c, khat, vhat, 64, B, H_q)
    assert status.item() == binding.SPARSE_ERR_BAD_INDEX
    assert torch.isfinite(O.float()).all()


def test_nsa_length_beyond_compressed_rows_is_reported():
    """seq_len needs more compressed rows than N_cap holds: reported, rows clamped."""
    B, H_q, H_kv, T_cap, k_cap, N_cap = 1, 8, 1, 12 * BLK, 4, 8
    c = _case(B, H_q, H_kv, T_cap, [12 * BLK], k_cap, N_cap, seed=10)
    _, _, khat, vhat = _rows_from_oracle(c, N_cap, B, H_kv)
    O, _, status = _gpu_nsa(c, khat, vhat, 64, B, H_q)
    assert status.item() == binding.SPARSE_ERR_BAD_INDEX
    assert torch.isfinite(O.float()).all()


@pytest.mark.parametrize("chunks", [[700], [64, 1, 63, 200, 5], [130, 1, 1, 1, 1]])
def test_append_kv_pools_values_and_rounds_rows(chunks):
    """sparse_pool_append_kv: caches bit-exact, ktil / vtil the oracle's means within
    fp32 rounding, khat / vhat the bf16 rounding of ktil / vtil and within one bf16
    rounding of the oracle's means."""
    B, H_kv, T_cap, N_cap = 2, 3, 12 * BLK, 12
    total = sum(chunks)
    Kall = wl.randn_bf16((B, H_kv, total, D), 501, "cuda")
    Vall = wl.randn_bf16((B, H_kv, total, D), 502, "cuda")
    kc = torch.zeros((B, H_kv, T_cap, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ktil = torch.zeros((B, H_kv, N_cap, D), dtype=torch.float32, device="cuda")
    vtil = torch.zeros_like(ktil)
    khat = torch.zeros((B, H_kv, N_cap, D), dtype=torch.bfloat16, device="cuda")
    vhat = torch.zeros_like(khat)
    t = 0
    for n in chunks:
        binding.sparse_pool_append_kv(kc, vc, ktil, vtil, Kall[:, :, t:t + n].contiguous(),
                                      Vall[:, :, t:t + n].contiguous(), t, khat=khat, vhat=vhat)
        t += n
    torch.cuda.synchronize()
    P = B * H_kv
    assert np.array_equal(bits(kc)[:, :, :total], bits(Kall))
    assert np.array_equal(bits(vc)[:, :, :total], bits(Vall))
    lens = np.full(P, total, np.int64)
    nb = (total + BLK - 1) // BLK
    for name, cache, til, hat in (("k", kc, ktil, khat), ("v", vc, vtil, vhat)):
        ref = oracle.pool(bits(cache).reshape(P, T_cap, D), lens, N_cap)[:, :nb]
        got = til.double().cpu().numpy().reshape(P, N_cap, D)[:, :nb]
        assert np.all(np.abs(got - ref) <= 1e-5 * (1 + np.abs(ref))), f"{name}til"
        hat_bits = bits(hat).reshape(P, N_cap, D)[:, :nb]
        assert np.array_equal(hat_bits, bits(til.to(torch.bfloat16)).reshape(P, N_cap, D)[:, :nb]), f"{name}hat"
        h = _bits_to_f64(hat_bits)
        assert np.all(np.abs(h - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6), f"{name}hat vs oracle"


def test_nsa_chain_append_then_decode():
    """The whole chain on the GPU (append_kv builds the caches and the bf16 compressed
    rows) against the oracle pooling in fp64."""
    B, H_q, H_kv, T_cap, k_cap, N_cap = 2, 32, 4, 24 * BLK, 8, 24
    lens_b = [24 * BLK - 5, 24 * BLK - 5]
    total = lens_b[0]
    K = wl.randn_bf16((B, H_kv, total, D), 601, "cuda")
    V = wl.randn_bf16((B, H_kv, total, D), 602, "cuda")
    kc = torch.zeros((B, H_kv, T_cap, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ktil = torch.zeros((B, H_kv, N_cap, D), dtype=torch.float32, device="cuda")
    vtil = torch.zeros_like(ktil)
    khat = torch.zeros((B, H_kv, N_cap, D), dtype=torch.bfloat16, device="cuda")
    vhat = torch.zeros_like(khat)
    binding.sparse_pool_append_kv(kc, vc, ktil, vtil, K[:, :, :total - 3].contiguous(),
                                  V[:, :, :total - 3].contiguous(), 0, khat=khat, vhat=vhat)
    for t in range(total - 3, total):
        binding.sparse_pool_append_kv(kc, vc, ktil, vtil, K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous(),
                                      t, khat=khat, vhat=vhat)
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=21)
    c["K"], c["V"] = kc, vc
    P = B * H_kv
    c["Kb"], c["Vb"] = bits(kc).reshape(P, T_cap, D), bits(vc).reshape(P, T_cap, D)
    O, _, status = _gpu_nsa(c, khat, vhat, 300, B, H_q)
    assert status.item() == 0
    kr = oracle.pool(c["Kb"], c["lens_p"], N_cap)
    vr = oracle.pool(c["Vb"], c["lens_p"], N_cap)
    ref = oracle.nsa(c["Qb"], c["Kb"], c["Vb"], kr, vr, c["idx_np"], c["cnt_np"], c["lens_p"], 300,
                     c["gates_np"].reshape(P, -1, 3))
    assert_attn_close(O, ref, "nsa chain")


def test_nsa_full_size_sampled_pairs():
    """The 128K decode shape (B=8, H_q=64, H_kv=8, 67 selected blocks, 512-token
    window, 2048 compressed rows) in the launch configuration of the bench; a sample of
    pairs checked against the oracle."""
    shape = wl.DECODE_128K
    B, H_q, H_kv, T = shape.B, shape.H_q, shape.H_kv, shape.T
    k_cap, N_cap, window = shape.n_init + shape.n_local + shape.k, shape.N_b, 512
    P = B * H_kv
    K = wl.randn_bf16((B, H_kv, T, D), 901, "cuda")
    V = wl.randn_bf16((B, H_kv, T, D), 902, "cuda")
    Q = wl.randn_bf16((B, H_q, D), 903, "cuda")
    kc, vc = torch.empty_like(K), torch.empty_like(V)
    ktil = torch.zeros((B, H_kv, N_cap, D), dtype=torch.float32, device="cuda")
    vtil = torch.zeros_like(ktil)
    khat = torch.zeros((B, H_kv, N_cap, D), dtype=torch.bfloat16, device="cuda")
    vhat = torch.zeros_like(khat)
    binding.sparse_pool_append_kv(kc, vc, ktil, vtil, K, V, 0, khat=khat, vhat=vhat)
    del K, V
    rng = np.random.default_rng(904)
    idx_np = np.stack([np.sort(rng.permutation(N_cap)[:k_cap]) for _ in range(P)]).astype(np.int32)
    cnt_np = np.full(P, k_cap, np.int32)
    gates_np = rng.uniform(0.0, 1.0, (B, H_q, 3))
    c = dict(Q=Q, K=kc, V=vc, idx=torch.from_numpy(idx_np).cuda().view(B, H_kv, k_cap),
             cnt=torch.from_numpy(cnt_np).cuda().view(B, H_kv),
             gates=torch.from_numpy(gates_np.astype(np.float32)).cuda(),
             seq=torch.full((B,), T, dtype=torch.int32, device="cuda"))
    O, _, status = _gpu_nsa(c, khat, vhat, window, B, H_q)
    assert status.item() == 0
    G = H_q // H_kv
    Qb = bits(Q).reshape(P, G, D)
    for p in (0, 9, 37, P - 1):
        b, g = divmod(p, H_kv)
        Kb = bits(kc[b, g]).reshape(1, T, D)
        Vb = bits(vc[b, g]).reshape(1, T, D)
        lens = np.array([T], np.int64)
        ref = oracle.nsa(Qb[p:p + 1], Kb, Vb, oracle.pool(Kb, lens, N_cap), oracle.pool(Vb, lens, N_cap),
                         idx_np[p:p + 1], cnt_np[p:p + 1], lens, window,
                         gates_np[b, g * G:(g + 1) * G].reshape(1, G, 3))
        assert_attn_close(O[b, g * G:(g + 1) * G], ref, f"nsa 128k pair {p}")


# ----------------------------------------------------------------------------- overlapping compression


def _round_rows(x64: np.ndarray) -> np.ndarray:
    return _to_bf16_bits(x64)


@pytest.mark.parametrize("cmp", [(32, 16), (64, 32), (16, 16), (48, 16)])
def test_compress_windows_match_the_oracle(cmp):
    """sparse_nsa_compress, fed in chunks: each completed window's row is the mean of
    its tokens rounded once to bf16 (within one bf16 rounding of the fp64 mean, nearly
    always equal to its rounding); rows of incomplete windows stay untouched."""
    l, s = cmp
    B, H_kv, T_cap = 2, 3, 700
    R = (T_cap - l) // s + 1
    K = wl.randn_bf16((B, H_kv, T_cap, D), 301, "cuda")
    V = wl.randn_bf16((B, H_kv, T_cap, D), 302, "cuda")
    khat = torch.full((B, H_kv, R + 2, D), 3.0, dtype=torch.bfloat16, device="cuda")
    vhat = torch.full_like(khat, 3.0)
    t = 0
    for n in (100, 1, 15, 17, 200, 0, 300):
        n = min(n, 650 - t)
        binding.sparse_nsa_compress(K, V, khat, vhat, t, n, cmp=cmp)
        t += n
    torch.cuda.synchronize()
    P = B * H_kv
    W = (t - l) // s + 1
    for X, hat in ((K, khat), (V, vhat)):
        ref = oracle.pool_windows(bits(X).reshape(P, T_cap, D), np.full(P, t), l, s, R + 2)
        got = _bits_to_f64(bits(hat).reshape(P, R + 2, D))
        assert np.all(np.abs(got[:, :W] - ref[:, :W]) <= 2.0 ** -8 * np.abs(ref[:, :W]) + 1e-7)
        same = np.mean(bits(hat).reshape(P, R + 2, D)[:, :W] == _round_rows(ref[:, :W]))
        assert same > 0.999, same
        assert np.all(got[:, W:] == 3.0)


def _route_case(B, H_q, H_kv, T_cap, lens_b, cmp, seed, n_rows=None):
    l, s = cmp
    P = B * H_kv
    G = H_q // H_kv
    K = wl.randn_bf16((B, H_kv, T_cap, D), seed, "cuda")
    Q = wl.randn_bf16((B, H_q, D), seed + 1, "cuda")
    lens_p = np.repeat(np.asarray(lens_b, np.int64), H_kv)
    if l == 0:
        R = n_rows or (T_cap + BLK - 1) // BLK
        rows64 = oracle.pool(bits(K).reshape(P, T_cap, D), lens_p, R)
    else:
        R = n_rows or (T_cap - l) // s + 1
        rows64 = oracle.pool_windows(bits(K).reshape(P, T_cap, D), lens_p, l, s, R)
    kb = _round_rows(rows64)
    khat = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda().view(B, H_kv, R, D)
    return dict(K=K, Q=Q, Qb=bits(Q).reshape(P, G, D), lens_p=lens_p, kb=kb, khat=khat, R=R,
                seq=torch.tensor(lens_b, dtype=torch.int32, device="cuda"))


def _assert_route_matches(idx_g, cnt_g, idx_r, cnt_r, sc, lens, n_init, n_local, k, rel=1e-4):
    """Identical lists except blocks whose oracle score lies within rel * s_k of the
    oracle's k-th candidate score (fp32 tensor-core scores against fp64)."""
    idx_g = idx_g.cpu().numpy().reshape(idx_r.shape)
    cnt_g = cnt_g.cpu().numpy().reshape(cnt_r.shape)
    exempt = 0
    for p in range(idx_r.shape[0]):
        assert cnt_g[p] == cnt_r[p], (p, cnt_g[p], cnt_r[p])
        c = cnt_r[p]
        g = idx_g[p, :c]
        assert np.all(np.diff(g) > 0) and np.all(idx_g[p, c:] == -1)
        if np.array_equal(g, idx_r[p, :c]):
            continue
        nb = (int(lens[p]) + BLK - 1) // BLK
        cand = [j for j in range(nb) if n_init <= j < nb - n_local]
        kth = sorted((sc[p, j] for j in cand), reverse=True)[k - 1]
        for j in set(g.tolist()) ^ set(idx_r[p, :c].tolist()):
            assert j in cand and abs(sc[p, j] - kth) <= rel * abs(kth), (p, j, sc[p, j], kth)
        exempt += 1
    return exempt


@pytest.mark.parametrize("cmp", [(32, 16), (0, 0), (64, 32)])
@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (64, 8), (32, 2), (3, 3)])
@pytest.mark.parametrize("k", [0, 1, 7, 40])
def test_nsa_select_matches_oracle(cmp, H_q, H_kv, k):
    B, T_cap = 2, 60 * BLK
    lens_b = [60 * BLK, 37 * BLK + 23]
    c = _route_case(B, H_q, H_kv, T_cap, lens_b, cmp, seed=400 + H_q + k)
    n_init, n_local = 1, 2
    k_tot = n_init + n_local + k
    idx = torch.full((B, H_kv, k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(c["Q"], c["khat"], c["seq"], n_init, n_local, k, idx, cnt, cmp=cmp, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kr = _bits_to_f64(c["kb"])
    if cmp[0] == 0:
        ir, cr, sc = oracle.select_heads(c["Qb"], kr, c["lens_p"], n_init, n_local, k, k_tot)
    else:
        ir, cr, sc = oracle.select_windows(c["Qb"], kr, c["lens_p"], cmp[0], cmp[1], n_init, n_local, k, k_tot,
                                           n_blocks_cap=60)
    _assert_route_matches(idx, cnt, ir, cr, sc, c["lens_p"], n_init, n_local, max(k, 1))


@pytest.mark.parametrize("n_blocks", [2723, 2724, 3000])
def test_nsa_select_register_and_radix_topk_boundary(n_blocks):
    """Block rows: up to 2720 candidates the top-k keeps them in registers across CTA 0's
    160 threads; 2721 and more take the radix threshold and the one-warp write."""
    B, H_q, H_kv, T_cap = 1, 8, 2, n_blocks * BLK
    lens_b = [T_cap]
    c = _route_case(B, H_q, H_kv, T_cap, lens_b, (0, 0), seed=470 + n_blocks)
    n_init, n_local, k = 1, 2, 64
    k_tot = n_init + n_local + k
    idx = torch.full((B, H_kv, k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(c["Q"], c["khat"], c["seq"], n_init, n_local, k, idx, cnt, cmp=(0, 0), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ir, cr, sc = oracle.select_heads(c["Qb"], _bits_to_f64(c["kb"]), c["lens_p"], n_init, n_local, k, k_tot)
    _assert_route_matches(idx, cnt, ir, cr, sc, c["lens_p"], n_init, n_local, k)


def test_nsa_select_short_and_empty_lengths():
    """No complete window (every block scores 0: ties to the lower index), one token,
    an empty sequence, n_local = 0."""
    B, H_q, H_kv, T_cap = 4, 8, 2, 20 * BLK
    lens_b = [0, 1, 40, 20 * BLK - 1]
    c = _route_case(B, H_q, H_kv, T_cap, lens_b, (32, 16), seed=430)
    k, n_init, n_local = 3, 0, 0
    idx = torch.full((B, H_kv, k), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(c["Q"], c["khat"], c["seq"], n_init, n_local, k, idx, cnt, cmp=(32, 16), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ir, cr, sc = oracle.select_windows(c["Qb"], _bits_to_f64(c["kb"]), c["lens_p"], 32, 16, n_init, n_local, k, k,
                                       n_blocks_cap=20)
    _assert_route_matches(idx, cnt, ir, cr, sc, c["lens_p"], n_init, n_local, k)


@pytest.mark.parametrize("flags", [0, binding.SPARSE_NSA_BRANCH_GRID])
@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (32, 2)])
def test_nsa_over_windows_matches_oracle(flags, H_q, H_kv):
    B, T_cap, k_cap = 2, 40 * BLK, 9
    lens_b = [40 * BLK, 27 * BLK + 13]
    l, s = 32, 16
    R = (T_cap - l) // s + 1
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, R, seed=500 + H_q)
    P = B * H_kv
    kb = _round_rows(oracle.pool_windows(c["Kb"], c["lens_p"], l, s, R))
    vb = _round_rows(oracle.pool_windows(c["Vb"], c["lens_p"], l, s, R))
    dev = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda().view(B, H_kv, R, D)
    O = torch.full((B, H_q, D), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = binding.nsa_workspace(B, H_q, H_kv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn_nsa(c["Q"], c["K"], c["V"], dev(kb), dev(vb), c["idx"], c["cnt"], c["seq"], 300,
                                   c["gates"], O, ws, flags=flags, status=status, cmp=(l, s))
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oracle.nsa(c["Qb"], c["Kb"], c["Vb"], _bits_to_f64(kb), _bits_to_f64(vb), c["idx_np"], c["cnt_np"],
                     c["lens_p"], 300, c["gates_np"].reshape(P, -1, 3), cmp=(l, s))
    assert_attn_close(O, ref, "nsa windows")


def test_nsa_windows_chain_append_compress_route_attend():
    """The decode chain on the GPU: append, compress the completed windows, route,
    three-branch attention; against the oracle's own chain (its fp64 windows and its
    selection).  Pairs whose selection differs near a tie are skipped for the output."""
    B, H_q, H_kv, T_cap = 2, 32, 4, 48 * BLK
    l, s = 32, 16
    R = (T_cap - l) // s + 1
    lens_b = [48 * BLK - 9, 48 * BLK - 9]
    total = lens_b[0]
    Kall = wl.randn_bf16((B, H_kv, total, D), 611, "cuda")
    Vall = wl.randn_bf16((B, H_kv, total, D), 612, "cuda")
    Q = wl.randn_bf16((B, H_q, D), 613, "cuda")
    kc = torch.zeros((B, H_kv, T_cap, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ktil = torch.zeros((B, H_kv, 48, D), dtype=torch.float32, device="cuda")
    khat = torch.zeros((B, H_kv, R, D), dtype=torch.bfloat16, device="cuda")
    vhat = torch.zeros_like(khat)
    t = 0
    for n in (total - 40, 7, 1, 32):
        binding.sparse_pool_append(kc, vc, ktil, Kall[:, :, t:t + n].contiguous(), Vall[:, :, t:t + n].contiguous(), t)
        binding.sparse_nsa_compress(kc, vc, khat, vhat, t, n, cmp=(l, s))
        t += n
    assert t == total
    n_init, n_local, k = 1, 2, 9
    k_tot = n_init + n_local + k
    seq = torch.tensor(lens_b, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, H_kv, k_tot), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H_kv), dtype=torch.int32, device="cuda")
    gates_np = np.random.default_rng(614).uniform(0, 1, (B, H_q, 3))
    gates = torch.from_numpy(gates_np.astype(np.float32)).cuda()
    O = torch.empty((B, H_q, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(Q, khat, seq, n_init, n_local, k, idx, cnt, cmp=(l, s), status=status)
    binding.sparse_decode_attn_nsa(Q, kc, vc, khat, vhat, idx, cnt, seq, 256, gates, O, None, status=status,
                                   cmp=(l, s))
    torch.cuda.synchronize()
    assert status.item() == 0
    P = B * H_kv
    G = H_q // H_kv
    Kb, Vb, Qb = bits(kc).reshape(P, T_cap, D), bits(vc).reshape(P, T_cap, D), bits(Q).reshape(P, G, D)
    lens_p = np.repeat(np.asarray(lens_b, np.int64), H_kv)
    kr = oracle.pool_windows(Kb, lens_p, l, s, R)
    vr = oracle.pool_windows(Vb, lens_p, l, s, R)
    ir, cr, sc = oracle.select_windows(Qb, kr, lens_p, l, s, n_init, n_local, k, k_tot, n_blocks_cap=48)
    exempt = _assert_route_matches(idx, cnt, ir, cr, sc, lens_p, n_init, n_local, k, rel=2e-2)
    ref = oracle.nsa(Qb, Kb, Vb, kr, vr, ir, cr, lens_p, 256, gates_np.reshape(P, G, 3), cmp=(l, s))
    same = [p for p in range(P) if np.array_equal(idx.cpu().numpy().reshape(P, k_tot)[p], ir[p])]
    assert len(same) >= P - exempt and len(same) > 0
    Og = O.view(B, H_kv, G, D).reshape(P, G, D)
    assert_attn_close(Og[same], ref[same], "nsa windows chain")


def test_nsa_select_full_size_sampled_pairs():
    """NSA routing on the 128K decode shape with 32/16 windows (8191 rows per pair) in
    the launch configuration of the bench; a sample of pairs checked by the oracle."""
    shape = wl.DECODE_128K
    B, H_q, H_kv, T = shape.B, shape.H_q, shape.H_kv, shape.T
    l, s = 32, 16
    R = (T - l) // s + 1
    P = B * H_kv
    G = H_q // H_kv
    rng = np.random.default_rng(931)
    kb = rng.standard_normal((P, R, D)).astype(np.float32) * 0.125
    kb = wl.bf16_bits(torch.from_numpy(kb).to(torch.bfloat16))
    khat = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda().view(B, H_kv, R, D)
    Q = wl.randn_bf16((B, H_q, D), 932, "cuda")
    seq = torch.full((B,), T, dtype=torch.int32, device="cuda")
    k_tot = shape.n_init + shape.n_local + shape.k
    idx = torch.empty((B, H_kv, k_tot), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H_kv), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(Q, khat, seq, shape.n_init, shape.n_local, shape.k, idx, cnt, cmp=(l, s), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Qb = bits(Q).reshape(P, G, D)
    sample = [0, 13, 38, P - 1]
    ir, cr, sc = oracle.select_windows(Qb[sample], _bits_to_f64(kb[sample]), np.full(len(sample), T), l, s,
                                       shape.n_init, shape.n_local, shape.k, k_tot, n_blocks_cap=shape.N_b)
    _assert_route_matches(idx.view(P, k_tot)[sample], cnt.view(P)[sample], ir, cr, sc, np.full(len(sample), T),
                          shape.n_init, shape.n_local, shape.k)


def test_nsa_select_many_queries_per_batch_element():
    """Routing of N_q verification queries per batch element (each its own lists),
    query by query against the oracle."""
    B, N_q, H_q, H_kv, T_cap = 2, 8, 16, 4, 45 * BLK
    l, s = 32, 16
    lens_b = [45 * BLK, 30 * BLK + 7]
    c = _route_case(B, H_q, H_kv, T_cap, lens_b, (l, s), seed=470)
    Qm = wl.randn_bf16((B, N_q, H_q, D), 471, "cuda")
    n_init, n_local, k = 1, 2, 6
    k_tot = n_init + n_local + k
    idx = torch.full((B, H_kv, N_q, k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv, N_q), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_nsa_select(Qm, c["khat"], c["seq"], n_init, n_local, k, idx, cnt, cmp=(l, s), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    P, G = B * H_kv, H_q // H_kv
    kr = _bits_to_f64(c["kb"])
    Qb = bits(Qm)   # [B][N_q][H_q][D]
    for q in range(N_q):
        Qq = Qb[:, q].reshape(P, G, D)
        ir, cr, sc = oracle.select_windows(Qq, kr, c["lens_p"], l, s, n_init, n_local, k, k_tot, n_blocks_cap=45)
        _assert_route_matches(idx[:, :, q], cnt[:, :, q], ir, cr, sc, c["lens_p"], n_init, n_local, k)
