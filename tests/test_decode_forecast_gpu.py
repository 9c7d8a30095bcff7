"""GPU parity of sparse_decode_attn_forecast: one decode layer, the attention of layer l
fused with the Forecast selection of layer l+1 (SparDA notes §4.1, §4.2 Alg.1 steps 2
and 4).

Checked against the fp64 oracle (selection: identical lists except near ties;
attention: the tolerances of parity_utils) and against the two calls it fuses
(sparse_select_topk scores with the same fp32 arithmetic, so its lists must be
identical; sparse_decode_attn with the same cluster split agrees within the
split-invariance bound of the decode tests).
Every input comes from the seeded generators."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl
from parity_utils import (BLK, D, assert_attn_close, assert_selection_matches, bits,
                          oracle_attn_on_taken_lists)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _lens_pair(lens_b, H_kv):
    return np.repeat(np.asarray(lens_b, dtype=np.int64), H_kv)


def _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed, ktil_np=None, F=None):
    """Seeded inputs: K/V/Q of layer l, a distinct ascending block list per pair, and
    the next layer's compressed keys and Forecast vectors."""
    P = B * H_kv
    rng = np.random.default_rng(seed)
    K = wl.randn_bf16((B, H_kv, T_cap, D), seed + 1, "cuda")
    V = wl.randn_bf16((B, H_kv, T_cap, D), seed + 2, "cuda")
    Q = wl.randn_bf16((B, H_q, D), seed + 3, "cuda")
    lens_p = _lens_pair(lens_b, H_kv)
    idx_np = np.full((P, k_cap), -1, np.int32)
    cnt_np = np.zeros(P, np.int32)
    for p in range(P):
        nb = (int(lens_p[p]) + BLK - 1) // BLK
        c = min(nb, k_cap) if p % 3 else min(nb, max(0, k_cap - 5))
        idx_np[p, :c] = np.sort(rng.permutation(nb)[:c])
        cnt_np[p] = c
    if ktil_np is None:
        ktil_np = rng.standard_normal((P, N_cap, D)).astype(np.float32)
    if F is None:
        F = wl.randn_bf16((B, H_kv, D), seed + 4, "cuda")
    return dict(K=K, V=V, Q=Q, idx_np=idx_np, cnt_np=cnt_np, ktil_np=ktil_np, F=F, lens_p=lens_p,
                idx=torch.from_numpy(idx_np).cuda().view(B, H_kv, k_cap),
                cnt=torch.from_numpy(cnt_np).cuda().view(B, H_kv),
                ktil=torch.from_numpy(ktil_np).cuda().view(B, H_kv, N_cap, D),
                seq=torch.tensor(lens_b, dtype=torch.int32, device="cuda"))


def _fused(c, B, H_q, H_kv, n_init, n_local, k, k_tot_next, n_split, with_F=True):
    O = torch.full((B, H_q, D), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H_q), dtype=torch.float32, device="cuda")
    idx_next = torch.full((B, H_kv, k_tot_next), -7, dtype=torch.int32, device="cuda")
    cnt_next = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn_forecast(c["Q"], c["K"], c["V"], c["idx"], c["cnt"], c["seq"], O, lse,
                                        F=c["F"] if with_F else None, ktil_next=c["ktil"], n_init=n_init,
                                        n_local=n_local, k=k, idx_next=idx_next, count_next=cnt_next,
                                        n_split=n_split, status=status)
    torch.cuda.synchronize()
    return O, lse, idx_next, cnt_next, status.item()


@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (64, 8), (32, 2)])
@pytest.mark.parametrize("n_split", [0, 1, 2, 4, 8])
def test_forecast_matches_oracle_and_the_separate_calls(H_q, H_kv, n_split):
    B, T_cap, k_cap, N_cap = 2, 700 * BLK, 21, 700
    lens_b = [700 * BLK, 611 * BLK + 9]
    n_init, n_local, k, k_tot_next = 1, 2, 32, 40
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=H_q + 13 * n_split)
    O, lse, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, n_init, n_local, k, k_tot_next, n_split)
    assert st == 0
    P, G = B * H_kv, H_q // H_kv
    # selection: identical to sparse_select_topk, and the oracle's up to near ties
    idx_sep = torch.full_like(idx_next, -7)
    cnt_sep = torch.full_like(cnt_next, -7)
    binding.sparse_select_topk(c["F"], c["ktil"], c["seq"], n_init, n_local, k, idx_sep, cnt_sep)
    torch.cuda.synchronize()
    assert torch.equal(idx_next, idx_sep) and torch.equal(cnt_next, cnt_sep)
    ridx, rcnt, rs = oracle.select(bits(c["F"]).reshape(P, D), c["ktil_np"].astype(np.float64), c["lens_p"], n_init,
                                   n_local, k, k_tot_next)
    assert_selection_matches(idx_next, cnt_next, ridx, rcnt, rs, c["lens_p"], n_init, n_local, k)
    # attention: the oracle's, and the cluster decode's (the fused kernel slices by k_tot,
    # the cluster kernel by count, so short lists may sum in another order)
    Oref, lref = oracle.attn(bits(c["Q"]).reshape(P, G, D), bits(c["K"]).reshape(P, T_cap, D),
                             bits(c["V"]).reshape(P, T_cap, D), c["idx_np"], c["cnt_np"], c["lens_p"])
    assert_attn_close(O, Oref.reshape(B, H_q, D))
    g, r = lse.cpu().double().numpy().reshape(lref.shape), lref
    assert np.array_equal(np.isfinite(g), np.isfinite(r))
    assert np.allclose(g[np.isfinite(r)], r[np.isfinite(r)], rtol=0, atol=2e-3)
    O_sep = torch.zeros_like(O)
    binding.sparse_decode_attn(c["Q"], c["K"], c["V"], c["idx"], c["cnt"], c["seq"], O_sep, n_split=n_split)
    torch.cuda.synchronize()
    assert (O.float() - O_sep.float()).abs().max().item() <= 2 ** -7


@pytest.mark.parametrize("k_cap", [7, 21, 67])
@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (64, 8)])
def test_forecast_sixteen_cta_clusters_with_short_lists(H_q, H_kv, k_cap):
    """Clusters of 16 CTAs with the group top-k: CTA 0 takes the next layer's top-k and
    attends over nothing, the other 15 share the list (7 blocks: 8 of them get none) and
    merge without CTA 0 (the pull form)."""
    B, T_cap, N_cap = 1, 700 * BLK, 700
    lens_b = [611 * BLK + 9]
    n_init, n_local, k, k_tot_next = 1, 2, 32, 40
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=H_q + k_cap)
    O, lse, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, n_init, n_local, k, k_tot_next, 16)
    assert st == 0
    P, G = B * H_kv, H_q // H_kv
    idx_sep = torch.full_like(idx_next, -7)
    cnt_sep = torch.full_like(cnt_next, -7)
    binding.sparse_select_topk(c["F"], c["ktil"], c["seq"], n_init, n_local, k, idx_sep, cnt_sep)
    torch.cuda.synchronize()
    assert torch.equal(idx_next, idx_sep) and torch.equal(cnt_next, cnt_sep)
    Oref, lref = oracle.attn(bits(c["Q"]).reshape(P, G, D), bits(c["K"]).reshape(P, T_cap, D),
                             bits(c["V"]).reshape(P, T_cap, D), c["idx_np"], c["cnt_np"], c["lens_p"])
    assert_attn_close(O, Oref.reshape(B, H_q, D))
    g, r = lse.cpu().double().numpy().reshape(lref.shape), lref
    assert np.array_equal(np.isfinite(g), np.isfinite(r))
    assert np.allclose(g[np.isfinite(r)], r[np.isfinite(r)], rtol=0, atol=2e-3)


def test_forecast_ties_go_to_the_lower_index_exactly():
    # integer scores: fp32 and fp64 agree exactly, so the tie rule alone decides
    B, H_q, H_kv, T_cap, k_cap, N_cap = 2, 16, 2, 300 * BLK, 9, 300
    lens_b = [300 * BLK, 77 * BLK + 5]
    P = B * H_kv
    rng = np.random.default_rng(7)
    ktil_np = np.zeros((P, N_cap, D), np.float32)
    ktil_np[:, :, 5] = rng.integers(-4, 5, size=(P, N_cap))
    F = torch.zeros((B, H_kv, D), dtype=torch.bfloat16, device="cuda")
    F[..., 5] = 1.0
    for kt in (ktil_np, np.zeros_like(ktil_np)):
        c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=31, ktil_np=kt, F=F)
        _, _, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, 1, 2, 16, 19, 0)
        assert st == 0
        ridx, rcnt, _ = oracle.select(bits(F).reshape(P, D), kt.astype(np.float64), c["lens_p"], 1, 2, 16, 19)
        assert np.array_equal(idx_next.cpu().numpy().reshape(ridx.shape), ridx)
        assert np.array_equal(cnt_next.cpu().numpy().reshape(rcnt.shape), rcnt)


def test_forecast_few_blocks_take_all_and_empty_lists():
    B, H_q, H_kv, T_cap, k_cap, N_cap = 5, 8, 2, 8 * BLK, 4, 8
    lens_b = [7 * BLK, 2 * BLK, 65, 1, 0]
    c = _case(B, H_q, H_kv, T_cap, lens_b, k_cap, N_cap, seed=3)
    O, lse, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, 1, 2, 4, 7, 0)
    assert st == 0
    P, G = B * H_kv, H_q // H_kv
    ridx, rcnt, _ = oracle.select(bits(c["F"]).reshape(P, D), c["ktil_np"].astype(np.float64), c["lens_p"], 1, 2, 4,
                                  7)
    assert np.array_equal(idx_next.cpu().numpy().reshape(ridx.shape), ridx)
    assert np.array_equal(cnt_next.cpu().numpy().reshape(rcnt.shape), rcnt)
    Oref, _ = oracle.attn(bits(c["Q"]).reshape(P, G, D), bits(c["K"]).reshape(P, T_cap, D),
                          bits(c["V"]).reshape(P, T_cap, D), c["idx_np"], c["cnt_np"], c["lens_p"])
    assert_attn_close(O, Oref.reshape(B, H_q, D))


@pytest.mark.parametrize("k", [0, 1, 5])
def test_forecast_small_k(k):
    B, H_q, H_kv, T_cap, k_cap, N_cap = 2, 16, 2, 100 * BLK, 7, 100
    c = _case(B, H_q, H_kv, T_cap, [100 * BLK, 37 * BLK + 2], k_cap, N_cap, seed=50 + k)
    _, _, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, 1, 2, k, 3 + k, 0)
    assert st == 0
    P = B * H_kv
    ridx, rcnt, rs = oracle.select(bits(c["F"]).reshape(P, D), c["ktil_np"].astype(np.float64), c["lens_p"], 1, 2,
                                   k, 3 + k)
    if k == 0:   # only B_init and B_local
        assert np.array_equal(idx_next.cpu().numpy().reshape(ridx.shape), ridx)
        assert np.array_equal(cnt_next.cpu().numpy().reshape(rcnt.shape), rcnt)
    else:
        assert_selection_matches(idx_next, cnt_next, ridx, rcnt, rs, c["lens_p"], 1, 2, k)


def test_forecast_without_F_is_the_decode_attention():
    B, H_q, H_kv, T_cap, k_cap = 2, 32, 4, 90 * BLK, 13
    c = _case(B, H_q, H_kv, T_cap, [90 * BLK, 50 * BLK + 3], k_cap, 90, seed=41)
    O, _, idx_next, _, st = _fused(c, B, H_q, H_kv, 1, 2, 8, 11, 4, with_F=False)
    assert st == 0 and (idx_next == -7).all()      # no selection written
    O_sep = torch.zeros_like(O)
    binding.sparse_decode_attn(c["Q"], c["K"], c["V"], c["idx"], c["cnt"], c["seq"], O_sep, n_split=4)
    torch.cuda.synchronize()
    assert (O.float() - O_sep.float()).abs().max().item() <= 2 ** -7


def test_forecast_reports_a_length_beyond_the_compressed_keys():
    B, H_q, H_kv, T_cap, k_cap, N_cap = 1, 8, 2, 20 * BLK, 5, 10
    c = _case(B, H_q, H_kv, T_cap, [20 * BLK], k_cap, N_cap, seed=5)
    _, _, idx_next, cnt_next, st = _fused(c, B, H_q, H_kv, 1, 2, 4, 7, 0)
    assert st == binding.SPARSE_ERR_BAD_INDEX
    assert (cnt_next <= 7).all() and (cnt_next >= 0).all()


def test_forecast_chain_of_layers_matches_the_oracle():
    """Layer 0 selects with sparse_select_topk; every layer then attends over the list
    the previous call selected and selects for the next layer (the decode chain of the
    SparDA notes, Alg.1), compared with the oracle's own chain."""
    L, B, H_q, H_kv, T = 4, 2, 32, 4, 256 * BLK
    n_init, n_local, k = 1, 2, 24
    k_tot = n_init + n_local + k
    P, G, N_cap = B * H_kv, H_q // H_kv, T // BLK
    lens_b = [T, T - 999]
    lens_p = _lens_pair(lens_b, H_kv)
    seq = torch.tensor(lens_b, dtype=torch.int32, device="cuda")
    Ks, Vs, kts = [], [], []
    for l in range(L):
        K = wl.randn_bf16((B, H_kv, T, D), 100 + l, "cuda")
        V = wl.randn_bf16((B, H_kv, T, D), 200 + l, "cuda")
        # compressed keys by the library's own append (the GPU side of the chain)
        kc, vc = torch.zeros_like(K), torch.zeros_like(V)
        kt = torch.zeros((B, H_kv, N_cap, D), dtype=torch.float32, device="cuda")
        for b in range(B):
            binding.sparse_pool_append(kc[b:b + 1], vc[b:b + 1], kt[b:b + 1], K[b:b + 1, :, :lens_b[b]].contiguous(),
                                       V[b:b + 1, :, :lens_b[b]].contiguous(), 0)
        Ks.append(kc)
        Vs.append(vc)
        kts.append(kt)
    Qs = [wl.randn_bf16((B, H_q, D), 300 + l, "cuda") for l in range(L)]
    Fs = [wl.randn_bf16((B, H_kv, D), 400 + l, "cuda") for l in range(L + 1)]
    idx = [torch.full((B, H_kv, k_tot), -7, dtype=torch.int32, device="cuda") for _ in range(L)]
    cnt = [torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda") for _ in range(L)]
    O = [torch.zeros((B, H_q, D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_select_topk(Fs[L], kts[0], seq, n_init, n_local, k, idx[0], cnt[0], status=status)
    for l in range(L):
        nxt = l + 1 < L
        binding.sparse_decode_attn_forecast(Qs[l], Ks[l], Vs[l], idx[l], cnt[l], seq, O[l],
                                            F=Fs[l] if nxt else None, ktil_next=kts[l + 1] if nxt else None,
                                            n_init=n_init, n_local=n_local, k=k,
                                            idx_next=idx[l + 1] if nxt else None,
                                            count_next=cnt[l + 1] if nxt else None, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    # the oracle's chain from the same generator inputs
    for l in range(L):
        Kb = bits(Ks[l]).reshape(P, T, D)
        ktil_ref = oracle.pool(Kb, lens_p, N_cap)
        F_sel = Fs[L] if l == 0 else Fs[l - 1]
        ridx, rcnt, rs = oracle.select(bits(F_sel).reshape(P, D), ktil_ref, lens_p, n_init, n_local, k, k_tot)
        exempt = assert_selection_matches(idx[l], cnt[l], ridx, rcnt, rs, lens_p, n_init, n_local, k)
        Qb, Vb = bits(Qs[l]).reshape(P, G, D), bits(Vs[l]).reshape(P, T, D)
        Oref, _ = oracle.attn(Qb, Kb, Vb, ridx, rcnt, lens_p)
        # every pair: over the oracle's list, or over the GPU's where a near tie let it differ
        Oown, _ = oracle_attn_on_taken_lists(idx[l], cnt[l], ridx, rcnt, Oref, Qb, Kb, Vb, lens_p)
        assert_attn_close(O[l], Oown.reshape(B, H_q, D), f"layer {l}")
        assert exempt <= 1


def test_forecast_128k_layer_all_pairs_at_full_size():
    """One physical layer of the 128K, B=8, G=8 workload at full size, in the launch
    configuration of the 80-layer bench step: sparse_select_topk picks this layer's
    blocks with F_0, then one sparse_decode_attn_forecast launch attends over them and
    selects again from the same compressed keys with F_10.  The oracle checks all 64
    pairs: both selections (near-tie rule) and the fused launch's attention (over the
    oracle's list, or over the GPU's where a validated near tie let it differ)."""
    from parity_utils import GpuLayer
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
    del Kb, Vb
    seq = torch.full((B,), sh.T, dtype=torch.int32, device="cuda")
    F0, F10 = wl.forecast(sh, 1, 0, "cuda"), wl.forecast(sh, 1, 10, "cuda")
    Q = wl.queries(sh, 1, "cuda")
    L.select(F0, seq)
    idx_next = torch.full_like(L.idx, -7)
    cnt_next = torch.full_like(L.count, -7)
    binding.sparse_decode_attn_forecast(Q, L.k_cache, L.v_cache, L.idx, L.count, seq, L.O, L.lse, F=F10,
                                        ktil_next=L.ktil, n_init=sh.n_init, n_local=sh.n_local, k=sh.k,
                                        idx_next=idx_next, count_next=cnt_next, status=L.status)
    torch.cuda.synchronize()
    assert L.status.item() == 0
    lens_p = [sh.T] * P
    Qb = bits(Q).reshape(P, G, D)
    ktil = oracle.pool(Kh, lens_p, sh.N_b)
    ridx, rcnt, rs = oracle.select(bits(F0).reshape(P, D), ktil, lens_p, sh.n_init, sh.n_local, sh.k)
    assert_selection_matches(L.idx, L.count, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
    Oref, _ = oracle.attn(Qb, Kh, Vh, ridx, rcnt, lens_p)
    Oown, _ = oracle_attn_on_taken_lists(L.idx, L.count, ridx, rcnt, Oref, Qb, Kh, Vh, lens_p)
    assert_attn_close(L.O, Oown.reshape(B, sh.H_q, D), "fused attention")
    nidx, ncnt, ns = oracle.select(bits(F10).reshape(P, D), ktil, lens_p, sh.n_init, sh.n_local, sh.k)
    assert_selection_matches(idx_next, cnt_next, nidx, ncnt, ns, lens_p, sh.n_init, sh.n_local, sh.k)
    for p in range(P):   # generator sanity: the planted blocks are the ones selected
        assert len(set(planted[1, p].tolist()) & set(nidx[p].tolist())) >= 40


@pytest.mark.parametrize("n_split", [0, 8, 16])
def test_b1_80layer_resident_sampled_layers(n_split):
    """The literal B = 1 variant of the 128K step (8 pairs per layer, all 80 layers
    resident in the bench): the bench's chain of launches -- sparse_select_topk for
    layer 0 with F^cur_0, then one sparse_decode_attn_forecast per layer -- run on the
    physical layers that sampled layers {0, 1, 39, 79} read and select for, each launch
    checked against the oracle: its attention over the list the previous launch chose
    and its selection for the next layer (none after the last)."""
    from parity_utils import oracle_attn_on_taken_lists
    sh = wl.DECODE_128K_B1
    B, H_kv, G, P = sh.B, sh.H_kv, sh.G, sh.pairs
    sample = (0, 1, 39, 79)
    phys = sorted({l for l in sample} | {l + 1 for l in sample if l + 1 < sh.layers})
    planted = wl.planted_sets(sh, sh.phys_layers)
    kc, vc, kt, Kh, Vh = {}, {}, {}, {}, {}
    for q in phys:
        kc[q] = torch.zeros((B, H_kv, sh.T, D), dtype=torch.bfloat16, device="cuda")
        vc[q] = torch.zeros_like(kc[q])
        kt[q] = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device="cuda")
        kn = torch.empty_like(kc[q])
        vn = torch.empty_like(kc[q])
        for p in range(P):
            kn[0, p], vn[0, p] = wl.kv_pair(sh, q, p, planted[q, p], "cuda")
        binding.sparse_pool_append(kc[q], vc[q], kt[q], kn, vn, 0)
        Kh[q], Vh[q] = bits(kn).reshape(P, sh.T, D), bits(vn).reshape(P, sh.T, D)
        del kn, vn
    seq = torch.full((B,), sh.T, dtype=torch.int32, device="cuda")
    lens_p = [sh.T] * P
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_tot = sh.k_tot
    ktil_ref = {q: oracle.pool(Kh[q], lens_p, sh.N_b) for q in phys}
    for q in phys:
        assert np.allclose(kt[q].view(P, sh.N_b, D).cpu().double().numpy(), ktil_ref[q], rtol=1e-5, atol=1e-6)
    for l in sample:
        # this layer's list: layer 0 from its own current-layer Forecast, later layers from
        # the previous layer's Forecast F_{l-1} (which targets layer l)
        F_prev = wl.forecast(sh, 0, -1, "cuda") if l == 0 else wl.forecast(sh, l, l - 1, "cuda")
        idx = torch.full((B, H_kv, k_tot), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
        binding.sparse_select_topk(F_prev, kt[l], seq, sh.n_init, sh.n_local, sh.k, idx, cnt, status=status)
        nxt = l + 1 < sh.layers
        F = wl.forecast(sh, l + 1, l, "cuda") if nxt else None
        Q = wl.queries(sh, l, "cuda")
        O = torch.zeros((B, sh.H_q, D), dtype=torch.bfloat16, device="cuda")
        idx_n = torch.full_like(idx, -7)
        cnt_n = torch.full_like(cnt, -7)
        binding.sparse_decode_attn_forecast(Q, kc[l], vc[l], idx, cnt, seq, O, F=F,
                                            ktil_next=kt[l + 1] if nxt else None, n_init=sh.n_init,
                                            n_local=sh.n_local, k=sh.k, idx_next=idx_n if nxt else None,
                                            count_next=cnt_n if nxt else None, n_split=n_split, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        ridx, rcnt, rs = oracle.select(bits(F_prev).reshape(P, D), ktil_ref[l], lens_p, sh.n_init, sh.n_local, sh.k)
        assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
        Qb = bits(Q).reshape(P, G, D)
        Oref, _ = oracle.attn(Qb, Kh[l], Vh[l], ridx, rcnt, lens_p)
        Oown, _ = oracle_attn_on_taken_lists(idx, cnt, ridx, rcnt, Oref, Qb, Kh[l], Vh[l], lens_p)
        assert_attn_close(O, Oown.reshape(B, sh.H_q, D), f"layer {l}")
        if nxt:
            nidx, ncnt, ns = oracle.select(bits(F).reshape(P, D), ktil_ref[l + 1], lens_p, sh.n_init, sh.n_local,
                                           sh.k)
            assert_selection_matches(idx_n, cnt_n, nidx, ncnt, ns, lens_p, sh.n_init, sh.n_local, sh.k)
            for p in range(P):   # generator sanity: the planted blocks are the ones selected
                assert len(set(planted[l + 1, p].tolist()) & set(nidx[p].tolist())) >= 40
        else:
            assert (idx_n == -7).all() and (cnt_n == -7).all()   # the last layer selects nothing
