"""GPU parity of sparse_prefill_select, the Forecast selection of every prefill position
(SparDA notes §4.3 eq.(16) with the per-position selection of eq.(6) / Alg.1 step 2).

Against the fp64 oracle: lists identical per position, except blocks whose score lies
within 1e-4 * max(|s_k|, 1) of the position's k-th candidate score (the scores are
fp32 tensor-core sums of exact products).  Small cases compare every position; long
ones (one CTA tile of 32 or 16 positions) a sample of positions.  Every input comes
from the seeded generators."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl
from parity_utils import BLK, D, bits

pytestmark = pytest.mark.gpu

TIE_REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _values(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _run(F, kt, lens_b, n_init, n_local, k):
    B, H_kv, T_cap, _ = F.shape
    k_tot = n_init + n_local + k
    idx = torch.full((B, H_kv, T_cap, k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv, T_cap), -7, dtype=torch.int32, device="cuda")
    seq = torch.tensor(lens_b, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_prefill_select(F, kt, seq, n_init, n_local, k, idx, cnt, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return idx, cnt


def _compare(idx_g, cnt_g, idx_r, cnt_r, Fv, ktv, rows, n_init, n_local, k):
    """idx_g/cnt_g: GPU rows [P][R]; idx_r/cnt_r: oracle rows; Fv [P][T][D] and ktv
    [P][N][D] fp64 values for the near-tie band."""
    exempt = 0
    for p in range(idx_r.shape[0]):
        for r, t in enumerate(rows):
            if cnt_r[p, r] < 0:
                continue
            c = cnt_r[p, r]
            assert cnt_g[p, r] == c, (p, t, cnt_g[p, r], c)
            g = idx_g[p, r, :c]
            assert np.all(np.diff(g) > 0) and np.all(idx_g[p, r, c:] == -1), (p, t)
            if np.array_equal(g, idx_r[p, r, :c]):
                continue
            nb = t // BLK + 1
            sc = ktv[p, :nb] @ Fv[p, t]
            cand = [j for j in range(nb) if n_init <= j < nb - n_local]
            kth = sorted((sc[j] for j in cand), reverse=True)[k - 1]
            for j in set(g.tolist()) ^ set(idx_r[p, r, :c].tolist()):
                assert j in cand and abs(sc[j] - kth) <= TIE_REL * max(abs(kth), 1.0), (p, t, j, sc[j], kth)
            exempt += 1
    return exempt


@pytest.mark.parametrize("n_init,n_local,k", [(1, 2, 3), (0, 1, 1), (2, 1, 0), (1, 2, 40), (1, 1, 7)])
def test_prefill_select_every_position(n_init, n_local, k):
    B, H_kv, T_cap, N = 2, 3, 1000, 16
    lens_b = [1000, 701]
    F = wl.randn_bf16((B, H_kv, T_cap, D), 700 + k, "cuda")
    kt = torch.randn((B, H_kv, N, D), generator=wl._gen("cuda", 701 + k), device="cuda")
    idx, cnt = _run(F, kt, lens_b, n_init, n_local, k)
    P = B * H_kv
    Fb = bits(F).reshape(P, T_cap, D)
    ktv = kt.double().cpu().numpy().reshape(P, N, D)
    lens_p = np.repeat(np.asarray(lens_b, np.int64), H_kv)
    ir, cr = oracle.prefill_select(Fb, ktv, lens_p, n_init, n_local, k)
    ig = idx.cpu().numpy().reshape(P, T_cap, -1)
    cg = cnt.cpu().numpy().reshape(P, T_cap)
    _compare(ig, cg, ir, cr, _values(Fb), ktv, list(range(T_cap)), n_init, n_local, max(k, 1))
    # positions past a length are not written
    assert np.all(cg[H_kv:, 701:] == -7)


def test_prefill_select_exact_ties_take_the_lower_block():
    """Unit Forecast vectors read one key dimension exactly: equal keys tie exactly in
    fp32, and the lower block wins."""
    B, H_kv, T_cap, N = 1, 2, 64 * 12, 12
    Fz = torch.zeros((B, H_kv, T_cap, D), dtype=torch.float32)
    Fz[..., 3] = 1.0
    F = Fz.to(torch.bfloat16).cuda()
    kt = torch.zeros((B, H_kv, N, D), dtype=torch.float32)
    kt[0, 0, :, 3] = torch.tensor([1.0, 5.0, 5.0, 2.0, 5.0, 5.0, 0.5, 5.0, 9.0, 5.0, 1.0, 1.0])
    kt[0, 1, :, 3] = torch.tensor([2.0] * N)
    kt = kt.cuda()
    idx, cnt = _run(F, kt, [T_cap], 1, 1, 3)
    P = B * H_kv
    ir, cr = oracle.prefill_select(bits(F).reshape(P, T_cap, D), kt.double().cpu().numpy().reshape(P, N, D),
                                   [T_cap] * P, 1, 1, 3)
    assert np.array_equal(idx.cpu().numpy().reshape(ir.shape), ir)
    assert np.array_equal(cnt.cpu().numpy().reshape(cr.shape), cr)


@pytest.mark.parametrize("T_cap,N", [(40000, 640), (100000, 1600), (131072, 2048)])
def test_prefill_select_long_sequences_sampled(T_cap, N):
    """Tiles of 32 and 16 positions (625 / 1563 / 2048 compressed keys); a sample of
    positions, including tile and block boundaries, checked by the oracle."""
    B, H_kv = 1, 2
    lens_b = [T_cap - 5]
    F = wl.randn_bf16((B, H_kv, T_cap, D), 710 + N, "cuda")
    kt = torch.randn((B, H_kv, N, D), generator=wl._gen("cuda", 711 + N), device="cuda")
    n_init, n_local, k = 1, 2, 32
    idx, cnt = _run(F, kt, lens_b, n_init, n_local, k)
    rng = np.random.default_rng(712)
    rows = sorted(set([0, 15, 16, 31, 32, 63, 64, 65, 127, 128, 4095, lens_b[0] - 1, lens_b[0] - 17] +
                      rng.integers(0, lens_b[0], 120).tolist()))
    P = B * H_kv
    Fb = bits(F).reshape(P, T_cap, D)
    ktv = kt.double().cpu().numpy().reshape(P, N, D)
    lens_p = np.repeat(np.asarray(lens_b, np.int64), H_kv)
    ir, cr = oracle.prefill_select(Fb, ktv, lens_p, n_init, n_local, k, rows=rows)
    ig = idx.cpu().numpy().reshape(P, T_cap, -1)[:, rows]
    cg = cnt.cpu().numpy().reshape(P, T_cap)[:, rows]
    _compare(ig, cg, ir, cr, _values(Fb), ktv, rows, n_init, n_local, k)


def test_prefill_select_bench_shape_sampled():
    """The bench's prefill workload (B = 4, H_kv = 8, 32K positions, 512 compressed keys,
    k = 32) in its launch configuration; sampled positions of a few pairs."""
    sh = wl.PREFILL_32K
    B, H_kv, T, N = sh.B, sh.H_kv, sh.T, sh.N_b
    x = wl.prefill_inputs(sh, "cuda")
    idx, cnt = _run(x["F"], x["ktil"], [T] * B, sh.n_init, sh.n_local, sh.k)
    P = B * H_kv
    rng = np.random.default_rng(713)
    rows = sorted(set([0, 64, 8191, T - 1] + rng.integers(0, T, 60).tolist()))
    for p in (0, 11, P - 1):
        b, g = divmod(p, H_kv)
        Fb = bits(x["F"][b, g]).reshape(1, T, D)
        ktv = x["ktil"][b, g].double().cpu().numpy().reshape(1, N, D)
        ir, cr = oracle.prefill_select(Fb, ktv, [T], sh.n_init, sh.n_local, sh.k, rows=rows)
        ig = idx[b, g].cpu().numpy()[None, rows]
        cg = cnt[b, g].cpu().numpy()[None, rows]
        _compare(ig, cg, ir, cr, _values(Fb), ktv, rows, sh.n_init, sh.n_local, sh.k)
