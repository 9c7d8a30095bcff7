"""sparse_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers of this library have no device allocator they may use at decode time:
a plain C host without a caching allocator (a cudaMalloc per call would synchronise
the device), or a serving engine whose device memory is planned up front.  For them
sparse_decode_attn_noalloc runs the stream-K decode path on scratch held in a fixed
4 MiB device array inside the library, so the call itself allocates nothing.

These tests call it through the C ABI twice in a row (the array keeps the previous
call's contents, so the second call shows the counters are cleared) and compare each
result with sparse_decode_attn on the same inputs, at the attention tolerance of the
other tests; and they check that sizes needing more scratch than the array holds are
rejected before anything is launched.  The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

D, BLK = 128, 64
MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _inputs(seed, B=8, H_q=64, H_kv=8, T=256 * BLK, k_cap=67):
    rng = np.random.default_rng(seed)
    P = B * H_kv
    K = wl.randn_bf16((B, H_kv, T, D), seed + 1, "cuda")
    V = wl.randn_bf16((B, H_kv, T, D), seed + 2, "cuda")
    Q = wl.randn_bf16((B, H_q, D), seed + 3, "cuda")
    nb = T // BLK
    idx = np.full((P, k_cap), -1, np.int32)
    cnt = np.zeros(P, np.int32)
    for p in range(P):
        c = k_cap if p % 5 else int(rng.integers(0, k_cap))
        idx[p, :c] = np.sort(rng.permutation(nb)[:c])
        cnt[p] = c
    idx_t = torch.from_numpy(idx).cuda().view(B, H_kv, k_cap)
    cnt_t = torch.from_numpy(cnt).cuda().view(B, H_kv)
    seq = torch.full((B,), T, dtype=torch.int32, device="cuda")
    return Q, K, V, idx_t, cnt_t, seq


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    for call, seed in enumerate((101, 202)):
        Q, K, V, idx, cnt, seq = _inputs(seed)
        ref = torch.zeros_like(Q)
        ref_lse = torch.zeros(Q.shape[:2], dtype=torch.float32, device="cuda")
        binding.sparse_decode_attn(Q, K, V, idx, cnt, seq, ref, ref_lse)
        out = torch.full_like(Q, 5.0)
        lse = torch.zeros_like(ref_lse)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.sparse_decode_attn_noalloc(Q, K, V, idx, cnt, seq, out, lse, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: status {status.item()}"
        err = (out.float() - ref.float()).abs()
        assert err.max().item() <= MAX_ABS, f"call {call}: max abs err {err.max().item():.3e}"
        assert err.mean().item() <= MEAN_ABS, f"call {call}: mean abs err {err.mean().item():.3e}"
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= 2e-3


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    Q, K, V, idx, cnt, seq = _inputs(7)
    out = torch.zeros_like(Q)
    with pytest.raises(binding.SparsePoolError) as e:
        # 1000 CTAs would need about 8 MB of partial states: more than the 4 MiB array
        binding.sparse_decode_attn_noalloc(Q, K, V, idx, cnt, seq, out, n_split=1000)
    assert e.value.status == binding.SPARSE_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert not out.any()


@pytest.mark.parametrize("n_split", [37, 304])
def test_noalloc_matches_the_oracle_at_other_splits(n_split):
    """The allocation-free call with other CTA counts (ranges that cut pairs at other
    points), against the fp64 oracle directly: the same tolerances as the decode tests."""
    import oracle
    Q, K, V, idx, cnt, seq = _inputs(303)
    B, H_q = Q.shape[:2]
    H_kv = K.shape[1]
    P, G, T = B * H_kv, H_q // H_kv, K.shape[2]
    out = torch.full_like(Q, 5.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.sparse_decode_attn_noalloc(Q, K, V, idx, cnt, seq, out, n_split=n_split, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Oref, _ = oracle.attn(wl.bf16_bits(Q).reshape(P, G, D), wl.bf16_bits(K).reshape(P, T, D),
                          wl.bf16_bits(V).reshape(P, T, D), idx.cpu().numpy().reshape(P, -1),
                          cnt.cpu().numpy().reshape(P), [T] * P)
    err = np.abs(out.float().cpu().double().numpy().reshape(Oref.shape) - Oref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"max {err.max():.3e} mean {err.mean():.3e}"


def test_noalloc_rejected_call_leaves_the_scratch_alone():
    """A call rejected by the argument checks launches nothing: a valid call right after
    it still gives the right result (its counters were not disturbed half-way)."""
    Q, K, V, idx, cnt, seq = _inputs(404)
    out = torch.zeros_like(Q)
    with pytest.raises(binding.SparsePoolError) as e:
        binding.sparse_decode_attn_noalloc(Q, K, V, idx, cnt, seq, out, flags=0x80)   # an unknown flag
    assert e.value.status == binding.SPARSE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not out.any()
    ref = torch.zeros_like(Q)
    binding.sparse_decode_attn(Q, K, V, idx, cnt, seq, ref)
    binding.sparse_decode_attn_noalloc(Q, K, V, idx, cnt, seq, out)
    torch.cuda.synchronize()
    assert (out.float() - ref.float()).abs().max().item() <= MAX_ABS
