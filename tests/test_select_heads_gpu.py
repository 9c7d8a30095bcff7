"""GPU parity of sparse_select_topk_heads, the InfLLM-V2 multi-head selector of the
SparDA notes' §4.3 comparison (eq.(8), Figure 3), against oracle.select_heads on
seeded inputs: identical lists except near ties (a differing block's oracle score
within 1e-4 * max(|s_(k)|, 1) of the oracle's k-th score)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import binding, build
from block_sparse_long_pool_gb300 import workloads as wl
from parity_utils import BLK, D, assert_selection_matches, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load()


def _run(lens_b, H_q, H_kv, N_cap, n_init, n_local, k, seed, scale=0.0, ktil_scale=1.0):
    B = len(lens_b)
    P, G = B * H_kv, H_q // H_kv
    rng = np.random.default_rng(seed)
    ktil_np = (rng.standard_normal((P, N_cap, D)) * ktil_scale).astype(np.float32)
    Q = wl.randn_bf16((B, H_q, D), seed + 1, "cuda")
    k_tot = n_init + n_local + k
    idx = torch.full((B, H_kv, k_tot), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H_kv), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq = torch.tensor(lens_b, dtype=torch.int32, device="cuda")
    binding.sparse_select_topk_heads(Q, torch.from_numpy(ktil_np).cuda().view(B, H_kv, N_cap, D), seq, n_init,
                                     n_local, k, idx, cnt, scale=scale, status=status)
    torch.cuda.synchronize()
    lens_p = np.repeat(np.asarray(lens_b, dtype=np.int64), H_kv)
    ref = oracle.select_heads(bits(Q).reshape(P, G, D), ktil_np.astype(np.float64), lens_p, n_init, n_local, k,
                              k_tot, scale=scale)
    return idx, cnt, ref, lens_p, status.item()


@pytest.mark.parametrize("H_q,H_kv", [(8, 8), (16, 4), (64, 8), (32, 2)])
@pytest.mark.parametrize("N_cap,lens_b,k", [(64, [4096, 3001, 65], 8), (513, [32769, 30000], 32),
                                            (2048, [131072, 100000], 64)])
def test_select_heads_matches_oracle(H_q, H_kv, N_cap, lens_b, k):
    idx, cnt, (ridx, rcnt, rs), lens_p, st = _run(lens_b, H_q, H_kv, N_cap, 1, 2, k, seed=N_cap + H_q)
    assert st == 0
    assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, 1, 2, k)


@pytest.mark.parametrize("N_cap", [2723, 2724, 3500])
def test_select_heads_register_and_radix_topk_boundary(N_cap):
    """The block-wide top-k keeps up to 17 candidates a thread in registers (2720 with the
    group's 160 threads); 2721 and more take the radix threshold and the one-warp write.
    N_cap = 2723 sits on the boundary (2720 candidates), 2724 just past it."""
    lens_b = [N_cap * BLK, N_cap * BLK - 100]
    idx, cnt, (ridx, rcnt, rs), lens_p, st = _run(lens_b, 8, 2, N_cap, 1, 2, 64, seed=N_cap)
    assert st == 0
    assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, 1, 2, 64)


def test_select_heads_scale_argument_and_sharp_softmax():
    # a large scale makes each head's softmax nearly one-hot: the sum then counts heads
    idx, cnt, (ridx, rcnt, rs), lens_p, st = _run([64 * 300, 64 * 250 + 7], 32, 4, 300, 1, 2, 12, seed=5,
                                                  scale=0.5, ktil_scale=0.2)
    assert st == 0
    assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, 1, 2, 12)


@pytest.mark.parametrize("k", [0, 1])
def test_select_heads_tiny_k_and_few_blocks(k):
    idx, cnt, (ridx, rcnt, rs), lens_p, st = _run([40 * BLK, 3 * BLK + 1, 65, 1, 0], 16, 2, 40, 1, 2, k, seed=9)
    assert st == 0
    if k == 0:
        assert np.array_equal(idx.cpu().numpy().reshape(ridx.shape), ridx)
        assert np.array_equal(cnt.cpu().numpy().reshape(rcnt.shape), rcnt)
    else:
        assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, 1, 2, k)


def test_select_heads_128k_layer_full_size():
    """The 128K decode layer's shape (B=8, H_q=64, H_kv=8, 2048 blocks, k=64) at full
    size, every pair checked against the oracle."""
    sh = wl.DECODE_128K
    idx, cnt, (ridx, rcnt, rs), lens_p, st = _run([sh.T] * sh.B, sh.H_q, sh.H_kv, sh.N_b, sh.n_init, sh.n_local,
                                                  sh.k, seed=77, ktil_scale=0.15)
    assert st == 0
    exempt = assert_selection_matches(idx, cnt, ridx, rcnt, rs, lens_p, sh.n_init, sh.n_local, sh.k)
    assert exempt <= 2
