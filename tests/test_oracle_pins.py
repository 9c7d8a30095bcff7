"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU, no GPU).

Each pin checks the oracle against something other than itself: closed forms, a
brute-force enumeration, a textbook/library routine (numpy mean, torch fp64 SDPA,
logsumexp), the SSV page's worked example, or the SSV saving formula on inputs
whose overlap is exact.  The mutation test at the end plants plausible mistakes in
a copy of the oracle's C source and checks that the pins catch every one.
"""
import itertools
import json
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_pool_gb300 import workloads as wl

D, BLK = 128, 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x) -> np.ndarray:
    """Float values that bf16 represents exactly -> uint16 bf16 bit patterns."""
    f = torch.as_tensor(np.asarray(x, dtype=np.float32))
    t = f.to(torch.bfloat16)
    assert torch.equal(t.float(), f), "test value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bits(shape, seed) -> np.ndarray:
    return wl.bf16_bits(wl.randn_bf16(shape, seed))


def values(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def unit_forecast(P, dims_weights):
    F = np.zeros((P, D), dtype=np.float32)
    for d, w in dims_weights:
        F[:, d] = w
    return bits(F)


# ----------------------------------------------------------------------------- pooling


def test_pool_single_token_is_the_bf16_value():
    K = rand_bits((3, 64, D), 1)
    out = oracle.pool(K, [1, 1, 1], 1)
    assert np.array_equal(out[:, 0], values(K)[:, 0])


def test_pool_constant_keys():
    K = bits(np.full((2, 256, D), 0.375))
    out = oracle.pool(K, [200, 130], 4)
    assert np.all(out[0] == 0.375)
    assert np.all(out[1, :3] == 0.375) and np.all(out[1, 3] == 0.0)


def test_pool_ramp_full_and_partial_blocks():
    # K[t][d] = ((t mod 64) + 64 (d mod 2)) / 128: a full block averages to
    # (31.5 + 64 (d mod 2)) / 128; a block holding r tokens to ((r-1)/2 + 64 (d mod 2)) / 128.
    T = 5 * BLK
    t = np.arange(T)[:, None]
    d = np.arange(D)[None, :]
    K = bits(((t % 64) + 64 * (d % 2)) / 128.0)[None]
    for r in (1, 17, 63, 64):
        length = 4 * BLK + r
        out = oracle.pool(K, [length], 5)[0]
        full = (31.5 + 64 * (np.arange(D) % 2)) / 128.0
        part = ((r - 1) / 2.0 + 64 * (np.arange(D) % 2)) / 128.0
        assert np.array_equal(out[:4], np.broadcast_to(full, (4, D)))
        assert np.allclose(out[4], part, rtol=0, atol=1e-15)


def test_pool_matches_numpy_block_means_ragged():
    K = rand_bits((3, 7 * BLK, D), 2)
    lens = [7 * BLK, 3 * BLK + 5, 1]
    out = oracle.pool(K, lens, 7)
    Kv = values(K)
    for p, n in enumerate(lens):
        for j in range(7):
            rows = Kv[p, j * BLK: min((j + 1) * BLK, n)]
            ref = rows.mean(axis=0) if len(rows) else np.zeros(D)
            assert np.allclose(out[p, j], ref, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- scores


def test_scores_unit_vector_reads_one_dimension():
    ktil = np.random.default_rng(3).standard_normal((2, 20, D))
    _, _, s = oracle.select(unit_forecast(2, [(5, 1.0)]), ktil, [20 * BLK] * 2, 1, 2, 4)
    assert np.array_equal(s, ktil[:, :, 5])


def test_scores_two_term_combination():
    ktil = np.random.default_rng(4).standard_normal((2, 9, D))
    _, _, s = oracle.select(unit_forecast(2, [(3, 2.0), (100, -0.5)]), ktil, [9 * BLK] * 2, 1, 2, 2)
    assert np.array_equal(s, 2.0 * ktil[:, :, 3] + (-0.5) * ktil[:, :, 100])


def test_scores_match_matrix_product():
    rng = np.random.default_rng(5)
    F = rand_bits((3, D), 5)
    ktil = rng.standard_normal((3, 33, D))
    _, _, s = oracle.select(F, ktil, [33 * BLK] * 3, 1, 2, 8)
    ref = np.einsum("pd,pjd->pj", values(F), ktil)
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- top-k


def _brute_topk(s, cands, k):
    """Best k-subset by exact total score; among equal totals the lexicographically
    smallest ascending tuple (equivalently: ties go to the lower block index)."""
    if len(cands) <= k:
        return tuple(sorted(cands))
    best = None
    for sub in itertools.combinations(sorted(cands), k):
        tot = sum(s[j] for j in sub)
        if best is None or tot > best[0] or (tot == best[0] and sub < best[1]):
            best = (tot, sub)
    return best[1]


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_brute_force_with_ties(seed):
    rng = np.random.default_rng(100 + seed)
    N, n_init, n_local, k = 13, 1, 2, 4
    ktil = np.zeros((1, N, D))
    ktil[0, :, 0] = rng.integers(-3, 4, size=N)      # small integers: many exact ties
    idx, count, s = oracle.select(unit_forecast(1, [(0, 1.0)]), ktil, [N * BLK], n_init, n_local, k)
    forced = set(range(n_init)) | set(range(N - n_local, N))
    cands = [j for j in range(N) if j not in forced]
    expect = sorted(forced | set(_brute_topk(s[0], cands, k)))
    assert count[0] == n_init + n_local + k
    assert list(idx[0, :count[0]]) == expect


def test_topk_all_equal_scores_take_lowest_indices():
    N = 40
    idx, count, _ = oracle.select(unit_forecast(1, [(7, 1.0)]), np.zeros((1, N, D)), [N * BLK], 1, 2, 5)
    assert list(idx[0, :count[0]]) == [0, 1, 2, 3, 4, 5, 38, 39]


def test_topk_excludes_init_and_local_blocks():
    N, k = 30, 6
    ktil = np.zeros((1, N, D))
    ktil[0, :, 0] = np.arange(N) * 0.25
    ktil[0, 0, 0] = 1e6          # init block scores highest ...
    ktil[0, N - 1, 0] = 1e6      # ... and so do the local blocks,
    ktil[0, N - 2, 0] = 1e6      # yet they must not take top-k slots
    idx, count, _ = oracle.select(unit_forecast(1, [(0, 1.0)]), ktil, [N * BLK], 1, 2, k)
    assert count[0] == 1 + 2 + k
    assert list(idx[0, :count[0]]) == [0] + list(range(N - 2 - k, N - 2)) + [N - 2, N - 1]


def test_local_blocks_follow_the_partial_last_block():
    # len = 10 blocks + 1 token: N_b = 11, local = blocks 9 and 10.
    N = 11
    ktil = np.zeros((1, 12, D))
    ktil[0, :N, 0] = -np.arange(N)   # candidate 1 scores best
    idx, count, _ = oracle.select(unit_forecast(1, [(0, 1.0)]), ktil, [10 * BLK + 1], 1, 2, 1)
    assert list(idx[0, :count[0]]) == [0, 1, 9, 10]


@pytest.mark.parametrize("N,expect", [(7, list(range(7))), (2, [0, 1]), (1, [0])])
def test_select_takes_every_block_when_few(N, expect):
    ktil = np.random.default_rng(6).standard_normal((1, 8, D))
    idx, count, _ = oracle.select(rand_bits((1, D), 6), ktil, [N * BLK], 1, 2, 8)
    assert list(idx[0, :count[0]]) == expect
    assert np.all(idx[0, count[0]:] == -1)


def test_select_empty_sequence():
    idx, count, _ = oracle.select(rand_bits((1, D), 7), np.zeros((1, 4, D)), [0], 1, 2, 3)
    assert count[0] == 0 and np.all(idx == -1)


def test_select_invariants_on_single_layer_workload():
    sh = wl.SINGLE_4K
    inp = wl.single_layer(sh)
    K = wl.bf16_bits(inp["K"]).reshape(sh.pairs, sh.T_cap, D)
    ktil = oracle.pool(K, [sh.T] * sh.pairs, sh.N_b)
    F = wl.bf16_bits(inp["F"]).reshape(sh.pairs, D)
    idx, count, _ = oracle.select(F, ktil, [sh.T] * sh.pairs, sh.n_init, sh.n_local, sh.k)
    for p in range(sh.pairs):
        sel = list(idx[p, :count[p]])
        assert count[p] == sh.k_tot == 11
        assert sel == sorted(set(sel))
        assert {0, sh.N_b - 2, sh.N_b - 1} <= set(sel)
        # sanity of the generator, not a pin: most planted blocks are the ones found
        assert len(set(inp["planted"][p].tolist()) & set(sel)) >= sh.n_planted - 2


# ----------------------------------------------------------------------------- attention


def _sdpa(Qv, Kv, Vv, token_mask, scale=None):
    """torch fp64 scaled_dot_product_attention; Qv [G][D], Kv/Vv [T][D], mask [T]."""
    q = torch.from_numpy(Qv)[None, :, None, :]                 # [1][G][1][D]
    k = torch.from_numpy(Kv)[None, None].expand(1, Qv.shape[0], -1, -1)
    v = torch.from_numpy(Vv)[None, None].expand(1, Qv.shape[0], -1, -1)
    m = torch.from_numpy(token_mask)[None, None, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    return o[0, :, 0].numpy()


def _lse(Qv, Kv, token_mask, scale):
    a = torch.from_numpy(Qv @ Kv[token_mask].T * scale)
    return torch.logsumexp(a, dim=-1).numpy()


def test_attn_all_blocks_equals_dense_sdpa():
    P, G, T = 3, 4, 5 * BLK + 17
    Q, K, V = rand_bits((P, G, D), 10), rand_bits((P, T, D), 11), rand_bits((P, T, D), 12)
    lens = [T, T - 40, 3 * BLK]
    nb = (T + BLK - 1) // BLK
    blocks = np.tile(np.arange(nb, dtype=np.int32), (P, 1))
    O, lse = oracle.attn(Q, K, V, blocks, [nb] * P, lens)
    for p in range(P):
        mask = np.arange(T) < lens[p]
        ref = _sdpa(values(Q[p]), values(K[p]), values(V[p]), mask)
        assert np.allclose(O[p], ref, rtol=1e-11, atol=1e-12)
        assert np.allclose(lse[p], _lse(values(Q[p]), values(K[p]), mask, 1 / math.sqrt(D)),
                           rtol=1e-12, atol=1e-12)


def test_attn_block_subset_equals_masked_sdpa_and_ignores_order_and_repeats():
    P, G, T = 2, 8, 9 * BLK
    Q, K, V = rand_bits((P, G, D), 13), rand_bits((P, T, D), 14), rand_bits((P, T, D), 15)
    blocks = np.array([[7, 2, 5, 2, -1], [8, 0, 3, 3, 6]], dtype=np.int32)
    O, _ = oracle.attn(Q, K, V, blocks, [5, 5], [T, T - 30])
    for p, n in enumerate([T, T - 30]):
        chosen = {j for j in blocks[p] if j >= 0}
        mask = np.array([(t // BLK) in chosen and t < n for t in range(T)])
        assert np.allclose(O[p], _sdpa(values(Q[p]), values(K[p]), values(V[p]), mask),
                           rtol=1e-11, atol=1e-12)


def test_attn_scale_argument_is_applied():
    Q, K, V = rand_bits((1, 2, D), 16), rand_bits((1, BLK, D), 17), rand_bits((1, BLK, D), 18)
    O, _ = oracle.attn(Q, K, V, np.zeros((1, 1), np.int32), [1], [BLK], scale=0.3)
    ref = _sdpa(values(Q[0]), values(K[0]), values(V[0]), np.ones(BLK, bool), scale=0.3)
    assert np.allclose(O[0], ref, rtol=1e-11, atol=1e-12)


def test_attn_equal_keys_give_mean_of_values():
    T = 4 * BLK
    K = np.repeat(rand_bits((1, 1, D), 19), T, axis=1)
    Q, V = rand_bits((1, 3, D), 20), rand_bits((1, T, D), 21)
    blocks = np.array([[1, 3]], dtype=np.int32)
    O, _ = oracle.attn(Q, K, V, blocks, [2], [T - 10])
    rows = [t for t in range(T) if t // BLK in (1, 3) and t < T - 10]
    assert np.allclose(O[0], np.broadcast_to(values(V[0, rows]).mean(axis=0), (3, D)),
                       rtol=1e-12, atol=1e-13)


def test_attn_constant_values_and_single_token():
    T = 2 * BLK
    Q, K = rand_bits((1, 4, D), 22), rand_bits((1, T, D), 23)
    V = bits(np.full((1, T, D), -1.25))
    O, _ = oracle.attn(Q, K, V, np.array([[0, 1]], np.int32), [2], [T])
    assert np.allclose(O, -1.25, rtol=0, atol=1e-14)
    V = rand_bits((1, T, D), 24)
    O, lse = oracle.attn(Q, K, V, np.array([[0, 1]], np.int32), [2], [1])
    assert np.array_equal(O[0], np.broadcast_to(values(V[0, 0]), (4, D)))
    assert np.allclose(lse[0], values(Q[0]) @ values(K[0, 0]) / math.sqrt(D), rtol=1e-13)


def test_attn_empty_set_gives_zero_and_minus_inf():
    Q, K, V = rand_bits((1, 2, D), 25), rand_bits((1, BLK, D), 26), rand_bits((1, BLK, D), 27)
    O, lse = oracle.attn(Q, K, V, np.full((1, 3), -1, np.int32), [0], [BLK])
    assert np.all(O == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------- verification


def test_verify_worked_example_of_the_ssv_page():
    ex = json.load(open(os.path.join(GOLDEN, "ssv_worked_example.json")))
    sets = ex["queries"]
    loads = {}
    for s in sets:
        for j in s:
            loads[j] = loads.get(j, 0) + 1
    for j, n in ex["printed_load_counts"].items():
        assert loads[int(j)] == n
    T = 24 * BLK
    Q, K, V = rand_bits((1, 4, 1, D), 30), rand_bits((1, 1, T, D), 31), rand_bits((1, 1, T, D), 32)
    I = np.array(sets, dtype=np.int32)[None, None]
    O, union, per_query = oracle.verify(Q, K, V, I, C=4, window_blocks=0, lens=[T])
    assert union == len(ex["derived"]["merged_union"]) == 10
    assert per_query == ex["derived"]["ungrouped_loads"] == 16


@pytest.mark.parametrize("gamma,n_sel,window", [(0.75, 16, 0), (0.75, 16, 512), (0.5, 8, 0),
                                                (0.875, 16, 0)])
def test_verify_saving_formula_on_core_private_overlap(gamma, n_sel, window):
    # SSV notes, grouping saving: merged / ungrouped = (1 + (C-1)(1-gamma)) / C.
    sh = wl.VerifyShape("t", B=2, H_q=4, H_kv=2, T=64 * BLK, N_q=8, n_sel=n_sel, gamma=gamma,
                        window_tokens=window, C=4)
    T = sh.T
    I = wl.verify_sets(sh).numpy()
    Q = rand_bits((sh.B, sh.N_q, sh.H_q, D), 33)
    K = rand_bits((sh.B, sh.H_kv, T, D), 34)
    _, union, per_query = oracle.verify(Q, K, K, I, sh.C, sh.window_blocks, [T] * sh.B)
    groups = sh.B * sh.H_kv * (sh.N_q // sh.C)
    w = sh.window_blocks
    assert union == groups * (n_sel * (1 + (sh.C - 1) * (1 - gamma)) + w)
    assert per_query == groups * sh.C * (n_sel + w)
    if w == 0:
        assert union / per_query == pytest.approx((1 + (sh.C - 1) * (1 - gamma)) / sh.C, abs=1e-15)
    if (gamma, n_sel, window) == (0.75, 16, 512):
        assert union / per_query == 36 / 96


def test_verify_equals_masked_sdpa_per_query():
    B, N_q, H_q, H_kv, T, C, wb = 1, 4, 4, 2, 12 * BLK, 2, 2
    G = H_q // H_kv
    Q, K, V = rand_bits((B, N_q, H_q, D), 35), rand_bits((B, H_kv, T, D), 36), rand_bits((B, H_kv, T, D), 37)
    I = np.array([[[[1, 4], [1, 5], [2, 4], [0, 9]], [[3, 6], [3, 7], [0, 6], [5, 8]]]], np.int32)
    O, union, per_query = oracle.verify(Q, K, V, I, C, wb, [T - 20])
    n = T - 20
    for g in range(H_kv):
        for q in range(N_q):
            chosen = set(I[0, g, q].tolist()) | {10, 11}
            mask = np.array([(t // BLK) in chosen and t < n for t in range(T)])
            ref = _sdpa(values(Q[0, q, g * G:(g + 1) * G]), values(K[0, g]), values(V[0, g]), mask)
            assert np.allclose(O[0, q, g * G:(g + 1) * G], ref, rtol=1e-11, atol=1e-12)
    assert per_query == 2 * 4 * 4


def test_verify_shared_layout_attends_over_the_first_query_set():
    # SSV notes, mode B: every query of a group uses its first query's layout
    B, N_q, H_q, H_kv, T, C, wb = 1, 4, 4, 2, 12 * BLK, 2, 2
    G = H_q // H_kv
    Q, K, V = rand_bits((B, N_q, H_q, D), 38), rand_bits((B, H_kv, T, D), 39), rand_bits((B, H_kv, T, D), 41)
    I = np.array([[[[1, 4], [1, 5], [2, 4], [0, 9]], [[3, 6], [3, 7], [0, 6], [5, 8]]]], np.int32)
    n = T - 20
    O, union, per_query = oracle.verify(Q, K, V, I, C, wb, [n], shared=True)
    for g in range(H_kv):
        for q in range(N_q):
            rep = (q // C) * C
            chosen = set(I[0, g, rep].tolist()) | {10, 11}
            mask = np.array([(t // BLK) in chosen and t < n for t in range(T)])
            ref = _sdpa(values(Q[0, q, g * G:(g + 1) * G]), values(K[0, g]), values(V[0, g]), mask)
            assert np.allclose(O[0, q, g * G:(g + 1) * G], ref, rtol=1e-11, atol=1e-12)
    # every group loads one layout: 2 selected + 2 window blocks
    assert union == H_kv * (N_q // C) * 4
    assert per_query == 2 * 4 * 4


def test_verify_shared_layout_with_singleton_groups_is_mode_a():
    sh = wl.VerifyShape("t", B=1, H_q=4, H_kv=2, T=64 * BLK, N_q=8, n_sel=8, gamma=0.5, window_tokens=128, C=4)
    I = wl.verify_sets(sh).numpy()
    Q = rand_bits((sh.B, sh.N_q, sh.H_q, D), 42)
    K, V = rand_bits((sh.B, sh.H_kv, sh.T, D), 43), rand_bits((sh.B, sh.H_kv, sh.T, D), 44)
    Oa, ua, pa = oracle.verify(Q, K, V, I, 1, sh.window_blocks, [sh.T])
    Ob, ub, pb = oracle.verify(Q, K, V, I, 1, sh.window_blocks, [sh.T], shared=True)
    assert np.array_equal(Oa, Ob) and (ua, pa) == (ub, pb)
    # and with C = 4 the shared layout loads n_sel + window per group
    _, u4, _ = oracle.verify(Q, K, V, I, 4, sh.window_blocks, [sh.T], shared=True)
    assert u4 == sh.H_kv * 2 * (sh.n_sel + sh.window_blocks)


def test_verify_shared_layout_on_the_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "ssv_worked_example.json")))
    T = 24 * BLK
    Q, K, V = rand_bits((1, 4, 1, D), 45), rand_bits((1, 1, T, D), 46), rand_bits((1, 1, T, D), 47)
    I = np.array(ex["queries"], dtype=np.int32)[None, None]
    _, union, per_query = oracle.verify(Q, K, V, I, C=4, window_blocks=0, lens=[T], shared=True)
    assert union == len(ex["queries"][0])          # the first query's blocks only
    assert per_query == ex["derived"]["ungrouped_loads"]


# ----------------------------------------------------------------------------- gather


def test_gather_is_a_plain_copy():
    P, T_host = 2, 5 * BLK + 9
    src = rand_bits((P, T_host, D), 40)
    idx = np.array([[4, 0, 5, -1], [2, 5, 1, 3]], dtype=np.int32)
    count = np.array([3, 4], np.int32)
    ring = oracle.gather(src, idx, count)
    for p in range(P):
        for i in range(count[p]):
            j = idx[p, i]
            rows = src[p, j * BLK: min((j + 1) * BLK, T_host)]
            assert np.array_equal(ring[p, i, :len(rows)], rows)
            assert np.all(ring[p, i, len(rows):] == 0)
    assert np.all(ring[0, 3] == 0)


# ----------------------------------------------------------------------------- multi-head selection


def _heads_case(seed, P=3, G=4, N=40, lens=(40 * 64, 23 * 64 + 5, 3 * 64)):
    rng = np.random.default_rng(seed)
    Q = rand_bits((P, G, D), seed + 100)
    ktil = rng.standard_normal((P, N, D)) * 0.3
    return Q, ktil, np.asarray(lens, dtype=np.int64)


def test_select_heads_with_one_head_is_the_forecast_selection():
    # softmax is monotone, so one head selects exactly what its raw scores select
    Q, ktil, lens = _heads_case(1, G=1)
    idx_h, cnt_h, _ = oracle.select_heads(Q, ktil, lens, 1, 2, 6)
    idx_f, cnt_f, _ = oracle.select(Q[:, 0], ktil, lens, 1, 2, 6)
    assert np.array_equal(idx_h, idx_f) and np.array_equal(cnt_h, cnt_f)


def test_select_heads_scores_are_a_sum_of_head_distributions():
    # each head contributes a distribution over the pair's blocks: the sum is G
    Q, ktil, lens = _heads_case(2, G=4)
    _, _, s = oracle.select_heads(Q, ktil, lens, 1, 2, 6)
    for p, n in enumerate(lens):
        nb = (int(n) + 63) // 64
        assert abs(s[p, :nb].sum() - 4.0) < 1e-12
        assert not s[p, nb:].any()


def test_select_heads_match_scipy_softmax_and_brute_force_topk():
    from scipy.special import softmax
    Q, ktil, lens = _heads_case(3, G=4)
    scale = 0.37
    idx, cnt, s = oracle.select_heads(Q, ktil, lens, 1, 2, 6, scale=scale)
    for p, n in enumerate(lens):
        nb = (int(n) + 63) // 64
        q = values(Q[p])                                           # [G][D]
        a = scale * q @ ktil[p, :nb].T                             # [G][nb]
        ref = softmax(a, axis=1).sum(axis=0)
        assert np.allclose(s[p, :nb], ref, rtol=1e-12, atol=1e-15)
        cand = [j for j in range(nb) if 1 <= j < nb - 2]
        top = sorted(cand, key=lambda j: (-ref[j], j))[:6]
        want = sorted(set(range(min(1, nb))) | set(range(max(nb - 2, 0), nb)) | set(top))
        assert list(idx[p, :cnt[p]]) == want


# ----------------------------------------------------------------------------- NSA three-branch output


def _nsa_case(seed):
    P, G, T, w = 2, 3, 10 * BLK + 21, 100
    lens = np.array([T, 6 * BLK + 3], np.int64)
    Q, K, V = rand_bits((P, G, D), seed), rand_bits((P, T, D), seed + 1), rand_bits((P, T, D), seed + 2)
    N = 11
    khat = oracle.pool(K, lens, N)
    vhat = oracle.pool(V, lens, N)
    blocks = np.array([[1, 4, 9, -1], [0, 2, -1, -1]], np.int32)
    count = np.array([3, 2], np.int32)
    return Q, K, V, khat, vhat, blocks, count, lens, w, G, N


def _nsa_with(gate, seed=50):
    Q, K, V, khat, vhat, blocks, count, lens, w, G, N = _nsa_case(seed)
    gates = np.broadcast_to(np.asarray(gate, np.float64), (2, G, 3)).copy()
    return oracle.nsa(Q, K, V, khat, vhat, blocks, count, lens, w, gates), (Q, K, V, khat, vhat, blocks, count,
                                                                            lens, w, G, N)


def test_nsa_selected_branch_is_sdpa_over_the_selected_tokens():
    O, (Q, K, V, _, _, blocks, count, lens, _, _, _) = _nsa_with((0.0, 1.0, 0.0))
    for p in range(2):
        chosen = set(blocks[p, :count[p]].tolist())
        mask = np.array([(t // BLK) in chosen and t < lens[p] for t in range(K.shape[1])])
        assert np.allclose(O[p], _sdpa(values(Q[p]), values(K[p]), values(V[p]), mask), rtol=1e-11, atol=1e-12)


def test_nsa_window_branch_is_sdpa_over_the_last_w_tokens():
    O, (Q, K, V, _, _, _, _, lens, w, _, _) = _nsa_with((0.0, 0.0, 1.0))
    for p in range(2):
        mask = np.array([lens[p] - w <= t < lens[p] for t in range(K.shape[1])])
        assert np.allclose(O[p], _sdpa(values(Q[p]), values(K[p]), values(V[p]), mask), rtol=1e-11, atol=1e-12)


def test_nsa_compressed_branch_is_sdpa_over_the_compressed_rows():
    O, (Q, _, _, khat, vhat, _, _, lens, _, _, _) = _nsa_with((1.0, 0.0, 0.0))
    for p in range(2):
        nb = (int(lens[p]) + BLK - 1) // BLK
        mask = np.arange(khat.shape[1]) < nb
        assert np.allclose(O[p], _sdpa(values(Q[p]), khat[p], vhat[p], mask), rtol=1e-11, atol=1e-12)


def test_nsa_output_is_linear_in_the_gates():
    Oc, _ = _nsa_with((1.0, 0.0, 0.0))
    Os, _ = _nsa_with((0.0, 1.0, 0.0))
    Ow, _ = _nsa_with((0.0, 0.0, 1.0))
    O, _ = _nsa_with((0.25, -0.5, 1.5))
    assert np.allclose(O, 0.25 * Oc - 0.5 * Os + 1.5 * Ow, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- overlapping compression (NSA)


def test_pool_windows_ramp_closed_form():
    """X[t] = t (exact in bf16 up to 256): window j of kernel 32, stride 16 has mean
    16 j + 15.5; rows past the complete windows are zero."""
    T = 200
    X = bits(np.repeat(np.arange(T, dtype=np.float32)[:, None], D, axis=1)[None])
    out = oracle.pool_windows(X, [T], 32, 16, 14)
    W = (T - 32) // 16 + 1
    for j in range(14):
        want = 16 * j + 15.5 if j < W else 0.0
        assert np.all(out[0, j] == want), j


def test_pool_windows_match_numpy_slices():
    P, T = 3, 300
    X = rand_bits((P, T, D), 71)
    lens = np.array([300, 47, 31], np.int64)
    for l, s in ((32, 16), (16, 8), (64, 32)):
        out = oracle.pool_windows(X, lens, l, s, 40)
        v = values(X)
        for p in range(P):
            W = 0 if lens[p] < l else (lens[p] - l) // s + 1
            for j in range(40):
                want = v[p, s * j:s * j + l].mean(axis=0) if j < W else np.zeros(D)
                assert np.allclose(out[p, j], want, rtol=1e-14, atol=1e-15), (l, s, p, j)


def test_pool_windows_with_the_block_kernel_are_the_complete_block_means():
    X = rand_bits((2, 320, D), 72)
    lens = np.array([320, 200], np.int64)
    win = oracle.pool_windows(X, lens, BLK, BLK, 5)
    blk = oracle.pool(X, lens, 5)
    for p in range(2):
        full = int(lens[p]) // BLK
        assert np.allclose(win[p, :full], blk[p, :full], rtol=1e-14, atol=1e-15)
        assert np.all(win[p, full:] == 0)


def _windows_case(seed, P=3, G=4, T=1000):
    X = rand_bits((P, T, D), seed)
    lens = np.array([T, 777, 300][:P], np.int64)
    kc = oracle.pool_windows(X, lens, 32, 16, (T - 32) // 16 + 1)
    Q = rand_bits((P, G, D), seed + 1)
    return Q, kc, lens


def test_select_windows_match_brute_force_softmax_and_max_pooling():
    from scipy.special import softmax
    Q, kc, lens = _windows_case(81)
    n_init, n_local, k = 1, 2, 4
    idx, cnt, sc = oracle.select_windows(Q, kc, lens, 32, 16, n_init, n_local, k, scale=0.1)
    qv = values(Q)
    for p in range(len(lens)):
        W = (int(lens[p]) - 32) // 16 + 1
        nb = (int(lens[p]) + BLK - 1) // BLK
        pj = sum(softmax(0.1 * (kc[p, :W] @ qv[p, h]), axis=0) for h in range(Q.shape[1]))
        sb = np.zeros(nb)
        for b in range(nb):
            over = [pj[j] for j in range(W) if 16 * j < 64 * b + 64 and 64 * b < 16 * j + 32]
            sb[b] = max(over) if over else 0.0
        assert np.allclose(sc[p, :nb], sb, rtol=1e-12, atol=1e-15)
        cand = [b for b in range(nb) if n_init <= b < nb - n_local]
        top = sorted(cand, key=lambda b: (-sb[b], b))[:k]
        want = sorted(set(range(min(n_init, nb))) | set(range(max(nb - n_local, 0), nb)) | set(top))
        assert list(idx[p, :cnt[p]]) == want


def test_select_windows_with_block_windows_is_the_multi_head_selection():
    """Kernel = stride = 64 and whole blocks: each block is one window, max-pooling is
    the identity and the routing is oracle_select_heads."""
    P, G, T = 2, 3, 64 * 40
    X = rand_bits((P, T, D), 82)
    lens = np.array([T, 64 * 23], np.int64)
    kc = oracle.pool_windows(X, lens, BLK, BLK, 40)
    Q = rand_bits((P, G, D), 83)
    a = oracle.select_windows(Q, kc, lens, BLK, BLK, 1, 2, 6, scale=0.2, n_blocks_cap=40)
    b = oracle.select_heads(Q, kc, lens, 1, 2, 6, scale=0.2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.allclose(a[2], b[2], rtol=1e-13, atol=1e-16)


def _nsa_windows_with(gate, seed=90):
    P, G, T, w = 2, 3, 10 * BLK + 21, 100
    lens = np.array([T, 6 * BLK + 3], np.int64)
    Q, K, V = rand_bits((P, G, D), seed), rand_bits((P, T, D), seed + 1), rand_bits((P, T, D), seed + 2)
    R = (T - 32) // 16 + 1
    kc, vc = oracle.pool_windows(K, lens, 32, 16, R), oracle.pool_windows(V, lens, 32, 16, R)
    blocks = np.array([[1, 4, 9, -1], [0, 2, -1, -1]], np.int32)
    count = np.array([3, 2], np.int32)
    gates = np.broadcast_to(np.asarray(gate, np.float64), (P, G, 3)).copy()
    O = oracle.nsa(Q, K, V, kc, vc, blocks, count, lens, w, gates, cmp=(32, 16))
    return O, (Q, K, V, kc, vc, blocks, count, lens, w, gates)


def test_nsa_windows_compressed_branch_is_sdpa_over_the_complete_windows():
    O, (Q, _, _, kc, vc, _, _, lens, _, _) = _nsa_windows_with((1.0, 0.0, 0.0))
    for p in range(2):
        W = (int(lens[p]) - 32) // 16 + 1
        mask = np.arange(kc.shape[1]) < W
        assert np.allclose(O[p], _sdpa(values(Q[p]), kc[p], vc[p], mask), rtol=1e-11, atol=1e-12)


def test_nsa_windows_leave_the_selected_and_window_branches_alone():
    O, (Q, K, V, kc, vc, blocks, count, lens, w, gates) = _nsa_windows_with((0.0, 0.7, 0.3))
    ref = oracle.nsa(Q, K, V, np.zeros((2, 11, D)), np.zeros((2, 11, D)), blocks, count, lens, w, gates)
    assert np.allclose(O, ref, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------- prefill selection


def _prefill_brute(Fv, kt, lens, n_init, n_local, k, k_tot):
    P, T, _ = Fv.shape
    idx = np.full((P, T, k_tot), -1, np.int32)
    cnt = np.full((P, T), -1, np.int32)
    for p in range(P):
        for t in range(int(lens[p])):
            nb = t // BLK + 1
            sc = kt[p, :nb] @ Fv[p, t]
            chosen = set(range(min(n_init, nb))) | set(range(max(nb - n_local, 0), nb))
            cand = [j for j in range(nb) if j not in chosen]
            chosen |= set(sorted(cand, key=lambda j: (-sc[j], j))[:k])
            sel = sorted(chosen)
            cnt[p, t] = len(sel)
            idx[p, t, :len(sel)] = sel
    return idx, cnt


def test_prefill_select_matches_brute_force_per_position():
    P, T, N = 2, 64 * 9 + 17, 10
    F = rand_bits((P, T, D), 91)
    kt = np.random.default_rng(92).standard_normal((P, N, D))
    lens = np.array([T, 64 * 5 + 3], np.int64)
    for n_init, n_local, k in ((1, 2, 3), (0, 1, 1), (2, 1, 5)):
        idx, cnt = oracle.prefill_select(F, kt, lens, n_init, n_local, k)
        bi, bc = _prefill_brute(values(F), kt, lens, n_init, n_local, k, n_init + n_local + k)
        assert np.array_equal(cnt, bc) and np.array_equal(idx, bi), (n_init, n_local, k)


def test_prefill_select_is_causal_and_matches_a_decode_of_the_prefix():
    """Row t depends only on the keys of blocks <= t // 64; with unit Forecast vectors
    the ranking is the closed-form order of one key dimension."""
    P, T, N = 1, 64 * 6, 6
    Fz = np.zeros((P, T, D), np.float32)
    Fz[:, :, 5] = 1.0
    F = bits(Fz)
    kt = np.zeros((P, N, D))
    kt[0, :, 5] = [0.5, 3.0, -1.0, 3.0, 2.0, 9.0]   # ties between blocks 1 and 3
    idx, cnt = oracle.prefill_select(F, kt, [T], 0, 1, 2)
    assert list(idx[0, 64 * 4 + 7, :cnt[0, 64 * 4 + 7]]) == [1, 3, 4]     # blocks 0..3 candidates, 4 local
    assert list(idx[0, 64 * 5 + 1, :cnt[0, 64 * 5 + 1]]) == [1, 3, 5]     # block 4 (2.0) below the tie pair
    kt2 = kt.copy()
    kt2[0, 5, 5] = -50.0   # a later block changes nothing for earlier rows
    idx2, _ = oracle.prefill_select(F, kt2, [T], 0, 1, 2)
    assert np.array_equal(idx[0, :320], idx2[0, :320])


def test_prefill_select_sampled_rows_equal_the_full_rows():
    P, T, N = 2, 500, 8
    F = rand_bits((P, T, D), 93)
    kt = np.random.default_rng(94).standard_normal((P, N, D))
    full_i, full_c = oracle.prefill_select(F, kt, [T, 333], 1, 2, 2)
    rows = [0, 64, 65, 200, 332, 499]
    si, sc = oracle.prefill_select(F, kt, [T, 333], 1, 2, 2, rows=rows)
    for r, t in enumerate(rows):
        assert np.array_equal(si[0, r], full_i[0, t]) and sc[0, r] == full_c[0, t]
    assert sc[1, rows.index(499)] == -1   # past the second pair's length


# ----------------------------------------------------------------------------- mutants

MUTANTS = [
    # pooling divides by the full block size instead of the tokens present
    ("sum[d] / (double)n", "sum[d] / (double)BLK"),
    # score reads the wrong operand dimension
    ("acc += Fp[d] * kj[d];", "acc += Fp[d] * kj[(d + 1) % D];"),
    # ties go to the higher block index
    ("return (x->j > y->j) - (x->j < y->j);", "return (x->j < y->j) - (x->j > y->j);"),
    # the local window is one block short
    ("for (int j = nb - n_local; j < nb; ++j)\n        if (j >= 0)\n            chosen[j] = 1;",
     "for (int j = nb - n_local + 1; j < nb; ++j)\n        if (j >= 0)\n            chosen[j] = 1;"),
    # the softmax scale is dropped
    ("a[n] = scale * dot;", "a[n] = dot;"),
    # values read from the key cache
    ("o[d] += w * bf16_value(Vp[", "o[d] += w * bf16_value(Kp["),
    # the length mask is off by one
    ("t < (long long)(j + 1) * BLK && t < len;", "t < (long long)(j + 1) * BLK && t <= len;"),
    # the verification window forgets its first block
    ("for (int j = nb - window_blocks; j < nb; ++j)", "for (int j = nb - window_blocks + 1; j < nb; ++j)"),
    # the bf16 widening uses the wrong half
    ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    # multi-head selection sums raw scores instead of per-head distributions
    ("s[j] += exp(a[j] - m) / z;", "s[j] += a[j];"),
    # multi-head softmax normalised over the candidates only
    ("z += exp(a[j] - m);", "z += j >= n_init ? exp(a[j] - m) : 0.0;"),
    # multi-head scores without the scale
    ("a[j] = scale * acc;", "a[j] = acc;"),
    # the NSA window starts one token late
    ("long long w0 = len[p] - window_tokens;", "long long w0 = len[p] - window_tokens + 1;"),
    # the NSA gates are swapped between the compressed and the selected branch
    ("o[d] = g[0] * oc[d] + g[1] * os[d] + g[2] * ow[d];", "o[d] = g[1] * oc[d] + g[0] * os[d] + g[2] * ow[d];"),
    # the NSA compressed branch forgets the last compressed row
    ("attend_rows(qd, kr, vr, nrows, scale, oc);", "attend_rows(qd, kr, vr, nrows - 1, scale, oc);"),
    # the compression windows start one token late
    ("for (long long t = (long long)s * j; t < (long long)s * j + l; ++t)",
     "for (long long t = (long long)s * j + 1; t < (long long)s * j + l; ++t)"),
    # max-pooling takes only the windows that lie inside the block
    ("if (w0 < b1 && b0 < w1 && pj[j] > best)", "if (w0 >= b0 && w1 <= b1 && pj[j] > best)"),
    # the window routing sums raw scores instead of per-head distributions
    ("pj[j] += exp(a[j] - m) / z;", "pj[j] += a[j];"),
    # the NSA window form attends over one row per block instead of the windows
    ("int nrows = cmp_len > 0 ? windows_of(len[p], cmp_len, cmp_stride) : nb;",
     "int nrows = cmp_len > 0 ? (nb < windows_of(len[p], cmp_len, cmp_stride) ? nb : windows_of(len[p], cmp_len, cmp_stride) - 1) : nb;"),
    # a prefill position sees one block too many (the block after its own)
    ("const int nb = (int)(t / BLK) + 1;", "const int nb = (int)(t / BLK) + 1 + (t % BLK == BLK - 1);"),
    # a prefill position reads the previous position's Forecast vector
    ("Fp[d] = bf16_value(F[((size_t)p * T_cap + t) * D + d]);",
     "Fp[d] = bf16_value(F[((size_t)p * T_cap + (t > 0 ? t - 1 : 0)) * D + d]);"),
    # mode B takes the group's last query as its representative
    ("const int *Ia = shared ? I + (((size_t)b * H_kv + g) * N_q + q0) * n_sel : Iq;",
     "const int *Ia = shared ? I + (((size_t)b * H_kv + g) * N_q + (q0 + C - 1 < N_q ? q0 + C - 1 : N_q - 1)) * n_sel : Iq;"),
]

PIN_TESTS = [
    test_pool_single_token_is_the_bf16_value, test_pool_constant_keys, test_pool_ramp_full_and_partial_blocks,
    test_pool_matches_numpy_block_means_ragged, test_scores_unit_vector_reads_one_dimension,
    test_scores_two_term_combination, test_scores_match_matrix_product,
    test_topk_all_equal_scores_take_lowest_indices, test_topk_excludes_init_and_local_blocks,
    test_local_blocks_follow_the_partial_last_block, test_attn_all_blocks_equals_dense_sdpa,
    test_attn_block_subset_equals_masked_sdpa_and_ignores_order_and_repeats,
    test_attn_scale_argument_is_applied, test_attn_equal_keys_give_mean_of_values,
    test_attn_constant_values_and_single_token, test_verify_worked_example_of_the_ssv_page,
    test_verify_equals_masked_sdpa_per_query, test_select_heads_with_one_head_is_the_forecast_selection,
    test_select_heads_scores_are_a_sum_of_head_distributions, test_select_heads_match_scipy_softmax_and_brute_force_topk,
    test_verify_shared_layout_attends_over_the_first_query_set, test_verify_shared_layout_with_singleton_groups_is_mode_a,
    test_verify_shared_layout_on_the_worked_example, test_nsa_selected_branch_is_sdpa_over_the_selected_tokens,
    test_nsa_window_branch_is_sdpa_over_the_last_w_tokens, test_nsa_compressed_branch_is_sdpa_over_the_compressed_rows,
    test_nsa_output_is_linear_in_the_gates, test_pool_windows_ramp_closed_form, test_pool_windows_match_numpy_slices,
    test_pool_windows_with_the_block_kernel_are_the_complete_block_means,
    test_select_windows_match_brute_force_softmax_and_max_pooling,
    test_select_windows_with_block_windows_is_the_multi_head_selection,
    test_nsa_windows_compressed_branch_is_sdpa_over_the_complete_windows,
    test_nsa_windows_leave_the_selected_and_window_branches_alone,
    test_prefill_select_matches_brute_force_per_position, test_prefill_select_is_causal_and_matches_a_decode_of_the_prefix,
    test_prefill_select_sampled_rows_equal_the_full_rows,
]


@pytest.mark.parametrize("m", range(len(MUTANTS)))
def test_pins_catch_planted_oracle_mistakes(m, tmp_path, monkeypatch):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    before, after = MUTANTS[m]
    assert before in src, f"mutant {m}: pattern not found"
    c_path, so_path = tmp_path / "mutant.c", tmp_path / "mutant.so"
    c_path.write_text(src.replace(before, after))
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", str(c_path), "-o",
                    str(so_path), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so_path)))
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError):
            caught.append(t.__name__)
    try:
        test_verify_saving_formula_on_core_private_overlap(0.75, 16, 512)
    except AssertionError:
        caught.append("saving_formula")
    for seed in range(3):
        try:
            test_topk_equals_brute_force_with_ties(seed)
        except AssertionError:
            caught.append("brute_force")
    assert caught, f"mutant {m} ({after!r}) passed every pin"
