"""Seeded synthetic inputs for the five decode workloads.

This module only draws inputs: shapes, random bf16 tensors, planted high-affinity
blocks and per-query block sets.  It holds none of the method's arithmetic (no
pooling, scoring, top-k or attention), so the CUDA path and the CPU oracle can both
be fed from it without sharing any computation.

Recipe (every tensor is seeded; bf16 values are N(0, 1) draws rounded once):

* Decode layers (SparDA notes §4.2 Alg.1 inputs): Q [B][H_q][128], one Forecast
  vector F per (batch, KV head) [B][H_kv][128], K/V caches [B][H_kv][T_cap][128]
  holding T tokens.  ``n_planted`` blocks per pair, drawn among the blocks that are
  neither init nor local at selection time, have their keys shifted by
  +0.5 * u / |u| before rounding, u the Forecast direction aimed at that layer, so
  that they are the blocks a Forecast vector should find (block affinity).
* 80-layer 128K workload: 80 logical layers backed by 10 physical KV layers
  (logical l uses physical l mod 10); each physical layer q has its own direction
  u_q per pair and 64 planted blocks, 38 of them (60 %) shared with physical q-1.
  F_l = u_{(l+1) mod 10} + 0.25 * noise (the Forecast of layer l targets layer l+1,
  SparDA notes eq.(6)); F^cur_0 = u_0 + 0.25 * noise (SparDA notes §4.6).  The B = 1
  variant keeps all 80 layers resident (80 physical layers, same recipe).
* Grouped verification (SSV notes, mechanism 1): per (batch, KV head, group of C
  queries) a core of round(gamma * n_sel) blocks shared by every query of the group
  plus n_sel - core private blocks per query, all distinct and drawn without
  replacement outside the sliding window, each query's list ascending.
* Prefill selection (SparDA notes §4.3 eq.(16), the 1.25x prefill workload's
  MiniCPM4.1-8B shape: G = 4): one Forecast vector per (batch, KV head, position)
  [B][H_kv][T][128] (bf16 N(0, 1)) and the prefill's compressed keys
  [B][H_kv][N_b][128] drawn directly as fp32 N(0, 1/64), the spread of a 64-token mean
  of N(0, 1) keys.
"""
from __future__ import annotations

import dataclasses

import torch

D = 128
BLK = 64


def n_blocks(tokens: int) -> int:
    return (tokens + BLK - 1) // BLK


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    """One block-sparse GQA decode workload."""
    name: str
    B: int
    H_q: int
    H_kv: int
    T: int                 # cached tokens before the step
    n_init: int
    n_local: int
    k: int
    n_planted: int
    n_new: int = 0         # tokens appended by the step (1 = decode append)
    layers: int = 1        # logical layers per step
    phys_layers: int = 1   # physical KV layers backing them (logical l -> l mod phys)
    shared_planted: int = 0
    seed: int = 1234

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def pairs(self) -> int:
        return self.B * self.H_kv

    @property
    def len_after(self) -> int:
        return self.T + self.n_new

    @property
    def N_b(self) -> int:
        return n_blocks(self.len_after)

    @property
    def k_tot(self) -> int:
        return min(self.N_b, self.n_init + self.n_local + self.k)

    @property
    def T_cap(self) -> int:
        # room for the appended tokens, rounded up to whole blocks
        return n_blocks(self.len_after) * BLK


@dataclasses.dataclass(frozen=True)
class VerifyShape:
    """Grouped speculative verification workload (SSV mode A)."""
    name: str
    B: int
    H_q: int
    H_kv: int
    T: int
    N_q: int
    n_sel: int
    gamma: float
    window_tokens: int
    C: int
    seed: int = 1238

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def window_blocks(self) -> int:
        return self.window_tokens // BLK

    @property
    def N_b(self) -> int:
        return n_blocks(self.T)


@dataclasses.dataclass(frozen=True)
class OffloadShape:
    """Offloaded-KV decode: full KV in pinned host memory, compressed keys in HBM."""
    name: str
    B: int
    H_q: int
    H_kv: int
    T: int
    layers: int
    n_init: int
    n_local: int
    k: int
    n_planted: int
    phys_layers: int
    seed: int = 1239

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def pairs(self) -> int:
        return self.B * self.H_kv

    @property
    def N_b(self) -> int:
        return n_blocks(self.T)

    @property
    def k_tot(self) -> int:
        return min(self.N_b, self.n_init + self.n_local + self.k)


# The five workloads (shapes of the pages' 32K-128K GQA decode and 64K verification).
SINGLE_4K = DecodeShape("single_layer_4k_b1_g4", B=1, H_q=8, H_kv=2, T=4096, n_init=1,
                        n_local=2, k=8, n_planted=8, seed=1235)
LLAMA8B_32K = DecodeShape("llama8b_32k_b8_append", B=8, H_q=32, H_kv=8, T=32768, n_init=1,
                          n_local=2, k=32, n_planted=26, n_new=1, seed=1236)
DECODE_128K = DecodeShape("decode_128k_70b_b8_80layers", B=8, H_q=64, H_kv=8, T=131072,
                          n_init=1, n_local=2, k=64, n_planted=64, layers=80, phys_layers=10,
                          shared_planted=38, seed=1237)
# The same 70B-shaped 128K decode at B = 1 with all 80 layers resident (80 x 537 MB =
# 42.9 GB, the footprint the SparDA notes print in eq.(2)): 8 pairs per layer.
DECODE_128K_B1 = DecodeShape("decode_128k_70b_b1_80layers_resident", B=1, H_q=64, H_kv=8, T=131072,
                             n_init=1, n_local=2, k=64, n_planted=64, layers=80, phys_layers=80,
                             shared_planted=38, seed=1241)
VERIFY_64K = VerifyShape("ssv_verify_64k_b4_c4", B=4, H_q=32, H_kv=8, T=65536, N_q=8, n_sel=16,
                         gamma=0.75, window_tokens=512, C=4, seed=1238)
OFFLOAD_128K = OffloadShape("offload_128k_b4_32layers", B=4, H_q=32, H_kv=8, T=131072, layers=32,
                            n_init=1, n_local=2, k=64, n_planted=64, phys_layers=32, seed=1239)


@dataclasses.dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    H_q: int
    H_kv: int
    T: int
    n_init: int
    n_local: int
    k: int
    seed: int

    @property
    def pairs(self) -> int:
        return self.B * self.H_kv

    @property
    def N_b(self) -> int:
        return n_blocks(self.T)

    @property
    def k_tot(self) -> int:
        return self.n_init + self.n_local + self.k


PREFILL_32K = PrefillShape("prefill_32k_b4_g4", B=4, H_q=32, H_kv=8, T=32768, n_init=1, n_local=2, k=32, seed=1240)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _subseed(seed: int, *parts: int) -> int:
    s = int(seed)
    for p in parts:
        s = (s * 1_000_003 + int(p) + 7) % (2 ** 61 - 1)
    return s


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def draw_blocks(n: int, lo: int, hi: int, seed: int, exclude=None) -> torch.Tensor:
    """n distinct block ids from [lo, hi) minus ``exclude``, ascending (CPU, seeded)."""
    pool = torch.arange(lo, hi, dtype=torch.int64)
    if exclude is not None and len(exclude) > 0:
        mask = torch.ones(hi - lo, dtype=torch.bool)
        ex = torch.as_tensor(exclude, dtype=torch.int64)
        ex = ex[(ex >= lo) & (ex < hi)] - lo
        mask[ex] = False
        pool = pool[mask]
    if n > pool.numel():
        raise ValueError(f"cannot draw {n} blocks from {pool.numel()}")
    perm = torch.randperm(pool.numel(), generator=_gen("cpu", seed))
    return pool[perm[:n]].sort().values


def planted_sets(shape: DecodeShape | OffloadShape, phys_layer_count: int | None = None):
    """Planted block ids per (physical layer, pair): LongTensor [P_phys][pairs][n_planted].

    Drawn among candidate blocks [n_init, N_b - n_local) at selection time; physical
    layer q keeps ``shared_planted`` of layer q-1's blocks."""
    P = phys_layer_count if phys_layer_count is not None else getattr(shape, "phys_layers", 1)
    lo, hi = shape.n_init, shape.N_b - shape.n_local
    shared = getattr(shape, "shared_planted", 0)
    out = torch.empty((P, shape.pairs, shape.n_planted), dtype=torch.int64)
    for p in range(shape.pairs):
        prev = None
        for q in range(P):
            s = _subseed(shape.seed, 11, q, p)
            if prev is None or shared == 0:
                cur = draw_blocks(shape.n_planted, lo, hi, s)
            else:
                keep_idx = torch.randperm(prev.numel(), generator=_gen("cpu", s))[:shared]
                keep = prev[keep_idx]
                fresh = draw_blocks(shape.n_planted - shared, lo, hi, s + 1, exclude=prev.tolist())
                cur = torch.cat([keep, fresh]).sort().values
            out[q, p] = cur
            prev = cur
    return out


def direction(shape, phys_layer: int, device="cpu") -> torch.Tensor:
    """Forecast direction u aimed at a physical layer: fp32 [pairs][128] (N(0,1))."""
    g = _gen(device, _subseed(shape.seed, 13, phys_layer))
    return torch.randn((shape.pairs, D), generator=g, device=device, dtype=torch.float32)


def forecast(shape, target_phys: int, logical: int, device="cpu") -> torch.Tensor:
    """F [B][H_kv][128] bf16 aimed at ``target_phys``: u + 0.25 * noise (multi-layer),
    or u itself for single-layer workloads."""
    u = direction(shape, target_phys, device)
    if getattr(shape, "layers", 1) > 1:
        g = _gen(device, _subseed(shape.seed, 17, logical))
        u = u + 0.25 * torch.randn(u.shape, generator=g, device=device, dtype=torch.float32)
    return u.to(torch.bfloat16).view(shape.B, shape.H_kv, D)


def queries(shape, logical: int, device="cpu") -> torch.Tensor:
    """Q [B][H_q][128] bf16 for one logical layer."""
    return randn_bf16((shape.B, shape.H_q, D), _subseed(shape.seed, 19, logical), device)


def kv_pair(shape, phys_layer: int, pair: int, planted: torch.Tensor | None, device="cpu",
            T_cap: int | None = None, tokens: int | None = None):
    """K and V of one (physical layer, pair): bf16 [T_cap][128] each, ``tokens`` rows drawn.

    Keys of planted blocks are shifted by +0.5 * u/|u| (u aimed at this layer) before
    rounding to bf16."""
    T = shape.T if tokens is None else tokens
    T_cap = T if T_cap is None else T_cap
    gk = _gen(device, _subseed(shape.seed, 23, phys_layer, pair))
    gv = _gen(device, _subseed(shape.seed, 29, phys_layer, pair))
    Kf = torch.randn((T, D), generator=gk, device=device, dtype=torch.float32)
    if planted is not None and planted.numel() > 0:
        u = direction(shape, phys_layer, device)[pair]
        # the selector sees the bf16 value of F; shift along that direction
        u = u.to(torch.bfloat16).to(torch.float32)
        shift = 0.5 * u / u.norm()
        rows = (planted.to(device).view(-1, 1) * BLK
                + torch.arange(BLK, device=device).view(1, -1)).reshape(-1)
        rows = rows[rows < T]
        Kf[rows] += shift
    K = torch.zeros((T_cap, D), dtype=torch.bfloat16, device=device)
    V = torch.zeros((T_cap, D), dtype=torch.bfloat16, device=device)
    K[:T] = Kf.to(torch.bfloat16)
    V[:T] = torch.randn((T, D), generator=gv, device=device, dtype=torch.float32).to(torch.bfloat16)
    return K, V


def new_tokens(shape: DecodeShape, phys_layer: int, step: int = 0, device="cpu"):
    """K_new, V_new [B][H_kv][n_new][128] bf16 for an append step."""
    k = randn_bf16((shape.B, shape.H_kv, shape.n_new, D), _subseed(shape.seed, 31, phys_layer, step), device)
    v = randn_bf16((shape.B, shape.H_kv, shape.n_new, D), _subseed(shape.seed, 37, phys_layer, step), device)
    return k, v


def single_layer(shape: DecodeShape, device="cpu"):
    """All inputs of a one-layer decode workload (configs with layers == 1).

    Returns a dict: K, V [B][H_kv][T_cap][128] (first T tokens filled), F, Q,
    k_new/v_new (when n_new > 0), planted [pairs][n_planted], seq_len_before/after."""
    planted = planted_sets(shape, 1)[0]
    K = torch.zeros((shape.B, shape.H_kv, shape.T_cap, D), dtype=torch.bfloat16, device=device)
    V = torch.zeros_like(K)
    for p in range(shape.pairs):
        b, h = divmod(p, shape.H_kv)
        K[b, h], V[b, h] = kv_pair(shape, 0, p, planted[p], device, T_cap=shape.T_cap)
    out = dict(K=K, V=V, F=forecast(shape, 0, 0, device), Q=queries(shape, 0, device),
               planted=planted, len_before=shape.T, len_after=shape.len_after)
    if shape.n_new > 0:
        out["k_new"], out["v_new"] = new_tokens(shape, 0, 0, device)
    return out


def verify_sets(shape: VerifyShape) -> torch.Tensor:
    """Per-query block sets I [B][H_kv][N_q][n_sel] int32 (core + private, ascending).

    Per (batch, KV head, group) a core of round(gamma * n_sel) blocks is shared by
    all C queries and every query adds n_sel - core private blocks; all are distinct
    and lie outside the window blocks [N_b - window_blocks, N_b)."""
    n_core = int(round(shape.gamma * shape.n_sel))
    n_priv = shape.n_sel - n_core
    hi = shape.N_b - shape.window_blocks
    I = torch.empty((shape.B, shape.H_kv, shape.N_q, shape.n_sel), dtype=torch.int32)
    for b in range(shape.B):
        for h in range(shape.H_kv):
            for q0 in range(0, shape.N_q, shape.C):
                nq = min(shape.C, shape.N_q - q0)
                s = _subseed(shape.seed, 41, b, h, q0)
                drawn = draw_blocks(n_core + nq * n_priv, 0, hi, s)
                perm = torch.randperm(drawn.numel(), generator=_gen("cpu", s + 1))
                drawn = drawn[perm]
                core = drawn[:n_core]
                for i in range(nq):
                    priv = drawn[n_core + i * n_priv: n_core + (i + 1) * n_priv]
                    I[b, h, q0 + i] = torch.cat([core, priv]).sort().values.to(torch.int32)
    return I


def verify_inputs(shape: VerifyShape, device="cpu"):
    """Q [B][N_q][H_q][128], K/V [B][H_kv][T][128], I, seq_len [B]."""
    K = torch.empty((shape.B, shape.H_kv, shape.T, D), dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    for b in range(shape.B):
        for h in range(shape.H_kv):
            K[b, h], V[b, h] = kv_pair(shape, 0, b * shape.H_kv + h, None, device)
    Q = randn_bf16((shape.B, shape.N_q, shape.H_q, D), _subseed(shape.seed, 43), device)
    I = verify_sets(shape).to(device)
    lens = torch.full((shape.B,), shape.T, dtype=torch.int32, device=device)
    return dict(Q=Q, K=K, V=V, I=I, seq_len=lens)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def prefill_inputs(shape: PrefillShape, device="cpu"):
    """Forecast vectors of every position and the prefill's compressed keys."""
    F = randn_bf16((shape.B, shape.H_kv, shape.T, D), _subseed(shape.seed, 1), device)
    ktil = torch.randn((shape.B, shape.H_kv, shape.N_b, D), generator=_gen(device, _subseed(shape.seed, 2)),
                       device=device, dtype=torch.float32) * 0.125
    return dict(F=F, ktil=ktil)
