#!/usr/bin/env python
"""Benchmark of the block-sparse GQA decode path on one GB300 (or N replicas).

Default workload: one 128K decode step of a 70B-shaped model (80 layers, B=8,
H_q=64, H_kv=8, d=128, T=131072, top-64 + 1 init + 2 local blocks).  A step runs, for
every layer l, the Forecast selection for layer l+1 (sparse_select_topk on a side
stream, allowed to start once attention of layer l-1 is done) overlapped with the
block-sparse attention of layer l (sparse_decode_attn on the main stream); layer 0
first selects with its own current-layer Forecast.  The 80-layer step is one CUDA
graph.  80 logical layers are backed by 10 physical KV layers (logical l reads
physical l mod 10): the literal B=8 x 80-layer x 128K cache is 343.6 GB.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample per step, and prints the same metric for it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn steps/sec and selected-KV HBM GB/s (fraction of 8 TB/s) at 128K"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
D, BLK = 128, 64
KV_BLOCK_BYTES = 2 * BLK * D * 2      # K + V of one selected block (bf16)
KTIL_ROW_BYTES = D * 4                # one fp32 compressed key


def n_candidates(sh):
    """Blocks the selection scores: every block but B_init and B_local (the pages' top-k
    is taken over the others), so the compressed keys it has to read."""
    return max(0, sh.N_b - sh.n_init - sh.n_local)


# ----------------------------------------------------------------------------- ranks


def dist_env():
    """(rank, world, local_rank) from the torchrun environment (1 process = 1 GPU)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a float over all ranks (replicas time independently; the slowest counts)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_steps_per_s(ms_per_step_max: float, world: int) -> float:
    """Replicas: every rank runs the full step on its own GPU, so the job completes
    ``world`` steps in the slowest rank's step time."""
    return world * 1000.0 / ms_per_step_max


# ----------------------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


ATTN_SOURCES = ("sparse_attn.cu", "attn_core.cuh", "attn_tc.cuh", "common.cuh")
FUSED_SOURCES = ("forecast.cu", "attn_core.cuh", "select_core.cuh", "select_layout.cuh", "common.cuh")


def kernel_source_hash(files=ATTN_SOURCES) -> str:
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, "block_sparse_long_pool_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_hash: str, name: str = "decode_attn_128k_traffic.txt"):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if it was
    taken on the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        kv = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha1") != kernel_hash:
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 25 ms during the timed region (a step
    of the default bench is ~3 ms, its timed region well under a second)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (the JSON line carries their summary); SPARSE_POOL_CLOCKS_DIR moves them
        out_dir = os.environ.get("SPARSE_POOL_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"sparse_pool_clocks_gpu{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- 128K decode workload


def step_config(sh, world: int) -> dict:
    """The workload the bench line is quoted on (both arms)."""
    layer_gb = sh.pairs * sh.T * D * 2 * 2 / 1e9
    return {"workload": sh.name, "B": sh.B, "H_q": sh.H_q, "H_kv": sh.H_kv, "d": D, "T": sh.T,
            "layers": sh.layers, "physical_kv_layers": sh.phys_layers, "block": BLK, "k": sh.k,
            "n_init": sh.n_init, "n_local": sh.n_local, "blocks_per_pair": sh.k_tot,
            "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {sh.phys_layers} physical layers x {layer_gb:.2f} GB, the same layer "
                  f"again after {sh.phys_layers * sh.pairs * (sh.k_tot * KV_BLOCK_BYTES + n_candidates(sh) * KTIL_ROW_BYTES) / 1e9:.2f}"
                  " GB of other reads"}


def l2_evict(buf):
    """Read a buffer larger than L2 (129 MB) so the next launch starts from a cold,
    clean L2."""
    import torch
    torch.sum(buf)


def step_distribution(per_step_ms):
    """Median and 10th / 90th percentiles of per-step times (ms)."""
    xs = sorted(per_step_ms)
    q = lambda f: xs[min(len(xs) - 1, int(f * len(xs)))]
    return {"median": round(statistics.median(xs), 4), "p10": round(q(0.1), 4), "p90": round(q(0.9), 4),
            "min": round(xs[0], 4), "max": round(xs[-1], 4), "steps": len(xs)}


class DecodeStep:
    """Device state of a multi-layer decode step (the 128K, 80-layer workloads) and its
    CUDA graph.

    mode "fused": layer 0 selects with sparse_select_topk, then every layer l is one
    sparse_decode_attn_forecast launch (attention of l + Forecast selection of l+1), all
    on one stream.  mode "separate": sparse_select_topk of layer l+1 on a side stream
    beside sparse_decode_attn of layer l (with a workspace: the split path)."""

    def __init__(self, device, shape=None, use_workspace=True, mode="fused", n_split=0):
        assert mode in ("fused", "separate")
        self.mode = mode
        import torch
        from block_sparse_long_pool_gb300 import binding
        from block_sparse_long_pool_gb300 import workloads as wl

        self.torch, self.binding, self.wl = torch, binding, wl
        sh = self.sh = shape if shape is not None else wl.DECODE_128K
        self.n_split = n_split
        self.dev = device
        B, H_kv, H_q, T = sh.B, sh.H_kv, sh.H_q, sh.T
        self.k_cap = sh.n_init + sh.n_local + sh.k
        P = sh.phys_layers
        planted = wl.planted_sets(sh, P)
        self.k_cache, self.v_cache, self.ktil = [], [], []
        for q in range(P):
            kc = torch.empty((B, H_kv, T, D), dtype=torch.bfloat16, device=device)
            vc = torch.empty_like(kc)
            kt = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device=device)
            for b in range(B):
                kn = torch.empty((1, H_kv, T, D), dtype=torch.bfloat16, device=device)
                vn = torch.empty_like(kn)
                for h in range(H_kv):
                    pr = b * H_kv + h
                    kn[0, h], vn[0, h] = wl.kv_pair(sh, q, pr, planted[q, pr], device)
                binding.sparse_pool_append(kc[b:b + 1], vc[b:b + 1], kt[b:b + 1], kn, vn, 0)
                del kn, vn
            self.k_cache.append(kc)
            self.v_cache.append(vc)
            self.ktil.append(kt)
        L = sh.layers
        # per-step inputs: Q_l and F_l (F_l targets layer l+1), F^cur_0; outputs O_l
        self.Q = torch.stack([wl.queries(sh, l, device) for l in range(L)])            # [L][B][H_q][D]
        self.F = torch.stack([wl.forecast(sh, (l + 1) % P, l, device) for l in range(L)])  # [L][B][H_kv][D]
        self.F0 = wl.forecast(sh, 0, -1, device)
        self.O = torch.zeros((L, B, H_q, D), dtype=torch.bfloat16, device=device)
        self.idx = torch.full((L, B, H_kv, self.k_cap), -1, dtype=torch.int32, device=device)
        self.count = torch.zeros((L, B, H_kv), dtype=torch.int32, device=device)
        self.seq = torch.full((B,), T, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.side = torch.cuda.Stream(device=device)
        self.workspace = (binding.decode_workspace(B, H_q, H_kv, self.k_cap, n_split, device=device)
                          if use_workspace else None)
        torch.cuda.synchronize(device)

    # bytes the method has to move per step
    def algorithmic_bytes(self):
        sh = self.sh
        attn = sh.layers * sh.pairs * sh.k_tot * KV_BLOCK_BYTES
        sel = (sh.layers) * sh.pairs * n_candidates(sh) * KTIL_ROW_BYTES     # layer-0 + layers 1..79
        return attn, sel

    def attn_bytes_per_launch(self):
        return self.sh.pairs * self.sh.k_tot * KV_BLOCK_BYTES

    def select_bytes_per_launch(self):
        return self.sh.pairs * n_candidates(self.sh) * KTIL_ROW_BYTES

    def fused_bytes_per_launch(self):
        return self.attn_bytes_per_launch() + self.select_bytes_per_launch()

    def launches_per_step(self):
        if self.mode == "fused":
            return 1 + self.sh.layers  # layer-0 selection + 80 fused layers
        return 2 * self.sh.layers      # 80 selections (incl. layer 0) + 80 attentions

    def _fused(self, l, stream):
        # attention of layer l over the list the previous launch selected, and the
        # Forecast selection of layer l+1 (none after the last layer)
        sh = self.sh
        q = l % sh.phys_layers
        nxt = l + 1 < sh.layers
        self.binding.sparse_decode_attn_forecast(
            self.Q[l], self.k_cache[q], self.v_cache[q], self.idx[l], self.count[l], self.seq, self.O[l],
            F=self.F[l] if nxt else None, ktil_next=self.ktil[(l + 1) % sh.phys_layers] if nxt else None,
            n_init=sh.n_init, n_local=sh.n_local, k=sh.k, idx_next=self.idx[l + 1] if nxt else None,
            count_next=self.count[l + 1] if nxt else None, n_split=self.n_split, status=self.status,
            stream=stream)

    def _select(self, l_target, F, stream):
        sh = self.sh
        self.binding.sparse_select_topk(F, self.ktil[l_target % sh.phys_layers], self.seq, sh.n_init, sh.n_local,
                                        sh.k, self.idx[l_target], self.count[l_target], status=self.status,
                                        stream=stream)

    def _attend(self, l, stream, count=None, workspace=True):
        # the block list of every layer comes from the side stream through an event, so
        # K/V streaming may start while the previous attention drains
        q = l % self.sh.phys_layers
        count = self.count[l] if count is None else count
        ws = self.workspace if workspace else None
        self.binding.sparse_decode_attn(self.Q[l], self.k_cache[q], self.v_cache[q], self.idx[l], count,
                                        self.seq, self.O[l], status=self.status,
                                        n_split=self.n_split if ws is not None else 0,
                                        flags=self.binding.SPARSE_ATTN_BLOCKS_READY, workspace=ws, stream=stream)

    def enqueue_step(self):
        """Enqueue one step on the current stream (+ the side stream in separate mode)."""
        torch = self.torch
        main = torch.cuda.current_stream(self.dev)
        L = self.sh.layers
        if self.mode == "fused":
            self._select(0, self.F0, main)           # layer 0: its own current-layer Forecast
            for l in range(L):
                self._fused(l, main)
            return
        sel_done = [None] * L
        self.side.wait_stream(main)
        self._select(0, self.F0, self.side)          # layer 0: its own current-layer Forecast
        ev0 = torch.cuda.Event()
        ev0.record(self.side)
        sel_done[0] = ev0
        after_prev_attn = torch.cuda.Event()
        after_prev_attn.record(main)
        for l in range(L):
            if l + 1 < L:
                self.side.wait_event(after_prev_attn)
                self._select(l + 1, self.F[l], self.side)
                ev = torch.cuda.Event()
                ev.record(self.side)
                sel_done[l + 1] = ev
            if sel_done[l] is not None:
                main.wait_event(sel_done[l])
            self._attend(l, main)
            after_prev_attn = torch.cuda.Event()
            after_prev_attn.record(main)
        main.wait_stream(self.side)

    def capture(self):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self.enqueue_step()           # warm the library (tensor maps, attributes) outside capture
        torch.cuda.synchronize(self.dev)
        with torch.cuda.graph(g, stream=s):
            self.enqueue_step()
        torch.cuda.synchronize(self.dev)
        return g


Decode128k = DecodeStep


def time_graph_steps(graph, K, world, dev, clocks_gpu):
    """K graph replays, barrier + synchronize on both sides, a CUDA event between
    consecutive replays (the per-step distribution) and clocks sampled meanwhile.
    Returns (max-over-ranks ms per step, per-step ms, clock summary)."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    with ClockSampler(clocks_gpu) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        # ~1 ms of GPU spinning ahead of the start event, during which the host enqueues
        # the replays: the timed region holds GPU work only, no wait for the host
        torch.cuda._sleep(2_000_000)
        evs[0].record()
        for i in range(K):
            graph.replay()
            evs[i + 1].record()
        torch.cuda.synchronize(dev)
        barrier(world)
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]
    ms = max_over_ranks(evs[0].elapsed_time(evs[K]), world, dev) / K
    return ms, per, clocks.summary()


def kernel_breakdown(wk, dev, peak):
    """Per-launch kernel times of the step's kernels, CUDA events on the launching
    stream: each launch alone after a 512 MB read that evicts L2 (a read leaves clean
    lines; a write would leave 129 MB of dirty lines for the timed kernel to write back),
    and the layers' launches back to back in one graph.  The block lists are the ones
    the step just selected."""
    import torch
    flush = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)
    cur = torch.cuda.current_stream(dev)
    L = wk.sh.layers
    reps_alone = 2 if L * 2 >= 160 else max(2, 160 // L)

    def time_alone(fn, reps=reps_alone, warmup=3):
        # synchronize, then the L2-evicting read (~85 us of GPU time), during which the
        # host enqueues the timed launch: the events bracket GPU work only, never a wait
        # for the host to submit the launch.  The untimed warm-up launches come first: the
        # first launch of a kernel in the process loads its module (~0.8 ms).
        for l in range(min(warmup, L)):
            fn(l)
        ev = []
        for _ in range(reps):
            for l in range(L):
                torch.cuda.synchronize(dev)
                l2_evict(flush)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn(l)
                b.record()
                ev.append((a, b))
        torch.cuda.synchronize(dev)
        t = sorted(a.elapsed_time(b) for a, b in ev)
        med = statistics.median(t)
        # a launch the host enqueued only after the evicting read had finished (a host
        # stall: the GPU idles between the start event and the kernel) reads many times
        # the median; such samples are left out of the mean and counted
        kept = [x for x in t if x <= 4.0 * med]
        dist = {"median_us": round(med * 1e3, 2), "p10_us": round(t[len(t) // 10] * 1e3, 2),
                "p90_us": round(t[(9 * len(t)) // 10] * 1e3, 2), "raw_mean_us": round(statistics.mean(t) * 1e3, 2),
                "host_stalls_dropped": len(t) - len(kept), "warmup_launches": min(warmup, L)}
        return statistics.mean(kept), len(t), dist

    def time_chain(fn, reps=5):
        # the L launches back to back in one graph (programmatic dependent launch
        # overlaps each launch's start with the previous one's end)
        g = torch.cuda.CUDAGraph()
        s_ = torch.cuda.Stream(device=dev)
        s_.wait_stream(cur)
        with torch.cuda.graph(g, stream=s_):
            for l in range(L):
                fn(l, s_)
        for _ in range(2):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / (reps * L)

    # the standalone decode attention (sparse_decode_attn, resident cache, no workspace)
    att_alone_ms, att_n, att_dist = time_alone(lambda l: wk._attend(l, cur, workspace=False))
    att_chain_ms = time_chain(lambda l, st_: wk._attend(l, st_, workspace=False))
    att_bytes = wk.attn_bytes_per_launch()
    att_hash = kernel_source_hash(ATTN_SOURCES)
    # what a launch costs without streaming: the same launch with every count 0 (list
    # fetch, Q load, merge, O write), and a one-element torch kernel timed the same way
    zero_count = torch.zeros_like(wk.count[0])
    att_empty_ms, _, _ = time_alone(lambda l: wk._attend(l, cur, count=zero_count, workspace=False), reps=1)
    tiny = torch.zeros(1, device=dev)
    floor_ms, _, _ = time_alone(lambda l: tiny.add_(1.0), reps=1)
    stream_ms = att_alone_ms - att_empty_ms
    attention = {"kernel": f"sparse_attn_kernel (sparse_decode_attn, decode, G={wk.sh.G})",
                 "algorithmic_bytes_per_launch": att_bytes,
                 "alone": {"avg_launch_us": round(att_alone_ms * 1e3, 2), "launches_timed": att_n, **att_dist,
                           "achieved": round(att_bytes / (att_alone_ms * 1e-3) / 1e9, 1),
                           "frac": round(att_bytes / (att_alone_ms * 1e-3) / 1e9 / peak, 4),
                           "empty_launch_us": round(att_empty_ms * 1e3, 2),
                           "event_floor_us": round(floor_ms * 1e3, 2),
                           "streaming_gbs": round(att_bytes / (stream_ms * 1e-3) / 1e9, 1) if stream_ms > 0 else None,
                           "streaming_frac": round(att_bytes / (stream_ms * 1e-3) / 1e9 / peak, 4)
                           if stream_ms > 0 else None,
                           "note": "empty_launch_us: the same launches with every count 0; event_floor_us: a "
                                   "one-element torch kernel timed the same way; streaming = bytes / (alone - "
                                   "empty)"},
                 "chained": {"avg_launch_us": round(att_chain_ms * 1e3, 2), "launches": L,
                             "achieved": round(att_bytes / (att_chain_ms * 1e-3) / 1e9, 1),
                             "frac": round(att_bytes / (att_chain_ms * 1e-3) / 1e9 / peak, 4),
                             "note": f"{L} launches back to back in a CUDA graph, one per layer"},
                 "traffic": profiled_traffic(att_hash) if wk.sh.name == "decode_128k_70b_b8_80layers" else None,
                 "kernel_source_sha1": att_hash}
    sel_alone_ms, sel_n, sel_dist = time_alone(lambda l: wk._select(l, wk.F[l - 1] if l else wk.F0, cur))
    sel_bytes = wk.select_bytes_per_launch()
    selection = {"kernel": "decode_forecast_kernel<1, false> (sparse_select_topk)",
                 "algorithmic_bytes_per_launch": sel_bytes,
                 "alone": {"avg_launch_us": round(sel_alone_ms * 1e3, 2), "launches_timed": sel_n, **sel_dist,
                           "achieved": round(sel_bytes / (sel_alone_ms * 1e-3) / 1e9, 1),
                           "frac": round(sel_bytes / (sel_alone_ms * 1e-3) / 1e9 / peak, 4)}}
    out = {"attention": attention, "selection": selection}
    if wk.mode == "fused":
        dom_alone_ms, dom_n, dom_dist = time_alone(lambda l: wk._fused(l, cur))
        dom_bytes = wk.fused_bytes_per_launch()
        out["dominant"] = {"kernel": "decode_forecast_kernel (sparse_decode_attn_forecast: attention of layer l + "
                                     f"Forecast selection of layer l+1, G={wk.sh.G})",
                           "algorithmic_bytes_per_launch": dom_bytes, "source": FUSED_SOURCES,
                           "alone_us": dom_alone_ms * 1e3, "alone_n": dom_n, "alone_dist": dom_dist}
    else:
        out["dominant"] = {"kernel": f"sparse_attn_kernel (sparse_decode_attn, G={wk.sh.G})",
                           "algorithmic_bytes_per_launch": att_bytes, "source": ATTN_SOURCES,
                           "alone_us": att_alone_ms * 1e3, "alone_n": att_n, "alone_dist": att_dist}
    del flush
    return out


def measure_decode_step(args, sh, rank, world, local_rank, with_e2e=True):
    """The multi-layer decode step of workload ``sh``: its CUDA graph timed over K
    replays, the roofline of the step, the per-kernel breakdown and (optionally) the
    end-to-end number with host copies.  Returns the fields of a JSON line."""
    import torch
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    import __graft_entry__
    __graft_entry__.build()

    wk = DecodeStep(dev, sh, use_workspace=args.workspace, mode=args.step_mode, n_split=args.n_split)
    graph = wk.capture()
    K, W = args.steps, args.warmup
    for _ in range(W):
        graph.replay()
    torch.cuda.synchronize(dev)
    assert wk.status.item() == 0, f"device status {wk.status.item()}"

    # ---- timed region: K graph replays (inputs resident in HBM, larger than L2)
    ms, per_step, clocks = time_graph_steps(graph, K, world, dev, local_rank)
    value = whole_job_steps_per_s(ms, world)
    attn_b, sel_b = wk.algorithmic_bytes()
    step_bytes = attn_b + sel_b
    peak, peak_src = measured_peaks()
    kb = kernel_breakdown(wk, dev, peak)
    dom = kb["dominant"]
    dom_hash = kernel_source_hash(dom["source"])
    dom_traffic = None
    if sh.name == "decode_128k_70b_b8_80layers":
        dom_traffic = (profiled_traffic(dom_hash, "decode_forecast_128k_traffic.txt") if wk.mode == "fused"
                       else profiled_traffic(dom_hash))
    elif sh.name == "decode_128k_70b_b1_80layers_resident" and wk.mode == "fused":
        dom_traffic = profiled_traffic(dom_hash, "decode_forecast_128k_b1_traffic.txt")
    launches = wk.launches_per_step()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    alone_gbs = dom["algorithmic_bytes_per_launch"] / (dom["alone_us"] * 1e-6) / 1e9
    roofline = {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "traffic": dom_traffic,
        "kernel": dom["kernel"] + ", inside the timed step",
        "achieved_is": "the step's algorithmic bytes (selected K/V + compressed keys of every launch) / the step's "
                       "CUDA-event time: per launch, the average algorithmic bytes of the step's launches / their "
                       "average duration",
        "peak_source": peak_src + " (the one HBM figure: a burst copy)",
        "algorithmic_bytes_per_step": step_bytes, "launches_per_step": launches,
        "avg_launch_us": round(ms * 1e3 / launches, 2),
        "algorithmic_bytes_per_launch": {"dominant": dom["algorithmic_bytes_per_launch"],
                                         "layer0_selection": wk.select_bytes_per_launch(),
                                         "average": round(step_bytes / launches)},
        "traffic_is": "dram__bytes_read.sum + dram__bytes_write.sum of one dominant launch (ncu), null unless "
                      "taken on the current kernel source",
        "alone": {"avg_launch_us": round(dom["alone_us"], 2), "launches_timed": dom["alone_n"], **dom["alone_dist"],
                  "achieved": round(alone_gbs, 1), "frac": round(alone_gbs / peak, 4),
                  "note": "each launch timed by itself after a 512 MB read that evicts L2, after 3 untimed "
                          "warm-up launches; the mean leaves out launches over 4x the median (host stalls)"},
        "kernel_source_sha1": dom_hash}
    line = {
        "value": round(value, 3), "unit": "steps/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms, 4), "step_ms": step_distribution(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, planted blocks)",
        "config": dict(step_config(sh, world), step_mode=wk.mode, n_split=args.n_split,
                       workspace=bool(args.workspace)),
        "selected_kv_gbs": round(world * step_bytes / (ms * 1e-3) / 1e9, 1),
        "hbm_frac_of_8tbs": round(step_bytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "hbm_frac_of_measured": round(step_bytes / (ms * 1e-3) / 1e9 / peak, 4),
        "bytes_per_step": {"selected_kv": attn_b, "compressed_keys": sel_b},
        "roofline": roofline,
        "attention_kernel": kb["attention"],
        "selection_kernel": kb["selection"],
        "gpu_launches": launches * K,
        "clocks": clocks,
    }
    if with_e2e:
        e2e_ms, h2d, d2h = measure_e2e(wk, graph, K, world, dev)
        line["e2e"] = {"value": round(world * 1000.0 / e2e_ms, 3), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h}
    assert wk.status.item() == 0, f"device status {wk.status.item()}"
    line["cpu_baseline"] = (cpu_baseline(wk, seconds=args.cpu_seconds)
                            if rank == 0 and not args.no_cpu_baseline else None)
    return line


def measure_e2e(wk, graph, K, world, dev):
    """End to end through the binding: Q and F from pinned host memory in, O out, every
    step inside the timed region.  Double-buffered: a second set of Q / F / O device
    buffers with its own graph; one stream moves step s+1's inputs in while step s runs,
    another moves step s's outputs out while step s+1 runs.  Returns (ms per step, H2D
    bytes per step, D2H bytes per step)."""
    import torch
    Qh = wk.Q.cpu().pin_memory()
    Fh = wk.F.cpu().pin_memory()
    F0h = wk.F0.cpu().pin_memory()
    Oh = torch.empty(wk.O.shape, dtype=wk.O.dtype).pin_memory()
    sets = [(wk.Q, wk.F, wk.F0, wk.O, graph)]
    wk.Q, wk.F, wk.F0, wk.O = (torch.empty_like(wk.Q), torch.empty_like(wk.F), torch.empty_like(wk.F0),
                               torch.empty_like(wk.O))
    wk.Q.copy_(sets[0][0])
    wk.F.copy_(sets[0][1])
    wk.F0.copy_(sets[0][2])
    sets.append((wk.Q, wk.F, wk.F0, wk.O, wk.capture()))
    main = torch.cuda.current_stream(dev)
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e_steps = max(4, K // 4)
    graph_done = [None, None]   # the last step of set i: its graph (inputs read, O written)
    d2h_done = [None, None]     # ... and the copy that read its O
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    for st in range(-2, e_steps):   # two untimed steps first: both graphs uploaded and warm
        if st == 0:
            main.wait_stream(h2d_s)
            main.wait_stream(d2h_s)
            torch.cuda.synchronize(dev)
            e0.record(main)
            h2d_s.wait_stream(main)
            d2h_s.wait_stream(main)
        i = st % 2
        Qd, Fd, F0d, Od, g_ = sets[i]
        with torch.cuda.stream(h2d_s):
            if graph_done[i] is not None:
                h2d_s.wait_event(graph_done[i])   # step st-2 has read this set's inputs
            Qd.copy_(Qh, non_blocking=True)
            Fd.copy_(Fh, non_blocking=True)
            F0d.copy_(F0h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(h2d_s)
        main.wait_event(ready)
        if d2h_done[i] is not None:
            main.wait_event(d2h_done[i])          # step st-2's O has been copied out
        g_.replay()
        done = torch.cuda.Event()
        done.record(main)
        graph_done[i] = done
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(done)
            Oh.copy_(Od, non_blocking=True)
            out = torch.cuda.Event()
            out.record(d2h_s)
            d2h_done[i] = out
    main.wait_stream(h2d_s)
    main.wait_stream(d2h_s)
    e1.record(main)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / e_steps
    wk.Q, wk.F, wk.F0, wk.O = sets[0][:4]
    h2d = Qh.numel() * 2 + Fh.numel() * 2 + F0h.numel() * 2
    d2h = Oh.numel() * 2
    return e2e_ms, h2d, d2h


def run_ours(args, rank, world, local_rank):
    from block_sparse_long_pool_gb300 import workloads as wl
    line = measure_decode_step(args, wl.DECODE_128K, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(dict({"metric": METRIC}, **line)), flush=True)


def run_b1_case(args, local_rank):
    """The literal B = 1 variant of the 128K step: all 80 layers resident (42.9 GB), 8
    pairs per layer, so a launch has 8 pairs to spread over the SMs."""
    import dataclasses
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wl.DECODE_128K_B1
    if args.layers:   # fewer resident layers (the 80 launches cycle over them): small profiling captures
        sh = dataclasses.replace(sh, name=f"{sh.name}_profiling_{args.layers}_physical", phys_layers=args.layers)
    line = measure_decode_step(args, sh, 0, 1, local_rank)
    print(json.dumps(dict({"case": "decode128k_b1", "metric": METRIC}, **line)), flush=True)


# ----------------------------------------------------------------------------- CPU oracle baseline


def _prepare_oracle_slice(wk, layer: int, batches, device=None):
    """Host copies of the inputs of one layer slice (the sampled batch elements): this
    layer's K/V and compressed keys, the next layer's compressed keys, Q_l and F_l.
    Pooling is not part of a decode step (the compressed keys are resident), so it
    happens here, outside any timing.  ``device`` draws the inputs there (the GPU arm
    draws them where its own kernels read them, so both see the same bytes)."""
    import numpy as np
    import oracle
    wl, sh = wk.wl, wk.sh
    dev = wk.dev if device is None else device
    q_cur, q_next = layer % sh.phys_layers, (layer + 1) % sh.phys_layers
    planted = wl.planted_sets(sh, sh.phys_layers)
    pairs = [b * sh.H_kv + h for b in batches for h in range(sh.H_kv)]
    Ks, Vs, Kn = [], [], []
    for p in pairs:
        k, v = wl.kv_pair(sh, q_cur, p, planted[q_cur, p], dev)
        Ks.append(wl.bf16_bits(k))
        Vs.append(wl.bf16_bits(v))
        kn, _ = wl.kv_pair(sh, q_next, p, planted[q_next, p], dev)
        Kn.append(wl.bf16_bits(kn))
    K, V, Knext = np.stack(Ks), np.stack(Vs), np.stack(Kn)
    lens = [sh.T] * len(pairs)
    ktil_cur = oracle.pool(K, lens, sh.N_b)
    ktil_next = oracle.pool(Knext, lens, sh.N_b)
    F = wl.bf16_bits(wl.forecast(sh, q_next, layer, "cpu")).reshape(sh.pairs, D)[pairs]
    Fc = wl.bf16_bits(wl.forecast(sh, q_cur, layer - 1, "cpu")).reshape(sh.pairs, D)[pairs]
    Q = wl.bf16_bits(wl.queries(sh, layer, "cpu")).reshape(sh.pairs, sh.G, D)[pairs]
    idx, cnt, _ = oracle.select(Fc, ktil_cur, lens, sh.n_init, sh.n_local, sh.k)   # this layer's blocks
    return dict(K=K, V=V, Q=Q, F=F, ktil_next=ktil_next, idx=idx, cnt=cnt, lens=lens, n=len(pairs), sh=sh)


def _time_oracle_slice(sl, threads: int):
    """Time the oracle's selection for layer l+1 and attention of layer l on a slice."""
    import oracle
    sh = sl["sh"]
    oracle.set_threads(threads)
    t0 = time.perf_counter()
    oracle.select(sl["F"], sl["ktil_next"], sl["lens"], sh.n_init, sh.n_local, sh.k)
    oracle.attn(sl["Q"], sl["K"], sl["V"], sl["idx"], sl["cnt"], sl["lens"])
    return time.perf_counter() - t0, sl["n"]


def _slice_geometry(sh):
    """Batch elements per oracle slice and threads: one OpenMP thread per pair, as many
    pairs as keep the host cores busy."""
    cores = len(os.sched_getaffinity(0))
    per_call = max(1, min(sh.B, cores // sh.H_kv))
    return per_call, min(cores, per_call * sh.H_kv)


def cpu_baseline(wk, seconds: float = 15.0, slices: int = 4):
    """The oracle on the host cores over a bounded sample of the decode step: layer
    slices of B_s batch elements (B_s x 8 pairs, one OpenMP thread per pair), repeated
    until that many seconds are spent, scaled to the step's layers x pairs."""
    per_call, threads = _slice_geometry(wk.sh)
    prepared = [_prepare_oracle_slice(wk, (7 * i) % wk.sh.layers,
                                      [(i * per_call + j) % wk.sh.B for j in range(per_call)])
                for i in range(slices)]
    spent, pair_layers, reps = 0.0, 0, 0
    while spent < seconds or reps < len(prepared):
        dt, n = _time_oracle_slice(prepared[reps % len(prepared)], threads)
        spent += dt
        pair_layers += n
        reps += 1
    step_s = spent / pair_layers * wk.sh.pairs * wk.sh.layers
    return {"value": round(1.0 / step_s, 6), "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} timed layer slices ({len(prepared)} distinct) of {per_call} batch element(s) x "
                      f"{wk.sh.H_kv} KV heads = {pair_layers} (pair, layer) units of select(l+1) + attention(l) "
                      f"in fp64 on {threads} threads, {spent:.1f} s, scaled to {wk.sh.pairs} pairs x "
                      f"{wk.sh.layers} layers"}


def run_reference(args, rank, world, local_rank):
    """The oracle as the reference arm, on the host cores only (no GPU, no CUDA
    library): every step is one bounded sample of the 128K step -- one layer slice of
    as many batch elements as keep the host cores busy (one thread per pair), the
    selection of layer l+1 and the attention of layer l -- drawn on the CPU.  The line
    reports the measured time per sample as ms_per_step and, as value, the steps/s of
    the whole 80-layer, 64-pair step extrapolated from it (the factor is stated)."""
    if rank != 0:
        return
    import oracle
    from block_sparse_long_pool_gb300 import workloads as wl
    oracle.build()

    class _Shim:  # just the fields the sampler needs
        pass
    wk = _Shim()
    wk.wl, wk.sh, wk.dev = wl, wl.DECODE_128K, "cpu"
    per_call, threads = _slice_geometry(wk.sh)
    t0 = time.perf_counter()
    prepared = [_prepare_oracle_slice(wk, (7 * i) % wk.sh.layers, [(i + j) % wk.sh.B for j in range(per_call)])
                for i in range(2)]
    prep_s = time.perf_counter() - t0
    times, n_pairs = [], 0
    for i in range(args.warmup + args.steps):
        dt, n = _time_oracle_slice(prepared[i % len(prepared)], threads)
        if i >= args.warmup:
            times.append(dt)
            n_pairs = n
    slice_s = statistics.mean(times)
    factor = wk.sh.pairs * wk.sh.layers / n_pairs
    value = 1.0 / (slice_s * factor)
    sample = (f"per step: one layer slice of {per_call} batch element(s) ({n_pairs} pairs) of {wk.sh.name}, "
              f"select(l+1) + attention(l) in fp64 on {threads} threads; value = 1 / (slice time x "
              f"{factor:g}), the whole step being {wk.sh.pairs} pairs x {wk.sh.layers} layers")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(slice_s * 1e3, 3),
            "ms_per_step_is": "the measured time of one timed sample (a layer slice), not of a whole step",
            "extrapolation_factor": factor, "full_step_ms_extrapolated": round(slice_s * factor * 1e3, 1),
            "timed_slices": len(times), "step_ms": step_distribution([t * 1e3 for t in times]),
            "input_prep_s": round(prep_s, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, planted blocks; drawn on the CPU)",
            "config": step_config(wk.sh, world),
            "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_layer_case(args, local_rank):
    """One physical layer of the 128K workload (4.3 GB of KV): selection then attention,
    serialised on one stream with a 512 MB L2-evicting read before each, every launch bracketed
    by CUDA events.  Used for isolated kernel times and small ncu captures."""
    import torch
    from block_sparse_long_pool_gb300 import binding
    from block_sparse_long_pool_gb300 import workloads as wl
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import dataclasses
    sh = wl.DECODE_128K
    if args.tokens:
        sh = dataclasses.replace(sh, T=args.tokens)
    B, H_kv, H_q, T = sh.B, sh.H_kv, sh.H_q, sh.T
    k_cap = sh.n_init + sh.n_local + sh.k
    planted = wl.planted_sets(sh, 1)
    select_only = args.case == "select"
    # the select-only case keeps just the compressed keys resident (KV built per batch element)
    kc = torch.empty((1 if select_only else B, H_kv, T, D), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kt = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device=dev)
    for b in range(B):
        kn = torch.empty((1, H_kv, T, D), dtype=torch.bfloat16, device=dev)
        vn = torch.empty_like(kn)
        for h in range(H_kv):
            kn[0, h], vn[0, h] = wl.kv_pair(sh, 0, b * H_kv + h, planted[0, b * H_kv + h], dev)
        cb = 0 if select_only else b
        binding.sparse_pool_append(kc[cb:cb + 1], vc[cb:cb + 1], kt[b:b + 1], kn, vn, 0)
    del kn, vn
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    idx = torch.empty((B, H_kv, k_cap), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H_kv), dtype=torch.int32, device=dev)
    O = torch.empty((B, H_q, D), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.ones(max(1, args.flush_mb) << 20 >> 2, dtype=torch.int32, device=dev)
    ws = None if args.no_workspace else binding.decode_workspace(B, H_q, H_kv, k_cap, args.n_split, device=dev)
    sel_ms, att_ms, fus_ms, hds_ms = [], [], [], []
    idx2, cnt2 = torch.empty_like(idx), torch.empty_like(cnt)
    idx3, cnt3 = torch.empty_like(idx), torch.empty_like(cnt)
    for i in range(args.warmup + args.steps):
        F = wl.forecast(sh, 0, i, dev)
        Q = wl.queries(sh, i, dev)
        torch.cuda.synchronize(dev)
        l2_evict(flush)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        binding.sparse_select_topk(F, kt, seq, sh.n_init, sh.n_local, sh.k, idx, cnt, status=status)
        e[1].record()
        torch.cuda.synchronize(dev)
        l2_evict(flush)
        e3 = torch.cuda.Event(enable_timing=True)
        e3.record()
        if not select_only:
            binding.sparse_decode_attn(Q, kc, vc, idx, cnt, seq, O, status=status, n_split=args.n_split,
                                       workspace=ws, flags=attn_flags(args))
        e[2].record()
        # one fused layer: this layer's attention and the selection from the same keys
        torch.cuda.synchronize(dev)
        l2_evict(flush)
        e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e4.record()
        if not select_only:
            binding.sparse_decode_attn_forecast(Q, kc, vc, idx, cnt, seq, O, F=F, ktil_next=kt, n_init=sh.n_init,
                                                n_local=sh.n_local, k=sh.k, idx_next=idx2, count_next=cnt2,
                                                n_split=args.n_split, status=status)
        e5.record()
        # the multi-head (InfLLM-V2) selector on the same compressed keys, for comparison
        torch.cuda.synchronize(dev)
        l2_evict(flush)
        e6, e7 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e6.record()
        binding.sparse_select_topk_heads(Q, kt, seq, sh.n_init, sh.n_local, sh.k, idx3, cnt3, status=status)
        e7.record()
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            hds_ms.append(e6.elapsed_time(e7))
            sel_ms.append(e[0].elapsed_time(e[1]))
            att_ms.append(e3.elapsed_time(e[2]))
            fus_ms.append(e4.elapsed_time(e5))
    assert status.item() == 0
    peak, src = measured_peaks()
    attn_bytes = sh.pairs * sh.k_tot * KV_BLOCK_BYTES
    sel_bytes = sh.pairs * n_candidates(sh) * KTIL_ROW_BYTES
    a, s_ = max(1e-6, statistics.median(att_ms)), statistics.median(sel_ms)
    f_ = max(1e-6, statistics.median(fus_ms)) if fus_ms else 1e-6
    h_ = statistics.median(hds_ms)
    if not select_only:
        assert torch.equal(idx2, idx) and torch.equal(cnt2, cnt), "fused selection differs from sparse_select_topk"
    line = {"case": "decode_128k_one_layer", "T": T, "steps": args.steps, "n_split": args.n_split,
            "attn_us": round(a * 1e3, 2), "attn_gbs": round(attn_bytes / a / 1e6, 1),
            "attn_frac": round(attn_bytes / a / 1e6 / peak, 4),
            "select_us": round(s_ * 1e3, 2), "select_gbs": round(sel_bytes / s_ / 1e6, 1),
            "select_frac": round(sel_bytes / s_ / 1e6 / peak, 4),
            "heads_select_us": round(h_ * 1e3, 2), "heads_over_forecast": round(h_ / s_, 3),
            "fused_us": round(f_ * 1e3, 2), "fused_gbs": round((attn_bytes + sel_bytes) / f_ / 1e6, 1),
            "fused_frac": round((attn_bytes + sel_bytes) / f_ / 1e6 / peak, 4),
            "peak_gbs": peak, "peak_source": src, "attention_contraction": contraction_name(args)}
    if select_only:   # only the selectors ran
        for key in ("attn_us", "attn_gbs", "attn_frac", "fused_us", "fused_gbs", "fused_frac"):
            line.pop(key)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- the other workloads
# One JSON line each (not the bench line): the 4K single layer, the 32K append step,
# grouped verification at 64K and the offloaded 128K decode.  Every timed iteration
# follows a 512 MB read that evicts L2 (these working sets fit in L2).


def _event_times(fn, steps, warmup, evict=None):
    """Per-iteration device time of fn() (CUDA events on the current stream), µs.  Each
    iteration starts from an idle GPU: synchronize, the L2-evicting read, during which
    the host enqueues fn's launches, so the events bracket GPU work only."""
    import torch
    pairs = []
    for i in range(warmup + steps):
        torch.cuda.synchronize()
        if evict is not None:
            l2_evict(evict)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        if i >= warmup:
            pairs.append((a, b))
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in pairs)
    q = lambda f: us[min(len(us) - 1, int(f * len(us)))]
    # the events of this GPU tick in steps of about a microsecond: the median sits on a
    # tick, the mean resolves finer
    return {"median_us": round(statistics.median(us), 2), "mean_us": round(statistics.mean(us), 2),
            "p10_us": round(q(0.1), 2), "p90_us": round(q(0.9), 2), "iterations": len(us)}


def _rate(nbytes, t_us, peak):
    gbs = nbytes / (t_us * 1e-6) / 1e9
    return round(gbs, 1), round(gbs / peak, 4)


def case_roofline(kernel, nbytes, t_us, peak, peak_src, traffic=None, note=None):
    """The roofline object of a case line: algorithmic bytes of one timed call over its
    median CUDA-event time, against the measured HBM copy bandwidth."""
    gbs = nbytes / (t_us * 1e-6) / 1e9
    out = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
           "traffic": traffic, "kernel": kernel, "algorithmic_bytes": int(nbytes), "median_us": t_us,
           "peak_source": peak_src}
    if note:
        out["note"] = note
    return out


def oracle_baseline(fn, seconds, units_per_call, unit, sample, min_reps=2):
    """The oracle (as it stands) on the host cores: fn() runs one bounded sample of the
    case's work in fp64, repeated for at least `seconds` of host time; value = units per second,
    the sample scaled by units_per_call (the part of the case's unit of work it is)."""
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    spent, reps = 0.0, 0
    while spent < seconds or reps < min_reps:
        t0 = time.perf_counter()
        fn()
        spent += time.perf_counter() - t0
        reps += 1
    per_call = spent / reps
    return {"value": round(units_per_call / per_call, 6), "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{sample}; {reps} timed calls, {spent:.1f} s, {per_call * 1e3:.2f} ms per call"}


class _Layer:
    """One decode layer on the device: cache, compressed keys, block lists, output."""

    def __init__(self, sh, dev, use_workspace=False, attn_flags=0):
        import torch
        from block_sparse_long_pool_gb300 import binding
        from block_sparse_long_pool_gb300 import workloads as wl
        self.sh, self.binding = sh, binding
        x = self.x = wl.single_layer(sh, dev)
        B, H_kv, H_q = sh.B, sh.H_kv, sh.H_q
        self.k_cache = torch.zeros_like(x["K"])
        self.v_cache = torch.zeros_like(x["V"])
        self.ktil = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device=dev)
        # bulk append of the cached tokens builds the compressed keys
        binding.sparse_pool_append(self.k_cache, self.v_cache, self.ktil, x["K"][:, :, :sh.T].contiguous(),
                                   x["V"][:, :, :sh.T].contiguous(), 0)
        self.F, self.Q = x["F"], x["Q"]
        self.k_new, self.v_new = x.get("k_new"), x.get("v_new")
        self.len_after = sh.len_after
        self.seq = torch.full((B,), sh.len_after, dtype=torch.int32, device=dev)
        self.idx = torch.empty((B, H_kv, sh.k_tot), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((B, H_kv), dtype=torch.int32, device=dev)
        self.O = torch.empty((B, H_q, D), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = binding.decode_workspace(B, H_q, H_kv, sh.k_tot, device=dev) if use_workspace else None
        self.attn_flags = attn_flags

    def step(self):
        sh, bd = self.sh, self.binding
        if sh.n_new > 0:
            # the same token written at the same position every step: the step is idempotent
            bd.sparse_pool_append(self.k_cache, self.v_cache, self.ktil, self.k_new, self.v_new, sh.T)
        # the append writes only the block of the new token, a local block: the selection
        # streams the candidates' keys while it runs
        local_only = sh.n_new > 0 and sh.T // BLK >= sh.N_b - sh.n_local
        bd.sparse_select_topk(self.F, self.ktil, self.seq, sh.n_init, sh.n_local, sh.k, self.idx, self.cnt,
                              status=self.status, flags=bd.SPARSE_SELECT_KEYS_READY if local_only else 0)
        bd.sparse_decode_attn(self.Q, self.k_cache, self.v_cache, self.idx, self.cnt, self.seq, self.O,
                              workspace=self.ws, status=self.status, flags=self.attn_flags)


def single_layer_oracle(lay, seconds):
    """The oracle on one decode step of a single-layer workload, all pairs: the
    compressed key of the block the appended token lands in (when the step appends),
    the Forecast selection and the attention, in fp64.  The compressed keys of the
    other blocks are resident (pooled outside the timing)."""
    import numpy as np
    import oracle
    from block_sparse_long_pool_gb300 import workloads as wl
    sh, x = lay.sh, lay.x
    P = sh.pairs
    K = wl.bf16_bits(x["K"]).reshape(P, sh.T_cap, D).copy()
    V = wl.bf16_bits(x["V"]).reshape(P, sh.T_cap, D).copy()
    if sh.n_new:
        K[:, sh.T:sh.len_after] = wl.bf16_bits(x["k_new"]).reshape(P, sh.n_new, D)
        V[:, sh.T:sh.len_after] = wl.bf16_bits(x["v_new"]).reshape(P, sh.n_new, D)
    lens = [sh.len_after] * P
    ktil = oracle.pool(K, lens, sh.N_b)
    F = wl.bf16_bits(x["F"]).reshape(P, D)
    Q = wl.bf16_bits(x["Q"]).reshape(P, sh.G, D)
    j0 = sh.T // BLK                     # the block the appended tokens land in
    blk = np.ascontiguousarray(K[:, j0 * BLK:(j0 + 1) * BLK]) if sh.n_new else None

    def step():
        if sh.n_new:
            oracle.pool(blk, [sh.len_after - j0 * BLK] * P, 1)
        idx, cnt, _ = oracle.select(F, ktil, lens, sh.n_init, sh.n_local, sh.k)
        oracle.attn(Q, K, V, idx, cnt, lens)
    what = ("append (the touched block's mean) + " if sh.n_new else "") + "select + attention"
    return oracle_baseline(step, seconds, 1.0, "steps/s", f"the whole step ({what}) of all {P} pairs in fp64")


def run_single_layer_case(args, dev, sh, name):
    import torch
    peak, src = measured_peaks()
    lay = _Layer(sh, dev, use_workspace=args.workspace, attn_flags=attn_flags(args))
    evict = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)
    with ClockSampler(dev.index or 0) as clk:
        t = _event_times(lay.step, args.steps, args.warmup, evict)
    torch.cuda.synchronize()
    assert lay.status.item() == 0, f"device status {lay.status.item()}"
    kv = sh.pairs * sh.k_tot * KV_BLOCK_BYTES
    sel = sh.pairs * n_candidates(sh) * KTIL_ROW_BYTES
    # append: new K/V rows read and written, the touched compressed key read and written
    app = sh.pairs * (sh.n_new * 2 * 2 * D * 2 + 2 * KTIL_ROW_BYTES) if sh.n_new else 0
    gbs, frac = _rate(kv + sel + app, t["median_us"], peak)
    launches = 3 if sh.n_new else 2
    line = {"case": name, "workload": sh.name, "decode_path": "split (workspace)" if args.workspace else "cluster",
            "attention_contraction": contraction_name(args),
            "unit_of_work": "one decode step (" +
            ("append + " if sh.n_new else "") + "select + attention)",
            "steps_per_s": round(1e6 / t["median_us"], 1), **t, "launches_per_step": launches,
            "algorithmic_bytes": {"selected_kv": kv, "compressed_keys": sel, "append": app},
            "achieved_gbs": gbs, "frac_of_measured_hbm": frac, "peak_gbs": peak, "peak_source": src,
            "roofline": case_roofline(f"the step's {launches} launches (" + ("pool_append_kernel, " if sh.n_new
                                      else "") + "decode_forecast_kernel<1, false>, sparse_attn_kernel)",
                                      kv + sel + app, t["median_us"], peak, src),
            "l2": "512 MB read evicts L2 before each step", "clocks": clk.summary(),
            "cpu_baseline": None if args.no_cpu_baseline else single_layer_oracle(lay, args.case_cpu_seconds)}
    print(json.dumps(line), flush=True)


def contraction_name(args):
    return "tcgen05.mma, tensor-memory accumulators" if getattr(args, "tensor_memory", False) else "mma.sync"


def attn_flags(args):
    """The attention calls' flag bits a case line's options ask for."""
    from block_sparse_long_pool_gb300 import binding
    return binding.SPARSE_ATTN_TENSOR_MEMORY if getattr(args, "tensor_memory", False) else 0


def run_verify_case(args, dev):
    import torch
    from block_sparse_long_pool_gb300 import binding
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wl.VERIFY_64K
    peak, src = measured_peaks()
    x = wl.verify_inputs(sh, dev)
    O = torch.empty_like(x["Q"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    evict = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)
    out = {"case": "verify64k", "workload": sh.name, "attention_contraction": contraction_name(args),
           "unit_of_work": "one verification round "
           f"({sh.N_q} queries x {sh.B * sh.H_kv} pairs)", "peak_gbs": peak, "peak_source": src,
           "l2": "512 MB read evicts L2 before each round"}
    clk = ClockSampler(dev.index or 0).__enter__()
    for C, key, shared in ((sh.C, "grouped", False), (1, "ungrouped", False), (sh.C, "shared_layout", True)):
        loaded = torch.zeros(1, dtype=torch.int64, device=dev)

        def run():
            binding.sparse_verify_attn_grouped(x["Q"], x["K"], x["V"], x["I"], C, sh.window_blocks, x["seq_len"], O,
                                               status=status, shared=shared, n_split=args.n_split,
                                               flags=attn_flags(args))
        binding.sparse_verify_attn_grouped(x["Q"], x["K"], x["V"], x["I"], C, sh.window_blocks, x["seq_len"], O,
                                           blocks_loaded=loaded, status=status, shared=shared, n_split=args.n_split,
                                           flags=attn_flags(args))
        t = _event_times(run, args.steps, args.warmup, evict)
        nbytes = int(loaded.item()) * KV_BLOCK_BYTES
        gbs, frac = _rate(nbytes, t["median_us"], peak)
        out[key] = {"C": C, "mode": "B (first query's layout)" if shared else "A (merged union)",
                    "blocks_loaded": int(loaded.item()), "bytes_loaded": nbytes, **t,
                    "achieved_gbs": gbs, "frac_of_measured_hbm": frac}
    # a model's verification round: 32 layers back to back in one CUDA graph (programmatic
    # dependent launch overlaps each launch's start with the previous one's end), over
    # 4 physical KV layers of 1.07 GB each (reuse distance far beyond L2)
    layers, phys = 32, 4
    Ks, Vs = [x["K"]], [x["V"]]
    for q_ in range(1, phys):
        Ks.append(wl.randn_bf16(tuple(x["K"].shape), wl._subseed(sh.seed, 90, q_), dev))
        Vs.append(wl.randn_bf16(tuple(x["V"].shape), wl._subseed(sh.seed, 91, q_), dev))
    cur = torch.cuda.current_stream(dev)
    for key, shared in (("grouped", False), ("shared_layout", True)):
        g_ = torch.cuda.CUDAGraph()
        s_ = torch.cuda.Stream(device=dev)
        s_.wait_stream(cur)
        with torch.cuda.graph(g_, stream=s_):
            for l in range(layers):
                # the lists are the round's own (routed before it): the union and the
                # K/V stream of layer l overlap the drain of layer l - 1
                binding.sparse_verify_attn_grouped(x["Q"], Ks[l % phys], Vs[l % phys], x["I"], sh.C, sh.window_blocks,
                                                   x["seq_len"], O, status=status, shared=shared, stream=s_,
                                                   n_split=args.n_split,
                                                   flags=binding.SPARSE_ATTN_BLOCKS_READY | attn_flags(args))
        for _ in range(2):
            g_.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps // 10)
        a.record()
        for _ in range(reps):
            g_.replay()
        b.record()
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(b) * 1e3 / (reps * layers)
        gbs, frac = _rate(out[key]["bytes_loaded"], us, peak)
        out[key]["chained"] = {"layers": layers, "physical_kv_layers": phys, "avg_launch_us": round(us, 2),
                               "achieved_gbs": gbs, "frac_of_measured_hbm": frac,
                               "rounds_per_s": round(1e6 / (us * layers), 1)}
    # the baseline of the SSV notes' kernel comparison: one decode-attention launch per
    # verification query, each over its own blocks and the window (no grouping)
    nb = (sh.T + BLK - 1) // BLK
    W = torch.arange(nb - sh.window_blocks, nb, dtype=torch.int32, device=dev)
    lists = [torch.cat([x["I"][:, :, q], W.expand(sh.B, sh.H_kv, sh.window_blocks)], dim=-1).sort(dim=-1).values
             .contiguous() for q in range(sh.N_q)]
    cnt_q = torch.full((sh.B, sh.H_kv), lists[0].shape[-1], dtype=torch.int32, device=dev)
    Qs = [x["Q"][:, q].contiguous() for q in range(sh.N_q)]
    Os = [torch.empty_like(Qs[0]) for _ in range(sh.N_q)]

    def per_query():
        for q in range(sh.N_q):
            binding.sparse_decode_attn(Qs[q], x["K"], x["V"], lists[q], cnt_q, x["seq_len"], Os[q], status=status,
                                       flags=attn_flags(args))
    t = _event_times(per_query, args.steps, args.warmup, evict)
    out["per_query_decode"] = {"launches": sh.N_q, **t,
                               "blocks_requested": sh.N_q * sh.B * sh.H_kv * int(lists[0].shape[-1]),
                               "grouped_speedup": round(t["median_us"] / out["grouped"]["median_us"], 3),
                               "shared_layout_speedup": round(t["median_us"] / out["shared_layout"]["median_us"], 3),
                               "note": "one sparse_decode_attn launch per verification query over its blocks and "
                                       "the window, back to back on one stream"}
    assert status.item() == 0, f"device status {status.item()}"
    g, u = out["grouped"], out["ungrouped"]
    out["bytes_ratio"] = round(g["bytes_loaded"] / u["bytes_loaded"], 4)
    out["bytes_ratio_bound"] = round((1 + (sh.C - 1) * (1 - sh.gamma)) / sh.C, 4)
    out["time_ratio"] = round(g["median_us"] / u["median_us"], 4)
    clk.__exit__(None, None, None)
    out["clocks"] = clk.summary()
    out["roofline"] = case_roofline("sparse_attn_kernel<2, true> (sparse_verify_attn_grouped, C = 4, G = 4)",
                                    g["bytes_loaded"], g["median_us"], peak, src,
                                    note="bytes = the blocks the grouped launch loads (blocks_loaded x 32 KB)")
    if not args.no_cpu_baseline:
        import oracle
        Qb, Kb, Vb = wl.bf16_bits(x["Q"]), wl.bf16_bits(x["K"]), wl.bf16_bits(x["V"])
        I = x["I"].cpu().numpy()
        out["cpu_baseline"] = oracle_baseline(
            lambda: oracle.verify(Qb, Kb, Vb, I, sh.C, sh.window_blocks, [sh.T] * sh.B), args.case_cpu_seconds,
            1.0, "rounds/s", f"the whole round (mode A, C = {sh.C}: {sh.N_q} queries x {sh.B * sh.H_kv} pairs) in fp64")
    else:
        out["cpu_baseline"] = None
    print(json.dumps(out), flush=True)


class Offload128k:
    """The offloaded 128K decode: K/V of every layer in pinned host memory, compressed
    keys resident, selected blocks gathered one layer ahead into a two-slot HBM ring."""

    def __init__(self, dev, layers=0):
        import dataclasses
        import torch
        from block_sparse_long_pool_gb300 import binding
        from block_sparse_long_pool_gb300 import workloads as wl
        self.torch, self.binding, self.dev = torch, binding, dev
        sh = self.sh = (dataclasses.replace(wl.OFFLOAD_128K, layers=layers, phys_layers=layers) if layers > 0
                        else wl.OFFLOAD_128K)
        B, H_kv, H_q, T, L = sh.B, sh.H_kv, sh.H_q, sh.T, sh.layers
        planted = wl.planted_sets(sh, L)
        self.k_host, self.v_host, self.ktil = [], [], []
        kc = torch.empty((B, H_kv, T, D), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        for l in range(L):
            kn = torch.empty_like(kc)
            vn = torch.empty_like(kc)
            for p in range(sh.pairs):
                b, h = divmod(p, H_kv)
                kn[b, h], vn[b, h] = wl.kv_pair(sh, l, p, planted[l, p], dev)
            kt = torch.zeros((B, H_kv, sh.N_b, D), dtype=torch.float32, device=dev)
            binding.sparse_pool_append(kc, vc, kt, kn, vn, 0)
            del kn, vn
            kh = torch.empty(kc.shape, dtype=torch.bfloat16, pin_memory=True)
            vh = torch.empty(kc.shape, dtype=torch.bfloat16, pin_memory=True)
            kh.copy_(kc)
            vh.copy_(vc)
            self.k_host.append(kh)
            self.v_host.append(vh)
            self.ktil.append(kt)
        del kc, vc
        self.Q = torch.stack([wl.queries(sh, l, dev) for l in range(L)])
        self.F = torch.stack([wl.forecast(sh, (l + 1) % L, l, dev) for l in range(L)])
        self.F0 = wl.forecast(sh, 0, -1, dev)
        kt_ = sh.k_tot
        self.k_ring = torch.zeros((2, B, H_kv, kt_, BLK, D), dtype=torch.bfloat16, device=dev)
        self.v_ring = torch.zeros_like(self.k_ring)
        self.slots = torch.arange(kt_, dtype=torch.int32, device=dev).repeat(B, H_kv, 1).contiguous()
        self.idx = torch.full((L, B, H_kv, kt_), -1, dtype=torch.int32, device=dev)
        self.count = torch.zeros((L, B, H_kv), dtype=torch.int32, device=dev)
        self.O = torch.zeros((L, B, H_q, D), dtype=torch.bfloat16, device=dev)
        self.seq = torch.full((B,), T, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self.copy = torch.cuda.Stream(device=dev)
        self.ws = binding.decode_workspace(B, H_q, H_kv, kt_, device=dev)
        torch.cuda.synchronize(dev)

    def link_bytes_per_layer(self):
        return self.sh.pairs * self.sh.k_tot * KV_BLOCK_BYTES

    def _select(self, l, F, stream):
        sh = self.sh
        self.binding.sparse_select_topk(F, self.ktil[l], self.seq, sh.n_init, sh.n_local, sh.k, self.idx[l],
                                        self.count[l], status=self.status, stream=stream)

    def _gather(self, l, stream):
        s = l % 2
        self.binding.sparse_gather_offloaded(self.k_host[l], self.v_host[l], self.idx[l], self.count[l],
                                             self.k_ring[s], self.v_ring[s], status=self.status, stream=stream)

    def _attend(self, l, stream):
        s = l % 2
        self.binding.sparse_decode_attn(self.Q[l], self.k_ring[s], self.v_ring[s], self.idx[l], self.count[l],
                                        self.seq, self.O[l], blk_slot=self.slots, status=self.status,
                                        flags=self.binding.SPARSE_ATTN_BLOCKS_READY, workspace=self.ws,
                                        stream=stream)

    def enqueue_step(self):
        torch = self.torch
        main = torch.cuda.current_stream(self.dev)
        L = self.sh.layers
        ev = lambda st: (lambda e: (e.record(st), e)[1])(torch.cuda.Event())
        self.side.wait_stream(main)
        self.copy.wait_stream(main)
        self._select(0, self.F0, self.side)
        self.copy.wait_event(ev(self.side))
        self._gather(0, self.copy)
        staged = [None] * L
        staged[0] = ev(self.copy)
        attn_done = [None] * L
        for l in range(L):
            if l + 1 < L:
                if l >= 1:
                    self.side.wait_event(attn_done[l - 1])    # F_l exists once layer l runs
                self._select(l + 1, self.F[l], self.side)
                self.copy.wait_event(ev(self.side))
                if l >= 1:
                    self.copy.wait_event(attn_done[l - 1])    # ring slot (l+1) % 2 is free again
                self._gather(l + 1, self.copy)
                staged[l + 1] = ev(self.copy)
            main.wait_event(staged[l])
            self._attend(l, main)
            attn_done[l] = ev(main)
        main.wait_stream(self.side)
        main.wait_stream(self.copy)


def run_offload_case(args, dev):
    import torch
    peak, src = measured_peaks()
    t0 = time.time()
    wk = Offload128k(dev, args.layers)
    setup_s = time.time() - t0
    sh = wk.sh
    # the link: one large pinned host -> device copy, and the gather kernel alone
    src_h = wk.k_host[0]
    dst = torch.empty(src_h.shape, dtype=src_h.dtype, device=dev)
    for _ in range(2):
        dst.copy_(src_h, non_blocking=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    reps = 4
    for _ in range(reps):
        dst.copy_(src_h, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    memcpy_gbs = reps * src_h.numel() * 2 / (a.elapsed_time(b) * 1e-3) / 1e9
    del dst
    wk._select(1, wk.F[0], torch.cuda.current_stream())
    evict = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)   # L2 may hold host lines too
    g = _event_times(lambda: wk._gather(1, torch.cuda.current_stream()), max(10, args.steps // 4), 3, evict)
    del evict
    gather_gbs = wk.link_bytes_per_layer() / (g["median_us"] * 1e-6) / 1e9
    # the 32-layer step as a CUDA graph
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        wk.enqueue_step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        wk.enqueue_step()
    steps = max(3, args.steps // 20)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        a.record()
        for _ in range(steps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
    assert wk.status.item() == 0, f"device status {wk.status.item()}"
    ms = a.elapsed_time(b) / steps
    link_step = sh.layers * wk.link_bytes_per_layer()
    hbm_step = sh.layers * (sh.pairs * n_candidates(sh) * KTIL_ROW_BYTES + 2 * wk.link_bytes_per_layer())
    line = {"case": "offload128k", "workload": sh.name, "unit_of_work": f"one decode step ({sh.layers} layers of "
            "select(l+1) -> gather(l+1) on a copy stream, beside attention(l) over the ring)",
            "steps_per_s": round(1000.0 / ms, 2), "ms_per_step": round(ms, 3), "steps_timed": steps,
            "link_bytes_per_step": link_step, "link_gbs": round(link_step / (ms * 1e-3) / 1e9, 1),
            "measured_h2d_memcpy_gbs": round(memcpy_gbs, 1),
            "frac_of_measured_link": round(link_step / (ms * 1e-3) / 1e9 / memcpy_gbs, 4),
            "gather_alone": {**g, "gbs": round(gather_gbs, 1)},
            "pcie5_x16_nominal_gbs": 64.0, "hbm_bytes_per_step": hbm_step,
            "hbm_frac_of_measured": round(hbm_step / (ms * 1e-3) / 1e9 / peak, 4), "peak_gbs": peak,
            "peak_source": src, "host_kv_gb": round(2 * sh.layers * wk.k_host[0].numel() * 2 / 1e9, 1),
            "setup_s": round(setup_s, 1),
            "roofline": {"bound": "host link", "achieved": round(link_step / (ms * 1e-3) / 1e9, 1),
                         "peak": round(memcpy_gbs, 1), "unit": "GB/s",
                         "frac": round(link_step / (ms * 1e-3) / 1e9 / memcpy_gbs, 4), "traffic": None,
                         "kernel": "gather_kernel (sparse_gather_offloaded) on the copy stream",
                         "peak_source": "a pinned host -> device copy of 1 GB measured in this run"},
            "clocks": clk.summary(),
            "cpu_baseline": None if args.no_cpu_baseline else offload_oracle(wk, args.case_cpu_seconds)}
    print(json.dumps(line), flush=True)


def offload_oracle(wk, seconds):
    """The oracle on one layer of the offloaded step, all pairs: the Forecast selection
    from the resident compressed keys, the staging copy of the selected blocks from the
    host cache into a ring, and the attention over the ring, in fp64; scaled to the
    step's layers."""
    import numpy as np
    import oracle
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wk.sh
    P, l = sh.pairs, 1
    Kh = wl.bf16_bits(wk.k_host[l]).reshape(P, sh.T, D)   # views of the pinned host cache
    Vh = wl.bf16_bits(wk.v_host[l]).reshape(P, sh.T, D)
    lens = [sh.T] * P
    ktil = oracle.pool(Kh, lens, sh.N_b)
    F = wl.bf16_bits(wk.F[l - 1]).reshape(P, D)
    Q = wl.bf16_bits(wk.Q[l]).reshape(P, sh.G, D)
    ring_k = np.zeros((P, sh.k_tot, BLK, D), np.uint16)
    ring_v = np.zeros_like(ring_k)

    def layer():
        idx, cnt, _ = oracle.select(F, ktil, lens, sh.n_init, sh.n_local, sh.k)
        oracle.gather(Kh, idx, cnt, ring_k)
        oracle.gather(Vh, idx, cnt, ring_v)
        # the same rows as the ring holds (a staged copy), read where the length mask is defined
        oracle.attn(Q, Kh, Vh, idx, cnt, lens)
    return oracle_baseline(layer, seconds, 1.0 / sh.layers, "steps/s",
                           f"one layer of all {P} pairs (select + staging copy of K and V + attention) in fp64, "
                           f"scaled to {sh.layers} layers")


NSA_WINDOW_TOKENS = 512


def run_nsa_case(args, dev):
    """NSA's gated three-branch decode on the 128K decode shape (8 x 8 pairs, G = 8,
    67 selected blocks, a 512-token window): with one compressed row per 64-token block
    (2048 per pair) and with NSA's overlapping 32/16 windows (8191 per pair).  For each:
    the routing (tensor-core sparse_nsa_select on the bf16 rows) and the one-launch
    three-branch attention, timed alone and as a layer; the fp32 multi-head selector
    (sparse_select_topk_heads) on the block rows for comparison."""
    import torch
    from block_sparse_long_pool_gb300 import binding
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wl.DECODE_128K
    peak, src = measured_peaks()
    B, H_q, H_kv = sh.B, sh.H_q, sh.H_kv
    T = args.tokens if args.tokens > 0 else sh.T   # a shorter cache only for small profiling captures
    N = (T + BLK - 1) // BLK
    k_tot, w = min(sh.k_tot, N), NSA_WINDOW_TOKENS
    kc = torch.empty((B, H_kv, T, D), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    ktil = torch.zeros((B, H_kv, N, D), dtype=torch.float32, device=dev)
    vtil = torch.zeros_like(ktil)
    khat = torch.zeros((B, H_kv, N, D), dtype=torch.bfloat16, device=dev)
    vhat = torch.zeros_like(khat)
    for b in range(B):   # one batch element at a time keeps the staging small
        kn = wl.randn_bf16((1, H_kv, T, D), wl._subseed(sh.seed, 71, b), dev)
        vn = wl.randn_bf16((1, H_kv, T, D), wl._subseed(sh.seed, 72, b), dev)
        binding.sparse_pool_append_kv(kc[b:b + 1], vc[b:b + 1], ktil[b:b + 1], vtil[b:b + 1], kn, vn, 0,
                                      khat=khat[b:b + 1], vhat=vhat[b:b + 1])
        del kn, vn
    Q = wl.randn_bf16((B, H_q, D), wl._subseed(sh.seed, 73), dev)
    gates = torch.rand((B, H_q, 3), generator=wl._gen(dev, wl._subseed(sh.seed, 74)), device=dev)
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    idx = torch.empty((B, H_kv, k_tot), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H_kv), dtype=torch.int32, device=dev)
    O = torch.empty((B, H_q, D), dtype=torch.bfloat16, device=dev)
    ws = binding.nsa_workspace(B, H_q, H_kv, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    evict = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)

    def select():
        binding.sparse_select_topk_heads(Q, ktil, seq, sh.n_init, sh.n_local, sh.k, idx, cnt, status=status)

    def attend():
        binding.sparse_decode_attn_nsa(Q, kc, vc, khat, vhat, idx, cnt, seq, w, gates, O, None,
                                       n_split=args.n_split, status=status)

    def attend_grid():
        binding.sparse_decode_attn_nsa(Q, kc, vc, khat, vhat, idx, cnt, seq, w, gates, O, ws, n_split=args.n_split,
                                       flags=binding.SPARSE_NSA_BRANCH_GRID, status=status)

    def route():
        binding.sparse_nsa_select(Q, khat, seq, sh.n_init, sh.n_local, sh.k, idx, cnt, cmp=(0, 0), status=status)

    def layer():
        route()
        attend()

    # NSA's overlapping compression: kernel 32, stride 16
    wl_, ws_ = 32, 16
    R = (T - wl_) // ws_ + 1
    kw = torch.empty((B, H_kv, R, D), dtype=torch.bfloat16, device=dev)
    vw = torch.empty_like(kw)
    binding.sparse_nsa_compress(kc, vc, kw, vw, 0, T, cmp=(wl_, ws_))

    def route_w():
        binding.sparse_nsa_select(Q, kw, seq, sh.n_init, sh.n_local, sh.k, idx, cnt, cmp=(wl_, ws_), status=status)

    def attend_w():
        binding.sparse_decode_attn_nsa(Q, kc, vc, kw, vw, idx, cnt, seq, w, gates, O, None, n_split=args.n_split,
                                       status=status, cmp=(wl_, ws_))

    def layer_w():
        route_w()
        attend_w()

    select()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        t_attn = _event_times(attend, args.steps, args.warmup, evict)
        t_grid = _event_times(attend_grid, args.steps, args.warmup, evict)
        t_sel = _event_times(select, args.steps, args.warmup, evict)
        t_route = _event_times(route, args.steps, args.warmup, evict)
        t_layer = _event_times(layer, args.steps, args.warmup, evict)
        t_route_w = _event_times(route_w, args.steps, args.warmup, evict)
        t_attn_w = _event_times(attend_w, args.steps, args.warmup, evict)
        t_layer_w = _event_times(layer_w, args.steps, args.warmup, evict)
        torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    pairs = B * H_kv
    w_blocks = (w + BLK - 1) // BLK
    nbytes = {"selected_kv": pairs * k_tot * KV_BLOCK_BYTES, "window_kv": pairs * w_blocks * KV_BLOCK_BYTES,
              "compressed_rows": pairs * N * 2 * D * 2, "q_o_gates": B * H_q * (2 * D * 2 + 12)}
    attn_bytes = sum(nbytes.values())
    gbs, frac = _rate(attn_bytes, t_attn["median_us"], peak)
    ggbs, gfrac = _rate(attn_bytes, t_grid["median_us"], peak)
    sel_bytes = pairs * N * KTIL_ROW_BYTES
    sgbs, sfrac = _rate(sel_bytes, t_sel["median_us"], peak)
    route_bytes = pairs * N * D * 2
    rgbs, rfrac = _rate(route_bytes, t_route["median_us"], peak)
    lgbs, lfrac = _rate(attn_bytes + route_bytes, t_layer["median_us"], peak)
    wbytes = dict(nbytes, compressed_rows=pairs * R * 2 * D * 2)
    attn_w_bytes = sum(wbytes.values())
    route_w_bytes = pairs * R * D * 2
    awgbs, awfrac = _rate(attn_w_bytes, t_attn_w["median_us"], peak)
    rwgbs, rwfrac = _rate(route_w_bytes, t_route_w["median_us"], peak)
    lwgbs, lwfrac = _rate(attn_w_bytes + route_w_bytes, t_layer_w["median_us"], peak)
    line = {"case": "nsa128k", "workload": f"nsa_decode_{T // 1024}k_b{B}_hq{H_q}_hkv{H_kv}_w{w}",
            "unit_of_work": "one NSA decode layer (multi-head routing + gated three-branch attention)",
            "attention": {"form": "fused (one cluster per pair, three branch states, one DSMEM merge)",
                          "launches": 1, **t_attn, "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
                          "frac_of_measured_hbm": frac},
            "attention_branch_grid": {"form": "a cluster per branch and pair, gates from the workspace",
                                      "launches": 1, **t_grid, "achieved_gbs": ggbs, "frac_of_measured_hbm": gfrac},
            "routing": {"call": "sparse_nsa_select (bf16 block rows, tensor cores)", **t_route,
                        "algorithmic_bytes": route_bytes, "achieved_gbs": rgbs, "frac_of_measured_hbm": rfrac},
            "routing_fp32_multi_head": {"call": "sparse_select_topk_heads (fp32 block rows)", **t_sel,
                                        "algorithmic_bytes": sel_bytes, "achieved_gbs": sgbs,
                                        "frac_of_measured_hbm": sfrac},
            "layer": {**t_layer, "achieved_gbs": lgbs, "frac_of_measured_hbm": lfrac,
                      "layers_per_s": round(1e6 / t_layer["median_us"], 1)},
            "windows_32_16": {
                "compressed_rows_per_pair": R,
                "routing": {**t_route_w, "algorithmic_bytes": route_w_bytes, "achieved_gbs": rwgbs,
                            "frac_of_measured_hbm": rwfrac},
                "attention": {**t_attn_w, "algorithmic_bytes": wbytes, "achieved_gbs": awgbs,
                              "frac_of_measured_hbm": awfrac},
                "layer": {**t_layer_w, "achieved_gbs": lwgbs, "frac_of_measured_hbm": lwfrac,
                          "layers_per_s": round(1e6 / t_layer_w["median_us"], 1)}},
            "peak_gbs": peak, "peak_source": src, "l2": "512 MB read evicts L2 before each timed call",
            "roofline": case_roofline("nsa_fused_kernel (sparse_decode_attn_nsa, block rows, G = 8)", attn_bytes,
                                      t_attn["median_us"], peak, src),
            "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle
        G = H_q // H_kv
        lens = [T] * H_kv
        Kb = wl.bf16_bits(kc[0]).reshape(H_kv, T, D)
        Vb = wl.bf16_bits(vc[0]).reshape(H_kv, T, D)
        kh64 = khat[0].float().double().cpu().numpy()
        vh64 = vhat[0].float().double().cpu().numpy()
        Qb = wl.bf16_bits(Q[0]).reshape(H_kv, G, D)
        gt = gates[0].double().cpu().numpy().reshape(H_kv, G, 3)

        def nsa_layer():
            ridx, rcnt, _ = oracle.select_windows(Qb, kh64, lens, BLK, BLK, sh.n_init, sh.n_local, sh.k, k_tot)
            oracle.nsa(Qb, Kb, Vb, kh64, vh64, ridx, rcnt, lens, w, gt)
        line["cpu_baseline"] = oracle_baseline(
            nsa_layer, args.case_cpu_seconds, 1.0 / B, "layers/s",
            f"batch element 0 ({H_kv} pairs) of one layer with block rows: the routing (per-head softmax over "
            f"the rows, summed, top-k) and the gated three-branch attention in fp64, scaled to {B} batch elements")
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


def run_prefill_case(args, dev):
    """The Forecast selection of every prefill position (SparDA notes eq.(16)) on the
    32K prefill shape: B = 4, H_kv = 8 (G = 4), 32768 positions, 512 compressed keys,
    k = 32.  One sparse_prefill_select launch per step."""
    import torch
    from block_sparse_long_pool_gb300 import binding
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wl.PREFILL_32K
    peak, src = measured_peaks()
    x = wl.prefill_inputs(sh, dev)
    B, H_kv, T, N = sh.B, sh.H_kv, sh.T, sh.N_b
    idx = torch.empty((B, H_kv, T, sh.k_tot), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H_kv, T), dtype=torch.int32, device=dev)
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    evict = torch.ones(512 << 20 >> 2, dtype=torch.int32, device=dev)

    def run():
        binding.sparse_prefill_select(x["F"], x["ktil"], seq, sh.n_init, sh.n_local, sh.k, idx, cnt, status=status)

    with ClockSampler(dev.index or 0) as clk:
        t = _event_times(run, args.steps, args.warmup, evict)
        torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    pairs = B * H_kv
    # scores: position t scores the candidates of the blocks it sees (causal)
    cand = sum(max(0, min(qb + 1 - sh.n_local, qb + 1) - sh.n_init) * min(BLK, T - qb * BLK)
               for qb in range(N))
    macs = pairs * cand * D
    nbytes = pairs * (T * D * 2 + N * D * 4 + T * (sh.k_tot + 1) * 4)
    sec = t["median_us"] * 1e-6
    tf = 2 * macs / sec / 1e12
    line = {"case": "prefill32k", "workload": sh.name, "unit_of_work": "the selection of all 32768 positions of "
            f"{pairs} (batch, KV head) pairs", **t, "positions_per_s": round(pairs * T / sec, 1),
            "scores": pairs * cand, "score_tflops": round(tf, 2),
            "score_tflops_note": "2 x (F . K~ multiply-adds); the kernel issues three bf16 mma per product "
                                 "(fp32 keys split into three bf16 terms)",
            "algorithmic_bytes": nbytes, "achieved_gbs": round(nbytes / sec / 1e9, 1),
            "frac_of_measured_hbm": round(nbytes / sec / 1e9 / peak, 4), "peak_gbs": peak, "peak_source": src,
            "l2": "512 MB read evicts L2 before each launch",
            "roofline": case_roofline("prefill_select_kernel (sparse_prefill_select)", nbytes, t["median_us"], peak,
                                      src, note="the kernel is instruction-bound by the per-position top-k "
                                                "(ncu: issue active ~60 %), not by its bytes"),
            "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle
        n_p, stride = 16, 16                 # 16 pairs (one thread each), every 16th position
        Fb = wl.bf16_bits(x["F"]).reshape(pairs, T, D)[:n_p]
        kt = x["ktil"].reshape(pairs, N, D)[:n_p].double().cpu().numpy()
        rows = list(range(stride - 1, T, stride))
        line["cpu_baseline"] = oracle_baseline(
            lambda: oracle.prefill_select(Fb, kt, [T] * n_p, sh.n_init, sh.n_local, sh.k, rows=rows),
            args.case_cpu_seconds, n_p * len(rows), "positions/s",
            f"{n_p} pairs x {len(rows)} positions (every {stride}th, spanning the causal range) of the selection "
            "in fp64; value = positions per second")
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


def run_refresh_case(args, dev):
    """SSV's refresh / reuse schedule (mechanism 2) on the 64K verification shape over a
    32-layer round: a refresh layer routes the 8 verification queries of every pair on
    the layer's compressed keys (sparse_nsa_select, NSA routing, the 8 window blocks as
    the local blocks and 16 routed blocks outside them) and verifies with those lists;
    a reuse layer verifies with the lists of the last refresh layer.  Each schedule is
    one CUDA graph of the 32 layers (4 physical KV layers, 1.07 GB each)."""
    import torch
    from block_sparse_long_pool_gb300 import binding
    from block_sparse_long_pool_gb300 import workloads as wl
    sh = wl.VERIFY_64K
    peak, src = measured_peaks()
    x = wl.verify_inputs(sh, dev)
    B, H_kv, T, N = sh.B, sh.H_kv, sh.T, sh.T // BLK
    layers, phys = 32, 4
    Ks, Vs = [x["K"]], [x["V"]]
    for q_ in range(1, phys):
        Ks.append(wl.randn_bf16(tuple(x["K"].shape), wl._subseed(sh.seed, 90, q_), dev))
        Vs.append(wl.randn_bf16(tuple(x["V"].shape), wl._subseed(sh.seed, 91, q_), dev))
    # compressed keys of each physical layer: one row per 64-token block
    khs = []
    for q_ in range(phys):
        kh = torch.empty((B, H_kv, N, D), dtype=torch.bfloat16, device=dev)
        vh = torch.empty_like(kh)
        binding.sparse_nsa_compress(Ks[q_], Vs[q_], kh, vh, 0, T, cmp=(BLK, BLK))
        khs.append(kh)
    k_tot = sh.window_blocks + sh.n_sel
    idx = torch.empty((B, H_kv, sh.N_q, k_tot), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H_kv, sh.N_q), dtype=torch.int32, device=dev)
    O = torch.empty_like(x["Q"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cur = torch.cuda.current_stream(dev)

    def layer(l, refresh, st):
        if refresh:
            binding.sparse_nsa_select(x["Q"], khs[l % phys], x["seq_len"], 0, sh.window_blocks, sh.n_sel, idx, cnt,
                                      cmp=(BLK, BLK), status=status, stream=st)
        # a reuse layer's lists were routed at least two launches back (the verification
        # kernel lets its successor start only after its own wait): its union and K/V
        # stream may overlap the previous layer's drain; a refresh layer's wait for the
        # routing just before it
        binding.sparse_verify_attn_grouped(x["Q"], Ks[l % phys], Vs[l % phys], idx, sh.C, sh.window_blocks,
                                           x["seq_len"], O, status=status, stream=st,
                                           flags=0 if refresh else binding.SPARSE_ATTN_BLOCKS_READY)

    def timed(schedule):
        g_ = torch.cuda.CUDAGraph()
        s_ = torch.cuda.Stream(device=dev)
        s_.wait_stream(cur)
        with torch.cuda.graph(g_, stream=s_):
            for l in range(layers):
                layer(l, schedule(l), s_)
        for _ in range(2):
            g_.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps // 10)
        a.record()
        for _ in range(reps):
            g_.replay()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3 / reps

    clk = ClockSampler(dev.index or 0).__enter__()
    t_all = timed(lambda l: True)
    t_none = timed(lambda l: l == 0)
    out = {"case": "refresh64k", "workload": sh.name + "_32layers",
           "unit_of_work": f"one verification round: {layers} layers x {sh.N_q} queries x {B * H_kv} pairs",
           "routing": "sparse_nsa_select: G heads per group, per-head softmax over the 1024 block rows, summed; "
                      "top-16 outside the 8 window blocks",
           "all_refresh_us": round(t_all, 1), "refresh_layer_us": round(t_all / layers, 2),
           "reuse_layer_us": round((t_none - t_all / layers) / (layers - 1), 2)}
    for r in (2, 4, 8):
        t_r = timed(lambda l, r=r: l % r == 0)
        out[f"refresh_every_{r}"] = {"round_us": round(t_r, 1), "rounds_per_s": round(1e6 / t_r, 1),
                                     "speedup_vs_all_refresh": round(t_all / t_r, 3)}
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    assert status.item() == 0, f"device status {status.item()}"
    # the bytes of one layer over the last routed lists: the merged unions it loads, plus
    # (refresh) the bf16 block rows the routing reads
    loaded = torch.zeros(1, dtype=torch.int64, device=dev)
    binding.sparse_verify_attn_grouped(x["Q"], Ks[0], Vs[0], idx, sh.C, sh.window_blocks, x["seq_len"], O,
                                       blocks_loaded=loaded, status=status)
    torch.cuda.synchronize()
    reuse_bytes = int(loaded.item()) * KV_BLOCK_BYTES
    route_bytes = B * H_kv * N * D * 2
    peak, src = measured_peaks()
    out["roofline"] = case_roofline("a refresh layer: nsa_route_kernel + sparse_attn_kernel<2, true>, chained",
                                    reuse_bytes + route_bytes, out["refresh_layer_us"], peak, src,
                                    note="per layer of the all-refresh round; bytes = the routed lists' merged "
                                         "unions (blocks_loaded x 32 KB) + the block rows routed over")
    out["clocks"] = clk.summary()
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        G = sh.G
        Qb, Kb, Vb = wl.bf16_bits(x["Q"]), wl.bf16_bits(Ks[0]), wl.bf16_bits(Vs[0])
        kh64 = khs[0].float().double().cpu().numpy().reshape(B * H_kv, N, D)
        lens_p = [T] * (B * H_kv)
        Qq = [np.ascontiguousarray(Qb[:, q].reshape(B * H_kv, G, D)) for q in range(sh.N_q)]

        def refresh_layer():
            I = np.empty((B * H_kv, sh.N_q, k_tot), np.int32)
            for q in range(sh.N_q):
                I[:, q], _, _ = oracle.select_windows(Qq[q], kh64, lens_p, BLK, BLK, 0, sh.window_blocks, sh.n_sel,
                                                      k_tot)
            oracle.verify(Qb, Kb, Vb, I.reshape(B, H_kv, sh.N_q, k_tot), sh.C, sh.window_blocks, [T] * B)
        out["cpu_baseline"] = oracle_baseline(
            refresh_layer, args.case_cpu_seconds, 1.0 / layers, "rounds/s",
            f"one refresh layer ({sh.N_q} queries x {B * H_kv} pairs routed over the block rows, then verified, "
            f"mode A) in fp64, scaled to an all-refresh round of {layers} layers")
    else:
        out["cpu_baseline"] = None
    print(json.dumps(out), flush=True)


OTHER_CASES = ("decode128k_b1", "single4k", "append32k", "verify64k", "offload128k", "nsa128k", "prefill32k",
               "refresh64k")


def run_other_case(args, local_rank):
    import torch
    from block_sparse_long_pool_gb300 import workloads as wl
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    if args.case == "single4k":
        run_single_layer_case(args, dev, wl.SINGLE_4K, "single4k")
    elif args.case == "append32k":
        run_single_layer_case(args, dev, wl.LLAMA8B_32K, "append32k")
    elif args.case == "verify64k":
        run_verify_case(args, dev)
    elif args.case == "nsa128k":
        run_nsa_case(args, dev)
    elif args.case == "prefill32k":
        run_prefill_case(args, dev)
    elif args.case == "refresh64k":
        run_refresh_case(args, dev)
    else:
        run_offload_case(args, dev)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["step", "layer", "select"] + list(OTHER_CASES), default="step",
                    help="step: the 80-layer decode step (the bench line); layer: one physical layer, "
                         "kernels serialised and timed alone (for profiling); select: selection only; "
                         "decode128k_b1: the 128K step at B = 1 with all 80 layers resident; "
                         "single4k / append32k / verify64k / offload128k / nsa128k / prefill32k / refresh64k: "
                         "the other workloads, one line each")
    ap.add_argument("--case-cpu-seconds", type=float, default=3.0,
                    help="other cases: host seconds of oracle work for their cpu_baseline")
    ap.add_argument("--layers", type=int, default=0,
                    help="offload128k: layers (default 32); decode128k_b1: resident physical layers (default 80); "
                         "fewer for profiling")
    ap.add_argument("--n-split", type=int, default=0)
    ap.add_argument("--no-workspace", action="store_true", help="layer case: attention without a workspace (cluster path)")
    ap.add_argument("--workspace", action="store_true",
                    help="step / single4k / append32k: attention with a workspace (split path)")
    ap.add_argument("--step-mode", choices=["fused", "separate"], default="fused",
                    help="fused: one sparse_decode_attn_forecast launch per layer; separate: sparse_select_topk "
                         "on a side stream beside sparse_decode_attn")
    ap.add_argument("--tokens", type=int, default=0, help="layer / nsa128k cases: cached tokens (default 131072)")
    ap.add_argument("--flush-mb", type=int, default=512, help="layer case: L2 flush buffer before each launch")
    ap.add_argument("--tensor-memory", action="store_true",
                    help="layer (with --no-workspace) / verify64k / single4k / append32k: the attention with "
                         "SPARSE_ATTN_TENSOR_MEMORY (tcgen05.mma, tensor-memory accumulators)")
    args = ap.parse_args()
    if args.tensor_memory and (args.workspace or (args.case == "layer" and not args.no_workspace)):
        ap.error("--tensor-memory runs the cluster path: no workspace")
    if args.warmup < 3 and args.case == "step":
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.case in ("layer", "select"):
        run_layer_case(args, local_rank)
    elif args.case == "decode128k_b1":
        run_b1_case(args, local_rank)
    elif args.case in OTHER_CASES:
        run_other_case(args, local_rank)
    elif args.impl == "reference":
        run_reference(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
