"""Thin ctypes binding of libsparsepool (include/sparse_pool.h) on torch tensors.

Argument marshalling only: every function checks dtype/device/shape/contiguity of
the tensors it is given, passes their data pointers and the current CUDA stream to
the C entry point of the same name, and raises ``SparsePoolError`` on a non-zero
status.  Every step of the computation runs in the CUDA kernels; there is no CPU
fallback, and a missing library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsparsepool.so")
_lock = threading.Lock()
_lib = None

D = 128
BLK = 64

SPARSE_OK = 0
SPARSE_ERR_INVALID_ARG = -1
SPARSE_ERR_UNSUPPORTED = -2
SPARSE_ERR_CUDA = -3
SPARSE_ERR_TIMEOUT = -4
SPARSE_ERR_NOT_READY = -5
SPARSE_ERR_BAD_INDEX = -6
SPARSE_ATTN_BLOCKS_READY = 1
SPARSE_ATTN_STREAM_K = 2
SPARSE_ATTN_TENSOR_MEMORY = 16
SPARSE_NSA_BRANCH_GRID = 4
SPARSE_SELECT_KEYS_READY = 8

# (name, restype, argtypes) of every entry point declared in include/sparse_pool.h
_P, _I, _LL, _F, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_uint
_SZ = ctypes.c_size_t
SIGNATURES = {
    "sparse_status_string": (ctypes.c_char_p, [_I]),
    "sparse_last_error": (ctypes.c_char_p, []),
    "sparse_version": (_I, []),
    "sparse_pool_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _LL, _I, _LL, _I, _P]),
    "sparse_pool_append_kv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _LL, _I, _LL, _I, _P]),
    "sparse_select_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]),
    "sparse_select_topk_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _U, _P, _P]),
    "sparse_select_topk_heads": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P, _P, _I, _P, _P]),
    "sparse_prefill_select": (_I, [_P, _LL, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]),
    "sparse_decode_attn": (_I, [_P, _P, _P, _LL, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P, _P, _I, _U, _P, _SZ,
                                _P, _P]),
    "sparse_decode_attn_ex": (_I, [_P, _P, _P, _LL, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P, _P, _I, _U, _P, _SZ,
                                   _P, _U, _LL, _P, _P]),
    "sparse_decode_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "sparse_decode_attn_noalloc": (_I, [_P, _P, _P, _LL, _P, _P, _P, _I, _P, _I, _I, _I, _F, _P, _P, _I, _U, _P,
                                        _P]),
    "sparse_decode_attn_forecast": (_I, [_P, _P, _P, _LL, _P, _P, _I, _P, _I, _I, _I, _F, _P, _P, _P, _P, _I, _I,
                                         _I, _I, _P, _P, _I, _I, _U, _P, _P]),
    "sparse_verify_attn_grouped": (_I, [_P, _P, _P, _LL, _P, _I, _I, _I, _I, _P, _I, _I, _I, _F, _P, _P, _I,
                                        _U, _P, _P]),
    "sparse_verify_attn_shared": (_I, [_P, _P, _P, _LL, _P, _I, _I, _I, _I, _P, _I, _I, _I, _F, _P, _P, _I,
                                       _U, _P, _P]),
    "sparse_gather_offloaded": (_I, [_P, _P, _LL, _P, _P, _I, _I, _I, _P, _P, _P, _I, _P, _P]),
    "sparse_decode_attn_nsa": (_I, [_P, _P, _P, _LL, _P, _P, _I, _I, _I, _P, _P, _I, _P, _I, _I, _I, _LL, _P, _F,
                                    _P, _P, _SZ, _I, _U, _P, _P]),
    "sparse_nsa_compress": (_I, [_P, _P, _LL, _I, _I, _LL, _I, _I, _I, _P, _P, _I, _P]),
    "sparse_nsa_select": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P, _P, _I, _P, _P]),
    "sparse_decode_attn_nsa_workspace_size": (_SZ, [_I, _I, _I]),
}


class SparsePoolError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def load(path: str = LIB_PATH):
    """Load libsparsepool.so (built in-tree by ``block_sparse_long_pool_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run `python -m block_sparse_long_pool_gb300.build` "
                               "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().sparse_status_string(int(status)).decode()


def _check(rc: int, name: str):
    if rc != SPARSE_OK:
        raise SparsePoolError(rc, f"{name}: {load().sparse_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device_ok=True, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device_ok and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def sparse_pool_append(k_cache, v_cache, ktil, k_new, v_new, len_before: int, stream=None):
    """Append k_new/v_new [B][H_kv][n_new][128] at len_before and update ktil."""
    B, H_kv, T_cap, _ = k_cache.shape
    n_new = k_new.shape[2]
    N_cap = ktil.shape[2]
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(v_cache, "v_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(ktil, "ktil", torch.float32, shape=(B, H_kv, N_cap, D))
    _need(k_new, "k_new", torch.bfloat16, shape=(B, H_kv, n_new, D))
    _need(v_new, "v_new", torch.bfloat16, shape=(B, H_kv, n_new, D))
    rc = load().sparse_pool_append(_ptr(k_cache), _ptr(v_cache), _ptr(ktil), _ptr(k_new), _ptr(v_new), B, H_kv,
                                   T_cap, N_cap, int(len_before), n_new, _stream(stream))
    _check(rc, "sparse_pool_append")


def sparse_pool_append_kv(k_cache, v_cache, ktil, vtil, k_new, v_new, len_before: int, khat=None, vhat=None,
                          stream=None):
    """Append k_new/v_new [B][H_kv][n_new][128] at len_before, update the pooled keys
    ktil and values vtil (fp32) and, when given, their bf16 copies khat / vhat."""
    B, H_kv, T_cap, _ = k_cache.shape
    n_new = k_new.shape[2]
    N_cap = ktil.shape[2]
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(v_cache, "v_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(ktil, "ktil", torch.float32, shape=(B, H_kv, N_cap, D))
    _need(vtil, "vtil", torch.float32, shape=(B, H_kv, N_cap, D))
    for t, n in ((khat, "khat"), (vhat, "vhat")):
        if t is not None:
            _need(t, n, torch.bfloat16, shape=(B, H_kv, N_cap, D))
    _need(k_new, "k_new", torch.bfloat16, shape=(B, H_kv, n_new, D))
    _need(v_new, "v_new", torch.bfloat16, shape=(B, H_kv, n_new, D))
    rc = load().sparse_pool_append_kv(_ptr(k_cache), _ptr(v_cache), _ptr(ktil), _ptr(vtil), _ptr(khat), _ptr(vhat),
                                      _ptr(k_new), _ptr(v_new), B, H_kv, T_cap, N_cap, int(len_before), n_new,
                                      _stream(stream))
    _check(rc, "sparse_pool_append_kv")


def sparse_select_topk(F, ktil, seq_len, n_init: int, n_local: int, k: int, idx_out, count_out,
                       status=None, stream=None, flags: int = 0):
    """Fill idx_out [B][H_kv][k_tot] and count_out [B][H_kv] from F [B][H_kv][128] and ktil.
    flags (SPARSE_SELECT_KEYS_READY) calls sparse_select_topk_ex."""
    B, H_kv, N_cap, _ = ktil.shape
    k_tot = idx_out.shape[2]
    _need(F, "F", torch.bfloat16, shape=(B, H_kv, D))
    _need(ktil, "ktil", torch.float32)
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(idx_out, "idx_out", torch.int32, shape=(B, H_kv, k_tot))
    _need(count_out, "count_out", torch.int32, shape=(B, H_kv))
    if status is not None:
        _need(status, "status", torch.int32)
    if flags:
        rc = load().sparse_select_topk_ex(_ptr(F), _ptr(ktil), _ptr(seq_len), B, H_kv, N_cap, n_init, n_local, k,
                                          _ptr(idx_out), _ptr(count_out), k_tot, int(flags), _ptr(status),
                                          _stream(stream))
        _check(rc, "sparse_select_topk_ex")
        return
    rc = load().sparse_select_topk(_ptr(F), _ptr(ktil), _ptr(seq_len), B, H_kv, N_cap, n_init, n_local, k,
                                   _ptr(idx_out), _ptr(count_out), k_tot, _ptr(status), _stream(stream))
    _check(rc, "sparse_select_topk")


def sparse_select_topk_heads(Q, ktil, seq_len, n_init: int, n_local: int, k: int, idx_out, count_out,
                             scale: float = 0.0, status=None, stream=None):
    """Multi-head (InfLLM-V2) selection: Q [B][H_q][128] bf16, ktil [B][H_kv][N_cap][128]
    fp32 -> idx_out [B][H_kv][k_tot], count_out [B][H_kv]."""
    B, H_kv, N_cap, _ = ktil.shape
    H_q = Q.shape[1]
    k_tot = idx_out.shape[2]
    _need(Q, "Q", torch.bfloat16, shape=(B, H_q, D))
    _need(ktil, "ktil", torch.float32)
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(idx_out, "idx_out", torch.int32, shape=(B, H_kv, k_tot))
    _need(count_out, "count_out", torch.int32, shape=(B, H_kv))
    if status is not None:
        _need(status, "status", torch.int32)
    rc = load().sparse_select_topk_heads(_ptr(Q), _ptr(ktil), _ptr(seq_len), B, H_q, H_kv, N_cap, float(scale),
                                         n_init, n_local, k, _ptr(idx_out), _ptr(count_out), k_tot, _ptr(status),
                                         _stream(stream))
    _check(rc, "sparse_select_topk_heads")


def _decode_args(Q, k_base, v_base, blk_logical, count, seq_len, O, lse, blk_slot):
    B, H_q, _ = Q.shape
    n_pairs, k_tot = blk_logical.shape[0] * blk_logical.shape[1], blk_logical.shape[2]
    H_kv = blk_logical.shape[1]
    pair_stride = k_base.numel() // (n_pairs * D)
    _need(Q, "Q", torch.bfloat16, shape=(B, H_q, D))
    _need(k_base, "k_base", torch.bfloat16)
    _need(v_base, "v_base", torch.bfloat16, shape=tuple(k_base.shape))
    if k_base.numel() != n_pairs * pair_stride * D:
        raise ValueError("k_base must hold B*H_kv pair regions of pair_stride x 128")
    _need(blk_logical, "blk_logical", torch.int32, shape=(B, H_kv, k_tot))
    if blk_slot is not None:
        _need(blk_slot, "blk_slot", torch.int32, shape=(B, H_kv, k_tot))
    _need(count, "count", torch.int32, shape=(B, H_kv))
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(O, "O", torch.bfloat16, shape=(B, H_q, D))
    if lse is not None:
        _need(lse, "lse", torch.float32, shape=(B, H_q))
    return B, H_q, H_kv, k_tot, pair_stride


def sparse_decode_attn_workspace_size(B: int, H_q: int, H_kv: int, k_tot: int, n_split: int = 0) -> int:
    """Bytes of the workspace of sparse_decode_attn (split and stream-K paths; 0: sizes
    that no workspace path serves)."""
    return int(load().sparse_decode_attn_workspace_size(B, H_q, H_kv, k_tot, n_split))


def decode_workspace(B: int, H_q: int, H_kv: int, k_tot: int, n_split: int = 0, device="cuda"):
    """A zeroed workspace tensor for sparse_decode_attn, or None when not needed."""
    n = sparse_decode_attn_workspace_size(B, H_q, H_kv, k_tot, n_split)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n > 0 else None


def _ws(workspace):
    if workspace is None:
        return None, 0
    _need(workspace, "workspace", torch.uint8)
    return _ptr(workspace), workspace.numel()


def sparse_decode_attn(Q, k_base, v_base, blk_logical, count, seq_len, O, lse=None, blk_slot=None,
                       scale: float = 0.0, n_split: int = 0, flags: int = 0, workspace=None, status=None,
                       stream=None):
    """O [B][H_q][128] = attention of Q over the listed blocks of k_base/v_base.

    k_base/v_base hold B*H_kv pair regions of pair_stride x 128 rows (a cache
    [B][H_kv][T_cap][128] or a ring slot [B][H_kv][k_tot][64][128]).  ``flags`` may be
    SPARSE_ATTN_BLOCKS_READY: the block list and K/V are not written by the previous
    kernel on ``stream`` (they are already complete while it runs), so K/V streaming may
    start while it drains; SPARSE_ATTN_TENSOR_MEMORY: both contractions as tcgen05.mma
    with tensor-memory accumulators (cluster path, no workspace)."""
    B, H_q, H_kv, k_tot, pair_stride = _decode_args(Q, k_base, v_base, blk_logical, count, seq_len, O, lse,
                                                    blk_slot)
    ws, ws_bytes = _ws(workspace)
    rc = load().sparse_decode_attn(_ptr(Q), _ptr(k_base), _ptr(v_base), pair_stride, _ptr(blk_slot),
                                   _ptr(blk_logical), _ptr(count), k_tot, _ptr(seq_len), B, H_q, H_kv,
                                   float(scale), _ptr(O), _ptr(lse), n_split, int(flags), ws, ws_bytes,
                                   _ptr(status), _stream(stream))
    _check(rc, "sparse_decode_attn")


def sparse_decode_attn_noalloc(Q, k_base, v_base, blk_logical, count, seq_len, O, lse=None, blk_slot=None,
                               scale: float = 0.0, n_split: int = 0, flags: int = 0, status=None, stream=None):
    """sparse_decode_attn without a workspace argument and without allocating: for
    callers that cannot allocate device memory (a host without a caching allocator, an
    engine whose device memory is planned up front).  The library's fixed 4 MiB device
    array serves as scratch; calls sharing it must not overlap on the GPU."""
    B, H_q, H_kv, k_tot, pair_stride = _decode_args(Q, k_base, v_base, blk_logical, count, seq_len, O, lse,
                                                    blk_slot)
    rc = load().sparse_decode_attn_noalloc(_ptr(Q), _ptr(k_base), _ptr(v_base), pair_stride, _ptr(blk_slot),
                                           _ptr(blk_logical), _ptr(count), k_tot, _ptr(seq_len), B, H_q, H_kv,
                                           float(scale), _ptr(O), _ptr(lse), n_split, int(flags), _ptr(status),
                                           _stream(stream))
    _check(rc, "sparse_decode_attn_noalloc")


def sparse_decode_attn_ex(Q, k_base, v_base, blk_logical, count, seq_len, O, ready_flag, ready_target: int,
                          timeout_ns: int, lse=None, blk_slot=None, scale: float = 0.0, n_split: int = 0,
                          flags: int = 0, workspace=None, status=None, stream=None):
    """sparse_decode_attn after a bounded check of a staging-ready word."""
    B, H_q, H_kv, k_tot, pair_stride = _decode_args(Q, k_base, v_base, blk_logical, count, seq_len, O, lse,
                                                    blk_slot)
    _need(ready_flag, "ready_flag", torch.int32)
    rc = load().sparse_decode_attn_ex(_ptr(Q), _ptr(k_base), _ptr(v_base), pair_stride, _ptr(blk_slot),
                                      _ptr(blk_logical), _ptr(count), k_tot, _ptr(seq_len), B, H_q, H_kv,
                                      float(scale), _ptr(O), _ptr(lse), n_split, int(flags), *_ws(workspace),
                                      _ptr(ready_flag),
                                      int(ready_target), int(timeout_ns), _ptr(status), _stream(stream))
    _check(rc, "sparse_decode_attn_ex")


def sparse_decode_attn_forecast(Q, k_cache, v_cache, blk_idx, count, seq_len, O, lse=None, F=None, ktil_next=None,
                                n_init: int = 1, n_local: int = 2, k: int = 0, idx_next=None, count_next=None,
                                scale: float = 0.0, n_split: int = 0, flags: int = 0, status=None, stream=None):
    """One decode layer in one kernel: O = attention of Q over blocks blk_idx of the
    resident cache k_cache / v_cache [B][H_kv][T_cap][128], and (when F is given) the
    Forecast selection of the next layer from ktil_next [B][H_kv][N_cap][128] into
    idx_next [B][H_kv][k_tot_next] / count_next [B][H_kv]."""
    B, H_q, H_kv, k_tot, T_cap = _decode_args(Q, k_cache, v_cache, blk_idx, count, seq_len, O, lse, None)
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    N_cap = k_tot_next = 0
    if F is not None:
        if ktil_next is None or idx_next is None or count_next is None:
            raise ValueError("F needs ktil_next, idx_next and count_next")
        N_cap = ktil_next.shape[2]
        k_tot_next = idx_next.shape[2]
        _need(F, "F", torch.bfloat16, shape=(B, H_kv, D))
        _need(ktil_next, "ktil_next", torch.float32, shape=(B, H_kv, N_cap, D))
        _need(idx_next, "idx_next", torch.int32, shape=(B, H_kv, k_tot_next))
        _need(count_next, "count_next", torch.int32, shape=(B, H_kv))
    if status is not None:
        _need(status, "status", torch.int32)
    rc = load().sparse_decode_attn_forecast(_ptr(Q), _ptr(k_cache), _ptr(v_cache), T_cap, _ptr(blk_idx), _ptr(count),
                                            k_tot, _ptr(seq_len), B, H_q, H_kv, float(scale), _ptr(O), _ptr(lse),
                                            _ptr(F), _ptr(ktil_next), N_cap, n_init, n_local, k, _ptr(idx_next),
                                            _ptr(count_next), k_tot_next, n_split, int(flags), _ptr(status),
                                            _stream(stream))
    _check(rc, "sparse_decode_attn_forecast")


def sparse_verify_attn_grouped(Q, k_cache, v_cache, idx_q, C: int, window_blocks: int, seq_len, O,
                               blocks_loaded=None, scale: float = 0.0, n_split: int = 0, status=None,
                               stream=None, shared: bool = False, flags: int = 0):
    """Grouped verification: Q [B][N_q][H_q][128], idx_q [B][H_kv][N_q][n_sel].  Mode A
    (each query over its own set), or with ``shared`` mode B (sparse_verify_attn_shared:
    every query over its group's first query's set)."""
    B, N_q, H_q, _ = Q.shape
    _, H_kv, T_cap, _ = k_cache.shape
    n_sel = idx_q.shape[3]
    _need(Q, "Q", torch.bfloat16, shape=(B, N_q, H_q, D))
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(v_cache, "v_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(idx_q, "idx_q", torch.int32, shape=(B, H_kv, N_q, n_sel))
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(O, "O", torch.bfloat16, shape=(B, N_q, H_q, D))
    if blocks_loaded is not None:
        _need(blocks_loaded, "blocks_loaded", torch.int64)
    fn = load().sparse_verify_attn_shared if shared else load().sparse_verify_attn_grouped
    rc = fn(_ptr(Q), _ptr(k_cache), _ptr(v_cache), T_cap, _ptr(idx_q), n_sel, N_q, C, window_blocks, _ptr(seq_len), B,
            H_q, H_kv, float(scale), _ptr(O), _ptr(blocks_loaded), n_split, int(flags), _ptr(status),
            _stream(stream))
    _check(rc, "sparse_verify_attn_shared" if shared else "sparse_verify_attn_grouped")


def sparse_gather_offloaded(k_host, v_host, idx, count, k_ring, v_ring, ready_flag=None, n_ctas: int = 0,
                            status=None, stream=None):
    """Stage blocks idx [B][H_kv][k_tot] of pinned host K/V [B][H_kv][T_host][128]
    into ring slots [B][H_kv][k_tot][64][128]."""
    B, H_kv, T_host, _ = k_host.shape
    k_tot = idx.shape[2]
    _need(k_host, "k_host", torch.bfloat16, device_ok=False, shape=(B, H_kv, T_host, D))
    _need(v_host, "v_host", torch.bfloat16, device_ok=False, shape=(B, H_kv, T_host, D))
    for t, n in ((k_host, "k_host"), (v_host, "v_host")):
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{n} must be pinned host memory (or device memory)")
    _need(idx, "idx", torch.int32, shape=(B, H_kv, k_tot))
    _need(count, "count", torch.int32, shape=(B, H_kv))
    _need(k_ring, "k_ring", torch.bfloat16, shape=(B, H_kv, k_tot, BLK, D))
    _need(v_ring, "v_ring", torch.bfloat16, shape=(B, H_kv, k_tot, BLK, D))
    if ready_flag is not None:
        _need(ready_flag, "ready_flag", torch.int32)
    rc = load().sparse_gather_offloaded(_ptr(k_host), _ptr(v_host), T_host, _ptr(idx), _ptr(count), k_tot, B,
                                        H_kv, _ptr(k_ring), _ptr(v_ring), _ptr(ready_flag), n_ctas, _ptr(status),
                                        _stream(stream))
    _check(rc, "sparse_gather_offloaded")


def sparse_decode_attn_nsa_workspace_size(B: int, H_q: int, H_kv: int) -> int:
    """Bytes of the sparse_decode_attn_nsa workspace (0: invalid sizes)."""
    return int(load().sparse_decode_attn_nsa_workspace_size(B, H_q, H_kv))


def nsa_workspace(B: int, H_q: int, H_kv: int, device="cuda"):
    """A zeroed workspace tensor for sparse_decode_attn_nsa."""
    return torch.zeros(sparse_decode_attn_nsa_workspace_size(B, H_q, H_kv), dtype=torch.uint8, device=device)


def sparse_decode_attn_nsa(Q, k_cache, v_cache, khat, vhat, blk_idx, count, seq_len, window_tokens: int, gates, O,
                           workspace, scale: float = 0.0, n_split: int = 0, flags: int = 0, status=None,
                           stream=None, cmp: tuple = (0, 0)):
    """NSA gated three-branch decode: Q [B][H_q][128], K/V [B][H_kv][T_cap][128],
    compressed rows khat/vhat [B][H_kv][N_cap][128] (one per 64-token block, or with
    ``cmp = (l, s)`` the complete overlapping windows), selected blocks blk_idx
    [B][H_kv][k_tot] with count [B][H_kv], gates [B][H_q][3] = (g_c, g_s, g_w) fp32;
    writes O [B][H_q][128] = g_c o_c + g_s o_s + g_w o_w."""
    B, H_q, _ = Q.shape
    _, H_kv, T_cap, _ = k_cache.shape
    N_cap = khat.shape[2]
    k_tot = blk_idx.shape[2]
    _need(Q, "Q", torch.bfloat16, shape=(B, H_q, D))
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(v_cache, "v_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(khat, "khat", torch.bfloat16, shape=(B, H_kv, N_cap, D))
    _need(vhat, "vhat", torch.bfloat16, shape=(B, H_kv, N_cap, D))
    _need(blk_idx, "blk_idx", torch.int32, shape=(B, H_kv, k_tot))
    _need(count, "count", torch.int32, shape=(B, H_kv))
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(gates, "gates", torch.float32, shape=(B, H_q, 3))
    _need(O, "O", torch.bfloat16, shape=(B, H_q, D))
    ws, ws_bytes = _ws(workspace)
    rc = load().sparse_decode_attn_nsa(_ptr(Q), _ptr(k_cache), _ptr(v_cache), T_cap, _ptr(khat), _ptr(vhat), N_cap,
                                       int(cmp[0]), int(cmp[1]), _ptr(blk_idx), _ptr(count), k_tot, _ptr(seq_len), B, H_q, H_kv,
                                       int(window_tokens), _ptr(gates), float(scale), _ptr(O), ws, ws_bytes,
                                       n_split, int(flags), _ptr(status), _stream(stream))
    _check(rc, "sparse_decode_attn_nsa")


def sparse_nsa_compress(k_cache, v_cache, khat, vhat, len_before: int, n_new: int, cmp=(32, 16), stream=None):
    """Rows of the overlapping windows completed by tokens [len_before, len_before + n_new)."""
    B, H_kv, T_cap, _ = k_cache.shape
    R = khat.shape[2]
    _need(k_cache, "k_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(v_cache, "v_cache", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(khat, "khat", torch.bfloat16, shape=(B, H_kv, R, D))
    _need(vhat, "vhat", torch.bfloat16, shape=(B, H_kv, R, D))
    rc = load().sparse_nsa_compress(_ptr(k_cache), _ptr(v_cache), T_cap, B, H_kv, int(len_before), int(n_new),
                                    int(cmp[0]), int(cmp[1]), _ptr(khat), _ptr(vhat), R, _stream(stream))
    _check(rc, "sparse_nsa_compress")


def sparse_nsa_select(Q, khat, seq_len, n_init: int, n_local: int, k: int, idx_out, count_out, cmp=(32, 16),
                      scale: float = 0.0, status=None, stream=None):
    """NSA routing: per-head softmax over the compressed rows khat [B][H_kv][R][128],
    summed over the group, max-pooled onto the 64-token blocks, top-k.  Q [B][H_q][128]
    (idx_out [B][H_kv][k_tot], count_out [B][H_kv]) or, for several queries per batch
    element, Q [B][N_q][H_q][128] (idx_out [B][H_kv][N_q][k_tot], count_out [B][H_kv][N_q])."""
    if Q.dim() == 3:
        B, H_q, _ = Q.shape
        N_q = 1
    else:
        B, N_q, H_q, _ = Q.shape
    _, H_kv, R, _ = khat.shape
    k_tot = idx_out.shape[-1]
    _need(Q, "Q", torch.bfloat16, shape=(B, H_q, D) if Q.dim() == 3 else (B, N_q, H_q, D))
    _need(khat, "khat", torch.bfloat16, shape=(B, H_kv, R, D))
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(idx_out, "idx_out", torch.int32, shape=(B, H_kv, k_tot) if Q.dim() == 3 else (B, H_kv, N_q, k_tot))
    _need(count_out, "count_out", torch.int32, shape=(B, H_kv) if Q.dim() == 3 else (B, H_kv, N_q))
    rc = load().sparse_nsa_select(_ptr(Q), _ptr(khat), R, int(cmp[0]), int(cmp[1]), _ptr(seq_len), B, N_q, H_q, H_kv,
                                  float(scale), n_init, n_local, k, _ptr(idx_out), _ptr(count_out), k_tot,
                                  _ptr(status), _stream(stream))
    _check(rc, "sparse_nsa_select")


def sparse_prefill_select(F, ktil, seq_len, n_init: int, n_local: int, k: int, idx_out, count_out, status=None,
                          stream=None):
    """Forecast selection of every prefill position: F [B][H_kv][T_cap][128] bf16, ktil
    [B][H_kv][N_cap][128] fp32 -> idx_out [B][H_kv][T_cap][k_tot], count_out [B][H_kv][T_cap]."""
    B, H_kv, T_cap, _ = F.shape
    N_cap = ktil.shape[2]
    k_tot = idx_out.shape[3]
    _need(F, "F", torch.bfloat16, shape=(B, H_kv, T_cap, D))
    _need(ktil, "ktil", torch.float32, shape=(B, H_kv, N_cap, D))
    _need(seq_len, "seq_len", torch.int32, shape=(B,))
    _need(idx_out, "idx_out", torch.int32, shape=(B, H_kv, T_cap, k_tot))
    _need(count_out, "count_out", torch.int32, shape=(B, H_kv, T_cap))
    rc = load().sparse_prefill_select(_ptr(F), T_cap, _ptr(ktil), N_cap, _ptr(seq_len), B, H_kv, n_init, n_local, k,
                                      _ptr(idx_out), _ptr(count_out), k_tot, _ptr(status), _stream(stream))
    _check(rc, "sparse_prefill_select")
