"""fp64 CPU oracle for block-sparse GQA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (``block_sparse_long_pool_gb300``) never
does, and the two share no code: the oracle is plain C (``oracle.c``) built with gcc
and called through ctypes on numpy arrays.

Arrays of bf16 values travel as ``numpy.uint16`` holding the bf16 bit patterns, so
the oracle sees the exact input values.  Every routine computes in double precision.
What each routine follows on the pages is stated in ``oracle.c``:

* ``pool``    -- SparDA notes, eq.(4): mean of each 64-token block's keys.
* ``select``  -- SparDA notes, eq.(6) and Alg.1 step 2: Forecast scores, top-k
  outside init/local blocks (ties to the lower index), union, ascending.
* ``attn``    -- SparDA notes, eq.(7), scale 1/sqrt(d) from the SSV notes' NSA step 3.
* ``verify``  -- SSV notes, mechanism 1, mode A (per-query sets plus window).
* ``gather``  -- SparDA notes, §4.5: staging is a plain copy.
* ``prefill_select`` -- SparDA notes, eq.(16): the Forecast selection of every prefill
  position over the blocks it can see.
* ``pool_windows`` / ``select_windows`` / ``nsa(..., cmp=(l, s))`` -- eq.(4) with an
  overlapping kernel and stride, NSA routing max-pooled onto the 64-token blocks, and
  NSA's compressed branch over those windows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

D = 128
BLK = 64


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` with gcc (OpenMP, -O2, IEEE math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Load an oracle build from ``path`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_get_threads.restype = i32
    lib.oracle_pool.argtypes = [P, i64, i32, P, i32, P]
    lib.oracle_select.argtypes = [P, P, i32, i32, P, i32, i32, i32, i32, P, P, P]
    lib.oracle_select.restype = i32
    lib.oracle_select_heads.argtypes = [P, i32, P, i32, i32, P, ctypes.c_double, i32, i32, i32, i32, P, P, P]
    lib.oracle_select_heads.restype = i32
    lib.oracle_attn.argtypes = [P, i32, P, P, i64, i32, P, P, i32, P, f64, P, P]
    lib.oracle_verify.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, i32, i32, i32, P,
                                  f64, P, P, P]
    lib.oracle_verify_shared.argtypes = lib.oracle_verify.argtypes
    lib.oracle_gather.argtypes = [P, i64, i32, P, P, i32, P]
    lib.oracle_nsa.argtypes = [P, i32, P, P, i64, i32, P, P, i32, P, P, i32, P, i64, P, f64, P]
    lib.oracle_nsa_windows.argtypes = [P, i32, P, P, i64, i32, P, P, i32, P, P, i32, P, i64, P, f64, i32, i32, P]
    lib.oracle_pool_windows.argtypes = [P, i64, i32, P, i32, i32, i32, P]
    lib.oracle_pool_windows.restype = i32
    lib.oracle_select_windows.argtypes = [P, i32, P, i32, i32, P, i32, i32, f64, i32, i32, i32, i32, P, P, P, i32]
    lib.oracle_select_windows.restype = i32
    lib.oracle_prefill_select.argtypes = [P, i64, P, i32, i32, P, P, i32, i32, i32, i32, i32, P, P]
    lib.oracle_prefill_select.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 inputs travel as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def threads() -> int:
    return int(_load().oracle_get_threads())


def pool(K, lens, n_blocks_cap: int) -> np.ndarray:
    """Compressed keys [P][n_blocks_cap][128] (fp64) from K [P][T_cap][128] (bf16 bits)."""
    K = _u16(K)
    lens = _i64(lens)
    P, T_cap, d = K.shape
    assert d == D and lens.shape == (P,)
    out = np.empty((P, n_blocks_cap, D), dtype=np.float64)
    _load().oracle_pool(_ptr(K), T_cap, P, _ptr(lens), n_blocks_cap, _ptr(out))
    return out


def select(F, ktil, lens, n_init: int, n_local: int, k: int, k_tot: int | None = None):
    """Block selection.  Returns (idx [P][k_tot] int32, count [P] int32, scores [P][N] fp64)."""
    F = _u16(F)
    ktil = np.ascontiguousarray(ktil, dtype=np.float64)
    lens = _i64(lens)
    P, n_cap, d = ktil.shape
    assert d == D and F.shape == (P, D) and lens.shape == (P,)
    if k_tot is None:
        k_tot = n_init + n_local + k
    idx = np.empty((P, k_tot), dtype=np.int32)
    count = np.empty((P,), dtype=np.int32)
    scores = np.empty((P, n_cap), dtype=np.float64)
    rc = _load().oracle_select(_ptr(F), _ptr(ktil), n_cap, P, _ptr(lens), n_init, n_local, k,
                               k_tot, _ptr(idx), _ptr(count), _ptr(scores))
    if rc != 0:
        raise ValueError("oracle_select: a pair needs more than k_tot or n_blocks_cap entries")
    return idx, count, scores


def select_heads(Q, ktil, lens, n_init: int, n_local: int, k: int, k_tot: int | None = None, scale: float = 0.0):
    """Multi-head (InfLLM-V2) block selection from Q [P][G][128] bf16 bits: per-head
    softmax of scale * q_h . ktil_j over the blocks, summed over heads, then the top-k.
    Returns (idx [P][k_tot] int32, count [P] int32, scores [P][N] fp64)."""
    Q = _u16(Q)
    ktil = np.ascontiguousarray(ktil, dtype=np.float64)
    lens = _i64(lens)
    P, n_cap, d = ktil.shape
    G = Q.shape[1]
    assert d == D and Q.shape == (P, G, D) and lens.shape == (P,)
    if k_tot is None:
        k_tot = n_init + n_local + k
    idx = np.empty((P, k_tot), dtype=np.int32)
    count = np.empty((P,), dtype=np.int32)
    scores = np.empty((P, n_cap), dtype=np.float64)
    rc = _load().oracle_select_heads(_ptr(Q), G, _ptr(ktil), n_cap, P, _ptr(lens), float(scale), n_init, n_local,
                                     k, k_tot, _ptr(idx), _ptr(count), _ptr(scores))
    if rc != 0:
        raise ValueError("oracle_select_heads: a pair needs more than k_tot or n_blocks_cap entries")
    return idx, count, scores


def prefill_select(F, ktil, lens, n_init: int, n_local: int, k: int, k_tot: int | None = None, rows=None):
    """Forecast selection of every prefill position (or of the positions in ``rows``):
    F [P][T][128] bf16 bits, ktil [P][N][128].  Returns (idx [P][R][k_tot] int32,
    count [P][R] int32) with R = T or len(rows); rows at or past a pair's length are -1 / -1."""
    F = _u16(F)
    ktil = np.ascontiguousarray(ktil, dtype=np.float64)
    lens = _i64(lens)
    P, T_cap, d = F.shape
    n_cap = ktil.shape[1]
    assert d == D and ktil.shape[0] == P and lens.shape == (P,)
    if k_tot is None:
        k_tot = n_init + n_local + k
    rr = None if rows is None else _i32(rows)
    R = T_cap if rr is None else len(rr)
    idx = np.full((P, R, k_tot), -1, dtype=np.int32)
    count = np.full((P, R), -1, dtype=np.int32)
    rc = _load().oracle_prefill_select(_ptr(F), T_cap, _ptr(ktil), n_cap, P, _ptr(lens), _ptr(rr), R, n_init, n_local,
                                       k, k_tot, _ptr(idx), _ptr(count))
    if rc != 0:
        raise ValueError("oracle_prefill_select: a position needs more than k_tot or n_blocks_cap entries")
    return idx, count


def attn(Q, K, V, blocks, count, lens, scale: float | None = None):
    """Attention of Q [P][G][128] over the listed blocks of K/V [P][T][128].

    Returns (O [P][G][128] fp64, lse [P][G] fp64)."""
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    blocks, count, lens = _i32(blocks), _i32(count), _i64(lens)
    P, G, d = Q.shape
    assert d == D and K.shape == V.shape and K.shape[0] == P and K.shape[2] == D
    k_tot = blocks.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.empty((P, G, D), dtype=np.float64)
    lse = np.empty((P, G), dtype=np.float64)
    _load().oracle_attn(_ptr(Q), G, _ptr(K), _ptr(V), K.shape[1], P, _ptr(blocks), _ptr(count),
                        k_tot, _ptr(lens), float(scale), _ptr(O), _ptr(lse))
    return O, lse


def verify(Q, K, V, I, C: int, window_blocks: int, lens, scale: float | None = None, shared: bool = False):
    """Grouped verification, mode A (each query over its own set; the group loads the
    merged union) or, with ``shared``, mode B (every query over its group's first
    query's set).  Q [B][N_q][H_q][128], K/V [B][H_kv][T][128], I [B][H_kv][N_q][n_sel].
    Returns (O [B][N_q][H_q][128], union_blocks, per_query_blocks)."""
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    I, lens = _i32(I), _i64(lens)
    B, N_q, H_q, d = Q.shape
    _, H_kv, T_cap, _ = K.shape
    n_sel = I.shape[3]
    assert d == D and I.shape[:3] == (B, H_kv, N_q) and lens.shape == (B,)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.empty((B, N_q, H_q, D), dtype=np.float64)
    u = np.zeros(1, dtype=np.int64)
    pq = np.zeros(1, dtype=np.int64)
    fn = _load().oracle_verify_shared if shared else _load().oracle_verify
    fn(_ptr(Q), _ptr(K), _ptr(V), T_cap, B, H_q, H_kv, N_q, _ptr(I), n_sel, C, window_blocks, _ptr(lens),
       float(scale), _ptr(O), _ptr(u), _ptr(pq))
    return O, int(u[0]), int(pq[0])


def windows(lens, l: int, s: int):
    """Complete compression windows [s*j, s*j + l) within each length."""
    lens = np.asarray(lens, dtype=np.int64)
    return np.where(lens < l, 0, (lens - l) // s + 1)


def pool_windows(X, lens, l: int, s: int, n_rows_cap: int) -> np.ndarray:
    """Overlapping compression: rows [P][n_rows_cap][128] (fp64), row j the mean of
    X[s*j : s*j + l] for the complete windows, zero beyond."""
    X = _u16(X)
    lens = _i64(lens)
    P, T_cap, d = X.shape
    assert d == D and lens.shape == (P,)
    out = np.empty((P, n_rows_cap, D), dtype=np.float64)
    rc = _load().oracle_pool_windows(_ptr(X), T_cap, P, _ptr(lens), int(l), int(s), int(n_rows_cap), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_pool_windows: more windows than n_rows_cap")
    return out


def select_windows(Q, kcmp, lens, l: int, s: int, n_init: int, n_local: int, k: int, k_tot: int | None = None,
                   scale: float = 0.0, n_blocks_cap: int | None = None):
    """NSA routing: per-head softmax over the compressed windows kcmp [P][R][128],
    summed over the G heads of Q [P][G][128], max-pooled onto the 64-token blocks,
    top-k.  Returns (idx [P][k_tot] int32, count [P] int32, block scores [P][n_blocks_cap])."""
    Q = _u16(Q)
    kcmp = np.ascontiguousarray(kcmp, dtype=np.float64)
    lens = _i64(lens)
    P, n_rows_cap, d = kcmp.shape
    G = Q.shape[1]
    assert d == D and Q.shape == (P, G, D) and lens.shape == (P,)
    if k_tot is None:
        k_tot = n_init + n_local + k
    if n_blocks_cap is None:
        n_blocks_cap = max(1, int((lens.max() + BLK - 1) // BLK))
    idx = np.empty((P, k_tot), dtype=np.int32)
    count = np.empty((P,), dtype=np.int32)
    scores = np.empty((P, n_blocks_cap), dtype=np.float64)
    rc = _load().oracle_select_windows(_ptr(Q), G, _ptr(kcmp), n_rows_cap, P, _ptr(lens), int(l), int(s),
                                       float(scale), n_init, n_local, k, k_tot, _ptr(idx), _ptr(count),
                                       _ptr(scores), int(n_blocks_cap))
    if rc != 0:
        raise ValueError("oracle_select_windows: a pair needs more than k_tot, n_rows_cap or n_blocks_cap entries")
    return idx, count, scores


def nsa(Q, K, V, khat, vhat, blocks, count, lens, window_tokens: int, gates, scale: float | None = None,
        cmp: tuple[int, int] | None = None):
    """NSA gated three-branch output: Q [P][G][128] bf16 bits, K/V [P][T][128] bf16 bits,
    khat/vhat [P][N][128] compressed rows, blocks [P][k_tot] selected, gates [P][G][3]
    = (g_c, g_s, g_w).  The compressed rows are one per 64-token block holding a token,
    or with ``cmp = (l, s)`` the complete windows of kernel l and stride s.
    Returns O [P][G][128] fp64."""
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    khat = np.ascontiguousarray(khat, dtype=np.float64)
    vhat = np.ascontiguousarray(vhat, dtype=np.float64)
    blocks, count, lens = _i32(blocks), _i32(count), _i64(lens)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    P, G, d = Q.shape
    T = K.shape[1]
    n_cap = khat.shape[1]
    assert d == D and K.shape == (P, T, D) and V.shape == K.shape and vhat.shape == khat.shape
    assert gates.shape == (P, G, 3) and blocks.shape[0] == P and lens.shape == (P,)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.empty((P, G, D), dtype=np.float64)
    if cmp is None:
        _load().oracle_nsa(_ptr(Q), G, _ptr(K), _ptr(V), T, P, _ptr(khat), _ptr(vhat), n_cap, _ptr(blocks),
                           _ptr(count), blocks.shape[1], _ptr(lens), int(window_tokens), _ptr(gates), float(scale),
                           _ptr(O))
    else:
        _load().oracle_nsa_windows(_ptr(Q), G, _ptr(K), _ptr(V), T, P, _ptr(khat), _ptr(vhat), n_cap, _ptr(blocks),
                                   _ptr(count), blocks.shape[1], _ptr(lens), int(window_tokens), _ptr(gates),
                                   float(scale), int(cmp[0]), int(cmp[1]), _ptr(O))
    return O


def gather(src, idx, count, ring=None):
    """Staging copy: src [P][T_host][128] bf16 bits -> ring [P][k_tot][64][128]."""
    src = _u16(src)
    idx, count = _i32(idx), _i32(count)
    P, T_host, d = src.shape
    k_tot = idx.shape[1]
    if ring is None:
        ring = np.zeros((P, k_tot, BLK, D), dtype=np.uint16)
    assert ring.shape == (P, k_tot, BLK, D) and ring.dtype == np.uint16 and ring.flags.c_contiguous
    _load().oracle_gather(_ptr(src), T_host, P, _ptr(idx), _ptr(count), k_tot, _ptr(ring))
    return ring
