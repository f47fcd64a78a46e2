"""CPU fp64 oracle for the multi-adapter LoRA path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It is independent of the CUDA library: it shares no
code with it, and its only common ground with it is the seeded input generator
(which holds none of the method's arithmetic).

The arithmetic lives in ``lora_oracle.c`` (plain C, IEEE double); this module
only marshals numpy arrays into it.  Each wrapped function names the passage
of the multi-LoRA pages it follows in the C source's header.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def load(path: str):
    """Load and type an oracle shared library (the default one, or a test's variant)."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    if _lib is None:
        # LORA_ORACLE_LIB lets the mutation tests point the pins at a planted-mistake build
        _lib = load(os.environ.get("LORA_ORACLE_LIB") or _build.build())
    return _lib


def _declare(L):
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    L.oracle_adapter_bytes.restype = i64
    L.oracle_adapter_bytes.argtypes = [i64, i64, i64, i64]
    L.oracle_pages_needed.restype = i64
    L.oracle_pages_needed.argtypes = [i64, i64, i64, i64]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_bf16_rne.argtypes = [ctypes.c_double]
    L.oracle_bf16_rne_array.restype = None
    L.oracle_bf16_rne_array.argtypes = [vp, vp, i64]
    L.oracle_unpack_matrix.restype = ctypes.c_int
    L.oracle_unpack_matrix.argtypes = [vp, i64, i64, vp, i64, i64, i64, i64, vp]
    L.oracle_lora_apply.restype = ctypes.c_int
    L.oracle_lora_apply.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i64, i64, vp, i64,
                                    vp, i32, i32, i64, i64]
    L.oracle_shrink.restype = ctypes.c_int
    L.oracle_shrink.argtypes = [vp, i64, vp, i64, i64, vp, vp, i64, i64, vp, i64, vp,
                                i32, i32, i64, i64]
    L.oracle_expand.restype = ctypes.c_int
    L.oracle_expand.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i64, i64, vp, i64, vp,
                                i32, i32, i64, i64]
    L.oracle_base_apply.restype = ctypes.c_int
    L.oracle_base_apply.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i64, i64, vp, i64,
                                    vp, i32, i32, i64, i64]
    L.oracle_lora_backward.restype = ctypes.c_int
    L.oracle_lora_backward.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp, vp, i64, i64, vp, i64,
                                       vp, i32, i32, i64, i64]
    L.oracle_segments_build.restype = i32
    L.oracle_segments_build.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.oracle_work_lists.restype = None
    L.oracle_work_lists.argtypes = [vp, i32, i32, i32, vp, vp, vp]


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def adapter_bytes(rank: int, d_in: int, d_out: int, bytes_per_param: int = 2) -> int:
    return int(lib().oracle_adapter_bytes(rank, d_in, d_out, bytes_per_param))


def pages_needed(rank: int, d_in: int, d_out: int, page_elems: int) -> int:
    return int(lib().oracle_pages_needed(rank, d_in, d_out, page_elems))


def bf16_rne(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_rne_array(_p(v), _p(out), v.size)
    return out


def unpack_matrix(pool, page0: int, rows: int, cols: int) -> np.ndarray:
    """Logical rows x cols matrix read back through the page table (bf16 bits)."""
    out = np.empty((rows, cols), dtype=np.uint16)
    pl = _c(pool.page_list, np.int32)
    pp = _c(pool.pool, np.uint16)
    rc = lib().oracle_unpack_matrix(_p(pp), pool.n_pages, pool.page_elems, _p(pl), pl.size,
                                    page0, rows, cols, _p(out))
    if rc:
        raise ValueError("page table points outside the pool")
    return out


def _pool_args(pool):
    pl = _c(pool.page_list, np.int32)
    pp = _c(pool.pool, np.uint16)
    desc = np.ascontiguousarray(pool.desc)
    return pl, pp, desc


def lora_apply(x, y0, ids, pool, d_in: int = None, d_out: int = None):
    """y (double [T, d_out]) and the error bits for y = y0 + s_i (x A_i) B_i per token."""
    d_in = pool.d_in if d_in is None else d_in
    d_out = pool.d_out if d_out is None else d_out
    x = _c(x, np.uint16)
    y0 = _c(y0, np.uint16)
    ids = _c(ids, np.int32)
    T = ids.size
    y = np.empty((T, d_out), dtype=np.float64)
    pl, pp, desc = _pool_args(pool)
    err = lib().oracle_lora_apply(_p(x), x.shape[1] if T else d_in, _p(y0),
                                  y0.shape[1] if T else d_out, _p(y), T, _p(ids), _p(pp),
                                  pool.n_pages, pool.page_elems, _p(pl), pl.size, _p(desc),
                                  desc.size, pool.max_rank, d_in, d_out)
    return y, int(err)


def base_apply(x, w0, ids, pool):
    """y (double [T, d_out]) and the error bits for y = x W0^T + s_i (x A_i) B_i per token;
    w0: bf16 bits [d_out, ldw >= d_in]."""
    x = _c(x, np.uint16)
    w0 = _c(w0, np.uint16)
    ids = _c(ids, np.int32)
    T = ids.size
    y = np.empty((T, pool.d_out), dtype=np.float64)
    pl, pp, desc = _pool_args(pool)
    err = lib().oracle_base_apply(_p(x), x.shape[1] if T else pool.d_in, _p(w0), w0.shape[1], _p(y), T, _p(ids),
                                  _p(pp), pool.n_pages, pool.page_elems, _p(pl), pl.size, _p(desc),
                                  desc.size, pool.max_rank, pool.d_in, pool.d_out)
    return y, int(err)


def shrink(x, ids, pool, h_init=None, ldh: int = None):
    """h (double [T, ldh]) = x . A_i^T per token (unscaled); untouched rows keep h_init."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    T = ids.size
    ldh = pool.max_rank if ldh is None else ldh
    h = np.zeros((T, ldh), dtype=np.float64) if h_init is None else _c(h_init, np.float64).copy()
    pl, pp, desc = _pool_args(pool)
    err = lib().oracle_shrink(_p(x), x.shape[1] if T else pool.d_in, _p(h), ldh, T, _p(ids),
                              _p(pp), pool.n_pages, pool.page_elems, _p(pl), pl.size, _p(desc),
                              desc.size, pool.max_rank, pool.d_in, pool.d_out)
    return h, int(err)


def expand(h, y0, ids, pool):
    """y (double [T, d_out]) = y0 + s_i * h . B_i per token, h given as fp32."""
    h = _c(h, np.float32)
    y0 = _c(y0, np.uint16)
    ids = _c(ids, np.int32)
    T = ids.size
    y = np.empty((T, pool.d_out), dtype=np.float64)
    pl, pp, desc = _pool_args(pool)
    err = lib().oracle_expand(_p(h), h.shape[1] if T else pool.max_rank, _p(y0),
                              y0.shape[1] if T else pool.d_out, _p(y), T, _p(ids), _p(pp),
                              pool.n_pages, pool.page_elems, _p(pl), pl.size, _p(desc),
                              desc.size, pool.max_rank, pool.d_in, pool.d_out)
    return y, int(err)


def lora_backward(x, g, ids, pool, grad=None):
    """(dx double [T, d_in], grad double [n_pages, page_elems], err): the gradients of the
    LoRA delta given g = dL/dy (bf16 bits); dA_i and dB_i are added into `grad` (a fresh
    zero array when None) at their elements' pool positions."""
    x = _c(x, np.uint16)
    g = _c(g, np.uint16)
    ids = _c(ids, np.int32)
    T = ids.size
    dx = np.empty((T, pool.d_in), dtype=np.float64)
    grad = np.zeros(pool.pool.shape, dtype=np.float64) if grad is None else _c(grad, np.float64)
    pl, pp, desc = _pool_args(pool)
    err = lib().oracle_lora_backward(_p(x), x.shape[1] if T else pool.d_in, _p(g),
                                     g.shape[1] if T else pool.d_out, _p(dx), _p(grad), T, _p(ids),
                                     _p(pp), pool.n_pages, pool.page_elems, _p(pl), pl.size,
                                     _p(desc), desc.size, pool.max_rank, pool.d_in, pool.d_out)
    return dx, grad, int(err)


def unpack_grad(grad, pool, page0: int, rows: int, cols: int) -> np.ndarray:
    """Logical rows x cols matrix of a gradient array laid out like the pool (read through
    the page table, as unpack_matrix reads the weights)."""
    P = pool.page_elems
    e = np.arange(rows * cols, dtype=np.int64)
    pos = pool.page_list[page0 + e // P].astype(np.int64) * P + e % P
    return np.asarray(grad).reshape(-1)[pos].reshape(rows, cols)


GROUP, CONTIGUOUS = 0, 1


def segments_build(ids, n_adapters: int, mode: int = GROUP):
    """(perm, indptr, seg_adapter, n_tokens, err) of the GROUP / CONTIGUOUS segmentation."""
    ids = _c(ids, np.int32)
    T = ids.size
    perm = np.full(max(T, 1), -1, dtype=np.int32)
    indptr = np.zeros(T + 1, dtype=np.int32)
    seg_ad = np.full(max(T, 1), -1, dtype=np.int32)
    nt = np.zeros(1, dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    ns = lib().oracle_segments_build(_p(ids), T, n_adapters, mode, _p(perm), _p(indptr),
                                     _p(seg_ad), _p(nt), _p(err))
    n_tok = int(nt[0])
    return perm[:n_tok].copy(), indptr[: ns + 1].copy(), seg_ad[:ns].copy(), n_tok, int(err[0])


def work_lists(indptr, short_max: int, tile_m: int):
    """(short_units [n_short], long_units [n_long, 2]) derived from the segments."""
    indptr = _c(indptr, np.int32)
    ns = indptr.size - 1
    total = int(indptr[-1]) if ns > 0 else 0
    short = np.zeros(max(ns, 1), dtype=np.int32)
    cap = total // max(tile_m, 1) + ns + 1
    long_ = np.zeros((cap, 2), dtype=np.int32)
    counts = np.zeros(2, dtype=np.int32)
    lib().oracle_work_lists(_p(indptr), ns, short_max, tile_m, _p(short), _p(long_), _p(counts))
    return short[: counts[0]].copy(), long_[: counts[1]].copy()
