"""Thin Python binding of liblora_sgmv.so (the C ABI in include/lora_sgmv.h and
include/lora_pool.h).

Argument marshalling only: every step of the LoRA path runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There is
no fallback: if the library cannot be built or loaded, every call raises.
"""

from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import build as _build

# ---------------------------------------------------------------- C structs --

LORA_OK = 0
LORA_ERR_INVALID_ARG = -1
LORA_ERR_UNSUPPORTED = -2
LORA_ERR_CUDA = -3
LORA_ERR_WORKSPACE = -4
LORA_DERR_BAD_ADAPTER = 1
LORA_DERR_BAD_PAGE = 2
LORA_DERR_BAD_RANK = 4
LORA_DERR_TIMEOUT = 8
LORA_MAX_RANK = 64
LORA_MAX_ADAPTERS = 32768
LORA_SHORT_MAX_TOKENS = 24
LORA_TILE_M = 128
LORA_BGMV_STATIC_ADAPTERS = 1
LORA_SEG_GROUP = 0
LORA_SEG_CONTIGUOUS = 1
LORA_FIXED_SCRATCH_MAX_TOKENS = 16384
LORA_MAX_PROJ = 4

EXPORTED = (
    "lora_segments_buffer_bytes",
    "lora_segments_carve",
    "lora_segments_build",
    "lora_sgmv_shrink",
    "lora_sgmv_expand",
    "lora_apply",
    "lora_apply_f32y",
    "lora_apply_multi",
    "lora_sgmv_backward",
    "lora_apply_fixed_scratch",
    "lora_bgmv",
    "lora_bgmv_ex",
    "lora_base_apply",
    "lora_pool_pages_needed",
    "lora_status_string",
    "lora_abi_version",
    "lora_launch_count",
    "lora_debug_wait_probe",
    "lora_debug_gather_width",
    "lora_pool_mgr_create",
    "lora_pool_mgr_destroy",
    "lora_pool_mgr_page_list_len",
    "lora_pool_mgr_free_pages",
    "lora_pool_resident_rank",
    "lora_pool_pin",
    "lora_pool_unpin",
    "lora_pool_mgr_reserve",
    "lora_pool_mgr_release",
    "lora_pool_load",
    "lora_pool_evict",
    "lora_pool_mgr_stats",
)


class lora_adapter_desc_t(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("scale", ctypes.c_float),
                ("a_page0", ctypes.c_int32), ("b_page0", ctypes.c_int32)]


class lora_pool_view_t(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("n_pages", ctypes.c_int64),
                ("page_list", ctypes.c_void_p), ("n_page_list", ctypes.c_int64),
                ("adapters", ctypes.c_void_p), ("n_adapters", ctypes.c_int32),
                ("page_elems", ctypes.c_int32), ("max_rank", ctypes.c_int32),
                ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32)]


class lora_proj_t(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("y", ctypes.c_void_p),
                ("ldy", ctypes.c_int64), ("view", lora_pool_view_t)]


class lora_pool_stats_t(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_int64), ("loads", ctypes.c_int64), ("refused", ctypes.c_int64),
                ("evictions", ctypes.c_int64), ("pages_loaded", ctypes.c_int64),
                ("resident", ctypes.c_int32), ("pinned", ctypes.c_int32)]


class lora_segments_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("max_long_units", ctypes.c_int32),
                ("token_perm", ctypes.c_void_p), ("seg_indptr", ctypes.c_void_p),
                ("seg_adapter", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("short_units", ctypes.c_void_p), ("long_units", ctypes.c_void_p),
                ("scratch", ctypes.c_void_p), ("h_scratch", ctypes.c_void_p),
                ("k_partials", ctypes.c_void_p)]


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))
        self.status = status


_lib = None


def lib():
    """The loaded library (built in-tree first if its sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.lora_launch_count.restype = ctypes.c_uint64
        L.lora_launch_count.argtypes = []
        L.lora_debug_wait_probe.restype = None
        L.lora_debug_wait_probe.argtypes = [ctypes.c_int64]
        L.lora_debug_gather_width.restype = ctypes.c_int32
        L.lora_debug_gather_width.argtypes = [ctypes.POINTER(lora_pool_view_t), ctypes.c_int32]
        L.lora_segments_buffer_bytes.restype = sz
        L.lora_segments_buffer_bytes.argtypes = [i32]
        L.lora_segments_carve.restype = i32
        L.lora_segments_carve.argtypes = [vp, sz, i32, ctypes.POINTER(lora_segments_t)]
        L.lora_segments_build.restype = i32
        L.lora_segments_build.argtypes = [vp, i32, i32, i32, ctypes.POINTER(lora_segments_t), vp, vp]
        seg_p = ctypes.POINTER(lora_segments_t)
        view_p = ctypes.POINTER(lora_pool_view_t)
        L.lora_sgmv_shrink.restype = i32
        L.lora_sgmv_shrink.argtypes = [vp, i64, vp, i64, seg_p, view_p, vp, vp]
        L.lora_sgmv_expand.restype = i32
        L.lora_sgmv_expand.argtypes = [vp, i64, vp, i64, seg_p, view_p, vp, vp]
        L.lora_apply.restype = i32
        L.lora_apply.argtypes = [vp, i64, vp, i64, seg_p, view_p, vp, vp]
        L.lora_apply_f32y.restype = i32
        L.lora_apply_f32y.argtypes = [vp, i64, vp, i64, vp, i64, seg_p, view_p, vp, vp]
        L.lora_sgmv_backward.restype = i32
        L.lora_sgmv_backward.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i64, seg_p, view_p, vp, vp]
        L.lora_apply_multi.restype = i32
        L.lora_apply_multi.argtypes = [ctypes.POINTER(lora_proj_t), i32, seg_p, vp, vp]
        L.lora_apply_fixed_scratch.restype = i32
        L.lora_apply_fixed_scratch.argtypes = [vp, i64, vp, i64, seg_p, view_p, vp, vp]
        L.lora_bgmv.restype = i32
        L.lora_bgmv.argtypes = [vp, i64, vp, i64, vp, i32, view_p, vp, vp]
        L.lora_base_apply.restype = i32
        L.lora_base_apply.argtypes = [vp, i64, vp, i64, vp, i64, vp, seg_p, view_p, vp, vp]
        L.lora_bgmv_ex.restype = i32
        L.lora_bgmv_ex.argtypes = [vp, i64, vp, i64, vp, i32, view_p, ctypes.c_uint32, vp, vp]
        L.lora_pool_pages_needed.restype = i64
        L.lora_pool_pages_needed.argtypes = [i32, i32, i32, i32]
        L.lora_status_string.restype = ctypes.c_char_p
        L.lora_status_string.argtypes = [i32]
        L.lora_abi_version.restype = i32
        L.lora_abi_version.argtypes = []
        i32p = ctypes.POINTER(ctypes.c_int32)
        L.lora_pool_mgr_create.restype = i32
        L.lora_pool_mgr_create.argtypes = [i64, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.lora_pool_mgr_destroy.restype = None
        L.lora_pool_mgr_destroy.argtypes = [vp]
        L.lora_pool_mgr_page_list_len.restype = i64
        L.lora_pool_mgr_page_list_len.argtypes = [vp]
        L.lora_pool_mgr_free_pages.restype = i64
        L.lora_pool_mgr_free_pages.argtypes = [vp]
        L.lora_pool_resident_rank.restype = i32
        L.lora_pool_resident_rank.argtypes = [vp, i32]
        L.lora_pool_pin.restype = i32
        L.lora_pool_pin.argtypes = [vp, i32]
        L.lora_pool_unpin.restype = i32
        L.lora_pool_unpin.argtypes = [vp, i32]
        L.lora_pool_mgr_reserve.restype = i32
        L.lora_pool_mgr_reserve.argtypes = [vp, i32, i32, i32p, i32, i32p, i32p, i32, i32p]
        L.lora_pool_mgr_release.restype = i32
        L.lora_pool_mgr_release.argtypes = [vp, i32]
        L.lora_pool_load.restype = i32
        L.lora_pool_load.argtypes = [vp, i32, i32, ctypes.c_float, vp, vp, view_p, vp]
        L.lora_pool_evict.restype = i32
        L.lora_pool_evict.argtypes = [vp, i32, view_p, vp]
        L.lora_pool_mgr_stats.restype = i32
        L.lora_pool_mgr_stats.argtypes = [vp, ctypes.POINTER(lora_pool_stats_t)]
        _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def status_string(status: int) -> str:
    return lib().lora_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != LORA_OK:
        raise LoraError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major tensor with unit column stride")
    return int(t.stride(0))


# ------------------------------------------------------------ device views --

class PoolView:
    """A projection's paged adapter pool on the device plus its C view."""

    def __init__(self, pool: torch.Tensor, page_list: torch.Tensor, adapters: torch.Tensor,
                 page_elems: int, max_rank: int, d_in: int, d_out: int):
        self.pool = pool  # bf16 (or int16 bits) [n_pages, page_elems]
        self.page_list = page_list  # int32
        self.adapters = adapters  # uint8 [n_adapters * 16] or int32 [n_adapters, 4]
        self.c = lora_pool_view_t(
            pool.data_ptr(), pool.numel() // page_elems, page_list.data_ptr(), page_list.numel(),
            adapters.data_ptr(), adapters.numel() * adapters.element_size() // 16, page_elems,
            max_rank, d_in, d_out)

    @classmethod
    def from_host(cls, host_pool, device="cuda"):
        """Upload a workloads.AdapterPool."""
        pool = torch.from_numpy(host_pool.pool.view(np.int16)).to(device).view(torch.bfloat16)
        pl = torch.from_numpy(np.ascontiguousarray(host_pool.page_list, dtype=np.int32)).to(device)
        desc = torch.from_numpy(np.ascontiguousarray(host_pool.desc).view(np.uint8)).to(device)
        return cls(pool, pl, desc, host_pool.page_elems, host_pool.max_rank, host_pool.d_in,
                   host_pool.d_out)

    @property
    def d_in(self):
        return self.c.d_in

    @property
    def d_out(self):
        return self.c.d_out


class Segments:
    """A device buffer carved into the segment arrays for T tokens."""

    def __init__(self, T: int, device="cuda"):
        nbytes = int(lib().lora_segments_buffer_bytes(T))
        self.buf = torch.zeros(max(nbytes, 16) // 4 + 4, dtype=torch.int32, device=device)
        self.c = lora_segments_t()
        _check(lib().lora_segments_carve(_ptr(self.buf), self.buf.numel() * 4, T, ctypes.byref(self.c)),
               "lora_segments_carve")
        self.T = T

    def _view(self, ptr_field: str, n: int) -> torch.Tensor:
        off = (getattr(self.c, ptr_field) - self.buf.data_ptr()) // 4
        return self.buf[off: off + n]

    @property
    def meta(self) -> torch.Tensor:
        return self._view("meta", 8)

    def host(self):
        """(perm, indptr, seg_adapter, n_tokens, short_units, long_units [n, 2]) on the host."""
        meta = self.meta.cpu().numpy()
        n_segs, n_tok, n_short, n_long = (int(v) for v in meta[:4])
        perm = self._view("token_perm", n_tok).cpu().numpy()
        indptr = self._view("seg_indptr", n_segs + 1).cpu().numpy()
        seg_ad = self._view("seg_adapter", n_segs).cpu().numpy()
        short = self._view("short_units", n_short).cpu().numpy()
        long_ = self._view("long_units", 2 * n_long).cpu().numpy().reshape(-1, 2)
        return perm, indptr, seg_ad, n_tok, short, long_


# ------------------------------------------------------------ entry points --

def lora_segments_buffer_bytes(T: int) -> int:
    return int(lib().lora_segments_buffer_bytes(T))


def lora_pool_pages_needed(rank: int, d_in: int, d_out: int, page_elems: int) -> int:
    return int(lib().lora_pool_pages_needed(rank, d_in, d_out, page_elems))


def lora_status_string(status: int) -> str:
    return status_string(status)


def lora_abi_version() -> int:
    return int(lib().lora_abi_version())


def lora_segments_build(token_adapter: torch.Tensor, n_adapters: int, seg: Segments,
                        mode: int = LORA_SEG_GROUP, err: Optional[torch.Tensor] = None, stream=None):
    T = int(token_adapter.numel())
    _check(lib().lora_segments_build(_ptr(token_adapter), T, n_adapters, mode, ctypes.byref(seg.c),
                                     _ptr(err), _stream(stream)), "lora_segments_build")


def lora_sgmv_shrink(x: torch.Tensor, h: torch.Tensor, seg: Segments, view: PoolView,
                     err: Optional[torch.Tensor] = None, stream=None):
    _check(lib().lora_sgmv_shrink(_ptr(x), _ld(x), _ptr(h), _ld(h), ctypes.byref(seg.c),
                                  ctypes.byref(view.c), _ptr(err), _stream(stream)),
           "lora_sgmv_shrink")


def lora_sgmv_expand(h: torch.Tensor, y: torch.Tensor, seg: Segments, view: PoolView,
                     err: Optional[torch.Tensor] = None, stream=None):
    _check(lib().lora_sgmv_expand(_ptr(h), _ld(h), _ptr(y), _ld(y), ctypes.byref(seg.c),
                                  ctypes.byref(view.c), _ptr(err), _stream(stream)),
           "lora_sgmv_expand")


def lora_apply(x: torch.Tensor, y: torch.Tensor, seg: Segments, view: PoolView,
               err: Optional[torch.Tensor] = None, stream=None):
    _check(lib().lora_apply(_ptr(x), _ld(x), _ptr(y), _ld(y), ctypes.byref(seg.c),
                            ctypes.byref(view.c), _ptr(err), _stream(stream)), "lora_apply")


def lora_apply_f32y(x: torch.Tensor, y0: torch.Tensor, yf: torch.Tensor, seg: Segments, view: PoolView,
                    err: Optional[torch.Tensor] = None, stream=None):
    """lora_apply with the result written as fp32 into yf (y0 bf16 is only read)."""
    _check(lib().lora_apply_f32y(_ptr(x), _ld(x), _ptr(y0), _ld(y0), _ptr(yf), _ld(yf),
                                 ctypes.byref(seg.c), ctypes.byref(view.c), _ptr(err), _stream(stream)),
           "lora_apply_f32y")


def lora_apply_multi(calls, seg: Segments, err: Optional[torch.Tensor] = None, stream=None):
    """Several projections on one batch in one grouped call: `calls` is a list of
    (x, y, view) with the same d_in; projections may share x."""
    arr = (lora_proj_t * len(calls))()
    for i, (x, y, view) in enumerate(calls):
        arr[i].x = _ptr(x).value
        arr[i].ldx = _ld(x)
        arr[i].y = _ptr(y).value
        arr[i].ldy = _ld(y)
        arr[i].view = view.c
    _check(lib().lora_apply_multi(arr, len(calls), ctypes.byref(seg.c), _ptr(err), _stream(stream)),
           "lora_apply_multi")


def lora_sgmv_backward(x: torch.Tensor, dy: torch.Tensor, dx: Optional[torch.Tensor], grad_pool: torch.Tensor,
                       hu: torch.Tensor, seg: Segments, view: PoolView, err: Optional[torch.Tensor] = None,
                       stream=None):
    """Adapter gradients: dA_i, dB_i added into grad_pool (fp32, the pool's page layout),
    dx += the adapter path's contribution (bf16 in place, or None).  hu: fp32 workspace
    [2 * T, ldh]."""
    ldh = _ld(hu)
    _check(lib().lora_sgmv_backward(_ptr(x), _ld(x), _ptr(dy), _ld(dy), _ptr(dx), _ld(dx) if dx is not None else 0,
                                    _ptr(grad_pool), _ptr(hu), ldh, ctypes.byref(seg.c), ctypes.byref(view.c),
                                    _ptr(err), _stream(stream)), "lora_sgmv_backward")


def apply_kernel_names():
    """Names of the kernels one lora_apply call may launch, in launch order."""
    return ["gather_kernel", "fused_tc_kernel"]


def lora_apply_fixed_scratch(x: torch.Tensor, y: torch.Tensor, seg: Segments, view: PoolView,
                             err: Optional[torch.Tensor] = None, stream=None):
    """lora_apply with its intermediate in the library's fixed device array: for callers
    that cannot allocate a workspace (see include/lora_sgmv.h).  Calls that may overlap on
    the GPU share that array and must be serialised by the caller."""
    _check(lib().lora_apply_fixed_scratch(_ptr(x), _ld(x), _ptr(y), _ld(y), ctypes.byref(seg.c),
                                          ctypes.byref(view.c), _ptr(err), _stream(stream)),
           "lora_apply_fixed_scratch")


def debug_wait_probe(cycles: int) -> None:
    """Test-only: arm (cycles > 0) or disarm the kernels' timeout probe."""
    lib().lora_debug_wait_probe(int(cycles))


def debug_gather_width(shapes) -> int:
    """Test-only, host only: the gather kernel's cluster width for a call over projections
    of the given (d_in, d_out) shapes, before the launcher's occupancy narrowing."""
    arr = (lora_pool_view_t * max(1, len(shapes)))()
    for i, (d_in, d_out) in enumerate(shapes):
        arr[i].d_in, arr[i].d_out = int(d_in), int(d_out)
    return int(lib().lora_debug_gather_width(arr, len(shapes)))


def launch_count() -> int:
    """Kernels the library has launched in this process (a recorded graph counts once)."""
    return int(lib().lora_launch_count())


def lora_base_apply(x: torch.Tensor, w0: torch.Tensor, y: torch.Tensor, token_adapter: torch.Tensor, seg: Segments,
                    view: PoolView, err: Optional[torch.Tensor] = None, stream=None):
    """y = bf16(x W0^T + s_i (x A_i^T) B_i), y written only; w0 bf16 [d_out, ldw >= d_in]."""
    _check(lib().lora_base_apply(_ptr(x), _ld(x), _ptr(w0), _ld(w0), _ptr(y), _ld(y), _ptr(token_adapter),
                                 ctypes.byref(seg.c), ctypes.byref(view.c), _ptr(err), _stream(stream)),
           "lora_base_apply")


def lora_bgmv(x: torch.Tensor, y: torch.Tensor, token_adapter: torch.Tensor, view: PoolView,
              err: Optional[torch.Tensor] = None, stream=None, static_adapters: bool = False):
    """static_adapters: lora_bgmv_ex with LORA_BGMV_STATIC_ADAPTERS (see include/lora_sgmv.h)."""
    T = int(token_adapter.numel())
    if static_adapters:
        _check(lib().lora_bgmv_ex(_ptr(x), _ld(x), _ptr(y), _ld(y), _ptr(token_adapter), T, ctypes.byref(view.c),
                                  LORA_BGMV_STATIC_ADAPTERS, _ptr(err), _stream(stream)), "lora_bgmv_ex")
    else:
        _check(lib().lora_bgmv(_ptr(x), _ld(x), _ptr(y), _ld(y), _ptr(token_adapter), T,
                               ctypes.byref(view.c), _ptr(err), _stream(stream)), "lora_bgmv")



# ---------------------------------------------------------- pool residency --

def _host_bits(m, rows: int, cols: int) -> tuple:
    """(pointer, owner) of a host bf16 matrix [rows, cols]: a contiguous CPU tensor of
    bfloat16 / int16 / uint16 or a numpy uint16 / int16 array."""
    if isinstance(m, torch.Tensor):
        if m.device.type != "cpu" or m.element_size() != 2 or not m.is_contiguous():
            raise ValueError("expected a contiguous 2-byte CPU tensor")
        if m.numel() != rows * cols:
            raise ValueError("expected %d x %d elements" % (rows, cols))
        return ctypes.c_void_p(m.data_ptr()), m
    a = np.ascontiguousarray(m)
    if a.dtype.itemsize != 2 or a.size != rows * cols:
        raise ValueError("expected a %d x %d array of 2-byte elements" % (rows, cols))
    return ctypes.c_void_p(a.ctypes.data), a


def lora_pool_mgr_create(n_pages: int, page_elems: int, n_adapters: int, max_rank: int,
                         d_in: int, d_out: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().lora_pool_mgr_create(n_pages, page_elems, n_adapters, max_rank, d_in, d_out,
                                      ctypes.byref(h)), "lora_pool_mgr_create")
    return h


def lora_pool_mgr_destroy(mgr: ctypes.c_void_p) -> None:
    lib().lora_pool_mgr_destroy(mgr)


def lora_pool_mgr_page_list_len(mgr) -> int:
    return int(lib().lora_pool_mgr_page_list_len(mgr))


def lora_pool_mgr_free_pages(mgr) -> int:
    return int(lib().lora_pool_mgr_free_pages(mgr))


def lora_pool_resident_rank(mgr, adapter: int) -> int:
    return int(lib().lora_pool_resident_rank(mgr, adapter))


def lora_pool_pin(mgr, adapter: int) -> None:
    _check(lib().lora_pool_pin(mgr, adapter), "lora_pool_pin")


def lora_pool_unpin(mgr, adapter: int) -> None:
    _check(lib().lora_pool_unpin(mgr, adapter), "lora_pool_unpin")


def lora_pool_mgr_reserve(mgr, adapter: int, rank: int, pages_cap: int, evicted_cap: int):
    """(pages, evicted) as int32 arrays: the pages the adapter now holds (empty if it was
    already resident with this rank) and the adapters evicted for them, in order."""
    pages = (ctypes.c_int32 * max(1, pages_cap))()
    evicted = (ctypes.c_int32 * max(1, evicted_cap))()
    n_p, n_e = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().lora_pool_mgr_reserve(mgr, adapter, rank, pages, pages_cap, ctypes.byref(n_p), evicted,
                                       evicted_cap, ctypes.byref(n_e)), "lora_pool_mgr_reserve")
    return (np.frombuffer(pages, dtype=np.int32)[: n_p.value].copy(),
            np.frombuffer(evicted, dtype=np.int32)[: n_e.value].copy())


def lora_pool_mgr_release(mgr, adapter: int) -> None:
    _check(lib().lora_pool_mgr_release(mgr, adapter), "lora_pool_mgr_release")


def lora_pool_load(mgr, adapter: int, rank: int, scale: float, A, B, view: PoolView, stream=None):
    """A: host bf16 [rank, d_in], B: host bf16 [rank, d_out] (tensors or uint16 arrays).  A
    pinned tensor is copied asynchronously: keep it unchanged until the stream passes."""
    pa, _ = _host_bits(A, rank, view.d_in)
    pb, _ = _host_bits(B, rank, view.d_out)
    _check(lib().lora_pool_load(mgr, adapter, rank, float(scale), pa, pb, ctypes.byref(view.c),
                                _stream(stream)), "lora_pool_load")


def lora_pool_mgr_stats(mgr) -> dict:
    st = lora_pool_stats_t()
    _check(lib().lora_pool_mgr_stats(mgr, ctypes.byref(st)), "lora_pool_mgr_stats")
    return {name: int(getattr(st, name)) for name, _ in lora_pool_stats_t._fields_}


def lora_pool_evict(mgr, adapter: int, view: PoolView, stream=None) -> None:
    _check(lib().lora_pool_evict(mgr, adapter, ctypes.byref(view.c), _stream(stream)), "lora_pool_evict")


class PoolManager:
    """One projection's pool residency (include/lora_pool.h): a host-side manager plus,
    from device_view(), the device pool, page list and descriptors it fills."""

    def __init__(self, n_pages: int, page_elems: int, n_adapters: int, max_rank: int,
                 d_in: int, d_out: int):
        self.h = lora_pool_mgr_create(n_pages, page_elems, n_adapters, max_rank, d_in, d_out)
        self.n_pages, self.page_elems, self.n_adapters = n_pages, page_elems, n_adapters
        self.max_rank, self.d_in, self.d_out = max_rank, d_in, d_out

    def close(self):
        if self.h is not None and self.h.value:
            lora_pool_mgr_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def page_list_len(self) -> int:
        return lora_pool_mgr_page_list_len(self.h)

    @property
    def slots_per_adapter(self) -> int:
        return self.page_list_len // self.n_adapters

    @property
    def free_pages(self) -> int:
        return lora_pool_mgr_free_pages(self.h)

    def stats(self) -> dict:
        """hits, loads, refused, evictions, pages_loaded, resident, pinned."""
        return lora_pool_mgr_stats(self.h)

    def resident_rank(self, adapter: int) -> int:
        return lora_pool_resident_rank(self.h, adapter)

    def pin(self, adapter: int):
        lora_pool_pin(self.h, adapter)

    def unpin(self, adapter: int):
        lora_pool_unpin(self.h, adapter)

    def reserve(self, adapter: int, rank: int):
        return lora_pool_mgr_reserve(self.h, adapter, rank, self.slots_per_adapter, self.n_adapters)

    def release(self, adapter: int):
        lora_pool_mgr_release(self.h, adapter)

    def device_view(self, device="cuda") -> PoolView:
        """A zeroed device pool, page list and descriptor array of this manager's geometry."""
        pool = torch.zeros(self.n_pages, self.page_elems, dtype=torch.bfloat16, device=device)
        pl = torch.zeros(self.page_list_len, dtype=torch.int32, device=device)
        desc = torch.zeros(self.n_adapters * 16, dtype=torch.uint8, device=device)
        return PoolView(pool, pl, desc, self.page_elems, self.max_rank, self.d_in, self.d_out)

    def load(self, adapter: int, rank: int, scale: float, A, B, view: PoolView, stream=None):
        lora_pool_load(self.h, adapter, rank, scale, A, B, view, stream)

    def evict(self, adapter: int, view: PoolView, stream=None):
        lora_pool_evict(self.h, adapter, view, stream)
