"""The C-ABI library on the host: it loads, exports every symbol include/*.h
declares, and rejects bad arguments before launching anything (no GPU needed)."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
from segmented_gather_gemm_lora_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    L = B.lib()
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(B.EXPORTED) == set(names)


def test_header_constants_match_the_binding():
    text = "".join(open(h).read() for h in HEADERS)
    defs = re.findall(r"#define\s+(LORA_[A-Z0-9_]+)\s+\(?(-?\d+)u?\)?", text)
    assert len(defs) >= 17
    for name, value in defs:
        if name in ("LORA_ABI_VERSION", "LORA_KSPLIT_MAX"):
            continue
        assert getattr(B, name) == int(value), name


def test_abi_version_and_status_strings():
    assert B.lora_abi_version() == 1
    assert B.lora_status_string(0) == "ok"
    assert "invalid" in B.lora_status_string(-1)
    assert "unsupported" in B.lora_status_string(-2)
    assert B.lora_status_string(-99) == "unknown status"


def test_struct_sizes_match_c_layout():
    assert ctypes.sizeof(B.lora_adapter_desc_t) == 16
    assert ctypes.sizeof(B.lora_pool_view_t) == 64
    assert ctypes.sizeof(B.lora_segments_t) == 8 + 9 * 8


@pytest.mark.parametrize("rank,d_in,d_out,P", [(16, 8192, 8192, 4096), (13, 5120, 11008, 4096),
                                                (64, 13824, 5120, 4096), (1, 8, 8, 64)])
def test_pages_needed_matches_oracle(rank, d_in, d_out, P):
    assert B.lora_pool_pages_needed(rank, d_in, d_out, P) == oracle.pages_needed(rank, d_in, d_out, P)


def test_carve_layout():
    L = B.lib()
    for T in (0, 1, 16, 64, 129, 9216):
        n = B.lora_segments_buffer_bytes(T)
        assert n % 16 == 0 and n >= 4 * (4 * T + 8) + 4 * 64 * T * (1 + 8)
        buf = (ctypes.c_uint8 * (n + 16))()
        base = (ctypes.addressof(buf) + 15) // 16 * 16
        s = B.lora_segments_t()
        assert L.lora_segments_carve(ctypes.c_void_p(base), n, T, ctypes.byref(s)) == 0
        assert s.T == T
        assert s.max_long_units == T // B.LORA_TILE_M + T // (B.LORA_SHORT_MAX_TOKENS + 1) + 1
        ptrs = [s.token_perm, s.seg_indptr, s.seg_adapter, s.meta, s.short_units, s.long_units, s.scratch,
                s.h_scratch, s.k_partials]
        assert all(p % 16 == 0 for p in ptrs)
        assert ptrs == sorted(ptrs) and ptrs[0] == base
        assert L.lora_segments_carve(ctypes.c_void_p(base), n - 16, T, ctypes.byref(s)) == B.LORA_ERR_WORKSPACE
        assert L.lora_segments_carve(ctypes.c_void_p(base + 4), n, T, ctypes.byref(s)) == B.LORA_ERR_INVALID_ARG


def fake_view(**kw):
    v = dict(pool=0x10000, n_pages=10, page_list=0x20000, n_page_list=10, adapters=0x30000,
             n_adapters=4, page_elems=4096, max_rank=16, d_in=256, d_out=256)
    v.update(kw)
    return B.lora_pool_view_t(v["pool"], v["n_pages"], v["page_list"], v["n_page_list"], v["adapters"],
                              v["n_adapters"], v["page_elems"], v["max_rank"], v["d_in"], v["d_out"])


def fake_seg(T=16):
    s = B.lora_segments_t()
    s.T = T
    s.max_long_units = T // B.LORA_TILE_M + T // (B.LORA_SHORT_MAX_TOKENS + 1) + 1
    for i, f in enumerate(("token_perm", "seg_indptr", "seg_adapter", "meta", "short_units",
                           "long_units", "scratch", "h_scratch", "k_partials")):
        setattr(s, f, 0x100000 + 0x1000 * i)
    return s


@pytest.mark.parametrize("bad,want", [
    (dict(pool=0x10008), B.LORA_ERR_INVALID_ARG),  # misaligned pool
    (dict(pool=0), B.LORA_ERR_INVALID_ARG),
    (dict(d_in=250), B.LORA_ERR_INVALID_ARG),  # not a multiple of 8
    (dict(d_out=0), B.LORA_ERR_INVALID_ARG),
    (dict(max_rank=0), B.LORA_ERR_INVALID_ARG),
    (dict(max_rank=65), B.LORA_ERR_UNSUPPORTED),
    (dict(page_elems=4004), B.LORA_ERR_INVALID_ARG),  # not a multiple of 8
    (dict(page_elems=3072), B.LORA_ERR_UNSUPPORTED),  # not a power of two
    (dict(page_elems=32), B.LORA_ERR_UNSUPPORTED),
    (dict(n_adapters=0), B.LORA_ERR_INVALID_ARG),
])
def test_apply_rejects_bad_views_without_launch(bad, want):
    L = B.lib()
    seg = fake_seg()
    v = fake_view(**bad)
    rc = L.lora_apply(ctypes.c_void_p(0x400000), 256, ctypes.c_void_p(0x800000), 256, ctypes.byref(seg),
                      ctypes.byref(v), None, None)
    assert rc == want


def test_apply_rejects_bad_activations_without_launch():
    L = B.lib()
    seg = fake_seg(16)
    v = fake_view()
    x, y = ctypes.c_void_p(0x400000), ctypes.c_void_p(0x800000)
    # misaligned, short stride, stride not a multiple of 8, x overlapping y
    assert L.lora_apply(ctypes.c_void_p(0x400002), 256, y, 256, ctypes.byref(seg), ctypes.byref(v), None, None) == -1
    assert L.lora_apply(x, 128, y, 256, ctypes.byref(seg), ctypes.byref(v), None, None) == -1
    assert L.lora_apply(x, 260, y, 256, ctypes.byref(seg), ctypes.byref(v), None, None) == -1
    assert L.lora_apply(x, 256, ctypes.c_void_p(0x400000 + 512 * 8), 256, ctypes.byref(seg),
                        ctypes.byref(v), None, None) == -1
    assert L.lora_apply(x, 256, y, 256, None, ctypes.byref(v), None, None) == -1
    # a segment buffer carved for more tokens than it can hold
    small = fake_seg(16)
    small.max_long_units -= 1  # one long unit fewer than 16 tokens can need
    assert L.lora_apply(x, 256, y, 256, ctypes.byref(small), ctypes.byref(v), None, None) == B.LORA_ERR_WORKSPACE


def test_other_entry_points_reject_bad_arguments():
    L = B.lib()
    seg = fake_seg(16)
    v = fake_view()
    x, y, h = ctypes.c_void_p(0x400000), ctypes.c_void_p(0x800000), ctypes.c_void_p(0xC00000)
    assert L.lora_sgmv_shrink(x, 256, h, 8, ctypes.byref(seg), ctypes.byref(v), None, None) == -1  # ldh < max_rank
    assert L.lora_sgmv_shrink(x, 256, h, 18, ctypes.byref(seg), ctypes.byref(v), None, None) == -1  # ldh % 4
    assert L.lora_sgmv_expand(h, 16, y, 100, ctypes.byref(seg), ctypes.byref(v), None, None) == -1
    assert L.lora_bgmv(x, 256, y, 256, None, 4, ctypes.byref(v), None, None) == -1
    assert L.lora_bgmv(x, 256, y, 256, ctypes.c_void_p(0x900000), -1, ctypes.byref(v), None, None) == -1
    assert L.lora_segments_build(ctypes.c_void_p(0x900000), 16, 4, 2, ctypes.byref(seg), None, None) == -1
    assert L.lora_segments_build(ctypes.c_void_p(0x900000), 16, 0, 0, ctypes.byref(seg), None, None) == -1
    assert L.lora_segments_build(ctypes.c_void_p(0x900000), 16, 40000, 0, ctypes.byref(seg), None, None) == -2
    assert L.lora_segments_build(ctypes.c_void_p(0x900000), 17, 4, 0, ctypes.byref(seg), None, None) == -1


def test_empty_batches_are_noops_without_launch():
    L = B.lib()
    seg = fake_seg(0)
    v = fake_view()
    assert L.lora_apply(None, 256, None, 256, ctypes.byref(seg), ctypes.byref(v), None, None) == 0
    assert L.lora_bgmv(None, 256, None, 256, None, 0, ctypes.byref(v), None, None) == 0
    assert L.lora_sgmv_shrink(None, 256, None, 16, ctypes.byref(seg), ctypes.byref(v), None, None) == 0


def test_apply_multi_rejects_bad_groups_on_the_host():
    """Argument checks of lora_apply_multi happen before any launch (no GPU needed)."""
    L = B.lib()
    seg = B.lora_segments_t()
    seg.T = 0  # nothing to launch even when the arguments pass
    projs = (B.lora_proj_t * 2)()
    for i in range(2):
        v = projs[i].view
        v.pool, v.n_pages, v.page_list, v.n_page_list = 0x100000, 4, 0x200000, 8
        v.adapters, v.n_adapters, v.page_elems, v.max_rank = 0x300000, 2, 4096, 16
        v.d_in, v.d_out = 4096, 1024
        projs[i].x, projs[i].ldx, projs[i].y, projs[i].ldy = 0x400000, 4096, 0x800000 + i * 0x100000, 1024
    assert L.lora_apply_multi(projs, 2, ctypes.byref(seg), None, None) == B.LORA_OK
    assert L.lora_apply_multi(projs, 0, ctypes.byref(seg), None, None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_apply_multi(projs, B.LORA_MAX_PROJ + 1, ctypes.byref(seg), None, None) == B.LORA_ERR_UNSUPPORTED
    projs[1].view.d_in = 2048
    assert L.lora_apply_multi(projs, 2, ctypes.byref(seg), None, None) == B.LORA_ERR_INVALID_ARG
    projs[1].view.d_in = 4096
    projs[1].view.max_rank = 65
    assert L.lora_apply_multi(projs, 2, ctypes.byref(seg), None, None) == B.LORA_ERR_UNSUPPORTED


def _width_rule(shapes):
    """The gather kernel's width rule restated: fewest 512-column stages per unit among
    w0 / 2 .. w0, ties to the wider."""
    d = max(max(a, b) for a, b in shapes)
    w0 = min(max(-(-d // 512), 1), 8)
    best, best_cost = w0, None
    for w in range(w0, max(1, w0 // 2) - 1, -1):
        cost = 0
        for a, b in shapes:
            kc = (-(-a // w) + 7) // 8 * 8
            nc = (-(-b // w) + 7) // 8 * 8
            cost += w * (-(-kc // 512) + -(-nc // 512))
        if best_cost is None or cost < best_cost:
            best, best_cost = w, cost
    return best


def test_gather_cluster_width():
    """The widths of the benchmark's projections (host only), a restatement of the rule on
    random shapes, and the argument checks."""
    assert B.debug_gather_width([(5120, 5120)] * 3) == 5  # 13B-shaped q, k, v: 1024 columns a CTA
    assert B.debug_gather_width([(5120, 13824)] * 2) == 5
    assert B.debug_gather_width([(13824, 5120)]) == 5
    assert B.debug_gather_width([(4096, 11008)]) == 8
    assert B.debug_gather_width([(11008, 4096)]) == 8
    assert B.debug_gather_width([(4096, 4096)]) == 8
    assert B.debug_gather_width([(256, 256)]) == 1
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(1, 4))
        shapes = [(8 * int(rng.integers(1, 2200)), 8 * int(rng.integers(1, 2200))) for _ in range(n)]
        assert B.debug_gather_width(shapes) == _width_rule(shapes), shapes
    assert B.debug_gather_width([]) == -1
    assert B.debug_gather_width([(4, 4096)]) == -1
    assert B.debug_gather_width([(4096, 4096)] * (B.LORA_MAX_PROJ + 1)) == -1
