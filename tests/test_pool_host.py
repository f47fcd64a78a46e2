"""Pool residency on the host (include/lora_pool.h): page accounting, least-recently-used
eviction, pins, and argument checks, against a plain Python model of the policy ("Multi-LoRA
Serving in Production", sections "Unified Paged Memory" and "Eviction and Replacement
Policies").  No GPU: every call here is host bookkeeping or is rejected before any launch."""

import ctypes
import threading

import numpy as np
import pytest

from segmented_gather_gemm_lora_gb300 import binding as B


def ceil_div(a, b):
    return -(-a // b)


class Model:
    """The policy as the header states it, written out plainly: free pages handed out lowest
    first; a reserve of a resident adapter with the same rank only refreshes its last use;
    otherwise its own pages (other rank) and then the least recently used unpinned adapters
    are released until enough pages are free, or nothing changes."""

    def __init__(self, n_pages, P, n_ad, max_rank, d_in, d_out):
        self.free = set(range(n_pages))
        self.P, self.n_ad, self.max_rank, self.d_in, self.d_out = P, n_ad, max_rank, d_in, d_out
        self.rank = {}
        self.pages = {}
        self.pins = {}
        self.order = []  # least recent first
        self.counts = dict(hits=0, loads=0, refused=0, evictions=0, pages_loaded=0)

    def need(self, r):
        return ceil_div(r * self.d_in, self.P) + ceil_div(r * self.d_out, self.P)

    def _release(self, a):
        self.free |= set(self.pages.pop(a))
        del self.rank[a]
        self.order.remove(a)

    def reserve(self, a, r):
        if not (0 <= a < self.n_ad and 1 <= r <= self.max_rank):
            return "invalid", None, None
        if self.rank.get(a) == r:
            self.order.remove(a)
            self.order.append(a)
            self.counts["hits"] += 1
            return "ok", [], []
        again = a in self.rank
        if again and self.pins.get(a, 0) > 0:
            return "invalid", None, None
        avail = len(self.free) + (len(self.pages[a]) if again else 0)
        ev = [a] if again else []
        for e in self.order:
            if avail >= self.need(r):
                break
            if e == a or self.pins.get(e, 0) > 0:
                continue
            avail += len(self.pages[e])
            ev.append(e)
        if avail < self.need(r):
            self.counts["refused"] += 1
            return "workspace", None, None
        for e in ev:
            self._release(e)
        got = sorted(self.free)[: self.need(r)]
        self.free -= set(got)
        self.pages[a] = got
        self.rank[a] = r
        self.order.append(a)
        self.counts["loads"] += 1
        self.counts["evictions"] += len(ev)
        self.counts["pages_loaded"] += len(got)
        return "ok", got, ev

    def pin(self, a):
        if a not in self.rank:
            return "invalid"
        self.pins[a] = self.pins.get(a, 0) + 1
        return "ok"

    def unpin(self, a):
        if self.pins.get(a, 0) <= 0:
            return "invalid"
        self.pins[a] -= 1
        return "ok"

    def release(self, a):
        if a not in self.rank:
            return "ok"
        if self.pins.get(a, 0) > 0:
            return "invalid"
        self._release(a)
        return "ok"


def status_of(fn, *args):
    try:
        out = fn(*args)
        return "ok", out
    except B.LoraError as e:
        return {B.LORA_ERR_INVALID_ARG: "invalid", B.LORA_ERR_WORKSPACE: "workspace"}[e.status], None


def test_geometry_and_slots():
    m = B.PoolManager(1000, 4096, 50, 64, 5120, 13824)
    per = ceil_div(64 * 5120, 4096) + ceil_div(64 * 13824, 4096)
    assert m.slots_per_adapter == per == 80 + 216
    assert m.page_list_len == 50 * per
    assert m.free_pages == 1000
    for r in (1, 8, 16, 33, 64):
        assert ceil_div(r * 5120, 4096) + ceil_div(r * 13824, 4096) == B.lora_pool_pages_needed(r, 5120, 13824, 4096)
    m.close()


@pytest.mark.parametrize("args", [
    (0, 4096, 8, 16, 1024, 1024),        # no pages
    (100, 3000, 8, 16, 1024, 1024),      # page size not a power of two
    (100, 32, 8, 16, 1024, 1024),        # page size below 64
    (100, 4096, 0, 16, 1024, 1024),      # no adapters
    (100, 4096, 40000, 16, 1024, 1024),  # too many adapters
    (100, 4096, 8, 65, 1024, 1024),      # rank above the build's maximum
    (100, 4096, 8, 16, 1020, 1024),      # d_in not a multiple of 8
    (1 << 31, 4096, 8, 16, 1024, 1024),  # page ids beyond int32
])
def test_bad_geometry_is_rejected(args):
    with pytest.raises(B.LoraError) as e:
        B.PoolManager(*args)
    assert e.value.status == B.LORA_ERR_INVALID_ARG


def check_invariants(m, model):
    held = []
    for a in range(model.n_ad):
        r = m.resident_rank(a)
        assert r == model.rank.get(a, 0)
        if r:
            held += model.pages[a]
    assert len(held) == len(set(held))
    assert all(0 <= p < m.n_pages for p in held)
    assert m.free_pages == m.n_pages - len(held) == len(model.free)


@pytest.mark.parametrize("seed", range(4))
def test_policy_matches_the_model_under_random_traffic(seed):
    rng = np.random.default_rng(seed)
    n_pages = int(rng.integers(40, 300))
    d_in, d_out = [(1024, 1024), (4096, 11008), (5120, 13824), (256, 512)][seed]
    P = [4096, 4096, 8192, 1024][seed]
    n_ad = 30
    m = B.PoolManager(n_pages, P, n_ad, 64, d_in, d_out)
    model = Model(n_pages, P, n_ad, 64, d_in, d_out)
    evictions = workspace = 0
    for step in range(3000):
        op = rng.random()
        a = int(rng.integers(-1, n_ad + 1))
        if op < 0.6:
            r = int(rng.choice([0, 8, 16, 32, 64, 65, int(rng.integers(1, 65))]))
            want = model.reserve(a, r)
            got, out = status_of(m.reserve, a, r)
            assert got == want[0], (step, a, r)
            if got == "ok":
                pages, ev = out
                assert list(pages) == want[1], step
                assert list(ev) == want[2], step
                evictions += len(ev)
            workspace += got == "workspace"
        elif op < 0.75:
            assert status_of(m.pin, a)[0] == (model.pin(a) if 0 <= a < n_ad else "invalid")
        elif op < 0.9:
            assert status_of(m.unpin, a)[0] == (model.unpin(a) if 0 <= a < n_ad else "invalid")
        else:
            assert status_of(m.release, a)[0] == (model.release(a) if 0 <= a < n_ad else "invalid")
        if step % 50 == 0:
            check_invariants(m, model)
    check_invariants(m, model)
    assert evictions > 20 and workspace > 0  # the traffic reached both paths
    want = dict(model.counts, resident=len(model.rank),
                pinned=sum(1 for a in model.rank if model.pins.get(a, 0) > 0))
    assert m.stats() == want
    m.close()


def test_lru_order_pins_and_rank_change():
    # 1024 x 1024, pages of 4096: a rank-16 adapter holds 4 + 4 pages
    m = B.PoolManager(24, 4096, 8, 32, 1024, 1024)
    for a in (0, 1, 2):
        pages, ev = m.reserve(a, 16)
        assert len(pages) == 8 and len(ev) == 0
    assert m.free_pages == 0
    assert list(m.reserve(0, 16)[0]) == []  # resident: only refreshed, so 1 is now the oldest
    m.pin(1)
    pages, ev = m.reserve(3, 16)  # 1 is pinned: 2 goes
    assert list(ev) == [2] and m.resident_rank(2) == 0
    assert sorted(pages) == list(range(16, 24))  # 2's pages, reused
    with pytest.raises(B.LoraError):
        m.reserve(1, 8)  # pinned, other rank
    with pytest.raises(B.LoraError):
        m.release(1)  # pinned
    m.pin(0)
    m.pin(3)
    with pytest.raises(B.LoraError) as e:
        m.reserve(4, 16)  # everything pinned
    assert e.value.status == B.LORA_ERR_WORKSPACE
    assert [m.resident_rank(a) for a in range(5)] == [16, 16, 0, 16, 0]  # unchanged
    m.unpin(3)
    with pytest.raises(B.LoraError):
        m.reserve(3, 32)  # its own 8 pages are not enough and 0 and 1 are pinned
    m.unpin(0)
    pages, ev = m.reserve(3, 32)  # rank change: its own pages go first, then the oldest unpinned (0)
    assert list(ev) == [3, 0] and m.resident_rank(3) == 32 and m.resident_rank(0) == 0
    assert list(pages) == list(range(0, 8)) + list(range(16, 24))
    with pytest.raises(B.LoraError):
        m.unpin(3)  # not pinned any more
    m.close()


def test_concurrent_threads_keep_the_books():
    m = B.PoolManager(200, 4096, 64, 64, 2048, 2048)

    def worker(seed):
        rng = np.random.default_rng(seed)
        for _ in range(2000):
            a = int(rng.integers(0, 64))
            if rng.random() < 0.8:
                try:
                    m.reserve(a, int(rng.choice([8, 16, 32, 64])))
                except B.LoraError:
                    pass
            else:
                m.release(a)

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(6)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    held = 0
    for a in range(64):
        r = m.resident_rank(a)
        held += B.lora_pool_pages_needed(r, 2048, 2048, 4096) if r else 0
    assert m.free_pages == 200 - held
    m.close()


def test_device_calls_reject_bad_arguments_before_any_launch():
    m = B.PoolManager(64, 4096, 8, 16, 1024, 1024)
    L = B.lib()
    host = np.zeros(16 * 1024, dtype=np.uint16)
    hp = ctypes.c_void_p(host.ctypes.data)

    def view(**kw):
        v = B.lora_pool_view_t(0x10000, 64, 0x20000, m.page_list_len, 0x30000, 8, 4096, 16, 1024, 1024)
        for k, val in kw.items():
            setattr(v, k, val)
        return v

    good = view()
    for bad in (view(n_pages=65), view(page_elems=8192), view(n_adapters=9), view(max_rank=32),
                view(d_in=2048), view(d_out=512), view(n_page_list=m.page_list_len - 1), view(pool=0),
                view(adapters=0)):
        assert L.lora_pool_load(m.h, 1, 16, 1.0, hp, hp, ctypes.byref(bad), None) == B.LORA_ERR_INVALID_ARG
        assert L.lora_pool_evict(m.h, 1, ctypes.byref(bad), None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_load(m.h, 1, 16, 1.0, None, hp, ctypes.byref(good), None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_load(m.h, 8, 16, 1.0, hp, hp, ctypes.byref(good), None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_load(m.h, 1, 17, 1.0, hp, hp, ctypes.byref(good), None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_load(None, 1, 16, 1.0, hp, hp, ctypes.byref(good), None) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_evict(m.h, 3, ctypes.byref(good), None) == B.LORA_OK  # not resident: nothing to do
    assert m.free_pages == 64
    assert L.lora_pool_mgr_page_list_len(None) == -1 and L.lora_pool_mgr_free_pages(None) == -1
    assert L.lora_pool_resident_rank(m.h, 8) == -1
    m.close()


def test_reserve_rejects_short_output_buffers_and_nulls():
    m = B.PoolManager(64, 4096, 8, 16, 1024, 1024)
    L = B.lib()
    S = m.slots_per_adapter
    pages = (ctypes.c_int32 * S)()
    ev = (ctypes.c_int32 * 8)()
    n_p, n_e = ctypes.c_int32(-7), ctypes.c_int32(-7)
    args = lambda pcap, ecap: (m.h, 1, 16, pages, pcap, ctypes.byref(n_p), ev, ecap, ctypes.byref(n_e))
    assert L.lora_pool_mgr_reserve(*args(S - 1, 8)) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_mgr_reserve(*args(S, 7)) == B.LORA_ERR_INVALID_ARG
    assert L.lora_pool_mgr_reserve(m.h, 1, 16, None, S, ctypes.byref(n_p), ev, 8, ctypes.byref(n_e)) == -1
    assert L.lora_pool_mgr_reserve(m.h, 1, 16, pages, S, None, ev, 8, ctypes.byref(n_e)) == -1
    assert L.lora_pool_mgr_reserve(None, 1, 16, pages, S, ctypes.byref(n_p), ev, 8, ctypes.byref(n_e)) == -1
    assert (n_p.value, n_e.value) == (-7, -7) and m.free_pages == 64  # nothing written, nothing taken
    assert L.lora_pool_mgr_reserve(*args(S, 8)) == B.LORA_OK and (n_p.value, n_e.value) == (8, 0)
    assert list(pages[:8]) == list(range(8))
    assert L.lora_pool_pin(None, 1) == -1 and L.lora_pool_unpin(m.h, 99) == -1
    assert L.lora_pool_mgr_stats(m.h, None) == -1 and L.lora_pool_mgr_release(m.h, -1) == -1
    m.close()
