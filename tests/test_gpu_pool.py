"""GPU: adapters made resident on demand by lora_pool_load (include/lora_pool.h), with
evictions along the way, then served by lora_apply and lora_bgmv.  The device pool holds each
resident adapter's A and B bit for bit (compared with the host matrices they were copied from),
and the outputs match the fp64 oracle run on a host-built pool of the same adapters
("Multi-LoRA Serving in Production", sections "Unified Paged Memory", "Tiered Storage
Hierarchy and Asynchronous Streaming" and "Eviction and Replacement Policies")."""

import dataclasses
import time

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import compare_bf16, cuda_or_skip, ids_dev, new_err, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

D_IN, D_OUT, P, N_AD = 1024, 2048, 4096, 24


@pytest.fixture(autouse=True)
def _cuda():
    cuda_or_skip()


def pinned(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()


def device_state(view):
    pool = to_host_bits(view.pool)
    pl = view.page_list.cpu().numpy()
    desc = view.adapters.cpu().numpy().view(W.DESC_DTYPE)
    return pool, pl, desc


def logical(pool, pl, slot0, n_elems):
    """A matrix read back through its page-list slots (host indexing of device bytes)."""
    npg = -(-n_elems // P)
    return np.concatenate([pool[pl[slot0 + k]] for k in range(npg)])[:n_elems]


def check_resident(mgr, view, ref):
    pool, pl, desc = device_state(view)
    held = []
    S = mgr.slots_per_adapter
    for a in range(N_AD):
        r = mgr.resident_rank(a)
        assert int(desc[a]["rank"]) == r, a
        if r == 0:
            continue
        na = -(-r * D_IN // P)
        nb = -(-r * D_OUT // P)
        assert (int(desc[a]["a_page0"]), int(desc[a]["b_page0"])) == (a * S, a * S + na)
        assert np.float32(desc[a]["scale"]) == np.float32(ref.desc[a]["scale"])
        assert np.array_equal(logical(pool, pl, a * S, r * D_IN), ref.A[a].reshape(-1)), a
        assert np.array_equal(logical(pool, pl, a * S + na, r * D_OUT), ref.B[a].reshape(-1)), a
        held += list(pl[a * S: a * S + na + nb])
    assert len(held) == len(set(held)) and all(0 <= p < mgr.n_pages for p in held)
    assert mgr.free_pages == mgr.n_pages - len(held)


def test_loads_with_evictions_serve_batches():
    rng = np.random.default_rng(71)
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=N_AD)
    ref = W.build_pool(rng, D_IN, D_OUT, ranks, max_rank=64)  # the oracle's pool
    host_A = [pinned(ref.A[a]) for a in range(N_AD)]
    host_B = [pinned(ref.B[a]) for a in range(N_AD)]
    # 200 pages: four rank-64 adapters (48 pages each) fit, the catalogue does not
    mgr = B.PoolManager(200, P, N_AD, 64, D_IN, D_OUT)
    view = mgr.device_view()
    copy = torch.cuda.Stream()
    err = new_err()
    seen_evicted = 0
    for rd in range(10):
        chosen = rng.choice(N_AD, size=4, replace=False)
        # two long segments (tensor-core path), short ones, and tokens without an adapter
        ids = np.concatenate([np.full(int(rng.integers(20, 150)), chosen[0]), np.full(40, chosen[1]),
                              rng.choice(chosen[2:], size=12), np.full(3, -1)]).astype(np.int32)
        ids = ids[rng.permutation(ids.size)] if rd % 2 else ids
        batch = W.make_batch(rng, ids, D_IN, D_OUT)
        before = [mgr.resident_rank(a) for a in range(N_AD)]
        with torch.cuda.stream(copy):
            for a in chosen:
                mgr.load(int(a), int(ranks[a]), float(ref.desc[a]["scale"]), host_A[a], host_B[a], view,
                         stream=copy)
                mgr.pin(int(a))
        ready = torch.cuda.Event()
        ready.record(copy)
        torch.cuda.current_stream().wait_event(ready)
        after = [mgr.resident_rank(a) for a in range(N_AD)]
        seen_evicted += sum(1 for a in range(N_AD) if before[a] and not after[a])
        x, y = to_dev_bits(batch.x), to_dev_bits(batch.y0)
        seg = B.Segments(len(ids))
        B.lora_segments_build(ids_dev(ids), N_AD, seg, mode=B.LORA_SEG_GROUP, err=err)
        B.lora_apply(x, y, seg, view, err=err)
        torch.cuda.synchronize()
        want, oerr = oracle.lora_apply(batch.x, batch.y0, ids, ref)
        assert int(err.item()) == oerr == 0, rd
        compare_bf16(to_host_bits(y)[:, :D_OUT], want, "pool round %d" % rd)
        check_resident(mgr, view, ref)
        for a in chosen:
            mgr.unpin(int(a))
    assert seen_evicted > 0


def test_evicted_adapter_is_flagged_and_its_rows_left_alone():
    rng = np.random.default_rng(72)
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=N_AD)
    ref = W.build_pool(rng, D_IN, D_OUT, ranks, max_rank=64)
    mgr = B.PoolManager(400, P, N_AD, 64, D_IN, D_OUT)
    view = mgr.device_view()
    for a in (2, 5, 7):  # pageable numpy sources
        mgr.load(a, int(ranks[a]), float(ref.desc[a]["scale"]), ref.A[a], ref.B[a], view)
    mgr.evict(5, view)
    ids = np.array([2, 5, 7, 5, -1, 2, 7, 7, 5, 2, 11], dtype=np.int32)
    batch = W.make_batch(rng, ids, D_IN, D_OUT)
    masked = dataclasses.replace(ref, desc=ref.desc.copy())
    for a in range(N_AD):
        if a not in (2, 7):
            masked.desc[a]["rank"] = 0  # not resident on the device either
    want, oerr = oracle.lora_apply(batch.x, batch.y0, ids, masked)
    assert oerr == B.LORA_DERR_BAD_RANK
    x, y = to_dev_bits(batch.x), to_dev_bits(batch.y0)
    err = new_err()
    B.lora_bgmv(x, y, ids_dev(ids), view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == oerr
    yh = to_host_bits(y)
    good = (ids == 2) | (ids == 7)
    compare_bf16(yh[good][:, :D_OUT], want[good], "resident rows next to evicted ones")
    assert np.array_equal(yh[~good], batch.y0[~good])
    check_resident(mgr, view, ref)


def test_load_throughput_from_pinned_host_memory():
    """Host-to-device rate of lora_pool_load for 48 rank-64 adapters of an MLP up projection
    (4096 -> 11008, 1.9 MB each) from pinned memory, one stream, timed with CUDA events."""
    rng = np.random.default_rng(73)
    d_in, d_out, n = 4096, 11008, 48
    per = -(-64 * d_in // P) + -(-64 * d_out // P)
    mgr = B.PoolManager(n * per, P, n, 64, d_in, d_out)
    view = mgr.device_view()
    A = pinned(rng.integers(0, 1 << 14, size=(64, d_in), dtype=np.uint16))
    Bm = pinned(rng.integers(0, 1 << 14, size=(64, d_out), dtype=np.uint16))
    s = torch.cuda.Stream()
    for a in range(4):  # warm-up: first launches, first copies
        mgr.load(a, 64, 0.25, A, Bm, view, stream=s)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(s)
    for a in range(4, n):
        mgr.load(a, 64, 0.25, A, Bm, view, stream=s)
    e1.record(s)
    torch.cuda.synchronize()
    host_s = time.perf_counter() - t0
    nbytes = (n - 4) * 64 * (d_in + d_out) * 2
    gbs = nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    print("\npool load: %d adapters, %.1f MB, %.1f GB/s on the device clock, %.1f GB/s host wall"
          % (n - 4, nbytes / 1e6, gbs, nbytes / host_s / 1e9))
    assert gbs > 1.0
    pool, pl, desc = device_state(view)
    S = mgr.slots_per_adapter
    for a in (4, n - 1):
        assert np.array_equal(logical(pool, pl, a * S, 64 * d_in), A.numpy().view(np.uint16).reshape(-1))
        assert np.array_equal(logical(pool, pl, a * S + 64, 64 * d_out), Bm.numpy().view(np.uint16).reshape(-1))
