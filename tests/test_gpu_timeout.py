"""The kernels' bounded waits, exercised without any fault: with the test-only
timeout probe armed, every CTA waits (about a millisecond at most) on a barrier that
nothing arrives on, gives up, flags LORA_DERR_TIMEOUT and writes nothing; the
context stays usable and the next call, with the probe disarmed, is correct."""

import numpy as np
import pytest
import torch

from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import compare_bf16, cuda_or_skip, ids_dev, new_err, oracle_apply, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

PROBE_CYCLES = 2_000_000  # about a millisecond at the GB300's clocks


@pytest.fixture(autouse=True)
def _cuda():
    cuda_or_skip()
    yield
    B.debug_wait_probe(0)  # never leave the probe armed for later tests


def mixed_batch(seed):
    """Long segments (fused tensor-core kernel) and short ones (gather kernel)."""
    rng = np.random.default_rng(seed)
    ranks = [16, 64, 8, 32]
    pool = W.build_pool(rng, 4096, 2048, ranks, max_rank=64)
    lens = [300, 3, 200, 1, 2, 140]
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    return pool, W.make_batch(rng, ids, 4096, 2048)


def test_timeout_flags_and_leaves_outputs_then_recovers():
    pool, batch = mixed_batch(61)
    view = B.PoolView.from_host(pool)
    x = to_dev_bits(batch.x)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), pool.n_adapters, seg, mode=B.LORA_SEG_GROUP, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    B.debug_wait_probe(PROBE_CYCLES)
    y = to_dev_bits(batch.y0)
    B.lora_apply(x, y, seg, view, err=err)  # gather kernel, then the fused kernel
    yb = to_dev_bits(batch.y0)
    errb = new_err()
    B.lora_bgmv(x, yb, ids_dev(batch.ids), view, err=errb)
    torch.cuda.synchronize()
    assert int(err.item()) & B.LORA_DERR_TIMEOUT
    assert int(errb.item()) & B.LORA_DERR_TIMEOUT
    assert np.array_equal(to_host_bits(y), batch.y0), "a CTA that gave up wrote output"
    assert np.array_equal(to_host_bits(yb), batch.y0)

    B.debug_wait_probe(0)
    err.zero_()
    y = to_dev_bits(batch.y0)
    B.lora_apply(x, y, seg, view, err=err)  # the same segment buffer: its counters are back at zero
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _ = oracle_apply(batch.x, batch.y0, batch.ids, pool)
    compare_bf16(to_host_bits(y), ref, "after the timeout probe")


@pytest.mark.parametrize("static", [False, True])
def test_timeout_on_the_decode_kernel(static):
    """The decode kernel (small adapters, one token per cluster) takes the same exit,
    with and without LORA_BGMV_STATIC_ADAPTERS; the next call is correct."""
    rng = np.random.default_rng(62)
    pool = W.build_pool(rng, 4096, 4096, [16, 8, 16, 4], max_rank=16)
    ids = rng.integers(-1, 4, size=24).astype(np.int32)
    batch = W.make_batch(rng, ids, 4096, 4096)
    view = B.PoolView.from_host(pool)
    x = to_dev_bits(batch.x)
    idt = ids_dev(ids)
    B.debug_wait_probe(PROBE_CYCLES)
    y = to_dev_bits(batch.y0)
    err = new_err()
    B.lora_bgmv(x, y, idt, view, err=err, static_adapters=static)
    torch.cuda.synchronize()
    assert int(err.item()) & B.LORA_DERR_TIMEOUT
    assert np.array_equal(to_host_bits(y), batch.y0), "a CTA that gave up wrote output"
    B.debug_wait_probe(0)
    err.zero_()
    B.lora_bgmv(x, y, idt, view, err=err, static_adapters=static)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _ = oracle_apply(batch.x, batch.y0, ids, pool)
    compare_bf16(to_host_bits(y), ref, "after the timeout probe")
