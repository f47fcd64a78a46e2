"""lora_apply_fixed_scratch: the entry point for callers that cannot allocate device
memory (their device memory is planned once by a host runtime, so they cannot size
or request the workspace the staged tensor-core path keeps its intermediate in).  It
must give the same outputs as lora_apply, bit for bit, call after call, although
every call reuses the one fixed array inside the library, and it must not touch the
caller's h_scratch (passed as NULL here, so a call that still used it would fail).

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import compare_bf16, cuda_or_skip, ids_dev, new_err, oracle_apply, to_dev_bits, to_host_bits


def batch_with_long_and_short_segments(seed):
    """Long segments (tensor-core path, which uses the scratch) next to short ones."""
    rng = np.random.default_rng(seed)
    ranks = [16, 64, 7, 32, 8]
    pool = W.build_pool(rng, 4096, 2048, ranks, max_rank=64)
    lens = [300, 129, 5, 200, 1, 2, 140]
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    ids = ids[rng.permutation(ids.size)] if seed % 2 else ids
    batch = W.make_batch(rng, ids, 4096, 2048)
    return pool, batch


def run(entry, pool, batch, view, no_h_scratch=False):
    x = to_dev_bits(batch.x)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), pool.n_adapters, seg, mode=B.LORA_SEG_GROUP, err=err)
    if no_h_scratch:
        seg.c.h_scratch = None  # the fixed-scratch call must not read or write it
    entry(x, y, seg, view, err=err)
    torch.cuda.synchronize()
    return to_host_bits(y), int(err.item())


@pytest.mark.gpu
def test_fixed_scratch_matches_lora_apply_on_two_calls_in_a_row():
    cuda_or_skip()
    cases = [batch_with_long_and_short_segments(s) for s in (1, 2)]
    views = [B.PoolView.from_host(pool) for pool, _ in cases]
    # two calls of the fixed-scratch entry point back to back, then the reference calls
    fixed = [run(B.lora_apply_fixed_scratch, pool, batch, view, no_h_scratch=True)
             for (pool, batch), view in zip(cases, views)]
    for ((pool, batch), view), (y_fixed, e_fixed) in zip(zip(cases, views), fixed):
        y_ref, e_ref = run(B.lora_apply, pool, batch, view)
        assert e_fixed == e_ref == 0
        assert np.array_equal(y_fixed, y_ref), "fixed scratch differs from lora_apply"
        ref, oerr = oracle_apply(batch.x, batch.y0, batch.ids, pool)
        assert oerr == 0
        compare_bf16(y_fixed, ref, "fixed scratch vs oracle")


def test_fixed_scratch_rejects_batches_above_its_limit():
    """Checked on the host before anything else, so no GPU is needed."""
    L = B.lib()
    T = B.LORA_FIXED_SCRATCH_MAX_TOKENS + 1
    seg = B.lora_segments_t()
    seg.T = T
    view = B.lora_pool_view_t()
    rc = L.lora_apply_fixed_scratch(ctypes.c_void_p(0x400000), 256, ctypes.c_void_p(0x800000), 256,
                                    ctypes.byref(seg), ctypes.byref(view), None, None)
    assert rc == B.LORA_ERR_UNSUPPORTED
