"""GPU parity of lora_base_apply (the base projection with the adapter term in its
epilogue, y written once) against the fp64 oracle on the same seeded inputs."""

import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import compare_bf16, cuda_or_skip, ids_dev, new_err, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    cuda_or_skip()


def oracle_base(x, w0, ids, pool):
    """oracle.base_apply over the rows, split across host threads (rows are independent)."""
    T = len(ids)
    n = max(1, min(16, os.cpu_count() or 1, T))
    cuts = np.linspace(0, T, n + 1).astype(int)
    with cf.ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda k: oracle.base_apply(x[cuts[k]:cuts[k + 1]], w0, ids[cuts[k]:cuts[k + 1]], pool),
                            range(n)))
    return np.concatenate([p[0] for p in parts]), int(np.bitwise_or.reduce([p[1] for p in parts]))


def make_case(seed, d_in, d_out, ranks, lens, ldw_pad=8, page_elems=4096, shuffle=True, none_frac=0.05):
    rng = np.random.default_rng(seed)
    pool = W.build_pool(rng, d_in, d_out, ranks, page_elems=page_elems, max_rank=max(ranks))
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    if shuffle:
        ids = ids[rng.permutation(ids.size)]
    ids[rng.random(ids.size) < none_frac] = -1
    batch = W.make_batch(rng, ids, d_in, d_out, ldx=d_in + 8, ldy=d_out + 8)
    w0 = W.f32_to_bf16_bits((rng.standard_normal((d_out, d_in + ldw_pad)) / np.sqrt(d_in)).astype(np.float32))
    return pool, batch, w0


def run_base(pool, batch, w0, mode=B.LORA_SEG_CONTIGUOUS):
    view = B.PoolView.from_host(pool)
    x = to_dev_bits(batch.x)
    y = torch.full((batch.T, batch.y0.shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    guard = to_dev_bits(batch.y0)[:, pool.d_out:]
    y[:, pool.d_out:] = guard  # the columns past d_out must stay as they are
    w = to_dev_bits(w0)
    seg = B.Segments(batch.T)
    err = new_err()
    idt = ids_dev(batch.ids)
    B.lora_segments_build(idt, pool.n_adapters, seg, mode=mode, err=err)
    B.lora_base_apply(x, w, y, idt, seg, view, err=err)
    torch.cuda.synchronize()
    yh = to_host_bits(y)
    assert np.array_equal(yh[:, pool.d_out:], batch.y0[:, pool.d_out:]), "columns past d_out written"
    return yh[:, : pool.d_out], int(err.item())


@pytest.mark.parametrize("mode", [B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS])
def test_base_apply_prefill_and_decode_mix(mode):
    """Long segments (tensor-core shrink), short ones (gather), -1 tokens; T not a multiple
    of 128; d_out a multiple of 256."""
    pool, batch, w0 = make_case(1, 1024, 768, [16, 8, 64, 32, 1], [300, 129, 5, 1, 200, 2, 40, 17], shuffle=False)
    y, err = run_base(pool, batch, w0, mode)
    ref, oerr = oracle_base(batch.x, w0, batch.ids, pool)
    assert err == oerr == 0
    compare_bf16(y, ref, "base apply")


def test_base_apply_ragged_shapes():
    """d_in not a multiple of the 64-column K step (zero-filled boxes), d_out not a multiple
    of the 256-column tile nor of 32, rows of B crossing 256-element pages, shuffled tokens."""
    pool, batch, w0 = make_case(2, 1000, 1016, [7, 16, 13, 3], [150, 3, 90, 1, 60], page_elems=256)
    y, err = run_base(pool, batch, w0, B.LORA_SEG_GROUP)
    ref, oerr = oracle_base(batch.x, w0, batch.ids, pool)
    assert err == oerr == 0
    compare_bf16(y, ref, "ragged base apply")


def test_base_apply_no_adapter_is_the_base_product():
    """Every id -1: y = bf16(x W0^T)."""
    pool, batch, w0 = make_case(3, 512, 256, [8], [70], none_frac=1.0)
    assert (batch.ids == -1).all()
    y, err = run_base(pool, batch, w0)
    ref = W.bf16_bits_to_f32(batch.x[:, :512]).astype(np.float64) @ W.bf16_bits_to_f32(w0[:, :512]).astype(np.float64).T
    assert err == 0
    compare_bf16(y, ref, "base product")


def test_base_apply_bad_adapters_keep_the_base_term():
    """Adapters with a rank above max_rank or a page outside the pool: their tokens get the
    base term alone and the error word carries both bits."""
    pool, batch, w0 = make_case(4, 512, 512, [16, 16, 16, 16], [40, 140, 30, 9], shuffle=True, none_frac=0.0)
    pool.desc[1]["rank"] = 32  # above max_rank 16
    pool.page_list[int(pool.desc[2]["b_page0"])] = pool.n_pages + 5
    y, err = run_base(pool, batch, w0, B.LORA_SEG_GROUP)
    ref, oerr = oracle_base(batch.x, w0, batch.ids, pool)
    assert err == oerr == B.LORA_DERR_BAD_RANK | B.LORA_DERR_BAD_PAGE
    compare_bf16(y, ref, "bad adapters")


def test_base_apply_prefill_shape_sampled():
    """The prefill configuration's shape (32 requests of 64-512 tokens, 4096 -> 4096, 200
    rank-16 adapters): every column of 192 sampled rows against the oracle."""
    wl = W.prefill(5)
    pool, b = wl.pools[0], wl.batch
    rng = np.random.default_rng(6)
    w0 = W.f32_to_bf16_bits((rng.standard_normal((4096, 4096)) / 64.0).astype(np.float32))
    batch = W.Batch(x=b.x, y0=b.y0, ids=b.ids, d_in=4096, d_out=4096)
    y, err = run_base(pool, batch, w0, B.LORA_SEG_CONTIGUOUS)
    assert err == 0
    rows = np.sort(rng.choice(batch.T, 192, replace=False))
    ref, oerr = oracle_base(batch.x[rows], w0, batch.ids[rows], pool)
    assert oerr == 0
    compare_bf16(y[rows], ref, "prefill-shaped base apply")
