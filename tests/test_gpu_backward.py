"""GPU parity of the backward pass (adapter training): dA_i and dB_i added into the
gradient pool and dx, through lora_sgmv_backward, against the fp64 oracle on the same
seeded inputs."""

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import (MAX_ABS, MAX_REL_L2, compare_bf16, cuda_or_skip, ids_dev, new_err, to_dev_bits,
                      to_host_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    cuda_or_skip()


def owned_positions(pool):
    """Pool positions of every adapter element (the gradient is defined there only)."""
    P = pool.page_elems
    pos = []
    for i in range(pool.n_adapters):
        r = int(pool.ranks[i])
        if r <= 0:
            continue
        for page0, cols in ((int(pool.desc[i]["a_page0"]), pool.d_in), (int(pool.desc[i]["b_page0"]), pool.d_out)):
            e = np.arange(r * cols, dtype=np.int64)
            pos.append(pool.page_list[page0 + e // P].astype(np.int64) * P + e % P)
    return np.concatenate(pos)


def run_backward(pool, batch, g, mode=B.LORA_SEG_GROUP, with_dx=True, grad0=None, dx0=None):
    view = B.PoolView.from_host(pool)
    T = batch.T
    seg = B.Segments(T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), pool.n_adapters, seg, mode=mode, err=err)
    x = to_dev_bits(batch.x)
    dy = to_dev_bits(g)
    dx = to_dev_bits(dx0 if dx0 is not None else np.zeros((T, pool.d_in), dtype=np.uint16)) if with_dx else None
    grad = torch.from_numpy(grad0.astype(np.float32)).cuda() if grad0 is not None else \
        torch.zeros(pool.pool.shape, dtype=torch.float32, device="cuda")
    hu = torch.full((2 * T, 64), float("nan"), dtype=torch.float32, device="cuda")
    B.lora_sgmv_backward(x, dy, dx, grad, hu, seg, view, err=err)
    torch.cuda.synchronize()
    return (to_host_bits(dx) if with_dx else None), grad.cpu().numpy().astype(np.float64), int(err.item())


def compare_grad(got, ref, pos, what):
    gv, rv = got.reshape(-1)[pos], ref.reshape(-1)[pos]
    assert np.isfinite(gv).all(), what
    err = np.abs(gv - rv)
    assert err.max(initial=0) <= MAX_ABS, "%s: max |err| %.4g" % (what, err.max())
    rel = np.linalg.norm(gv - rv) / max(np.linalg.norm(rv), 1e-30)
    assert rel <= MAX_REL_L2, "%s: rel L2 %.3g" % (what, rel)


def case(seed, d_in, d_out, ranks, lens, shuffle=True):
    rng = np.random.default_rng(seed)
    pool = W.build_pool(rng, d_in, d_out, ranks, max_rank=64)
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    if shuffle:
        ids = ids[rng.permutation(ids.size)]
    ids[rng.random(ids.size) < 0.03] = -1
    batch = W.make_batch(rng, ids, d_in, d_out)
    g = W._normal_bf16(rng, (ids.size, d_out), 1.0)
    return pool, batch, g


@pytest.mark.parametrize("d_in,d_out,ranks,lens", [
    (1024, 2048, [16, 64, 8, 32], [300, 3, 200, 1, 2, 140, 9]),   # long and short segments
    (4096, 4096, [16, 16, 16], [300, 260, 129]),                  # prefill-shaped
    (4096, 11008, [8, 16, 32, 64] * 5, [1, 2, 1, 1] * 5),         # decode-shaped, mixed ranks
    (256, 256, [8, 8, 8, 8], [3, 5, 1, 7]),                       # the tiny shape
])
def test_backward_matches_oracle(d_in, d_out, ranks, lens):
    pool, batch, g = case(71, d_in, d_out, ranks, lens)
    dx0 = W._normal_bf16(np.random.default_rng(72), (batch.T, d_in), 1.0)
    dx, grad, err = run_backward(pool, batch, g, dx0=dx0)
    assert err == 0
    rdx, rgrad, oerr = oracle.lora_backward(batch.x, g, batch.ids, pool)
    assert oerr == 0
    compare_grad(grad, rgrad, owned_positions(pool), "gradients %dx%d" % (d_in, d_out))
    compare_bf16(dx, W.bf16_bits_to_f32(dx0).astype(np.float64) + rdx, "dx %dx%d" % (d_in, d_out))
    none = batch.ids < 0
    assert np.array_equal(dx[none], dx0[none])


def test_backward_contiguous_segments_and_accumulation():
    """CONTIGUOUS segments (an adapter in several segments), no dx, and gradients added
    into a non-zero gradient pool."""
    pool, batch, g = case(73, 2048, 1024, [16, 32], [150, 140, 5, 200, 3], shuffle=False)
    grad0 = np.random.default_rng(74).standard_normal(pool.pool.shape)
    dx, grad, err = run_backward(pool, batch, g, mode=B.LORA_SEG_CONTIGUOUS, with_dx=False,
                                 grad0=grad0)
    assert err == 0 and dx is None
    _, rgrad, _ = oracle.lora_backward(batch.x, g, batch.ids, pool, grad=grad0.astype(np.float32).astype(np.float64))
    compare_grad(grad, rgrad, owned_positions(pool), "accumulated gradients")


def test_backward_group_sums_are_repeatable_bitwise():
    pool, batch, g = case(75, 1024, 1024, [16, 64, 8], [300, 2, 150, 1])
    outs = [run_backward(pool, batch, g) for _ in range(3)]
    for dx, grad, err in outs[1:]:
        assert err == 0
        assert np.array_equal(dx, outs[0][0]) and np.array_equal(grad, outs[0][1])


@pytest.mark.parametrize("mode", [B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS])
def test_backward_long_segments(mode):
    """Segments of 2 000, 1 100 and 900 tokens (many 32-token steps of the gradient
    kernel, a partial last step) next to short ones: against the oracle, and, with GROUP
    segments, bit for bit the same on a second call."""
    pool, batch, g = case(78, 1024, 1024, [16, 64, 8, 32, 16, 8], [2000, 2, 1100, 1, 40, 900],
                          shuffle=(mode == B.LORA_SEG_GROUP))
    dx0 = W._normal_bf16(np.random.default_rng(79), (batch.T, 1024), 1.0)
    dx, grad, err = run_backward(pool, batch, g, mode=mode, dx0=dx0)
    assert err == 0
    rdx, rgrad, oerr = oracle.lora_backward(batch.x, g, batch.ids, pool)
    assert oerr == 0
    compare_grad(grad, rgrad, owned_positions(pool), "long-segment gradients")
    compare_bf16(dx, W.bf16_bits_to_f32(dx0).astype(np.float64) + rdx, "dx beside long segments")
    if mode == B.LORA_SEG_GROUP:
        dx2, grad2, err2 = run_backward(pool, batch, g, mode=mode, dx0=dx0)
        assert err2 == 0 and np.array_equal(dx2, dx) and np.array_equal(grad2, grad)


def test_backward_bad_adapters_add_nothing():
    pool, batch, g = case(76, 1024, 1024, [16, 16, 16], [140, 3, 150])
    pool.desc[1]["rank"] = 0  # not resident
    dx0 = W._normal_bf16(np.random.default_rng(77), (batch.T, 1024), 1.0)
    dx, grad, err = run_backward(pool, batch, g, dx0=dx0)
    assert err == B.LORA_DERR_BAD_RANK
    ids = np.where(batch.ids == 1, -1, batch.ids).astype(np.int32)
    rdx, rgrad, _ = oracle.lora_backward(batch.x, g, ids, pool)
    compare_grad(grad, rgrad, owned_positions(pool), "gradients next to a bad adapter")
    bad = batch.ids == 1
    assert np.array_equal(dx[bad], dx0[bad])
    compare_bf16(dx[~bad], W.bf16_bits_to_f32(dx0[~bad]).astype(np.float64) + rdx[~bad], "dx next to a bad adapter")
