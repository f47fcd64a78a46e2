"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same
seeded inputs -- bit-exact for segments and work lists, within the stated tolerance
for the LoRA outputs -- plus the invariants that must hold on the GPU too."""

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_lora_gb300 import binding as B
from segmented_gather_gemm_lora_gb300 import workloads as W
from gpu_util import (compare_bf16, compare_f32, cuda_or_skip, ids_dev, new_err, oracle_apply, run_apply,
                      run_apply_f32y, run_bgmv, to_dev_bits, to_host_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    cuda_or_skip()


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ segments --

def segment_cases():
    rng = np.random.default_rng(100)
    cases = [
        ("empty", np.array([], dtype=np.int32), 4),
        ("all_none", np.full(33, -1, dtype=np.int32), 4),
        ("one_adapter", np.zeros(300, dtype=np.int32), 1),
        ("all_distinct", np.arange(1500, dtype=np.int32)[::-1].copy(), 1500),
        ("max_id", np.full(40, 999, dtype=np.int32), 1000),
        ("runs_broken", np.array([3, 3, 1, 1, 3, -1, 3, 0, 0, 3, 3, 3], dtype=np.int32), 4),
        ("tile_edges", np.repeat(np.arange(8, dtype=np.int32), [8, 9, 24, 25, 127, 128, 129, 1024]), 8),
    ]
    for i in range(12):
        T = int(rng.integers(1, 5000))
        n = int(rng.integers(1, 2000))
        cases.append(("rand%d" % i, rng.integers(-1, n, size=T).astype(np.int32), n))
        k = int(rng.integers(1, 60))
        runs = np.repeat(rng.integers(-1, n, size=k), rng.integers(1, 400, size=k)).astype(np.int32)
        cases.append(("runs%d" % i, runs, n))
    cases.append(("decode", W.decode(0).batch.ids, 100))
    cases.append(("prefill", W.prefill(0).batch.ids, 200))
    cases.append(("hetero", W.hetero(0, which="up").batch.ids, 500))
    rng2 = np.random.default_rng(0)
    W.mixed13b_ranks(rng2)
    cases.append(("mixed13b", W.mixed13b_ids(rng2), 1000))
    cases.append(("big_catalogue", rng.integers(0, 32768, size=3000).astype(np.int32), 32768))
    cases.append(("long_batch", np.repeat(rng.integers(0, 50, size=40), 1200).astype(np.int32), 50))
    for T in (1, 2, 3, 5, 4097, 9999):  # every id valid (the identity order of maximal runs)
        cases.append(("valid%d" % T, np.sort(rng.integers(0, 30, size=T)).astype(np.int32)[::-1].copy(), 30))
    # the kernel's shared memory (16 bytes a token, 4 a GROUP adapter) just under and
    # just over 48 KB, where the launch needs the opt-in limit with its static part
    for T, n in ((3040, 64), (3072, 64), (3073, 64), (3000, 200)):
        cases.append(("smem%d_%d" % (T, n), np.repeat(rng.integers(-1, n, size=T // 48 + 1), 48)[:T].astype(np.int32), n))
    return cases


@pytest.mark.parametrize("mode", [B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS])
def test_segments_bit_exact(mode):
    for name, ids, n_ad in segment_cases():
        seg = B.Segments(len(ids))
        err = new_err()
        B.lora_segments_build(ids_dev(ids), n_ad, seg, mode=mode, err=err)
        torch.cuda.synchronize()
        perm, indptr, seg_ad, n_tok, short, long_ = seg.host()
        o_perm, o_indptr, o_ad, o_ntok, o_err = oracle.segments_build(ids, n_ad, mode)
        o_short, o_long = oracle.work_lists(o_indptr, B.LORA_SHORT_MAX_TOKENS, B.LORA_TILE_M)
        assert n_tok == o_ntok, name
        assert np.array_equal(perm, o_perm), name
        assert np.array_equal(indptr, o_indptr), name
        assert np.array_equal(seg_ad, o_ad), name
        assert np.array_equal(short, o_short), name
        assert np.array_equal(long_, o_long), name
        assert int(err.item()) == o_err, name


def test_segments_flag_bad_ids():
    ids = np.array([0, 7, -5, 1, 1, 2], dtype=np.int32)
    seg = B.Segments(len(ids))
    err = new_err()
    B.lora_segments_build(ids_dev(ids), 3, seg, err=err)
    torch.cuda.synchronize()
    perm, indptr, seg_ad, n_tok, _, _ = seg.host()
    assert int(err.item()) == B.LORA_DERR_BAD_ADAPTER
    assert perm.tolist() == [0, 3, 4, 5]
    assert seg_ad.tolist() == [0, 1, 2]


# -------------------------------------------------------------------- apply --

def check_untouched(y_bits, batch, pool, rows):
    """Rows in `rows` and every guard column must equal y0 bit for bit."""
    assert np.array_equal(y_bits[rows], batch.y0[rows])
    assert np.array_equal(y_bits[:, pool.d_out:], batch.y0[:, pool.d_out:])


@pytest.mark.parametrize("seed", range(5))
def test_apply_tiny(seed):
    wl = W.tiny(seed)
    pool = wl.pools[0]
    y, err, _ = run_apply(wl.batch, pool, wl.mode, wl.n_adapters)
    ref, oerr = oracle.lora_apply(wl.batch.x, wl.batch.y0, wl.batch.ids, pool)
    assert err == oerr == 0
    compare_bf16(y[:, : pool.d_out], ref, "tiny seed %d" % seed)


@pytest.mark.parametrize("seed", range(3))
def test_apply_decode(seed):
    wl = W.decode(seed)
    pool = wl.pools[0]
    y, err, _ = run_apply(wl.batch, pool, wl.mode, wl.n_adapters)
    ref, _ = oracle.lora_apply(wl.batch.x, wl.batch.y0, wl.batch.ids, pool)
    assert err == 0
    compare_bf16(y, ref, "decode seed %d" % seed)


@pytest.mark.parametrize("mode", [B.LORA_SEG_CONTIGUOUS, B.LORA_SEG_GROUP])
def test_apply_prefill_small(mode):
    wl = W.prefill(1, n_requests=5)
    pool = wl.pools[0]
    y, err, _ = run_apply(wl.batch, pool, mode, wl.n_adapters)
    ref, _ = oracle.lora_apply(wl.batch.x, wl.batch.y0, wl.batch.ids, pool)
    assert err == 0
    compare_bf16(y, ref, "prefill(5 requests)")


@pytest.mark.parametrize("which", ["up", "down"])
def test_apply_hetero(which):
    wl = W.hetero(0, which=which)
    pool = wl.pools[0]
    rng = np.random.default_rng(7)
    batch = W.make_batch(rng, wl.batch.ids, pool.d_in, pool.d_out, ldx=pool.d_in + 16,
                         ldy=pool.d_out + 8)
    y, err, _ = run_apply(batch, pool, wl.mode, wl.n_adapters)
    ref, _ = oracle.lora_apply(batch.x, batch.y0, batch.ids, pool)
    assert err == 0
    compare_bf16(y[:, : pool.d_out], ref, "hetero " + which)
    check_untouched(y, batch, pool, np.where(batch.ids < 0)[0])


@pytest.mark.parametrize("n_units", [600, 1500])
def test_gather_claim_order_many_units_mixed_ranks(n_units):
    """Short segments of mixed ranks: with a few hundred units the gather kernel claims them
    largest adapter first; beyond 1024 claimable units it claims them in segment order.
    Either way every token's output matches the oracle, and every unit runs once."""
    rng = np.random.default_rng(40 + n_units)
    ranks = rng.choice(np.array([1, 8, 16, 17, 32, 33, 48, 64], dtype=np.int32), size=n_units)
    pool = W.build_pool(rng, 512, 768, ranks, max_rank=64)
    ids = rng.permutation(np.repeat(np.arange(n_units, dtype=np.int32), rng.integers(1, 3, size=n_units)))
    ids[rng.random(ids.size) < 0.05] = -1
    batch = W.make_batch(rng, ids, 512, 768)
    ref, oerr = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, n_units)
    assert err == oerr == 0
    compare_bf16(y, ref, "claim order, %d units" % n_units)
    assert np.array_equal(y[ids < 0], batch.y0[ids < 0])


def test_apply_odd_shapes_and_ranks():
    """Ranks that divide nothing, widths that are not multiples of the page, rows that
    straddle pages, segment lengths around the dispatch thresholds, and -1 tokens."""
    rng = np.random.default_rng(11)
    ranks = [1, 7, 13, 33, 64, 8, 16]
    pool = W.build_pool(rng, 5120, 1000, ranks, page_elems=4096, max_rank=64)
    lens = [1, 2, 7, 8, 9, 23, 24, 25, 127, 128, 129, 300]
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    ids[rng.choice(ids.size, 20, replace=False)] = -1
    batch = W.make_batch(rng, ids, 5120, 1000, ldx=5128, ldy=1016)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, len(ranks))
        ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
        assert err == 0
        compare_bf16(y[:, :1000], ref, "odd shapes mode %d" % mode)
        check_untouched(y, batch, pool, np.where(ids < 0)[0])


def test_apply_small_pages():
    rng = np.random.default_rng(12)
    pool = W.build_pool(rng, 256, 512, [8, 24, 64], page_elems=64, max_rank=64)
    ids = rng.integers(-1, 3, size=200).astype(np.int32)
    batch = W.make_batch(rng, ids, 256, 512)
    y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, 3)
    ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    assert err == 0
    compare_bf16(y, ref, "64-element pages")


def test_gather_page_cache_edges():
    """Short segments and one-token calls on adapters whose page-list slots fill the gather
    kernel's per-unit cache exactly, exceed it by a few, or by far (then the producers read
    the page list from global memory): d_in 256, d_out 384 and 64-element pages, so an
    adapter of rank r takes 10 r slots -- rank 32 takes 320, rank 33 330, rank 64 640."""
    rng = np.random.default_rng(31)
    ranks = [32, 33, 64, 8, 64, 33]
    pool = W.build_pool(rng, 256, 384, ranks, page_elems=64, max_rank=64)
    ids = np.repeat(np.arange(len(ranks), dtype=np.int32), [1, 3, 2, 1, 3, 2])  # at most 3 tokens an adapter
    ids = np.concatenate([ids, np.array([-1, -1], dtype=np.int32)])
    rng.shuffle(ids)
    batch = W.make_batch(rng, ids, 256, 384)
    ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, len(ranks))
        assert err == 0
        compare_bf16(y[:, :384], ref, "page cache edges, segments mode %d" % mode)
    y, err = run_bgmv(batch, pool)  # max_rank 64: the gather kernel's one-token form
    assert err == 0
    compare_bf16(y[:, :384], ref, "page cache edges, one-token form")


MIXED13B_PROJ = [p[0] for p in W.PROJ_13B]


def mixed13b_cases():
    """(layer, projection, all rows?) pairs of the 13B-shaped check: every projection of
    layers 0, 19 and 39 (one projection per layer on all 4224 rows, the rest on a sample)
    plus eight random (layer, projection) pairs."""
    full = {0: "q", 19: "gate", 39: "down"}
    cases = [(layer, name, full[layer] == name) for layer in (0, 19, 39) for name in MIXED13B_PROJ]
    rng = np.random.default_rng(1313)
    for _ in range(8):
        cases.append((int(rng.integers(0, 40)), MIXED13B_PROJ[int(rng.integers(0, 7))], False))
    return cases


@pytest.mark.parametrize("layer,name,all_rows", mixed13b_cases())
def test_apply_mixed13b(layer, name, all_rows):
    """13B-shaped mixed batch (4 prefill requests of 1024 tokens + 128 decode tokens, GROUP
    segments, T = 4224), one (layer, projection) call at full size.  The oracle checks
    every row, or all 128 decode rows plus 160 prefill rows; rows of the full case are
    also checked through lora_apply_f32y against the literal bounds."""
    pool, batch, n_ad = W.mixed13b_projection(0, layer, name)
    ids = batch.ids
    view = B.PoolView.from_host(pool)
    y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, n_ad, view=view)
    assert err == 0
    if all_rows:
        rows = np.arange(batch.T)
    else:
        rng = np.random.default_rng([layer, MIXED13B_PROJ.index(name)])
        rows = np.sort(np.concatenate([rng.choice(4096, 160, replace=False), 4096 + np.arange(128)]))
    ref, oerr = oracle_apply(batch.x[rows], batch.y0[rows], ids[rows], pool)
    assert oerr == 0
    compare_bf16(y[rows], ref, "13B layer %d %s" % (layer, name))
    if all_rows:
        yf, errf = run_apply_f32y(batch, pool, B.LORA_SEG_GROUP, n_ad, view=view)
        assert errf == 0
        compare_f32(yf, ref, "13B f32y layer %d %s" % (layer, name))


@pytest.mark.parametrize("seed", range(5))
def test_apply_prefill_full(seed):
    """The prefill configuration at full size (32 requests of 64..512 tokens), every row,
    CONTIGUOUS segments as the configuration states (and GROUP for seed 0)."""
    wl = W.prefill(seed)
    pool = wl.pools[0]
    ref, _ = oracle_apply(wl.batch.x, wl.batch.y0, wl.batch.ids, pool)
    for mode in ([B.LORA_SEG_CONTIGUOUS, B.LORA_SEG_GROUP] if seed == 0 else [B.LORA_SEG_CONTIGUOUS]):
        y, err, _ = run_apply(wl.batch, pool, mode, wl.n_adapters)
        assert err == 0
        compare_bf16(y, ref, "prefill seed %d mode %d" % (seed, mode))


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("which", ["up", "down"])
def test_apply_hetero_seeds(seed, which):
    """Heterogeneous ranks at full size (256 decode tokens, 500 adapters of rank 8..64,
    MLP up 4096 -> 11008 or down 11008 -> 4096), every row, seeds 0-4."""
    wl = W.hetero(seed, which=which)
    pool = wl.pools[0]
    batch = W.make_batch(np.random.default_rng([seed, 7]), wl.batch.ids, pool.d_in, pool.d_out)
    y, err, _ = run_apply(batch, pool, wl.mode, wl.n_adapters)
    assert err == 0
    ref, _ = oracle_apply(batch.x, batch.y0, batch.ids, pool)
    compare_bf16(y, ref, "hetero %s seed %d" % (which, seed))


def f32y_cases():
    cases = []
    for seed in range(5):
        cases += [("tiny", seed), ("decode", seed), ("prefill", seed), ("hetero_up", seed), ("hetero_down", seed)]
    return cases


@pytest.mark.parametrize("name,seed", f32y_cases())
def test_f32y_literal_bounds(name, seed):
    """Every configuration through lora_apply_f32y (the same kernels as lora_apply, fp32
    output): max |err| <= 2e-2 and relative L2 <= 5e-3 against the oracle, with no
    allowance for output rounding; rows of tokens without an adapter stay unwritten.
    The bf16 outputs of lora_apply equal the fp32 ones rounded to nearest even."""
    if name.startswith("hetero"):
        which = name.split("_")[1]
        wl = W.hetero(seed, which=which)
        pool = wl.pools[0]
        ids = wl.batch.ids.copy()
        ids[::11] = -1
        batch = W.make_batch(np.random.default_rng([seed, 7]), ids, pool.d_in, pool.d_out)
    else:
        wl = W.WORKLOADS[name](seed)
        pool = wl.pools[0]
        batch = wl.batch
        if name == "decode":
            batch.ids[::9] = -1
    view = B.PoolView.from_host(pool)
    yf, err = run_apply_f32y(batch, pool, wl.mode, wl.n_adapters, view=view)
    assert err == 0
    ref, _ = oracle_apply(batch.x, batch.y0, batch.ids, pool)
    on = batch.ids >= 0
    compare_f32(yf[on], ref[on], "f32y %s seed %d" % (name, seed))
    assert np.isnan(yf[~on]).all()
    y, err2, _ = run_apply(batch, pool, wl.mode, wl.n_adapters, view=view)
    assert err2 == 0
    rounded = W.f32_to_bf16_bits(yf[on])
    assert np.array_equal(y[on][:, : pool.d_out], rounded)


# --------------------------------------------------------------------- bgmv --

@pytest.mark.parametrize("name", ["tiny", "decode", "hetero"])
def test_bgmv_parity(name):
    wl = {"tiny": W.tiny, "decode": W.decode, "hetero": lambda s: W.hetero(s, which="up")}[name](0)
    pool = wl.pools[0]
    ids = wl.batch.ids.copy()
    ids[::7] = -1
    y, err = run_bgmv(wl.batch, pool, ids=ids)
    ref, _ = oracle.lora_apply(wl.batch.x, wl.batch.y0, ids, pool)
    assert err == 0
    compare_bf16(y[:, : pool.d_out], ref, "bgmv " + name)
    assert np.array_equal(y[ids < 0], wl.batch.y0[ids < 0])


def test_bgmv_matches_apply_and_is_batch_invariant():
    """lora_bgmv (the decode kernel's fp32 sums) and lora_apply (the gather kernel's
    tensor-core sums) on the same batch, with a repeated adapter and a -1 id, both
    agree with the oracle; and a token's lora_bgmv output does not depend on the other
    tokens of its call: the batch's first dozen tokens, alone, give the same bits."""
    wl = W.decode(1)
    pool = wl.pools[0]
    ids = wl.batch.ids.copy()
    ids[3] = ids[7]
    ids[5] = -1
    b = W.Batch(x=wl.batch.x, y0=wl.batch.y0, ids=ids, d_in=wl.batch.d_in, d_out=wl.batch.d_out)
    yb, eb = run_bgmv(b, pool)
    ya, ea, _ = run_apply(b, pool, B.LORA_SEG_GROUP, wl.n_adapters)
    assert eb == ea == 0
    ref, _ = oracle_apply(b.x, b.y0, ids, pool)
    compare_bf16(yb, ref, "bgmv")
    compare_bf16(ya, ref, "apply")
    sub = W.Batch(x=b.x[:12], y0=b.y0[:12], ids=ids[:12], d_in=b.d_in, d_out=b.d_out)
    ys, es = run_bgmv(sub, pool)
    assert es == 0
    assert np.array_equal(ys, yb[:12])


def test_bgmv_static_adapters_chain_in_graph():
    """With LORA_BGMV_STATIC_ADAPTERS the decode kernel reads the ids and the pool, and
    stages the adapters, before the kernel ahead of it has finished, but x and y only
    after.  Four calls back to back in one CUDA graph, each reading the previous call's
    y as its x, equal the same chain run call by call without the flag and with a
    synchronisation in between, bit for bit, replay after replay; the first call also
    matches the oracle."""
    rng = np.random.default_rng(83)
    d = 4096
    pool = W.build_pool(rng, d, d, [16, 8, 16, 4, 12, 16, 1, 16] * 3, max_rank=16)
    ids = rng.integers(-1, pool.n_adapters, size=64).astype(np.int32)
    batch = W.make_batch(rng, ids, d, d)
    view = B.PoolView.from_host(pool)
    x0 = to_dev_bits(batch.x)
    y0 = to_dev_bits(batch.y0)
    idt = ids_dev(ids)
    err = new_err()
    ys = [torch.empty_like(y0) for _ in range(4)]

    def chain(static, sync):
        for y in ys:
            y.copy_(y0)
        prev = x0
        for y in ys:
            B.lora_bgmv(prev, y, idt, view, err=err, static_adapters=static)
            if sync:
                torch.cuda.synchronize()
            prev = y

    chain(False, True)
    torch.cuda.synchronize()
    want = [y.clone() for y in ys]
    assert int(err.item()) == 0
    ref, oerr = oracle_apply(batch.x, batch.y0, ids, pool)
    assert oerr == 0
    compare_bf16(to_host_bits(want[0]), ref, "first call of the chain")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain(True, False)
    for _ in range(30):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for y, w in zip(ys, want):
            assert torch.equal(y.view(torch.int16), w.view(torch.int16))
    assert int(err.item()) == 0


def test_bgmv_rows_independent_of_the_batch():
    """A few adapters shared by many tokens (runs of one adapter included), -1 ids and a
    bad id, at T = 256 and 257: against the oracle, with the oracle's error word; every
    token's row is the same, bit for bit, when the batch is shuffled, and when the same
    256 tokens come with 44 more -1 tokens after them."""
    rng = np.random.default_rng(4242)
    d = 2048
    pool = W.build_pool(rng, d, d, [16, 4, 9, 16, 1, 12], max_rank=16)
    for T in (256, 257):
        ids = rng.integers(-1, pool.n_adapters, size=T).astype(np.int32)
        ids[T - 9:] = 2
        ids[17] = pool.n_adapters + 3
        batch = W.make_batch(rng, ids, d, d, ldx=d + 8, ldy=d + 24)
        y, err = run_bgmv(batch, pool)
        ref, oerr = oracle_apply(batch.x, batch.y0, ids, pool)
        assert err == oerr == B.LORA_DERR_BAD_ADAPTER
        compare_bf16(y[:, :d], ref, "decode kernel T=%d" % T)
        assert np.array_equal(y[ids < 0], batch.y0[ids < 0])
        assert np.array_equal(y[:, d:], batch.y0[:, d:])
        perm = rng.permutation(T)
        shuf = W.Batch(x=batch.x[perm], y0=batch.y0[perm], ids=ids[perm], d_in=d, d_out=d)
        ys, es = run_bgmv(shuf, pool)
        assert es == err
        assert np.array_equal(ys, y[perm]), "a token's row depends on its place in the batch (T=%d)" % T
    ids = rng.integers(0, 3, size=256).astype(np.int32)
    batch = W.make_batch(rng, ids, d, d)
    yg, eg = run_bgmv(batch, pool)
    pad = np.full(44, -1, dtype=np.int32)
    big = W.Batch(x=np.concatenate([batch.x, batch.x[:44]]), y0=np.concatenate([batch.y0, batch.y0[:44]]),
                  ids=np.concatenate([ids, pad]), d_in=d, d_out=d)
    yu, eu = run_bgmv(big, pool)
    assert eg == eu == 0
    assert np.array_equal(yg, yu[:256]), "a token's row depends on the batch's size"


def test_bgmv_decode_kernel_shapes_and_pages():
    """The decode kernel on the shapes it takes: one CTA (d = 256), slices narrower than
    a sub-slice, d_in != d_out, 1024-element pages, rows that cross pages (d = 1000),
    clusters of five and eight CTAs (5120 -> 8192),
    ranks 1..16 with max_rank 16, strides wider than the rows; and a view with more page
    slots than the kernel caches (256-element pages), which lora_bgmv runs on the gather
    kernel.  Against the oracle; -1 rows and the guard columns untouched."""
    for seed, (d_in, d_out, page) in enumerate([(256, 256, 4096), (1024, 2048, 4096), (4096, 1024, 1024),
                                                (1000, 4096, 4096), (5120, 8192, 4096), (2048, 4096, 256)]):
        rng = np.random.default_rng(900 + seed)
        ranks = [1, 16, 3, 8, 16, 5, 12, 2]
        pool = W.build_pool(rng, d_in, d_out, ranks, max_rank=16, page_elems=page)
        ids = rng.integers(-1, len(ranks), size=40).astype(np.int32)
        batch = W.make_batch(rng, ids, d_in, d_out, ldx=d_in + 16, ldy=d_out + 8)
        y, err = run_bgmv(batch, pool)
        ref, oerr = oracle_apply(batch.x, batch.y0, ids, pool)
        assert err == oerr == 0
        compare_bf16(y[:, :d_out], ref, "decode kernel %dx%d page %d" % (d_in, d_out, page))
        assert np.array_equal(y[ids < 0], batch.y0[ids < 0])
        assert np.array_equal(y[:, d_out:], batch.y0[:, d_out:])


# ------------------------------------------------------------ shrink/expand --

def test_shrink_parity_and_chain_equals_apply():
    wl = W.hetero(1, which="down")
    pool = wl.pools[0]
    rng = np.random.default_rng(15)
    batch = W.make_batch(rng, wl.batch.ids, pool.d_in, pool.d_out)
    view = B.PoolView.from_host(pool)
    x = to_dev_bits(batch.x)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), wl.n_adapters, seg, err=err)
    ldh = 64
    h = torch.full((batch.T, ldh), 7.0, dtype=torch.float32, device="cuda")
    B.lora_sgmv_shrink(x, h, seg, view, err=err)
    B.lora_sgmv_expand(h, y, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hh = h.cpu().numpy()
    href, _ = oracle.shrink(batch.x, batch.ids, pool, h_init=np.full((batch.T, ldh), 7.0), ldh=ldh)
    np.testing.assert_allclose(hh, href, rtol=1e-4, atol=1e-4)
    ya, _, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, wl.n_adapters, view=view)
    assert np.array_equal(to_host_bits(y), ya)


def test_expand_parity_random_h():
    wl = W.hetero(2, which="up")
    pool = wl.pools[0]
    rng = np.random.default_rng(16)
    batch = W.make_batch(rng, wl.batch.ids, pool.d_in, pool.d_out)
    hin = rng.standard_normal((batch.T, 64), dtype=np.float32)
    view = B.PoolView.from_host(pool)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), wl.n_adapters, seg, err=err)
    B.lora_sgmv_expand(torch.from_numpy(hin).cuda(), y, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _ = oracle.expand(hin, batch.y0, batch.ids, pool)
    compare_bf16(to_host_bits(y), ref, "expand")


# --------------------------------------------------------------- invariants --

def test_zero_B_leaves_y0():
    rng = np.random.default_rng(17)
    pool = W.build_pool(rng, 4096, 4096, [16] * 20, zero_B=True)
    ids = rng.integers(-1, 20, size=300).astype(np.int32)
    batch = W.make_batch(rng, ids, 4096, 4096)
    y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, 20)
    assert err == 0
    assert np.array_equal(W.bf16_bits_to_f32(y), W.bf16_bits_to_f32(batch.y0))


def test_zero_padded_rank_equals_unpadded():
    rng = np.random.default_rng(18)
    d_in, d_out = 4096, 2048
    base = W.build_pool(rng, d_in, d_out, [8, 16, 5], max_rank=64)
    A, Bm, ranks = [], [], []
    for i, r in enumerate(base.ranks):
        rp = int(r) + 24
        a = np.zeros((rp, d_in), dtype=np.uint16)
        b = np.zeros((rp, d_out), dtype=np.uint16)
        a[:r] = base.A[i]
        b[:r] = base.B[i]
        A.append(a)
        Bm.append(b)
        ranks.append(rp)
    padded = W.pack_pool(A, Bm, np.array(ranks), d_in, d_out, rng, scales=base.scales, max_rank=64)
    ids = np.repeat(rng.integers(0, 3, size=30), rng.integers(1, 40, size=30)).astype(np.int32)
    batch = W.make_batch(rng, ids, d_in, d_out)
    y1, e1, _ = run_apply(batch, base, B.LORA_SEG_GROUP, 3)
    y2, e2, _ = run_apply(batch, padded, B.LORA_SEG_GROUP, 3)
    assert e1 == e2 == 0
    assert np.array_equal(W.bf16_bits_to_f32(y1), W.bf16_bits_to_f32(y2))


def test_request_order_invariance_bitwise():
    wl = W.prefill(3, n_requests=6)
    pool = wl.pools[0]
    ids = wl.batch.ids
    # split into requests (runs) and reverse their order
    starts = np.flatnonzero(np.r_[True, ids[1:] != ids[:-1]])
    ends = np.r_[starts[1:], ids.size]
    order = np.concatenate([np.arange(s, e) for s, e in list(zip(starts, ends))[::-1]])
    b2 = W.Batch(x=wl.batch.x[order], y0=wl.batch.y0[order], ids=ids[order], d_in=4096, d_out=4096)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y1, _, _ = run_apply(wl.batch, pool, mode, wl.n_adapters)
        y2, _, _ = run_apply(b2, pool, mode, wl.n_adapters)
        assert np.array_equal(y1[order], y2)


def test_group_equals_contiguous_bitwise():
    wl = W.prefill(4, n_requests=8)
    pool = wl.pools[0]
    y1, _, _ = run_apply(wl.batch, pool, B.LORA_SEG_GROUP, wl.n_adapters)
    y2, _, _ = run_apply(wl.batch, pool, B.LORA_SEG_CONTIGUOUS, wl.n_adapters)
    assert np.array_equal(y1, y2)


# ---------------------------------------------------------------- error paths --

def test_device_errors_flag_and_skip():
    rng = np.random.default_rng(19)
    pool = W.build_pool(rng, 1024, 1024, [16, 16, 16, 16], max_rank=16)
    pool.desc[1]["rank"] = 32  # above max_rank
    pool.page_list[int(pool.desc[2]["b_page0"]) + 1] = pool.n_pages + 3  # page outside the pool
    pool.desc[3]["rank"] = 0  # not resident
    ids = np.array([0, 1, 2, 3, 0, -1, 1, 0], dtype=np.int32)
    batch = W.make_batch(rng, ids, 1024, 1024)
    ref, oerr = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, 4)
    assert err == oerr == B.LORA_DERR_BAD_RANK | B.LORA_DERR_BAD_PAGE
    good = ids == 0
    compare_bf16(y[good], ref[good], "good rows next to bad ones")
    assert np.array_equal(y[~good], batch.y0[~good])
    yb, errb = run_bgmv(batch, pool)
    assert errb == oerr
    assert np.array_equal(yb[~good], batch.y0[~good])
    ids2 = ids.copy()
    ids2[2] = 9
    yc, errc = run_bgmv(batch, pool, ids=ids2)
    assert errc & B.LORA_DERR_BAD_ADAPTER
    assert np.array_equal(yc[2], batch.y0[2])


def test_segment_ids_beyond_the_view_flag_and_skip():
    """Segments built for more adapters than the pool view holds: the compute calls
    check every segment's adapter id against the view (short segments on the gather
    path, long ones on the tensor-core path) and skip those outside it."""
    rng = np.random.default_rng(31)
    pool = W.build_pool(rng, 2048, 2048, [16, 16, 16], max_rank=16)
    ids = np.repeat(np.array([5, 0, 7, 1, 2, 6], dtype=np.int32), [3, 20, 150, 4, 140, 1])
    batch = W.make_batch(rng, ids, 2048, 2048)
    bad = ids >= 3
    ref, oerr = oracle.lora_apply(batch.x, batch.y0, np.where(bad, -1, ids).astype(np.int32), pool)
    assert oerr == 0
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, 8)
        assert err == B.LORA_DERR_BAD_ADAPTER
        compare_bf16(y[~bad], ref[~bad], "rows next to out-of-view adapters")
        assert np.array_equal(y[bad], batch.y0[bad])


def test_graph_chain_sees_every_row_of_the_previous_call():
    """Two lora_apply calls in one CUDA graph, the second reading the first's y as its x,
    over a batch with both short segments (gather kernel) and long ones (tensor-core
    kernels), replayed many times: every replay equals the chain run call by call with
    a synchronisation in between, bit for bit.  The tensor-core shrink starts without
    waiting for the same call's gather kernel, so this checks that the next call still
    sees the gather's rows."""
    rng = np.random.default_rng(53)
    d = 1024
    pool = W.build_pool(rng, d, d, [16, 32, 8, 64] * 8, max_rank=64)
    ids = np.concatenate([np.full(300, 3, dtype=np.int32), rng.permutation(np.arange(4, 32, dtype=np.int32)),
                          np.full(140, 1, dtype=np.int32), np.arange(4, 12, dtype=np.int32)])
    ids = rng.permutation(ids).astype(np.int32)
    batch = W.make_batch(rng, ids, d, d)
    view = B.PoolView.from_host(pool)
    x0 = to_dev_bits(batch.x)
    y0 = to_dev_bits(batch.y0)
    idt = ids_dev(ids)
    seg = B.Segments(len(ids))
    err = new_err()
    y1 = torch.empty_like(y0)
    y2 = torch.empty_like(y0)

    def chain(sync):
        y1.copy_(y0)
        y2.copy_(y0)
        B.lora_segments_build(idt, 32, seg, mode=B.LORA_SEG_GROUP, err=err)
        B.lora_apply(x0, y1, seg, view, err=err)
        if sync:
            torch.cuda.synchronize()
        B.lora_apply(y1, y2, seg, view, err=err)

    chain(True)
    torch.cuda.synchronize()
    want = y2.clone()
    assert int(err.item()) == 0
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain(False)
    for _ in range(40):
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int16), want.view(torch.int16))
    assert int(err.item()) == 0


def test_empty_batch_is_noop():
    wl = W.tiny(0)
    view = B.PoolView.from_host(wl.pools[0])
    seg = B.Segments(0)
    err = new_err()
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    B.lora_segments_build(empty, 4, seg, err=err)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    B.lora_apply(x, y, seg, view, err=err)
    B.lora_bgmv(x, y, empty, view, err=err)
    torch.cuda.synchronize()
    assert int(seg.meta[0].item()) == 0
    assert int(err.item()) == 0


# ------------------------------------------------------ tensor-core long path --

def long_segment_batch(seed, ranks, lens, d_in, d_out, page_elems=4096):
    rng = np.random.default_rng(seed)
    pool = W.build_pool(rng, d_in, d_out, ranks, page_elems=page_elems, max_rank=64)
    ids = np.concatenate([np.full(n, i % len(ranks), dtype=np.int32) for i, n in enumerate(lens)])
    batch = W.make_batch(rng, ids, d_in, d_out, ldx=d_in + 64, ldy=d_out + 8)
    return pool, batch


@pytest.mark.parametrize("mode", [B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS])
def test_tc_odd_ranks_and_tile_edges(mode):
    """Long segments on the tensor cores with ranks that are not multiples of 16 and
    segment lengths around the 128-token tile."""
    ranks = [1, 7, 13, 33, 64, 16, 48]
    lens = [25, 127, 128, 129, 256, 300, 40, 1, 3, 24]
    pool, batch = long_segment_batch(21, ranks, lens, 4096, 1024)
    y, err, _ = run_apply(batch, pool, mode, len(ranks))
    ref, _ = oracle.lora_apply(batch.x, batch.y0, batch.ids, pool)
    assert err == 0
    compare_bf16(y[:, :1024], ref, "tensor-core tiles mode %d" % mode)
    check_untouched(y, batch, pool, np.array([], dtype=int))


def test_tc_wide_shapes():
    """d_in = 13824 (27 chunks per CTA) and d_out = 13824 (108 column chunks), rank 64."""
    for d_in, d_out in ((13824, 5120), (5120, 13824)):
        pool, batch = long_segment_batch(22, [64, 32], [200, 140], d_in, d_out)
        y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, 2)
        ref, _ = oracle.lora_apply(batch.x, batch.y0, batch.ids, pool)
        assert err == 0
        compare_bf16(y[:, :d_out], ref, "tensor-core %dx%d" % (d_in, d_out))


def test_tc_shrink_expand_chain_equals_apply():
    wl = W.prefill(5, n_requests=6)
    pool = wl.pools[0]
    batch = wl.batch
    view = B.PoolView.from_host(pool)
    x = to_dev_bits(batch.x)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), wl.n_adapters, seg, mode=B.LORA_SEG_GROUP, err=err)
    h = torch.full((batch.T, 64), 3.0, dtype=torch.float32, device="cuda")
    B.lora_sgmv_shrink(x, h, seg, view, err=err)
    B.lora_sgmv_expand(h, y, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    href, _ = oracle.shrink(batch.x, batch.ids, pool, h_init=np.full((batch.T, 64), 3.0), ldh=64)
    np.testing.assert_allclose(h.cpu().numpy(), href, rtol=1e-4, atol=1e-4)
    ya, _, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, wl.n_adapters, view=view)
    assert np.array_equal(to_host_bits(y), ya)


def test_tc_expand_parity_random_h():
    pool, batch = long_segment_batch(23, [16, 64, 5], [150, 200, 64], 2048, 4096)
    rng = np.random.default_rng(24)
    hin = rng.standard_normal((batch.T, 64), dtype=np.float32)
    view = B.PoolView.from_host(pool)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), 3, seg, err=err)
    B.lora_sgmv_expand(torch.from_numpy(hin).cuda(), y, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _ = oracle.expand(hin, batch.y0, batch.ids, pool)
    compare_bf16(to_host_bits(y)[:, :4096], ref, "tensor-core expand")


def test_tc_device_errors_in_long_tiles():
    rng = np.random.default_rng(25)
    pool = W.build_pool(rng, 2048, 2048, [16, 16, 16], max_rank=16)
    pool.desc[1]["rank"] = 32
    pool.page_list[int(pool.desc[2]["a_page0"]) + 3] = -7
    ids = np.repeat(np.array([0, 1, 2, 0], dtype=np.int32), [150, 140, 130, 20])
    batch = W.make_batch(rng, ids, 2048, 2048)
    ref, oerr = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, 3)
        assert err == oerr == B.LORA_DERR_BAD_RANK | B.LORA_DERR_BAD_PAGE
        good = ids == 0
        compare_bf16(y[good], ref[good], "long tiles next to bad ones")
        assert np.array_equal(y[~good], batch.y0[~good])


def test_fused_shrink_only_bad_adapters_and_counters():
    """lora_sgmv_shrink on long tiles (the fused kernel's shrink-only form): an adapter
    whose rank is above the view's max_rank and one with a page slot outside the pool
    write no h (their rows keep the caller's values) and set the oracle's error bits;
    the good adapters' h match the oracle; two calls in a row on one segment buffer give
    the same h, and a lora_apply on that buffer afterwards equals one on a fresh buffer
    bit for bit (the work counter is back at zero after each call)."""
    rng = np.random.default_rng(31)
    pool = W.build_pool(rng, 4096, 1024, [16, 16, 16, 64], max_rank=64)
    pool.desc[1]["rank"] = 80
    pool.page_list[int(pool.desc[2]["a_page0"]) + 2] = pool.n_pages + 9
    ids = np.repeat(np.array([0, 1, 2, 3, 0], dtype=np.int32), [300, 140, 130, 200, 40])
    batch = W.make_batch(rng, ids, 4096, 1024)
    view = B.PoolView.from_host(pool)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(ids), 4, seg, mode=B.LORA_SEG_GROUP, err=err)
    href, oerr = oracle.shrink(batch.x, ids, pool, h_init=np.full((batch.T, 64), -3.0), ldh=64)
    assert oerr == B.LORA_DERR_BAD_RANK | B.LORA_DERR_BAD_PAGE
    outs = []
    for _ in range(2):
        err.zero_()
        h = torch.full((batch.T, 64), -3.0, dtype=torch.float32, device="cuda")
        B.lora_sgmv_shrink(to_dev_bits(batch.x), h, seg, view, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == oerr
        hh = h.cpu().numpy()
        np.testing.assert_allclose(hh, href, rtol=1e-4, atol=1e-4)
        outs.append(hh)
    assert np.array_equal(outs[0], outs[1])
    y = to_dev_bits(batch.y0)
    B.lora_apply(to_dev_bits(batch.x), y, seg, view, err=err)
    torch.cuda.synchronize()
    fresh, e2, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, 4, view=view)
    assert e2 == oerr
    assert np.array_equal(to_host_bits(y), fresh)


def test_tc_segments_reused_across_calls_and_shapes():
    """One segment buffer serves several projections of different d_in in a row (the
    tensor-core kernels' work counters must be back at zero after each call);
    every result equals a fresh run bit for bit."""
    rng = np.random.default_rng(26)
    ranks = [16, 64, 7]
    lens = [256, 300, 129]
    ids = np.concatenate([np.full(n, i, dtype=np.int32) for i, n in enumerate(lens)])
    seg = B.Segments(ids.size)
    err = new_err()
    B.lora_segments_build(ids_dev(ids), len(ranks), seg, mode=B.LORA_SEG_GROUP, err=err)
    for d_in, d_out in ((4096, 1024), (1024, 2048), (8192, 1024), (4096, 1024)):
        pool = W.build_pool(rng, d_in, d_out, ranks, max_rank=64)
        batch = W.make_batch(rng, ids, d_in, d_out)
        view = B.PoolView.from_host(pool)
        outs = []
        for _ in range(2):
            y = to_dev_bits(batch.y0)
            B.lora_apply(to_dev_bits(batch.x), y, seg, view, err=err)
            torch.cuda.synchronize()
            outs.append(to_host_bits(y))
        assert int(err.item()) == 0
        fresh, e2, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, len(ranks), view=view)
        assert e2 == 0
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], fresh)
        ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
        compare_bf16(fresh, ref, "reused segments %dx%d" % (d_in, d_out))


@pytest.mark.parametrize("d_in", [1024, 4096])
def test_tc_shrink_caller_h_odd_stride_and_ranks(d_in):
    """Caller's h with a row stride of 72 and ranks that are not multiples of 4, with
    d_in in one slice (h written straight from tensor memory) and in four slices
    (partials summed by the tile's last slice)."""
    pool, batch = long_segment_batch(27, [7, 13, 33, 64], [200, 150, 130, 300], d_in, 1024)
    view = B.PoolView.from_host(pool)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), 4, seg, err=err)
    hbuf = torch.full((batch.T, 72), -5.0, dtype=torch.float32, device="cuda")
    B.lora_sgmv_shrink(to_dev_bits(batch.x), hbuf, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    href, _ = oracle.shrink(batch.x, batch.ids, pool, h_init=np.full((batch.T, 72), -5.0), ldh=72)
    got = hbuf.cpu().numpy().astype(np.float64)
    scale = np.abs(href).max()
    np.testing.assert_allclose(got, href, rtol=1e-4, atol=1e-5 * scale)


def test_tc_interleaved_tokens_full_tiles():
    """Segments of 300 tokens whose rows are interleaved in x (every third row), so full
    tiles take the row-by-row copies, next to a run of 256 consecutive tokens."""
    rng = np.random.default_rng(28)
    ranks = [32, 8, 64, 16]
    ids = np.concatenate([np.arange(900, dtype=np.int32) % 3, np.full(256, 3, dtype=np.int32)])
    pool = W.build_pool(rng, 2048, 4096, ranks, max_rank=64)
    batch = W.make_batch(rng, ids, 2048, 4096, ldx=2048 + 8, ldy=4096 + 64)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, len(ranks))
        ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
        assert err == 0
        compare_bf16(y[:, :4096], ref, "interleaved tiles mode %d" % mode)


def test_tc_expand_caller_h_odd_stride():
    pool, batch = long_segment_batch(29, [5, 13, 64], [130, 256, 140], 1024, 2048)
    rng = np.random.default_rng(30)
    hin = rng.standard_normal((batch.T, 68), dtype=np.float32)
    view = B.PoolView.from_host(pool)
    y = to_dev_bits(batch.y0)
    seg = B.Segments(batch.T)
    err = new_err()
    B.lora_segments_build(ids_dev(batch.ids), 3, seg, err=err)
    B.lora_sgmv_expand(torch.from_numpy(hin).cuda(), y, seg, view, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _ = oracle.expand(hin, batch.y0, batch.ids, pool)
    compare_bf16(to_host_bits(y)[:, :2048], ref, "tensor-core expand, h stride 68")


def test_tc_single_full_tile():
    """T = 128, one adapter: the tile is the whole of x and y."""
    pool, batch = long_segment_batch(31, [64], [128], 4096, 4096)
    for mode in (B.LORA_SEG_GROUP, B.LORA_SEG_CONTIGUOUS):
        y, err, _ = run_apply(batch, pool, mode, 1)
        ref, _ = oracle.lora_apply(batch.x, batch.y0, batch.ids, pool)
        assert err == 0
        compare_bf16(y[:, :4096], ref, "single tile mode %d" % mode)


def test_gather_multi_token_units_mixed_subslice_widths():
    """d = 5120 gives every CTA of an 8-CTA cluster a 512- and a 128-column sub-slice;
    units of 2..8 tokens with ranks 32 and 64 use the expand accumulator across both.
    Repeated runs: the warps of a CTA meet at no barrier between chunks, so a warp
    that owned another warp's accumulator entries would show up as a varying error."""
    rng = np.random.default_rng(32)
    ranks = [32, 64, 48, 32, 64, 16, 40]
    counts = [3, 2, 4, 5, 8, 3, 7]
    ids = np.concatenate([np.full(n, i, dtype=np.int32) for i, n in enumerate(counts)])
    ids = ids[rng.permutation(ids.size)]
    pool = W.build_pool(rng, 5120, 5120, ranks, max_rank=64)
    batch = W.make_batch(rng, ids, 5120, 5120)
    ref, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    first = None
    for rep in range(4):
        y, err, _ = run_apply(batch, pool, B.LORA_SEG_GROUP, len(ranks))
        assert err == 0
        compare_bf16(y, ref, "gather 5120x5120, run %d" % rep)
        first = y if first is None else first
        assert np.array_equal(y, first)


# ------------------------------------------------------ multi-projection call --

def multi_case(seed, d_in, d_outs, n_long=3, n_short=20):
    """Projections on one batch (shared x, one pool per projection, mixed ranks) with long
    segments (tensor-core path) and short ones (gather path)."""
    rng = np.random.default_rng(seed)
    n_ad = 12
    ranks = rng.choice(np.array([8, 16, 32, 64], dtype=np.int32), size=n_ad)
    lens = list(rng.integers(129, 400, size=n_long)) + list(rng.integers(1, 8, size=n_short))
    ids = np.concatenate([np.full(n, i % n_ad, dtype=np.int32) for i, n in enumerate(lens)])
    ids = ids[rng.permutation(ids.size)]
    ids[rng.random(ids.size) < 0.03] = -1
    T = ids.size
    x = W._normal_bf16(rng, (T, d_in), 1.0)
    pools, y0s = [], []
    for d_out in d_outs:
        pools.append(W.build_pool(rng, d_in, d_out, ranks, max_rank=64))
        y0s.append(W._normal_bf16(rng, (T, d_out), 1.0))
    return ids, x, pools, y0s, n_ad


@pytest.mark.parametrize("d_in,d_outs", [(5120, (5120, 5120, 5120)), (4096, (1024, 2048)),
                                         (1024, (4096, 4096, 512, 1536))])
def test_apply_multi_matches_separate_calls_and_oracle(d_in, d_outs):
    ids, x, pools, y0s, n_ad = multi_case(41, d_in, d_outs)
    seg = B.Segments(ids.size)
    err = new_err()
    B.lora_segments_build(ids_dev(ids), n_ad, seg, mode=B.LORA_SEG_GROUP, err=err)
    views = [B.PoolView.from_host(p) for p in pools]
    xd = to_dev_bits(x)
    ys = [to_dev_bits(y0) for y0 in y0s]
    B.lora_apply_multi([(xd, y, v) for y, v in zip(ys, views)], seg, err=err)
    sep = []
    for y0, v in zip(y0s, views):
        y = to_dev_bits(y0)
        B.lora_apply(xd, y, seg, v, err=err)
        sep.append(y)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    perm, indptr, seg_ad, n_tok, short, long_ = seg.host()
    long_tok = np.zeros(ids.size, dtype=bool)
    for s_, m0 in long_:
        lo = indptr[s_] + m0
        long_tok[perm[lo:min(lo + 128, indptr[s_ + 1])]] = True
    for g, (pool, y0) in enumerate(zip(pools, y0s)):
        got, want = to_host_bits(ys[g]), to_host_bits(sep[g])
        assert np.array_equal(got[long_tok], want[long_tok]), "projection %d, tensor-core rows" % g
        ref, _ = oracle_apply(x, y0, ids, pool)
        compare_bf16(got, ref, "multi projection %d" % g)
        assert np.array_equal(got[ids < 0], y0[ids < 0])


def test_apply_multi_mixed13b_qkv_and_gate_up():
    """The 13B-shaped batch's q, k, v (one x) and gate, up (one x) as two grouped calls on
    one segment build, every row against the oracle for v and up, sampled rows otherwise."""
    rng = np.random.default_rng(77)
    for names in (("q", "k", "v"), ("gate", "up")):
        parts = [W.mixed13b_projection(0, 5, n) for n in names]
        ids = parts[0][1].ids
        x = parts[0][1].x  # one input for the group
        seg = B.Segments(ids.size)
        err = new_err()
        B.lora_segments_build(ids_dev(ids), 1000, seg, mode=B.LORA_SEG_GROUP, err=err)
        xd = to_dev_bits(x)
        ys = [to_dev_bits(b.y0) for _, b, _ in parts]
        B.lora_apply_multi([(xd, y, B.PoolView.from_host(p)) for (p, _, _), y in zip(parts, ys)], seg, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for k, ((pool, b, _), y) in enumerate(zip(parts, ys)):
            rows = np.arange(ids.size) if k == len(parts) - 1 else \
                np.sort(np.concatenate([rng.choice(4096, 128, replace=False), 4096 + np.arange(128)]))
            ref, _ = oracle_apply(x[rows], b.y0[rows], ids[rows], pool)
            compare_bf16(to_host_bits(y)[rows], ref, "13B grouped %s" % names[k])
