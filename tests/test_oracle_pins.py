"""Pins for the CPU oracle: each check ties it to something other than itself --
the pages' worked numbers, a library routine (numpy float64 matmul, Python's
stable sort), closed forms, the merged-weight identity and exact invariants.

A plausible slip in the oracle (a dropped scale, a transposed operand, a wrong
page index, an unstable grouping) fails at least one of these.
"""

import itertools

import numpy as np
import pytest

import oracle
from segmented_gather_gemm_lora_gb300 import workloads as W
from conftest import read_golden


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------- sizing --

def test_sizing_llama3_70b_table():
    """Memory-per-adapter table, Llama-3-70B r=16 ("Multi-LoRA serving: the single
    translator...", section "The maths that matters")."""
    rows = read_golden("sizing_llama3_70b_r16.txt")
    total = 0
    per = {}
    for r in rows:
        if r[0] in ("SUM", "LAYERS", "TOTAL_MIB"):
            per[r[0]] = int(r[1])
            continue
        name, d_in, d_out, rank, want = r[0], int(r[1]), int(r[2]), int(r[3]), int(r[4])
        got = oracle.adapter_bytes(rank, d_in, d_out, 2)
        assert got == want, name
        # with 4096-element bf16 pages every matrix fills whole pages: no rounding slack
        assert oracle.pages_needed(rank, d_in, d_out, 4096) * 4096 * 2 == want, name
        total += got
    assert total == per["SUM"]
    assert round(per["LAYERS"] * total / 2**20) == per["TOTAL_MIB"]


def test_sizing_llama3_8b_params():
    """Adapter parameter count, Llama-3-8B attention r=8 ("QLoRA and multi-LoRA at the
    limit on small models", section "The maths that matters")."""
    (L, m, d, r, want_m, want_mb), = read_golden("sizing_llama3_8b_attn_r8.txt")
    L, m, d, r = int(L), int(m), int(d), int(r)
    bytes_one = oracle.adapter_bytes(r, d, d, 2)  # one square matrix pair
    params = L * m * bytes_one // 2
    assert round(params / 1e6, 1) == float(want_m)
    assert round(params * 2 / 1e6, 1) == float(want_mb)


def test_sizing_qwen25_7b():
    """Per-rank adapter parameters and adapter sizes for Qwen2.5-7B ("Multi-LoRA Serving:
    Many Adapters on One GPU", sections "GPU memory budget", "Rank and slot sizing")."""
    rows = read_golden("sizing_qwen25_7b.txt")
    projs = {r[1]: (int(r[2]), int(r[3])) for r in rows if r[0] == "proj"}
    kv = {r[0]: r[1] for r in rows if r[0] != "proj"}
    per_rank = sum(oracle.adapter_bytes(1, di, do, 1) for di, do in projs.values())
    assert per_rank == int(kv["per_layer_per_rank"])
    L = int(kv["layers"])
    assert per_rank * L == int(kv["total_per_rank"])
    qv = sum(oracle.adapter_bytes(16, *projs[p], 2) for p in ("q", "v")) * L
    assert round(qv / 1e6, 1) == float(kv["qv_r16_MB"])
    all16 = sum(oracle.adapter_bytes(16, di, do, 2) for di, do in projs.values()) * L
    assert round(all16 / 1e6, 1) == float(kv["all_r16_MB"])
    all64 = sum(oracle.adapter_bytes(64, di, do, 2) for di, do in projs.values()) * L
    assert round(all64 / 1e6) == float(kv["all_r64_MB"])
    assert round(8 * all64 / 1e9, 2) == float(kv["slots8_r64_GB"])


def test_pages_needed_rounding():
    # one page partly used per matrix when r*d is not a multiple of the page
    assert oracle.pages_needed(13, 5120, 11008, 4096) == -(-13 * 5120 // 4096) + -(-13 * 11008 // 4096)
    assert oracle.pages_needed(1, 8, 8, 4096) == 2


# ------------------------------------------------------------------- bf16 --

def test_bf16_rne_identity_on_all_finite_values():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_bits_to_f32(bits)
    finite = np.isfinite(v)
    back = oracle.bf16_rne(v[finite].astype(np.float64))
    want = bits[finite].copy()
    want[want == 0x8000] = 0x8000  # -0 stays -0
    assert np.array_equal(back, want)


def test_bf16_rne_ties_to_even_and_nearest():
    rng = np.random.default_rng(5)
    bits = rng.integers(0x0080, 0x7F00, size=4000).astype(np.uint16)  # positive normals
    lo = W.bf16_bits_to_f32(bits).astype(np.float64)
    hi = W.bf16_bits_to_f32(bits + np.uint16(1)).astype(np.float64)
    mid = (lo + hi) / 2  # exact in double
    even = np.where(bits % 2 == 0, bits, bits + np.uint16(1)).astype(np.uint16)
    assert np.array_equal(oracle.bf16_rne(mid), even)
    assert np.array_equal(oracle.bf16_rne(-mid), even | np.uint16(0x8000))
    eps = (hi - lo) * 1e-3
    assert np.array_equal(oracle.bf16_rne(mid - eps), bits)
    assert np.array_equal(oracle.bf16_rne(mid + eps), bits + np.uint16(1))


# ----------------------------------------------------------- page table --

def test_unpack_equals_logical_matrices():
    rng = np.random.default_rng(1)
    pool = W.build_pool(rng, 40, 24, [1, 7, 13, 0, 5], page_elems=64)
    for i, r in enumerate(pool.ranks):
        if r == 0:
            continue
        a = oracle.unpack_matrix(pool, int(pool.desc[i]["a_page0"]), int(r), pool.d_in)
        b = oracle.unpack_matrix(pool, int(pool.desc[i]["b_page0"]), int(r), pool.d_out)
        assert np.array_equal(a, pool.A[i])
        assert np.array_equal(b, pool.B[i])


# -------------------------------------------------------------- the delta --

def numpy_reference(batch, pool):
    """Per token: y0 + s_i * (x . A_i^T) . B_i via numpy float64 matmuls on the logical
    (unpaged) matrices."""
    T = batch.T
    y = f64(batch.y0[:, : pool.d_out]).copy()
    x = f64(batch.x[:, : pool.d_in])
    for t in range(T):
        i = int(batch.ids[t])
        if i < 0:
            continue
        A = f64(pool.A[i])
        B = f64(pool.B[i])
        s = float(pool.scales[i])
        y[t] += s * ((x[t] @ A.T) @ B)
    return y


@pytest.mark.parametrize("page_elems", [64, 4096])
def test_apply_matches_numpy_matmul_mixed_ranks(page_elems):
    rng = np.random.default_rng(2)
    ranks = [8, 1, 13, 64, 16, 0]
    pool = W.build_pool(rng, 72, 40, ranks, page_elems=page_elems, max_rank=64)
    ids = np.array([0, 1, 2, 3, 4, -1, 2, 2, 0, 3, 1, 4], dtype=np.int32)
    batch = W.make_batch(rng, ids, 72, 40, ldx=80, ldy=48)
    y, err = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    assert err == 0
    ref = numpy_reference(batch, pool)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_single_adapter_reduces_to_dense_product():
    """Every token on one adapter: one dense Y0 + s (X A^T) B product (library matmul)."""
    rng = np.random.default_rng(3)
    pool = W.build_pool(rng, 256, 256, [8, 8, 8, 8])
    ids = np.full(16, 2, dtype=np.int32)
    batch = W.make_batch(rng, ids, 256, 256)
    y, err = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    X = f64(batch.x)
    ref = f64(batch.y0) + float(pool.scales[2]) * (X @ f64(pool.A[2]).T) @ f64(pool.B[2])
    assert err == 0
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_merged_weight_identity():
    """x (W0 + s A B) == x W0 + s (x A) B ("Multi-LoRA Serving in Production", section
    "Mathematical Formulation and the Batching Challenge"): W0 and x take values in
    {-1, 0, 1}, so x W0 is an integer of magnitude <= 256 and exact in bf16."""
    rng = np.random.default_rng(4)
    d = 256
    pool = W.build_pool(rng, d, d, [8, 16, 4])
    T = 12
    ids = rng.integers(0, 3, size=T).astype(np.int32)
    xv = rng.integers(-1, 2, size=(T, d)).astype(np.float32)
    W0 = rng.integers(-1, 2, size=(d, d)).astype(np.float64)
    y0v = (xv.astype(np.float64) @ W0)
    assert np.abs(y0v).max() <= 256
    x = W.f32_to_bf16_bits(xv)
    y0 = W.f32_to_bf16_bits(y0v.astype(np.float32))
    assert np.array_equal(f64(y0), y0v)
    y, err = oracle.lora_apply(x, y0, ids, pool)
    assert err == 0
    for t in range(T):
        i = ids[t]
        Wm = W0 + float(pool.scales[i]) * f64(pool.A[i]).T @ f64(pool.B[i])
        merged = xv[t].astype(np.float64) @ Wm
        np.testing.assert_allclose(y[t], merged, rtol=1e-11, atol=1e-11)


def test_rank_one_closed_form():
    rng = np.random.default_rng(6)
    pool = W.build_pool(rng, 96, 48, [1])
    ids = np.zeros(5, dtype=np.int32)
    batch = W.make_batch(rng, ids, 96, 48)
    y, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    a = f64(pool.A[0])[0]
    b = f64(pool.B[0])[0]
    s = float(pool.scales[0])
    for t in range(5):
        dot = float(np.dot(f64(batch.x[t]), a))
        np.testing.assert_allclose(y[t] - f64(batch.y0[t]), s * dot * b, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("which", ["A", "B"])
def test_zero_adapter_leaves_y0(which):
    rng = np.random.default_rng(7)
    pool = W.build_pool(rng, 64, 64, [8, 16], zero_A=(which == "A"), zero_B=(which == "B"))
    ids = np.array([0, 1, 1, 0, -1], dtype=np.int32)
    batch = W.make_batch(rng, ids, 64, 64)
    y, err = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    assert err == 0
    assert np.array_equal(y, f64(batch.y0))


def test_zero_padded_rank_equals_unpadded_exactly():
    """Padding an adapter to a higher rank with zero rows, same scale, changes nothing
    (the padded slot buffers of "Multi-LoRA Serving: Many Adapters on One GPU", section
    "Rank and slot sizing", waste memory, not accuracy)."""
    rng = np.random.default_rng(8)
    d_in, d_out = 128, 80
    base = W.build_pool(rng, d_in, d_out, [5, 16])
    A, B, ranks = [], [], []
    for i, r in enumerate(base.ranks):
        rp = int(r) + 11
        a = np.zeros((rp, d_in), dtype=np.uint16)
        b = np.zeros((rp, d_out), dtype=np.uint16)
        a[:r] = base.A[i]
        b[:r] = base.B[i]
        A.append(a)
        B.append(b)
        ranks.append(rp)
    padded = W.pack_pool(A, B, np.array(ranks), d_in, d_out, rng, scales=base.scales,
                         max_rank=32)
    ids = np.array([0, 1, 0, 1, 1], dtype=np.int32)
    batch = W.make_batch(rng, ids, d_in, d_out)
    y1, _ = oracle.lora_apply(batch.x, batch.y0, ids, base)
    y2, _ = oracle.lora_apply(batch.x, batch.y0, ids, padded)
    assert np.array_equal(y1, y2)


def test_token_order_invariance_exact():
    rng = np.random.default_rng(9)
    pool = W.build_pool(rng, 64, 32, [8, 4, 12])
    ids = rng.integers(-1, 3, size=20).astype(np.int32)
    batch = W.make_batch(rng, ids, 64, 32)
    y, _ = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    p = rng.permutation(20)
    yp, _ = oracle.lora_apply(batch.x[p], batch.y0[p], ids[p], pool)
    assert np.array_equal(yp, y[p])


def test_linearity_in_scale_and_x_exact():
    rng = np.random.default_rng(10)
    pool = W.build_pool(rng, 64, 32, [8, 4])
    ids = np.array([0, 1, 1, 0], dtype=np.int32)
    batch = W.make_batch(rng, ids, 64, 32)
    zero = np.zeros_like(batch.y0)
    y, _ = oracle.lora_apply(batch.x, zero, ids, pool)
    pool2 = W.pack_pool(pool.A, pool.B, pool.ranks, 64, 32, rng, scales=2 * pool.scales)
    y2, _ = oracle.lora_apply(batch.x, zero, ids, pool2)
    assert np.array_equal(y2, 2 * y)
    x2 = W.f32_to_bf16_bits(2 * W.bf16_bits_to_f32(batch.x))
    yx, _ = oracle.lora_apply(x2, zero, ids, pool)
    assert np.array_equal(yx, 2 * y)


def test_bad_inputs_keep_y0_and_flag():
    rng = np.random.default_rng(11)
    pool = W.build_pool(rng, 32, 32, [4, 4, 4], max_rank=8)
    pool.desc[1]["rank"] = 9  # above max_rank
    pool.page_list[int(pool.desc[2]["b_page0"])] = pool.n_pages + 5  # page outside the pool
    ids = np.array([0, 7, 1, 2, -2, -1], dtype=np.int32)
    batch = W.make_batch(rng, ids, 32, 32)
    y, err = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    assert err == 1 | 2 | 4
    assert np.array_equal(y[1:], f64(batch.y0[1:]))
    assert not np.array_equal(y[0], f64(batch.y0[0]))


def test_shrink_expand_compose_to_apply():
    rng = np.random.default_rng(12)
    pool = W.build_pool(rng, 128, 64, [8, 16, 3], max_rank=16)
    ids = np.array([2, 0, 1, -1, 1, 0], dtype=np.int32)
    batch = W.make_batch(rng, ids, 128, 64)
    h, e1 = oracle.shrink(batch.x, ids, pool)
    X = f64(batch.x)
    for t, i in enumerate(ids):
        if i >= 0:
            np.testing.assert_allclose(h[t, : pool.ranks[i]], X[t] @ f64(pool.A[i]).T, rtol=1e-12,
                                       atol=1e-13)
    y_chain, e2 = oracle.expand(h.astype(np.float32), batch.y0, ids, pool)
    y, e3 = oracle.lora_apply(batch.x, batch.y0, ids, pool)
    assert e1 == e2 == e3 == 0
    np.testing.assert_allclose(y_chain, y, rtol=1e-6, atol=1e-6)  # h passed through fp32


# ------------------------------------------------------------- segments --

def brute_segments(ids, n_adapters, mode):
    ids = list(ids)
    valid = [t for t in range(len(ids)) if 0 <= ids[t] < n_adapters]
    if mode == oracle.GROUP:
        perm = sorted(valid, key=lambda t: ids[t])  # Python's sort is stable
        groups = [list(g) for _, g in itertools.groupby(perm, key=lambda t: ids[t])]
    else:
        groups = []
        for key, g in itertools.groupby(range(len(ids)), key=lambda t: ids[t]):
            g = list(g)
            if 0 <= key < n_adapters:
                groups.append(g)
        perm = [t for g in groups for t in g]
    indptr = np.cumsum([0] + [len(g) for g in groups])
    seg_ad = [ids[g[0]] for g in groups]
    return np.array(perm), indptr, np.array(seg_ad)


@pytest.mark.parametrize("mode", [0, 1])
def test_segments_match_brute_force(mode):
    rng = np.random.default_rng(13)
    cases = [
        np.array([], dtype=np.int32),
        np.full(7, -1, dtype=np.int32),
        np.zeros(9, dtype=np.int32),
        np.arange(10, dtype=np.int32),
        np.array([3, 3, 1, 1, 3, -1, 3, 0, 0, 9], dtype=np.int32),
    ]
    for _ in range(40):
        T = int(rng.integers(1, 200))
        n = int(rng.integers(1, 20))
        cases.append(rng.integers(-1, n, size=T).astype(np.int32))
        cases.append(np.repeat(rng.integers(-1, n, size=T // 5 + 1), rng.integers(1, 9, size=T // 5 + 1)).astype(np.int32))
    for ids in cases:
        n_ad = 10 if ids.size == 0 else max(int(ids.max()) + 1, 1)
        perm, indptr, seg_ad, n_tok, err = oracle.segments_build(ids, n_ad, mode)
        bp, bi, ba = brute_segments(ids, n_ad, mode)
        assert err == 0
        assert np.array_equal(perm, bp)
        assert np.array_equal(indptr, bi)
        assert np.array_equal(seg_ad, ba)
        assert n_tok == int((ids >= 0).sum())


def test_segments_flag_invalid_ids():
    ids = np.array([0, 5, -3, 1, 1], dtype=np.int32)
    perm, indptr, seg_ad, n_tok, err = oracle.segments_build(ids, 4, oracle.GROUP)
    assert err == 1
    assert perm.tolist() == [0, 3, 4]
    assert seg_ad.tolist() == [0, 1]


def test_work_lists_brute_force():
    rng = np.random.default_rng(14)
    for _ in range(30):
        lens = rng.integers(1, 400, size=int(rng.integers(1, 12)))
        indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        short_max, tile = 8, 128
        s, l = oracle.work_lists(indptr, short_max, tile)
        want_s = [i for i, n in enumerate(lens) if n <= short_max]
        want_l = [(i, m0) for i, n in enumerate(lens) if n > short_max for m0 in range(0, n, tile)]
        assert s.tolist() == want_s
        assert [tuple(v) for v in l.tolist()] == want_l


def test_group_and_contiguous_give_same_outputs():
    """GROUP vs CONTIGUOUS segmentation changes the schedule, not the result: the
    per-token delta depends only on the token's own adapter."""
    rng = np.random.default_rng(15)
    ids = np.repeat(rng.integers(0, 5, size=12), rng.integers(1, 6, size=12)).astype(np.int32)
    for mode in (0, 1):
        perm, indptr, seg_ad, n_tok, _ = oracle.segments_build(ids, 5, mode)
        # every token sits in exactly one segment, whose adapter is its own
        seen = np.zeros(ids.size, dtype=int)
        for s in range(len(seg_ad)):
            for t in perm[indptr[s]: indptr[s + 1]]:
                seen[t] += 1
                assert ids[t] == seg_ad[s]
        assert (seen == 1).all()


# -------------------------------------------------------------- gradients --
#
# The backward oracle gives dL/dA_i, dL/dB_i (added at the pool positions of A_i
# and B_i) and dL/dx for L = sum_{t,n} g[t,n] y[t,n].  y is exactly linear in each
# adapter element and in each x element, so a finite difference of the forward
# oracle between two bf16 values of one element is exact up to fp64 rounding.

def backward_case(seed, d_in=64, d_out=48, ranks=(3, 5, 8), T=12, page_elems=64):
    rng = np.random.default_rng(seed)
    pool = W.build_pool(rng, d_in, d_out, list(ranks), page_elems=page_elems, max_rank=16)
    ids = rng.integers(-1, len(ranks), size=T).astype(np.int32)
    ids[:len(ranks)] = np.arange(len(ranks))  # every adapter used at least once
    batch = W.make_batch(rng, ids, d_in, d_out)
    g = W._normal_bf16(rng, (T, d_out), 1.0)
    return pool, batch, g


def loss(pool, batch, g):
    y, err = oracle.lora_apply(batch.x, batch.y0, batch.ids, pool)
    assert err == 0
    return float((f64(g) * y).sum())


def with_element(bits, idx, step):
    out = bits.copy()
    out[idx] = np.uint16(int(out[idx]) + step)
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_finite_differences(seed):
    pool, batch, g = backward_case(seed)
    dx, grad, err = oracle.lora_backward(batch.x, g, batch.ids, pool)
    assert err == 0
    L0 = loss(pool, batch, g)
    rng = np.random.default_rng(100 + seed)
    flat = pool.pool.reshape(-1)
    for i in range(pool.n_adapters):
        r = int(pool.ranks[i])
        for page0, rows, cols in ((int(pool.desc[i]["a_page0"]), r, pool.d_in),
                                  (int(pool.desc[i]["b_page0"]), r, pool.d_out)):
            for _ in range(4):
                e = int(rng.integers(0, rows * cols))
                q = int(pool.page_list[page0 + e // pool.page_elems]) * pool.page_elems + e % pool.page_elems
                p2 = W.AdapterPool(**{**pool.__dict__, "pool": with_element(flat, q, 37).reshape(pool.pool.shape)})
                delta = float(f64(p2.pool.reshape(-1)[q]) - f64(flat[q]))
                fd = (loss(p2, batch, g) - L0) / delta
                assert fd == pytest.approx(grad.reshape(-1)[q], rel=1e-7, abs=1e-9), (i, page0, e)
    for _ in range(6):  # dx through the adapter path (y0 is fixed)
        t, k = int(rng.integers(0, batch.T)), int(rng.integers(0, pool.d_in))
        b2 = W.Batch(x=with_element(batch.x, (t, k), 37), y0=batch.y0, ids=batch.ids, d_in=batch.d_in,
                     d_out=batch.d_out)
        delta = float(f64(b2.x[t, k]) - f64(batch.x[t, k]))
        fd = (loss(pool, b2, g) - L0) / delta
        assert fd == pytest.approx(dx[t, k], rel=1e-7, abs=1e-9), (t, k)


def test_backward_single_adapter_is_dense_products():
    """One adapter for every token: dB = s H^T G, dA = s U^T X, dx = s U A with H = X A^T,
    U = G B^T, checked against numpy float64 matmul on the logical matrices."""
    rng = np.random.default_rng(5)
    pool = W.build_pool(rng, 96, 80, [8], page_elems=64, max_rank=8)
    ids = np.zeros(20, dtype=np.int32)
    batch = W.make_batch(rng, ids, 96, 80)
    g = W._normal_bf16(rng, (20, 80), 1.0)
    dx, grad, err = oracle.lora_backward(batch.x, g, ids, pool)
    assert err == 0
    A, Bm = f64(pool.A[0]), f64(pool.B[0])
    X, G = f64(batch.x), f64(g)
    s = float(pool.scales[0])
    H, U = X @ A.T, G @ Bm.T
    d = pool.desc[0]
    np.testing.assert_allclose(oracle.unpack_grad(grad, pool, int(d["b_page0"]), 8, 80), s * H.T @ G, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(oracle.unpack_grad(grad, pool, int(d["a_page0"]), 8, 96), s * U.T @ X, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(dx, s * U @ A, rtol=1e-12, atol=1e-12)


def test_backward_zero_gradient_and_untouched_tokens():
    pool, batch, g = backward_case(3)
    dx, grad, _ = oracle.lora_backward(batch.x, np.zeros_like(g), batch.ids, pool)
    assert not dx.any() and not grad.any()
    dx, grad, _ = oracle.lora_backward(batch.x, g, batch.ids, pool)
    none = batch.ids < 0
    assert not dx[none].any()
    keep = ~none  # tokens without an adapter contribute nothing
    dx2, grad2, _ = oracle.lora_backward(batch.x[keep], g[keep], batch.ids[keep], pool)
    np.testing.assert_array_equal(grad2, grad)
    # gradients accumulate into the array given
    _, grad3, _ = oracle.lora_backward(batch.x, g, batch.ids, pool, grad=grad.copy())
    np.testing.assert_allclose(grad3, 2 * grad, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ base projection and delta --

def base_case(seed, d_in=72, d_out=40, ranks=(8, 1, 13, 16), T=12, ldw=None, page_elems=64):
    rng = np.random.default_rng(seed)
    pool = W.build_pool(rng, d_in, d_out, list(ranks), page_elems=page_elems, max_rank=16)
    ids = rng.integers(-1, len(ranks), size=T).astype(np.int32)
    batch = W.make_batch(rng, ids, d_in, d_out, ldx=d_in + 8)
    ldw = d_in + 16 if ldw is None else ldw
    w0 = W.f32_to_bf16_bits((rng.standard_normal((d_out, ldw)) / np.sqrt(d_in)).astype(np.float32))
    return pool, batch, w0


def test_base_apply_matches_numpy_matmul():
    """y = X W0^T + s_i (x A_i^T) B_i per token, against numpy float64 matmuls on the logical
    matrices (W0 read through its row stride, the pool through its pages)."""
    pool, batch, w0 = base_case(40)
    y, err = oracle.base_apply(batch.x, w0, batch.ids, pool)
    assert err == 0
    X = f64(batch.x[:, : pool.d_in])
    ref = X @ f64(w0[:, : pool.d_in]).T
    for t, i in enumerate(batch.ids):
        if i >= 0:
            ref[t] += float(pool.scales[i]) * ((X[t] @ f64(pool.A[i]).T) @ f64(pool.B[i]))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_base_apply_merged_weight_identity():
    """x (W0 + s A^T B)^T == x W0^T + s (x A^T) B for every token of adapter i ("Multi-LoRA
    Serving in Production", section "Mathematical Formulation and the Batching Challenge")."""
    pool, batch, w0 = base_case(41, d_in=64, d_out=56, ranks=(4, 16, 2))
    y, err = oracle.base_apply(batch.x, w0, batch.ids, pool)
    assert err == 0
    X = f64(batch.x[:, :64])
    W0 = f64(w0[:, :64])
    for t, i in enumerate(batch.ids):
        Wm = W0 if i < 0 else W0 + float(pool.scales[i]) * (f64(pool.B[i]).T @ f64(pool.A[i]))
        np.testing.assert_allclose(y[t], X[t] @ Wm.T, rtol=1e-11, atol=1e-11)


def test_base_apply_reduces_to_lora_apply_and_to_the_base():
    """W0 = 0 gives lora_apply's result on y0 = 0 exactly; no adapter (every id -1) gives
    the base product alone; a bad adapter keeps the base term and flags its bit."""
    pool, batch, w0 = base_case(42)
    zero = np.zeros_like(w0)
    y, err = oracle.base_apply(batch.x, zero, batch.ids, pool)
    y0 = np.zeros((batch.T, pool.d_out), dtype=np.uint16)
    want, werr = oracle.lora_apply(batch.x, y0, batch.ids, pool)
    assert err == werr == 0
    np.testing.assert_array_equal(y, want)
    none = np.full(batch.T, -1, dtype=np.int32)
    yb, eb = oracle.base_apply(batch.x, w0, none, pool)
    assert eb == 0
    np.testing.assert_allclose(yb, f64(batch.x[:, : pool.d_in]) @ f64(w0[:, : pool.d_in]).T, rtol=1e-12,
                               atol=1e-12)
    bad = batch.ids.copy()
    bad[0] = pool.n_adapters + 2
    y2, e2 = oracle.base_apply(batch.x, w0, bad, pool)
    assert e2 == 1  # bad adapter id
    np.testing.assert_array_equal(y2[0], yb[0])
    np.testing.assert_array_equal(y2[1:], oracle.base_apply(batch.x, w0, batch.ids, pool)[0][1:])
