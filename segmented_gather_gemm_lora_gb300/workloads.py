"""Seeded synthetic inputs for the multi-adapter LoRA path.

This module only *draws* inputs: activations x, base outputs y0, per-token
adapter ids, adapter matrices A_i / B_i and a paged adapter pool that holds
them.  It contains none of the method's arithmetic (no shrink, no expand, no
segment grouping); both the CPU oracle and the CUDA library consume what it
returns, so the two see identical bf16 bits.

Value distributions (the five workload shapes of the multi-LoRA serving pages:
tiny SGMV, decode BGMV, prefill SGMV, heterogeneous ranks, 13B-shaped mixed
batch):

* every value is drawn in fp32 from ``numpy.random.default_rng(seed)``
  (PCG64) and rounded once to bf16 with round-to-nearest-even;
* x ~ N(0, 1), y0 ~ N(0, 1), A_i ~ N(0, 1/d_in), B_i ~ N(0, 1/r_i);
* adapter popularity follows Zipf(s): p(k) ~ k^-s for k = 1..N, mapped to
  adapter id k-1 (benchmark protocol of "Multi-LoRA Serving: Many Adapters
  on One GPU", section "Benchmark protocol", items 1-2);
* alpha = 16 for every adapter, so scale_i = 16 / r_i (the PEFT example in
  "QLoRA and multi-LoRA at the limit", LoraConfig table).

Storage orientation (both row-major, bf16):

* A_i is stored as r_i rows of d_in elements: row j is column j of the
  d_in x r_i matrix of "Multi-LoRA Serving in Production", section
  "Mathematical Formulation and the Batching Challenge".
* B_i is stored as r_i rows of d_out elements (the r_i x d_out matrix of the
  same section, as is).

Paged pool ("Multi-LoRA Serving in Production", section "Unified Paged
Memory"): the pool is ``n_pages`` pages of ``page_elems`` bf16 elements.  An
adapter matrix with E = r * d elements occupies ceil(E / page_elems) pages,
listed in order in ``page_list`` starting at ``a_page0`` (A) or ``b_page0``
(B); logical element e lives on page ``page_list[page0 + e // P]`` at offset
``e % P``.  Physical pages are a random permutation of the pool, so an adapter
is never contiguous.  Every pool element that no adapter owns (spare pages and
the tail of each adapter's last page) is filled with a bf16 NaN so that a read
of unowned memory poisons the result.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

DESC_DTYPE = np.dtype(
    [("rank", "<i4"), ("scale", "<f4"), ("a_page0", "<i4"), ("b_page0", "<i4")]
)
"""Per-adapter descriptor, byte-compatible with the C struct lora_adapter_desc_t."""


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return f32_to_bf16_bits(v)


def zipf_ids(rng: np.random.Generator, n_catalogue: int, s: float, size: int) -> np.ndarray:
    """Draw adapter ids from Zipf(s) over a finite catalogue of n_catalogue adapters."""
    k = np.arange(1, n_catalogue + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    return rng.choice(n_catalogue, size=size, p=p).astype(np.int32)


@dataclasses.dataclass
class AdapterPool:
    """One projection's paged adapter pool (a lora_pool_view_t on the host)."""

    d_in: int
    d_out: int
    page_elems: int
    desc: np.ndarray  # DESC_DTYPE [n_adapters]; rank 0 = not resident
    page_list: np.ndarray  # int32 [n_page_list]
    pool: np.ndarray  # uint16 [n_pages, page_elems]
    A: List[Optional[np.ndarray]]  # logical uint16 [r_i, d_in] or None
    B: List[Optional[np.ndarray]]  # logical uint16 [r_i, d_out] or None
    max_rank: int

    @property
    def n_adapters(self) -> int:
        return int(self.desc.shape[0])

    @property
    def n_pages(self) -> int:
        return int(self.pool.shape[0])

    @property
    def ranks(self) -> np.ndarray:
        return self.desc["rank"]

    @property
    def scales(self) -> np.ndarray:
        return self.desc["scale"]


@dataclasses.dataclass
class Batch:
    """Token activations, base outputs and per-token adapter ids."""

    x: np.ndarray  # uint16 [T, ldx]; columns >= d_in are padding
    y0: np.ndarray  # uint16 [T, ldy]; columns >= d_out are guard values
    ids: np.ndarray  # int32 [T]; -1 = no adapter
    d_in: int
    d_out: int

    @property
    def T(self) -> int:
        return int(self.ids.shape[0])


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def build_pool(
    rng: np.random.Generator,
    d_in: int,
    d_out: int,
    ranks: Sequence[int],
    *,
    alpha: float = 16.0,
    page_elems: int = 4096,
    max_rank: Optional[int] = None,
    spare_pages: int = 3,
    zero_B: bool = False,
    zero_A: bool = False,
    scales: Optional[Sequence[float]] = None,
    shuffle_pages: bool = True,
) -> AdapterPool:
    """Draw adapters of the given ranks (0 = not resident) and pack them into pages."""
    n = len(ranks)
    ranks = np.asarray(ranks, dtype=np.int32)
    A: List[Optional[np.ndarray]] = []
    B: List[Optional[np.ndarray]] = []
    for r in ranks:
        r = int(r)
        if r <= 0:
            A.append(None)
            B.append(None)
            continue
        a = _normal_bf16(rng, (r, d_in), (1.0 / d_in) ** 0.5)
        b = _normal_bf16(rng, (r, d_out), (1.0 / r) ** 0.5)
        if zero_A:
            a[:] = 0
        if zero_B:
            b[:] = 0
        A.append(a)
        B.append(b)
    return pack_pool(A, B, ranks, d_in, d_out, rng, alpha=alpha, page_elems=page_elems,
                     max_rank=max_rank, spare_pages=spare_pages, scales=scales,
                     shuffle_pages=shuffle_pages)


def pack_pool(
    A: List[Optional[np.ndarray]],
    B: List[Optional[np.ndarray]],
    ranks: np.ndarray,
    d_in: int,
    d_out: int,
    rng: np.random.Generator,
    *,
    alpha: float = 16.0,
    page_elems: int = 4096,
    max_rank: Optional[int] = None,
    spare_pages: int = 3,
    scales: Optional[Sequence[float]] = None,
    shuffle_pages: bool = True,
) -> AdapterPool:
    """Lay logical adapter matrices out on physical pages: a random permutation of the
    pool (default), or in order when shuffle_pages is False."""
    P = int(page_elems)
    n = len(ranks)
    desc = np.zeros(n, dtype=DESC_DTYPE)
    counts = []
    for i, r in enumerate(ranks):
        r = int(r)
        na = _ceil_div(r * d_in, P) if r > 0 else 0
        nb = _ceil_div(r * d_out, P) if r > 0 else 0
        counts.append((na, nb))
    n_list = sum(na + nb for na, nb in counts)
    n_pages = n_list + spare_pages
    phys = rng.permutation(n_pages).astype(np.int32) if shuffle_pages else np.arange(n_pages, dtype=np.int32)
    page_list = phys[:n_list].copy()
    pool = np.full((n_pages, P), BF16_NAN, dtype=np.uint16)
    flat = pool.reshape(-1)
    cursor = 0
    for i, r in enumerate(ranks):
        r = int(r)
        na, nb = counts[i]
        desc[i]["rank"] = r
        if scales is not None:
            desc[i]["scale"] = np.float32(scales[i])
        else:
            desc[i]["scale"] = np.float32(alpha / r) if r > 0 else np.float32(0.0)
        desc[i]["a_page0"] = cursor
        desc[i]["b_page0"] = cursor + na
        for mat, npg, start in ((A[i], na, cursor), (B[i], nb, cursor + na)):
            if mat is None or npg == 0:
                continue
            src = mat.reshape(-1)
            for p in range(npg):
                lo = p * P
                hi = min(lo + P, src.size)
                base = int(page_list[start + p]) * P
                flat[base: base + (hi - lo)] = src[lo:hi]
        cursor += na + nb
    mr = int(max_rank) if max_rank is not None else max(1, int(ranks.max(initial=1)))
    return AdapterPool(d_in=d_in, d_out=d_out, page_elems=P, desc=desc, page_list=page_list,
                       pool=pool, A=A, B=B, max_rank=mr)


def make_batch(
    rng: np.random.Generator,
    ids: np.ndarray,
    d_in: int,
    d_out: int,
    *,
    ldx: Optional[int] = None,
    ldy: Optional[int] = None,
) -> Batch:
    """Draw x ~ N(0,1) and y0 ~ N(0,1) for the given per-token adapter ids."""
    T = int(len(ids))
    ldx = d_in if ldx is None else ldx
    ldy = d_out if ldy is None else ldy
    x = np.zeros((T, ldx), dtype=np.uint16)
    y0 = np.full((T, ldy), np.uint16(0x4049), dtype=np.uint16)  # guard columns: 3.140625
    x[:, :d_in] = _normal_bf16(rng, (T, d_in), 1.0)
    y0[:, :d_out] = _normal_bf16(rng, (T, d_out), 1.0)
    return Batch(x=x, y0=y0, ids=np.asarray(ids, dtype=np.int32).copy(), d_in=d_in, d_out=d_out)


# ---------------------------------------------------------------------------
# The five workload shapes.
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    batch: Batch
    pools: List[AdapterPool]  # one per projection call (same batch ids)
    mode: int  # 0 = GROUP segments, 1 = CONTIGUOUS segments
    n_adapters: int
    note: str = ""


def tiny(seed: int = 0) -> Workload:
    """d_in = d_out = 256, 4 adapters of rank 8, alpha 16, 16 tokens in segments [3,5,1,7]."""
    rng = np.random.default_rng(seed)
    ids = np.repeat(np.arange(4, dtype=np.int32), [3, 5, 1, 7])
    pool = build_pool(rng, 256, 256, [8, 8, 8, 8])
    batch = make_batch(rng, ids, 256, 256)
    return Workload("tiny", batch, [pool], mode=0, n_adapters=4)


def decode(seed: int = 0, T: int = 64) -> Workload:
    """64 decode tokens (one per request), q_proj 4096 -> 4096, 100 adapters of rank 16."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, 100, size=T).astype(np.int32)
    pool = build_pool(rng, 4096, 4096, [16] * 100)
    batch = make_batch(rng, ids, 4096, 4096)
    return Workload("decode", batch, [pool], mode=0, n_adapters=100)


def prefill_lengths(rng: np.random.Generator, n_requests: int = 32, lo: int = 64, hi: int = 512):
    return rng.integers(lo, hi + 1, size=n_requests)


def prefill(seed: int = 0, n_requests: int = 32) -> Workload:
    """32 requests of 64..512 tokens, 4096 -> 4096, 200 rank-16 adapters, Zipf(1.1) popularity."""
    rng = np.random.default_rng(seed)
    lengths = prefill_lengths(rng, n_requests)
    req_ad = zipf_ids(rng, 200, 1.1, n_requests)
    ids = np.repeat(req_ad, lengths).astype(np.int32)
    pool = build_pool(rng, 4096, 4096, [16] * 200)
    batch = make_batch(rng, ids, 4096, 4096)
    return Workload("prefill", batch, [pool], mode=1, n_adapters=200)


def hetero(seed: int = 0, T: int = 256, which: str = "both") -> Workload:
    """256 decode tokens, 500 adapters with ranks in {8,16,32,64}, MLP up 4096->11008 and
    down 11008->4096 as two separate calls (two pools, two batches sharing the ids)."""
    rng = np.random.default_rng(seed)
    ranks = rng.choice(np.array([8, 16, 32, 64], dtype=np.int32), size=500)
    ids = rng.integers(0, 500, size=T).astype(np.int32)
    pools = []
    if which in ("both", "up"):
        pools.append(build_pool(rng, 4096, 11008, ranks, max_rank=64))
    if which in ("both", "down"):
        pools.append(build_pool(rng, 11008, 4096, ranks, max_rank=64))
    batch = make_batch(rng, ids, 4096, 11008)
    return Workload("hetero", batch, pools, mode=0, n_adapters=500,
                    note="batch is for the up projection; use make_batch(...) for down")


PROJ_13B = (
    ("q", 5120, 5120),
    ("k", 5120, 5120),
    ("v", 5120, 5120),
    ("o", 5120, 5120),
    ("gate", 5120, 13824),
    ("up", 5120, 13824),
    ("down", 13824, 5120),
)


def mixed13b_ids(rng: np.random.Generator, n_decode: int = 128, n_prefill: int = 4,
                 prefill_len: int = 1024, n_catalogue: int = 1000):
    """Per-token ids of the 13B-shaped mixed batch: 4 prefill requests of 1024 tokens followed
    by 128 decode tokens, each request's adapter drawn from Zipf(1.1) over 1000 adapters."""
    pre = zipf_ids(rng, n_catalogue, 1.1, n_prefill)
    dec = zipf_ids(rng, n_catalogue, 1.1, n_decode)
    ids = np.concatenate([np.repeat(pre, prefill_len), dec]).astype(np.int32)
    return ids


def mixed13b_ranks(rng: np.random.Generator, n_catalogue: int = 1000) -> np.ndarray:
    return rng.choice(np.array([16, 32, 64], dtype=np.int32), size=n_catalogue)


def mixed13b(seed: int = 0, layers: Sequence[int] = (0,), projections: Sequence[str] = None,
             n_decode: int = 128) -> Workload:
    """13B-shaped mixed batch: only the adapters the batch references are resident (rank 0 for
    the rest of the 1000-adapter catalogue).  Returns the pools of the requested layers and
    projections, in (layer, projection) order; each has its own adapter matrices."""
    rng = np.random.default_rng(seed)
    ranks = mixed13b_ranks(rng)
    ids = mixed13b_ids(rng, n_decode=n_decode)
    referenced = np.zeros(1000, dtype=bool)
    referenced[np.unique(ids)] = True
    resident = np.where(referenced, ranks, 0).astype(np.int32)
    names = [p[0] for p in PROJ_13B] if projections is None else list(projections)
    pools = [mixed13b_pool(seed, resident, layer, name) for layer in layers for name in names]
    batch = make_batch(rng, ids, 5120, 5120)
    return Workload("mixed13b", batch, pools, mode=0, n_adapters=1000)


def mixed13b_pool(seed: int, resident: np.ndarray, layer: int, name: str) -> AdapterPool:
    """One (layer, projection) pool of the 13B-shaped batch; its draws depend only on the
    seed, the layer and the projection's place in the layer."""
    order = [p[0] for p in PROJ_13B]
    _, d_in, d_out = PROJ_13B[order.index(name)]
    prng = np.random.default_rng([seed, 1 + int(layer), 1 + order.index(name)])
    return build_pool(prng, d_in, d_out, resident, max_rank=64)


def mixed13b_projection(seed: int, layer: int, name: str):
    """(pool, batch, n_adapters) of one (layer, projection) call of the 13B-shaped batch:
    the pool as mixed13b draws it and a batch of that projection's shape on the batch's
    ids (x and y0 drawn from the seed, the layer and the projection)."""
    rng = np.random.default_rng(seed)
    ranks = mixed13b_ranks(rng)
    ids = mixed13b_ids(rng)
    resident = np.zeros(1000, dtype=np.int32)
    used = np.unique(ids)
    resident[used] = ranks[used]
    pool = mixed13b_pool(seed, resident, layer, name)
    order = [p[0] for p in PROJ_13B]
    brng = np.random.default_rng([seed, 101 + int(layer), 1 + order.index(name)])
    return pool, make_batch(brng, ids, pool.d_in, pool.d_out), 1000


WORKLOADS = {
    "tiny": tiny,
    "decode": decode,
    "prefill": prefill,
    "hetero": hetero,
    "mixed13b": mixed13b,
}
