// Tensor-core path for long segments (tcgen05 MMA, accumulators in tensor
// memory).
//
// "Multi-LoRA serving: the single translator with a thousand glossaries",
// section "SGMV: the kernel that holds it all up": for large segments (several
// requests on one adapter) the product goes through the tensor cores.  The
// multi-size gather GEMM of "Multi-LoRA Serving in Production", section
// "S-LoRA: MBGMV and MBGMM Kernels", tiles the token dimension and the
// projection dimensions per segment; here a tile is LORA_TILE_M = 128 tokens
// of one segment (rows gathered through the segment's token list) and the
// inner dimension is the adapter's own rank r_i, padded only to the MMA's
// granularity of 16 inside shared memory (never in the pool).
//
// Two persistent, warp-specialized kernels, one CTA per SM: loader warps feed
// rings of shared-memory stages (16-byte asynchronous copies signal their
// stage's mbarrier as they land, TMA copies count their bytes on it), one warp
// issues the MMAs, the other warps run the epilogue.  Two tensor-memory
// accumulators let one unit's epilogue overlap the next unit's loads and MMAs.
//
//  shrink_tc  H[128, r] = X[128, d_in] . A_i^T.  A unit is (tile, slice of
//             about 512 columns of d_in).  64-column chunks of x and of A_i
//             stream through a 6-stage ring in 128-byte-swizzle K-major form
//             into tcgen05.mma M = 128, N = r padded to 16.  With one slice per
//             tile the epilogue writes h; otherwise each unit writes an fp32
//             partial and reduce_partials sums a tile's partials in slice order,
//             so the result does not depend on timing.
//  expand_tc  Y[128, n0:n0+128] = bf16(Y0 + (s_i H) . B_i[:, n0:n0+128]).
//             A unit is (tile, 128-column chunk), so the expand, which carries
//             two thirds of the bytes, spreads over every SM.  s_i H is split
//             into bf16 hi + lo parts (two MMAs accumulating into the same fp32
//             columns), keeping the rank-r intermediate at about fp32
//             accuracy.  B_i rows are MN-major operands (r_i rows of d_out
//             contiguous elements, as stored).  y0 arrives by TMA tensor
//             copies for tiles of 128 consecutive tokens, by 16-byte
//             asynchronous copies otherwise; y leaves by coalesced 16-byte
//             stores.
//
// Tokens of one segment are listed in increasing order (the segment builder's
// order is stable), so a tile whose first and last tokens are 127 apart is the
// consecutive rows row0 .. row0 + 127 of x and y.
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc.cuh"

namespace lora {

// Four consecutive fp32 values to h[j .. j + 3], only those below r.
__device__ __forceinline__ void store_h4(float* hrow, int j, int r, float a, float b, float c, float d) {
  if (j + 3 < r) {
    *reinterpret_cast<float4*>(hrow + j) = make_float4(a, b, c, d);
  } else {
    const float v[4] = {a, b, c, d};
    for (int e = 0; e < 4 && j + e < r; ++e) hrow[j + e] = v[e];
  }
}

// Wait on the last (up to) `depth` phases a producer completed on a ring of
// `depth` barriers, so no asynchronous copy is still landing when the CTA ends.
__device__ __forceinline__ void drain_ring(uint64_t* ring, uint32_t issued, uint32_t depth) {
  for (uint32_t gg = issued > depth ? issued - depth : 0; gg < issued; ++gg)
    mbar_wait(smem_u32(&ring[gg % depth]), (gg / depth) & 1);
}

// ---------------------------------------------------------------- shrink_tc --
//
// Warp roles: 0-1 schedule (each claims units from a counter in the segment
// buffer and resolves tile, adapter and pages), 2-5 load, 6 issues MMAs, 7-10
// epilogue.  Units pass from the schedulers to the loaders through a 4-slot
// queue in shared memory (scheduler s fills slots s and s + 2), chunks from the
// loaders to the MMA warp through a 6-stage ring whose stages carry a record
// of their chunk, and finished units from the MMA warp to the epilogue with
// their accumulator.  Only the schedulers read the segment and adapter tables.
//
// A TMA tensor copy moves 128-byte box rows at a fixed rate per SM, so of a
// full tile's 128 x rows per chunk the first 64 come by TMA and the rest, with
// the adapter rows, by the four loader warps' 16-byte asynchronous copies; the
// two engines run side by side.

constexpr int kSThreads = 352;
constexpr int kSSched = 2, kSLoad = 4;
constexpr int kSWarpLoad0 = 2, kSWarpMma = 6;  // epilogue: warps 7-10
constexpr int kSStages = 6;
constexpr int kSXBytes = kTM * 128;  // x tile: 128 rows x 64 bf16
constexpr int kSABytes = 64 * 128;   // A tile: up to 64 rank rows x 64 bf16
constexpr int kSStageBytes = kSXBytes + kSABytes;
constexpr int kSTmaRows = 64;    // x rows of a full tile that come by TMA
static_assert(kSTmaRows % 16 == 0 && kSTmaRows <= kTM, "x rows split between TMA and the loader warps");
constexpr int kSMaxChunks = 64;  // 64-column chunks per unit
constexpr int kRecEnd = 1, kRecTma = 2, kRecNewTile = 4;

struct SUnit {  // scheduler -> loaders
  int tile, q, r, rpad, nch, kbeg, p0, cnt, row0, flags;
};
struct SRec {  // loaders -> MMA warp, one per stage
  int tile, q, r, rpad, c, nch, p0, cnt, flags;
};
struct ARec {  // MMA warp -> epilogue, one per accumulator
  int tile, q, r, rpad, p0, cnt, flags;
};

constexpr int kSSlotBytes = 64 + kTM * 4 + 64 * kSMaxChunks * 4;  // record, x rows, A pages
constexpr size_t kSOffQ = (size_t)kSStages * kSStageBytes;
constexpr size_t kSOffRec = kSOffQ + 4 * (size_t)kSSlotBytes;
constexpr size_t kSOffARec = kSOffRec + (size_t)kSStages * 64;
constexpr size_t kSOffBars = kSOffARec + 2 * 64;
constexpr size_t kShrinkSmem = kSOffBars + 64 * 8 + 1024;  // + alignment slack

struct ShrinkArgs {
  CUtensorMap xmap;  // x as [T rows, d_in columns], 64 x 64 boxes, 128-byte swizzle
  const uint16_t* x;
  long long ldx;
  float* h;
  long long ldh;
  int h_by_token;  // h rows by token (caller's h) or by segment position (scratch)
  int use_tma;
  // Launched right after this call's gather kernel, which waited for every earlier
  // grid before releasing this one and writes only y / h rows of short segments
  // and its own counter: nothing to wait for.
  int after_gather;
  float* part;  // [ksplit][T][LORA_MAX_RANK] partial sums by segment position
  int32_t* counter;  // work counter (zero between calls)
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* err;
  int T;
  int ksplit;  // slices of d_in per tile
  int klen;    // columns per slice (a multiple of 64)
};

__device__ __forceinline__ void named_sync_load() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kSThreads, 1) shrink_tc_kernel(const __grid_constant__ ShrinkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto slot_at = [&](int q) { return sm + kSOffQ + (size_t)q * kSSlotBytes; };
  auto srec_at = [&](uint32_t s) { return reinterpret_cast<SRec*>(sm + kSOffRec + (size_t)s * 64); };
  auto arec_at = [&](uint32_t b) { return reinterpret_cast<ARec*>(sm + kSOffARec + (size_t)b * 64); };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSOffBars);
  uint64_t* full_tma = bars;                // [stages] lead loader (+ TMA bytes)
  uint64_t* full_cp = bars + kSStages;      // [stages] 128 loader threads' copies landed
  uint64_t* empty = bars + 2 * kSStages;    // [stages] MMA done with the stage
  uint64_t* uq_full = bars + 3 * kSStages;  // [4] 32 scheduler lanes
  uint64_t* uq_empty = uq_full + 4;         // [4] 4 loader warps
  uint64_t* acc_full = uq_empty + 4;        // [2] MMAs of the unit done
  uint64_t* acc_empty = acc_full + 2;       // [2] 4 epilogue warps done
  uint64_t* rec_full = acc_empty + 2;       // [2] unit record written
  uint64_t* mma_done = rec_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  if (tid == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(smem_u32(&full_tma[s]), 1);
      mbar_init(smem_u32(&full_cp[s]), 32 * kSLoad);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(smem_u32(&uq_full[q]), 32);
      mbar_init(smem_u32(&uq_empty[q]), kSLoad);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
      mbar_init(smem_u32(&rec_full[b]), 1);
    }
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == kSWarpMma) tmem_alloc(smem_u32(tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_enter(a.after_gather != 0);

  const int ks = a.ksplit;
  bool ok = true;

  if (warp < kSSched) {
    // ---------------- schedulers ----------------
    const int sid = warp;
    const int n_work = a.meta[3] * ks;
    const int shift = v.page_shift;
    // Claims: unit sid * grid + block first, then units 2 * grid + counter.  Every
    // scheduler over-claims the counter exactly once; the last claim of all
    // puts it back to zero for the next call.  A scheduler claims its next unit
    // only once the loaders are done with its previous one (they meanwhile
    // load the other scheduler's unit), so when the units run out no CTA holds
    // more than one in reserve.
    const int g2 = kSSched * (int)gridDim.x;
    const int n_dyn = max(0, n_work - g2);
    int u = sid * (int)gridDim.x + (int)blockIdx.x;
    int claim = 0;      // lane 0: the counter's last answer
    bool over = false;  // lane 0: this scheduler's over-claim is made
    auto advance = [&]() {
      int c = 0;
      if (lane == 0) {
        claim = atomicAdd(a.counter, 1);
        c = claim;
        over = c >= n_dyn;
      }
      c = __shfl_sync(0xffffffffu, c, 0);
      u = c < n_dyn ? g2 + c : n_work;
    };
    for (uint32_t k = 0;;) {
      const bool end = u >= n_work;
      if (end && lane == 0) {
        if (!over) claim = atomicAdd(a.counter, 1);  // the first unit was already past the end
        if (claim == n_dyn + g2 - 1) *a.counter = 0;
      }
      TileInfo ti{};
      lora_adapter_desc_t d{};
      int tile = 0, q = 0;
      if (!end) {
        tile = u / ks;
        q = u - tile * ks;
        ti = load_tile(a.long_units, a.seg_adapter, a.indptr, a.perm, tile, a.use_tma);
        d = adapter_desc(v, ti.ad);
        const int bad = check_adapter_warp(v, ti.ad, d, lane);
        if (bad) {
          if (lane == 0 && q == 0) report(a.err, bad);
          advance();
          continue;
        }
      }
      const int qs = sid + 2 * (k & 1);
      if (k >= 2 && !mbar_wait(smem_u32(&uq_empty[qs]), ((k >> 1) - 1) & 1)) ok = false;
      uint8_t* slot = slot_at(qs);
      SUnit* su = reinterpret_cast<SUnit*>(slot);
      if (end) {
        if (lane == 0) su->flags = kRecEnd;
      } else {
        const int r = d.rank;
        const int kbeg = q * a.klen, nch = (min(v.d_in, kbeg + a.klen) - kbeg) / 64;
        if (lane == 0) {
          su->tile = tile;
          su->q = q;
          su->r = r;
          su->rpad = (r + 15) & ~15;
          su->nch = nch;
          su->kbeg = kbeg;
          su->p0 = ti.p0;
          su->cnt = ti.cnt;
          su->row0 = ti.row0;
          su->flags = ti.tma ? kRecTma : 0;
        }
        int* rows = reinterpret_cast<int*>(slot + 64);  // x row of each tile row, -1 past the tile
        int rv[kTM / 32];  // every lane's loads in flight before the stores
#pragma unroll
        for (int i = 0; i < kTM / 32; ++i) {
          const int m = lane + 32 * i;
          rv[i] = m >= ti.cnt ? -1 : ti.tma ? ti.row0 + m : a.perm[ti.p0 + m];
        }
#pragma unroll
        for (int i = 0; i < kTM / 32; ++i) rows[lane + 32 * i] = rv[i];
        int* pg = reinterpret_cast<int*>(slot + 64 + kTM * 4);  // [64][kSMaxChunks]
        for (int i0 = 0; i0 < r * nch; i0 += 32 * 8) {  // eight page-list reads in flight per lane
          int pv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = i0 + 32 * k + lane, jr = i / nch, c = i - jr * nch;
            const long long e = (long long)jr * v.d_in + kbeg + 64 * c;
            pv[k] = i < r * nch ? v.page_list[d.a_page0 + (e >> shift)] : 0;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = i0 + 32 * k + lane, jr = i / nch, c = i - jr * nch;
            if (i < r * nch) pg[jr * kSMaxChunks + c] = pv[k];
          }
        }
      }
      mbar_arrive(smem_u32(&uq_full[qs]));  // each lane after its own writes
      ++k;
      if (end) break;
      if (!mbar_wait(smem_u32(&uq_empty[qs]), ((k - 1) >> 1) & 1)) ok = false;  // the loaders are done with it
      advance();
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp < kSWarpMma) {
    // ---------------- loaders ----------------
    const int lw = warp - kSWarpLoad0;  // 0 leads: records, stage barrier, TMA
    const bool lead = lw == 0 && lane == 0;
    const int shift = v.page_shift;
    const long long pmask = (1LL << shift) - 1;
    if (lead && a.use_tma) prefetch_tensormap(&a.xmap);
    uint32_t g = 0, n0 = 0, n1 = 0;  // stages used; units read from each scheduler
    bool done0 = false, done1 = false;
    auto take_stage = [&]() -> uint32_t {
      const uint32_t st = g % kSStages;
      if (g >= kSStages && !mbar_wait(smem_u32(&empty[st]), ((g / kSStages) - 1) & 1)) ok = false;
      return st;
    };
    for (int s = 0; !(done0 && done1); s ^= 1) {
      if (s ? done1 : done0) continue;
      const uint32_t ns = s ? n1 : n0;
      const int qs = s + 2 * (ns & 1);
      if (!mbar_wait(smem_u32(&uq_full[qs]), (ns >> 1) & 1)) ok = false;
      if (s) ++n1; else ++n0;
      const uint8_t* slot = slot_at(qs);
      const SUnit su = *reinterpret_cast<const SUnit*>(slot);
      if (su.flags & kRecEnd) {
        if (s) done1 = true; else done0 = true;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&uq_empty[qs]));
        continue;
      }
      const bool tma = su.flags & kRecTma;
      const int* rows = reinterpret_cast<const int*>(slot + 64);
      const int* pg = reinterpret_cast<const int*>(slot + 64 + kTM * 4);
      // x rows of this thread: m = base + (lane >> 3) + 4 t, 16-byte piece lane & 7
      const int p = lane & 7;
      constexpr int kXPer = (kTM - kSTmaRows) / kSLoad;  // cp.async x rows per loader warp, TMA tiles
      const int xbase = tma ? kSTmaRows + kXPer * lw : 32 * lw;
      const int xcnt = tma ? kXPer / 4 : 8;
      const uint16_t* xsrc[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int rw = t < xcnt ? rows[xbase + (lane >> 3) + 4 * t] : -1;
        xsrc[t] = rw < 0 ? nullptr : a.x + (long long)rw * a.ldx + su.kbeg + 8 * p;
      }
      for (int c = 0; c < su.nch; ++c, ++g) {
        const uint32_t st = take_stage();
        const uint32_t xs = smem_u32(sm + st * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
        const int kcol = su.kbeg + 64 * c;
        if (lead) {
          SRec* rc = srec_at(st);
          rc->tile = su.tile;
          rc->q = su.q;
          rc->r = su.r;
          rc->rpad = su.rpad;
          rc->c = c;
          rc->nch = su.nch;
          rc->p0 = su.p0;
          rc->cnt = su.cnt;
          rc->flags = 0;
          if (tma) {
            mbar_arrive_expect_tx(smem_u32(&full_tma[st]), kSTmaRows * 128);
            tma_load_2d(xs, &a.xmap, kcol, su.row0, smem_u32(&full_tma[st]));
          } else {
            mbar_arrive(smem_u32(&full_tma[st]));
          }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < xcnt) {
            const int m = xbase + (lane >> 3) + 4 * t;
            cp_async16(xs + sw128_offset(m, p), xsrc[t] ? xsrc[t] + 64 * c : a.x, xsrc[t] != nullptr);
          }
        }
        // adapter rows j = 4 ((lane >> 3) + 4 t) + lw, piece lane & 7
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int jr = 4 * ((lane >> 3) + 4 * t) + lw;
          if (jr < su.rpad) {
            const bool real = jr < su.r;
            const long long e = real ? ((long long)jr * v.d_in + kcol) : 0;
            const uint16_t* src =
                real ? v.pool + ((long long)pg[jr * kSMaxChunks + c] << shift) + (e & pmask) + 8 * p : v.pool;
            cp_async16(as + sw128_offset(jr, p), src, real);
          }
        }
        cp_async_arrive_noinc(smem_u32(&full_cp[st]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&uq_empty[qs]));
    }
    {  // the end, for the MMA warp: a record with no data on the next stage
      const uint32_t st = take_stage();  // every loader thread, so no arrival runs ahead of the stage
      if (lead) {
        srec_at(st)->flags = kRecEnd;
        mbar_arrive(smem_u32(&full_tma[st]));
      }
      mbar_arrive(smem_u32(&full_cp[st]));
      ++g;
    }
    // nothing may still be landing in shared memory when the CTA ends
    cp_async_commit();
    cp_async_wait<0>();
    if (lead) {
      drain_ring(full_tma, g, kSStages);
      drain_ring(full_cp, g, kSStages);
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp == kSWarpMma) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      uint32_t nunit = 0;
      for (uint32_t g = 0;; ++g) {
        const uint32_t st = g % kSStages, ph = (g / kSStages) & 1;
        if (!mbar_wait(smem_u32(&full_tma[st]), ph) || !mbar_wait(smem_u32(&full_cp[st]), ph)) {
          ok = false;
          break;
        }
        const SRec rc = *srec_at(st);
        if (rc.flags & kRecEnd) break;
        const uint32_t b = nunit & 1, k = nunit >> 1;
        if (rc.c == 0) {
          if (k >= 1 && !mbar_wait(smem_u32(&acc_empty[b]), (k - 1) & 1)) ok = false;
          ARec* ar = arec_at(b);
          ar->tile = rc.tile;
          ar->q = rc.q;
          ar->r = rc.r;
          ar->rpad = rc.rpad;
          ar->p0 = rc.p0;
          ar->cnt = rc.cnt;
          ar->flags = 0;
          mbar_arrive(smem_u32(&rec_full[b]));
        }
        fence_proxy_async_smem();  // asynchronous-copy writes, seen here, before the tensor cores read them
        tc_fence_after();
        const uint32_t xs = smem_u32(sm + st * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
        const uint32_t idesc = idesc_bf16(kTM, rc.rpad, 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem + b * 64, sdesc_sw128(xs + 32 * kk, 16, 1024), sdesc_sw128(as + 32 * kk, 16, 1024), idesc,
                   (rc.c | kk) != 0);
        mma_commit(smem_u32(&empty[st]));
        if (rc.c == rc.nch - 1) {
          mma_commit(smem_u32(&acc_full[b]));
          ++nunit;
        }
      }
      // the end, passed on through the next accumulator record
      const uint32_t b = nunit & 1, k = nunit >> 1;
      if (k >= 1 && !mbar_wait(smem_u32(&acc_empty[b]), (k - 1) & 1)) ok = false;
      arec_at(b)->flags = kRecEnd;
      mbar_arrive(smem_u32(&rec_full[b]));
      if (nunit > 0) {  // every MMA of this CTA has completed before tensor memory is freed
        mma_commit(smem_u32(mma_done));
        mbar_wait(smem_u32(mma_done), 0);
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: h, or this slice's partial H ----------------
    const int quarter = warp & 3;  // tensor-memory lanes this warp may read
    const int m = quarter * 32 + lane;
    for (uint32_t nunit = 0;; ++nunit) {
      const uint32_t b = nunit & 1, k = nunit >> 1;
      if (!mbar_wait(smem_u32(&rec_full[b]), k & 1)) {
        ok = false;
        break;
      }
      const ARec ar = *arec_at(b);
      if (ar.flags & kRecEnd) break;
      if (!mbar_wait(smem_u32(&acc_full[b]), k & 1)) ok = false;
      tc_fence_after();
      const int r = ar.r, rpad = ar.rpad;
      const bool mine = m < ar.cnt;
      float* dst = ks == 1 ? a.h + (long long)(a.h_by_token ? (mine ? a.perm[ar.p0 + m] : 0) : ar.p0 + m) * a.ldh
                           : a.part + ((long long)ar.q * a.T + ar.p0 + m) * LORA_MAX_RANK;
      for (int c0 = 0; c0 < rpad; c0 += 16) {
        float vals[16];
        tmem_ld16(tmem + b * 64 + ((uint32_t)(quarter * 32) << 16) + c0, vals);
        if (mine) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            if (ks == 1)
              store_h4(dst, c0 + i, r, vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
            else
              *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));  // accumulator and record both free
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kSWarpMma) tmem_dealloc(tmem, 128);
  pdl_exit(a.after_gather != 0);
}

// ---------------------------------------------------------------- expand_tc --
//
// Warp roles: 0 schedules (claims groups of kEGroup consecutive units, resolves
// tile, adapter and B pages), 1-4 load, 5 issues MMAs, 6-13 epilogue, 14
// builds each new tile's H operand, s_i h as bf16 hi + lo, into one of two
// buffers, a tile ahead of the MMAs.  Units pass from the scheduler to the loaders through a 4-slot
// queue; the loaders' 3-stage ring carries a record of each unit to the MMA
// warp and the epilogue.  A unit's y0 comes by two TMA tensor copies when the
// tile is 128 consecutive tokens (the y stores and the B rows keep the load /
// store units busy meanwhile), by the loader warps' 16-byte asynchronous copies
// otherwise.

constexpr int kEThreads = 480;
constexpr int kEWarpH = 14;
constexpr int kELoad = 4;
constexpr int kEWarpLoad0 = 1, kEWarpMma = 5, kEWarpEpi0 = 6;
constexpr int kEEpiWarps = 8;  // (tensor-memory lane quarter, 64-column half) each
constexpr int kENC = 128;      // output columns per unit
constexpr int kEGroup = 4;     // units per claim
constexpr int kEStages = 3;
constexpr int kEQ = 4;                    // unit queue slots
constexpr int kEYBytes = kTM * kENC * 2;  // y0 / y tile: 2 atoms of 128 rows x 64 columns
constexpr int kEAtom = kTM * 128;         // one 128 x 64 bf16 atom column
constexpr int kEBBytes = 64 * kENC * 2;   // B tile: up to 64 rank rows x 128 columns
constexpr int kEStageBytes = kEYBytes + kEBBytes;
constexpr int kEHBytes = 2 * kTM * 128;  // one H operand: hi then lo

struct EUnit {  // scheduler -> loaders -> MMA warp and epilogue
  int tile, n0, r, rpad, p0, cnt, row0, flags, hbuf;
};
constexpr int kERecBytes = 64 + kTM * 4;          // record, y row of each tile row
constexpr int kESlotBytes = kERecBytes + 64 * 4;  // record, rows, B pages
constexpr size_t kEOffH = (size_t)kEStages * kEStageBytes;
constexpr size_t kEOffQ = kEOffH + 2 * (size_t)kEHBytes;
constexpr size_t kEOffRec = kEOffQ + (size_t)kEQ * kESlotBytes;
struct HReq {  // scheduler -> H builder, one per tile
  int p0, cnt, r, flags;
  float scale;
};
constexpr size_t kEOffHq = kEOffRec + (size_t)kEStages * kERecBytes;  // 2 requests: record, h rows
constexpr size_t kEOffBars = kEOffHq + 2 * (size_t)kERecBytes;
constexpr size_t kExpandSmem = kEOffBars + 64 * 8 + 1024;

struct ExpandArgs {
  CUtensorMap ymap;  // y as [T rows, d_out columns], 128 x 64 boxes, 128-byte swizzle
  uint16_t* y;
  long long ldy;
  float* yf;  // non-null: fp32 output rows (y is then read only, for y0)
  long long ldyf;
  const float* h;
  long long ldh;
  int h_by_token;
  int use_tma;
  int after_gather;  // expand-only call, launched right after its gather kernel: no wait
  int32_t* counter;  // work counter (zero between calls)
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* err;
};

__global__ void __launch_bounds__(kEThreads, 1) expand_tc_kernel(const __grid_constant__ ExpandArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto hbuf_at = [&](int hb) { return sm + kEOffH + (size_t)hb * kEHBytes; };
  auto slot_at = [&](uint32_t q) { return sm + kEOffQ + (size_t)q * kESlotBytes; };
  auto rec_at = [&](uint32_t st) { return sm + kEOffRec + (size_t)st * kERecBytes; };
  auto hq_at = [&](uint32_t q) { return sm + kEOffHq + (size_t)q * kERecBytes; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kEOffBars);
  uint64_t* full_tma = bars;                // [stages] lead loader (+ TMA bytes of y0)
  uint64_t* full_cp = bars + kEStages;      // [stages] 128 loader threads' copies landed
  uint64_t* empty = bars + 2 * kEStages;    // [stages] MMA commit + 8 epilogue warps
  uint64_t* uq_full = bars + 3 * kEStages;  // [kEQ] 32 scheduler lanes
  uint64_t* uq_empty = uq_full + kEQ;       // [kEQ] 4 loader warps
  uint64_t* acc_full = uq_empty + kEQ;      // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2] 8 epilogue warps
  uint64_t* h_ready = acc_empty + 2;        // [2] 32 scheduler lanes
  uint64_t* h_free = h_ready + 2;           // [2] MMA commit when it leaves the buffer's tile
  uint64_t* hq_full = h_free + 2;           // [2] 32 scheduler lanes
  uint64_t* hq_empty = hq_full + 2;         // [2] H builder
  uint64_t* mma_done = hq_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  if (tid == 0) {
    for (int s = 0; s < kEStages; ++s) {
      mbar_init(smem_u32(&full_tma[s]), 1);
      mbar_init(smem_u32(&full_cp[s]), 32 * kELoad);
      mbar_init(smem_u32(&empty[s]), 1 + kEEpiWarps);
    }
    for (int q = 0; q < kEQ; ++q) {
      mbar_init(smem_u32(&uq_full[q]), 32);
      mbar_init(smem_u32(&uq_empty[q]), kELoad);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kEEpiWarps);
      mbar_init(smem_u32(&h_ready[b]), 32);
      mbar_init(smem_u32(&h_free[b]), 1);
      mbar_init(smem_u32(&hq_full[b]), 32);
      mbar_init(smem_u32(&hq_empty[b]), 1);
    }
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == kEWarpMma) tmem_alloc(smem_u32(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_enter(a.after_gather != 0);
  bool ok = true;

  if (warp == 0) {
    // ---------------- scheduler ----------------
    const int n_nc = v.d_out / kENC;
    const int n_work = a.meta[3] * n_nc;
    const int n_claims = (n_work + kEGroup - 1) / kEGroup;
    const int shift = v.page_shift;
    uint32_t j = 0, tcount = 0;
    int cur = -1, bad = 0;
    TileInfo ti{};
    lora_adapter_desc_t d{};
    int rows[4] = {-1, -1, -1, -1};
    bool new_tile = false;
    auto take_slot = [&]() -> uint8_t* {
      const uint32_t qs = j % kEQ;
      if (j >= kEQ && !mbar_wait(smem_u32(&uq_empty[qs]), ((j / kEQ) - 1) & 1)) ok = false;
      return slot_at(qs);
    };
    // Claims: group blockIdx.x first, then groups grid + counter.  The scheduler
    // over-claims the counter exactly once; the last claim of all puts it back
    // to zero for the next call.  The next group is claimed once the loaders
    // are done with all but the last two units of this one, so that when the
    // groups run out no CTA holds much more than the group it is on.
    const int n_dyn = max(0, n_claims - (int)gridDim.x);
    int c = blockIdx.x;
    int claim = 0;      // lane 0: the counter's last answer
    bool over = false;  // lane 0: the over-claim is made
    for (;;) {
      if (c >= n_claims) {
        if (lane == 0) {
          if (!over) claim = atomicAdd(a.counter, 1);  // the first group was already past the end
          if (claim == n_dyn + (int)gridDim.x - 1) *a.counter = 0;
        }
        uint8_t* slot = take_slot();
        if (lane == 0) reinterpret_cast<EUnit*>(slot)->flags = kRecEnd;
        mbar_arrive(smem_u32(&uq_full[j % kEQ]));
        ++j;
        const int hq = tcount & 1;  // and the H builder's end
        if (tcount >= 2 && !mbar_wait(smem_u32(&hq_empty[hq]), ((tcount >> 1) - 1) & 1)) ok = false;
        if (lane == 0) reinterpret_cast<HReq*>(hq_at(hq))->flags = kRecEnd;
        mbar_arrive(smem_u32(&hq_full[hq]));
        break;
      }
      for (int w = c * kEGroup; w < min(n_work, (c + 1) * kEGroup); ++w) {
        const int tile = w / n_nc, n0 = (w - tile * n_nc) * kENC;
        if (tile != cur) {
          cur = tile;
          ti = load_tile(a.long_units, a.seg_adapter, a.indptr, a.perm, tile, a.use_tma);
          d = adapter_desc(v, ti.ad);
          bad = check_adapter_warp(v, ti.ad, d, lane);
          if (bad && lane == 0 && n0 == 0) report(a.err, bad);
          if (!bad) {
            new_tile = true;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int m = lane + 32 * i;
              rows[i] = m >= ti.cnt ? -1 : ti.tma ? ti.row0 + m : a.perm[ti.p0 + m];
            }
            // the tile's H operand, built by the H warp into buffer tcount & 1
            const int hq = tcount & 1;
            if (tcount >= 2 && !mbar_wait(smem_u32(&hq_empty[hq]), ((tcount >> 1) - 1) & 1)) ok = false;
            uint8_t* req = hq_at(hq);
            if (lane == 0) {
              HReq* hr = reinterpret_cast<HReq*>(req);
              hr->p0 = ti.p0;
              hr->cnt = ti.cnt;
              hr->r = d.rank;
              hr->flags = 0;
              hr->scale = d.scale;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) reinterpret_cast<int*>(req + 64)[lane + 32 * i] = rows[i];
            mbar_arrive(smem_u32(&hq_full[hq]));  // each lane after its own writes
            ++tcount;
          }
        }
        if (bad) continue;
        uint8_t* slot = take_slot();
        if (lane == 0) {
          EUnit* eu = reinterpret_cast<EUnit*>(slot);
          eu->tile = tile;
          eu->n0 = n0;
          eu->r = d.rank;
          eu->rpad = (d.rank + 15) & ~15;
          eu->p0 = ti.p0;
          eu->cnt = ti.cnt;
          eu->row0 = ti.row0;
          eu->flags = (ti.tma ? kRecTma : 0) | (new_tile ? kRecNewTile : 0);
          eu->hbuf = (tcount - 1) & 1;
        }
        new_tile = false;
        int* srows = reinterpret_cast<int*>(slot + 64);
#pragma unroll
        for (int i = 0; i < 4; ++i) srows[lane + 32 * i] = rows[i];
        int* pgb = reinterpret_cast<int*>(slot + kERecBytes);
        int pv[LORA_MAX_RANK / 32];  // both reads in flight before the stores
#pragma unroll
        for (int i = 0; i < LORA_MAX_RANK / 32; ++i) {
          const int jr = lane + 32 * i;
          pv[i] = jr < d.rank ? v.page_list[d.b_page0 + (((long long)jr * v.d_out + n0) >> shift)] : 0;
        }
#pragma unroll
        for (int i = 0; i < LORA_MAX_RANK / 32; ++i)
          if (lane + 32 * i < d.rank) pgb[lane + 32 * i] = pv[i];
        mbar_arrive(smem_u32(&uq_full[j % kEQ]));  // each lane after its own writes
        ++j;
      }
      if (j >= 2) {
        const uint32_t jd = j - 2;
        if (!mbar_wait(smem_u32(&uq_empty[jd % kEQ]), (jd / kEQ) & 1)) ok = false;
      }
      int cn = 0;
      if (lane == 0) {
        claim = atomicAdd(a.counter, 1);
        cn = claim;
        over = cn >= n_dyn;
      }
      cn = __shfl_sync(0xffffffffu, cn, 0);
      c = cn < n_dyn ? (int)gridDim.x + cn : n_claims;
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp < kEWarpMma) {
    // ---------------- loaders ----------------
    const int lw = warp - kEWarpLoad0;  // 0 leads: record, stage barrier, TMA
    const bool lead = lw == 0 && lane == 0;
    const int ltid = tid - 32 * kEWarpLoad0;
    const int shift = v.page_shift;
    const long long pmask = (1LL << shift) - 1;
    if (lead && a.use_tma) prefetch_tensormap(&a.ymap);
    uint32_t g = 0;
    const int p = lane & 7;
    for (uint32_t j = 0;; ++j, ++g) {
      const uint32_t qs = j % kEQ;
      if (!mbar_wait(smem_u32(&uq_full[qs]), (j / kEQ) & 1)) ok = false;
      const uint8_t* slot = slot_at(qs);
      const EUnit eu = *reinterpret_cast<const EUnit*>(slot);
      const uint32_t st = g % kEStages;
      if (g >= kEStages && !mbar_wait(smem_u32(&empty[st]), ((g / kEStages) - 1) & 1)) ok = false;
      uint8_t* rec = rec_at(st);
      // the unit's record and y rows travel with the stage
      if (lead) *reinterpret_cast<EUnit*>(rec) = eu;
      const int* srows = reinterpret_cast<const int*>(slot + 64);
      reinterpret_cast<int*>(rec + 64)[ltid] = srows[ltid];
      named_sync_load();  // every loader's writes before the lead's arrival publishes them
      const bool tma = eu.flags & kRecTma;
      if (lead) {
        if (tma && !(eu.flags & kRecEnd)) {
          mbar_arrive_expect_tx(smem_u32(&full_tma[st]), kEYBytes);
          tma_load_2d(smem_u32(sm + st * kEStageBytes), &a.ymap, eu.n0, eu.row0, smem_u32(&full_tma[st]));
          tma_load_2d(smem_u32(sm + st * kEStageBytes) + kEAtom, &a.ymap, eu.n0 + 64, eu.row0,
                      smem_u32(&full_tma[st]));
        } else {
          mbar_arrive(smem_u32(&full_tma[st]));
        }
      }
      if (eu.flags & kRecEnd) {
        mbar_arrive(smem_u32(&full_cp[st]));
        ++g;
        break;
      }
      const uint32_t ys = smem_u32(sm + st * kEStageBytes);
      const uint32_t bs = ys + kEYBytes;
      // y0 rows of other tiles: m = 32 lw + (lane >> 3) + 4 t, piece lane & 7 of each 64-column atom
      if (!tma) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int m = 32 * lw + (lane >> 3) + 4 * t;
          const int rw = srows[m];
          if (rw < 0) continue;
          const uint16_t* src = a.y + (long long)rw * a.ldy + eu.n0 + 8 * p;
          cp_async16(ys + sw128_offset(m, p), src);
          cp_async16(ys + kEAtom + sw128_offset(m, p), src + 64);
        }
      }
      // B rows j = 4 ((lane >> 4) + 2 t) + lw: MN-major operand, 2 atoms of 64
      // columns, 8 rank rows per 1024-byte group, 128-byte swizzle; zero beyond r
      const int* pgb = reinterpret_cast<const int*>(slot + kERecBytes);
      const int kg = eu.rpad / 8, p16 = lane & 15;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int jr = 4 * ((lane >> 4) + 2 * t) + lw;
        if (jr < eu.rpad) {
          const bool real = jr < eu.r;
          const long long e = real ? ((long long)jr * v.d_out + eu.n0) : 0;
          const uint16_t* src = real ? v.pool + ((long long)pgb[jr] << shift) + (e & pmask) + 8 * p16 : v.pool;
          cp_async16(bs + (uint32_t)((((p16 >> 3) * kg) + (jr >> 3)) * 1024) + sw128_offset(jr & 7, p16 & 7), src,
                     real);
        }
      }
      cp_async_arrive_noinc(smem_u32(&full_cp[st]));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&uq_empty[qs]));
    }
    cp_async_commit();
    cp_async_wait<0>();
    if (lead) {
      drain_ring(full_tma, g, kEStages);
      drain_ring(full_cp, g, kEStages);
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp == kEWarpMma) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      uint32_t uc = 0, tcount = 0;
      int hb = 0;
      for (uint32_t g = 0;; ++g) {
        const uint32_t st = g % kEStages, ph = (g / kEStages) & 1;
        if (!mbar_wait(smem_u32(&full_tma[st]), ph) || !mbar_wait(smem_u32(&full_cp[st]), ph)) {
          ok = false;
          break;
        }
        const EUnit rc = *reinterpret_cast<const EUnit*>(rec_at(st));
        if (rc.flags & kRecEnd) break;
        const uint32_t b = uc & 1, k = uc >> 1;
        if (rc.flags & kRecNewTile) {
          if (tcount > 0) mma_commit(smem_u32(&h_free[hb]));  // the previous tile's H is free once its MMAs end
          hb = rc.hbuf;
          if (!mbar_wait(smem_u32(&h_ready[hb]), (tcount >> 1) & 1)) ok = false;
          ++tcount;
        }
        if (k >= 1 && !mbar_wait(smem_u32(&acc_empty[b]), (k - 1) & 1)) ok = false;
        fence_proxy_async_smem();  // asynchronous-copy writes, seen here, before the tensor cores read them
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kTM, 64, 1);
        const uint32_t bs = smem_u32(sm + st * kEStageBytes) + kEYBytes;
        const uint32_t hhi = smem_u32(hbuf_at(hb)), hlo = hhi + kTM * 128;
        const int kg = rc.rpad / 8;
        for (int na = 0; na < kENC / 64; ++na) {
          int first = 1;
          for (int part = 0; part < 2; ++part) {
            const uint32_t abase = part ? hlo : hhi;
            for (int kk = 0; kk < rc.rpad / 16; ++kk) {
              mma_bf16(tmem + b * 128 + (uint32_t)(na * 64), sdesc_sw128(abase + 32 * kk, 16, 1024),
                       sdesc_sw128(bs + (uint32_t)((na * kg) * 1024 + kk * 2048), 0, 1024), idesc, first ? 0u : 1u);
              first = 0;
            }
          }
        }
        mma_commit(smem_u32(&acc_full[b]));
        mma_commit(smem_u32(&empty[st]));
        ++uc;
      }
      if (uc > 0) {
        mma_commit(smem_u32(mma_done));
        mbar_wait(smem_u32(mma_done), 0);
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kEWarpH) {
    // ---------------- H builder ----------------
    // Tile t's H into buffer t & 1 once the MMA warp has left tile t - 2: s * h
    // in two bf16 parts, K-major, 128-byte swizzle, one atom; zero beyond r
    // and beyond the tile's rows.  Lane l builds rows l + 32 i; every load of
    // a batch of eight 8-column chunks is in flight before the batch's stores.
    for (uint32_t t = 0;; ++t) {
      const int hq = t & 1;
      if (!mbar_wait(smem_u32(&hq_full[hq]), (t >> 1) & 1)) {
        ok = false;
        break;
      }
      const uint8_t* req = hq_at(hq);
      const HReq hr = *reinterpret_cast<const HReq*>(req);
      if (hr.flags & kRecEnd) break;
      if (t >= 2 && !mbar_wait(smem_u32(&h_free[hq]), ((t >> 1) - 1) & 1)) ok = false;
      uint8_t* hhi = hbuf_at(hq);
      uint8_t* hlo = hhi + kTM * 128;
      const int r = hr.r, nq8 = ((r + 15) & ~15) / 8, npair = 4 * nq8;
      const float* hrows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = lane + 32 * i;
        const long long row = m >= hr.cnt ? -1
                              : a.h_by_token ? (long long)reinterpret_cast<const int*>(req + 64)[m]
                                             : (long long)(hr.p0 + m);
        hrows[i] = row < 0 ? nullptr : a.h + row * a.ldh;
      }
      for (int t0 = 0; t0 < npair; t0 += 8) {
        float hv[8][8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int tp = t0 + b, i = tp / nq8, qq = tp - i * nq8;
          const float* hrow = tp >= npair ? nullptr : i == 0 ? hrows[0] : i == 1 ? hrows[1] : i == 2 ? hrows[2] : hrows[3];
#pragma unroll
          for (int e4 = 0; e4 < 2; ++e4) {
            const int jj = qq * 8 + 4 * e4;
            if (hrow != nullptr && jj + 3 < r) {
              const float4 f = *reinterpret_cast<const float4*>(hrow + jj);
              hv[b][4 * e4] = f.x;
              hv[b][4 * e4 + 1] = f.y;
              hv[b][4 * e4 + 2] = f.z;
              hv[b][4 * e4 + 3] = f.w;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) hv[b][4 * e4 + e] = (hrow != nullptr && jj + e < r) ? hrow[jj + e] : 0.f;
            }
          }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int tp = t0 + b, i = tp / nq8, qq = tp - i * nq8;
          if (tp >= npair) continue;
          const int m = lane + 32 * i;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float s0 = hr.scale * hv[b][2 * e], s1 = hr.scale * hv[b][2 * e + 1];
            hi[e] = pack_bf16x2(s0, s1);
            lo[e] = pack_bf16x2(s0 - bf_lo(hi[e]), s1 - bf_hi(hi[e]));
          }
          *reinterpret_cast<uint4*>(hhi + sw128_offset(m, qq)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(hlo + sw128_offset(m, qq)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&h_ready[hq]));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&hq_empty[hq]));
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else {
    // ---------------- epilogue: y = y0 + accumulator, per unit ----------------
    const int quarter = warp & 3;                 // tensor-memory lanes this warp may read
    const int half = (warp - kEWarpEpi0) >> 2;    // 64-column half of the unit (one swizzle atom)
    const int m = quarter * 32 + lane;            // tile row
    for (uint32_t g = 0, uc = 0;; ++g, ++uc) {
      const uint32_t st = g % kEStages, ph = (g / kEStages) & 1;
      if (!mbar_wait(smem_u32(&full_tma[st]), ph) || !mbar_wait(smem_u32(&full_cp[st]), ph)) {
        ok = false;
        break;
      }
      const uint8_t* rec = rec_at(st);
      const EUnit rc = *reinterpret_cast<const EUnit*>(rec);
      if (rc.flags & kRecEnd) break;
      const int tok_m = reinterpret_cast<const int*>(rec + 64)[m];
      const uint32_t b = uc & 1, k = uc >> 1;
      if (!mbar_wait(smem_u32(&acc_full[b]), k & 1)) ok = false;
      tc_fence_after();
      uint8_t* atom = sm + st * kEStageBytes + half * kEAtom;
      uint32_t acc[64];
      const uint32_t taddr = tmem + b * 128 + half * 64 + ((uint32_t)(quarter * 32) << 16);
      tmem_ld32_nowait(taddr, acc);
      tmem_ld32_nowait(taddr + 32, acc + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
      if (a.yf != nullptr) {  // fp32 output (diagnostic form): the same sums, not rounded to bf16
        if (ok && m < rc.cnt) {
          float* frow = a.yf + (long long)tok_m * a.ldyf + rc.n0 + half * 64;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float y0[8];
            unpack8(*reinterpret_cast<const uint4*>(atom + sw128_offset(m, cc)), y0);
            float4* o4 = reinterpret_cast<float4*>(frow + 8 * cc);
            o4[0] = make_float4(y0[0] + __uint_as_float(acc[8 * cc]), y0[1] + __uint_as_float(acc[8 * cc + 1]),
                                y0[2] + __uint_as_float(acc[8 * cc + 2]), y0[3] + __uint_as_float(acc[8 * cc + 3]));
            o4[1] = make_float4(y0[4] + __uint_as_float(acc[8 * cc + 4]), y0[5] + __uint_as_float(acc[8 * cc + 5]),
                                y0[6] + __uint_as_float(acc[8 * cc + 6]), y0[7] + __uint_as_float(acc[8 * cc + 7]));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
        continue;
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4* qp = reinterpret_cast<uint4*>(atom + sw128_offset(m, cc));
        float y0[8], dv[8];
        unpack8(*qp, y0);
#pragma unroll
        for (int e = 0; e < 8; ++e) dv[e] = __uint_as_float(acc[8 * cc + e]);
        uint4 o;
        o.x = pack_bf16x2(y0[0] + dv[0], y0[1] + dv[1]);
        o.y = pack_bf16x2(y0[2] + dv[2], y0[3] + dv[3]);
        o.z = pack_bf16x2(y0[4] + dv[4], y0[5] + dv[5]);
        o.w = pack_bf16x2(y0[6] + dv[6], y0[7] + dv[7]);
        *qp = o;
      }
      // 8 lanes per 128-byte row piece, four rows at a time, rows this warp wrote
      __syncwarp();
      if (ok) {
#pragma unroll
        for (int rr = 0; rr < 32; rr += 4) {
          const int sub = rr + (lane >> 3), mr = quarter * 32 + sub, pp = lane & 7;
          const int tk = __shfl_sync(0xffffffffu, tok_m, sub);
          if (mr < rc.cnt)
            *reinterpret_cast<uint4*>(a.y + (long long)tk * a.ldy + rc.n0 + half * 64 + 8 * pp) =
                *reinterpret_cast<const uint4*>(atom + sw128_offset(mr, pp));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEWarpMma) tmem_dealloc(tmem, 256);
  pdl_exit(a.after_gather != 0);
}

// ---------------------------------------------------------- reduce_partials --
//
// h of a tile split over several slices of d_in: the sum of the slices'
// partials in slice order (the order does not depend on which CTA finished
// first).  One CTA per tile at a time; (row, 4-column group) pairs spread over
// the threads, every slice's load in flight before the sums.

constexpr int kRThreads = 256;
constexpr int kRRows = 32;              // rows of a tile per work item
constexpr int kRGroups = kTM / kRRows;  // work items per tile

struct ReduceArgs {
  const float* part;
  float* h;
  long long ldh;
  int h_by_token;
  int T;
  int ks;
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
};

__global__ void __launch_bounds__(kRThreads) reduce_partials_kernel(const __grid_constant__ ReduceArgs a) {
  __shared__ int info[4];  // p0, cnt, rank, skip
  pdl_wait_then_release();
  const int n_tiles = a.meta[3];
  const int tid = threadIdx.x;
  // work item: (tile, group of kRRows rows), so a batch of few tiles still spreads
  // over many CTAs
  for (int w = blockIdx.x; w < n_tiles * kRGroups; w += gridDim.x) {
    const int tile = w / kRGroups, rg = w - tile * kRGroups;
    if (tid < 32) {
      const int s = a.long_units[2 * tile], m0 = a.long_units[2 * tile + 1];
      const int ad = a.seg_adapter[s];
      const lora_adapter_desc_t d = adapter_desc(a.v, ad);
      const int bad = check_adapter_warp(a.v, ad, d, tid);  // the tiles the shrink skipped
      if (tid == 0) {
        info[0] = a.indptr[s] + m0;
        info[1] = min(kTM, a.indptr[s + 1] - info[0]);
        info[2] = d.rank;
        info[3] = bad;
      }
    }
    __syncthreads();
    const int p0 = info[0], cnt = info[1], r = info[2], skip = info[3];
    __syncthreads();
    if (skip || rg * kRRows >= cnt) continue;
    const int rbase = rg * kRRows, nq4 = (r + 3) / 4, npairs = min(kRRows, cnt - rbase) * nq4;
    for (int i0 = tid; i0 < npairs; i0 += 2 * kRThreads) {
      float4 pv[LORA_KSPLIT_MAX][2];
      long long hrow[2];
#pragma unroll
      for (int b2 = 0; b2 < 2; ++b2) {
        const int i = i0 + kRThreads * b2;
        const int row = rbase + i / nq4, j = (i % nq4) * 4;
        hrow[b2] = i < npairs ? (a.h_by_token ? (long long)a.perm[p0 + row] : (long long)(p0 + row)) : 0;
#pragma unroll
        for (int qq = 0; qq < LORA_KSPLIT_MAX; ++qq)
          pv[qq][b2] = (qq < a.ks && i < npairs)
                           ? __ldcg(reinterpret_cast<const float4*>(
                                 a.part + ((long long)qq * a.T + p0 + row) * LORA_MAX_RANK + j))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int b2 = 0; b2 < 2; ++b2) {
        const int i = i0 + kRThreads * b2;
        if (i >= npairs) continue;
        float4 s4 = pv[0][b2];
#pragma unroll
        for (int qq = 1; qq < LORA_KSPLIT_MAX; ++qq) {
          if (qq < a.ks) {
            s4.x += pv[qq][b2].x;
            s4.y += pv[qq][b2].y;
            s4.z += pv[qq][b2].z;
            s4.w += pv[qq][b2].w;
          }
        }
        store_h4(a.h + hrow[b2] * a.ldh, (i % nq4) * 4, r, s4.x, s4.y, s4.z, s4.w);
      }
    }
  }
}

// ---------------------------------------------------------------- launchers --

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool looked = false;
  if (!looked) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    looked = true;
  }
  return fn;
}

}  // namespace

bool make_act_map(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <typename Args>
void fill_common(Args* a, const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err) {
  make_dev_view(view, &a->v);
  a->perm = seg->token_perm;
  a->indptr = seg->seg_indptr;
  a->seg_adapter = seg->seg_adapter;
  a->long_units = seg->long_units;
  a->meta = seg->meta;
  a->err = err;
}

}  // namespace

void shrink_split(int d_in, int* ks, int* klen) {
  int k = d_in / 512;
  if (k < 1) k = 1;
  if (k > kMaxKSplit) k = kMaxKSplit;
  const int len = ((d_in + k - 1) / k + 63) / 64 * 64;
  *klen = len;
  *ks = (d_in + len - 1) / len;
}

bool tc_shrink_ok(const lora_pool_view_t* v) {
  int ks, klen;
  shrink_split(v->d_in, &ks, &klen);
  return v->d_in % 64 == 0 && v->page_elems >= 128 && klen / 64 <= kSMaxChunks;
}

bool tc_expand_ok(const lora_pool_view_t* v) { return v->d_out % kENC == 0 && v->page_elems >= kENC; }

lora_status_t launch_shrink_tc(const void* x, long long ldx, float* h, long long ldh, int h_by_token, int after_gather,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  ShrinkArgs a;
  shrink_split(view->d_in, &a.ksplit, &a.klen);
  const long long upper = (long long)seg->max_long_units * a.ksplit;
  long long grid = sm_count();
  if (upper < grid) grid = upper;
  if (grid <= 0) return LORA_OK;
  a.use_tma = make_act_map(&a.xmap, x, seg->T, view->d_in, ldx, kSTmaRows) ? 1 : 0;
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.h = h;
  a.ldh = ldh;
  a.h_by_token = h_by_token;
  a.after_gather = after_gather;
  a.part = seg->k_partials;
  a.counter = seg->meta + 5;
  a.T = seg->T;
  fill_common(&a, seg, view, err);
  if (ensure_smem_attr((const void*)shrink_tc_kernel, kShrinkSmem) != cudaSuccess) return LORA_ERR_CUDA;
  if (launch_pdl((const void*)shrink_tc_kernel, dim3((unsigned)grid), dim3(kSThreads), kShrinkSmem, stream, 0, &a) !=
      cudaSuccess)
    return LORA_ERR_CUDA;
  if (a.ksplit == 1) return LORA_OK;
  ReduceArgs ra;
  ra.part = a.part;
  ra.h = h;
  ra.ldh = ldh;
  ra.h_by_token = h_by_token;
  ra.T = a.T;
  ra.ks = a.ksplit;
  ra.v = a.v;
  ra.perm = a.perm;
  ra.indptr = a.indptr;
  ra.seg_adapter = a.seg_adapter;
  ra.long_units = a.long_units;
  ra.meta = a.meta;
  long long rgrid = (long long)sm_count() * 4;
  if ((long long)seg->max_long_units * kRGroups < rgrid) rgrid = (long long)seg->max_long_units * kRGroups;
  return launch_pdl((const void*)reduce_partials_kernel, dim3((unsigned)rgrid), dim3(kRThreads), 0, stream, 0,
                    &ra) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status_t launch_expand_tc(const float* h, long long ldh, int h_by_token, int after_gather, void* y, long long ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream, float* yf, long long ldyf) {
  ExpandArgs a;
  a.yf = yf;
  a.ldyf = ldyf;
  const long long upper = (long long)seg->max_long_units * (view->d_out / kENC);
  long long grid = sm_count();
  if (upper < grid) grid = upper;
  if (grid <= 0) return LORA_OK;
  a.use_tma = make_act_map(&a.ymap, y, seg->T, view->d_out, ldy, kTM) ? 1 : 0;
  a.counter = seg->meta + 6;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.h_by_token = h_by_token;
  a.after_gather = after_gather;
  fill_common(&a, seg, view, err);
  if (ensure_smem_attr((const void*)expand_tc_kernel, kExpandSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)expand_tc_kernel, dim3((unsigned)grid), dim3(kEThreads), kExpandSmem, stream, 0,
                    &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
