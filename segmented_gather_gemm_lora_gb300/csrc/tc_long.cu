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
//             d_in).  64-column chunks of x and of A_i stream through two
//             3-stage rings in 128-byte-swizzle K-major form into tcgen05.mma
//             M = 128, N = r padded to 16.  x arrives as one TMA tensor copy
//             per chunk when the tile is 128 consecutive tokens, as 16-byte
//             asynchronous copies of the listed rows otherwise; A_i page by
//             page.  With one slice per tile the epilogue writes h directly;
//             otherwise each unit writes an fp32 partial and the unit that
//             finishes its tile last (a per-tile ticket) sums the partials in
//             slice order, so the result does not depend on timing.
//  expand_tc  Y[128, n0:n0+128] = bf16(Y0 + (s_i H) . B_i[:, n0:n0+128]).
//             A unit is (tile, 128-column chunk), so the expand, which carries
//             two thirds of the bytes, spreads over every SM.  s_i H is split
//             into bf16 hi + lo parts (two MMAs accumulating into the same fp32
//             columns), keeping the rank-r intermediate at about fp32
//             accuracy.  B_i rows are MN-major operands (r_i rows of d_out
//             contiguous elements, as stored).  y0 arrives and y leaves by TMA
//             tensor copies for tiles of 128 consecutive tokens, by 16-byte
//             pieces otherwise.
//
// Tokens of one segment are listed in increasing order (the segment builder's
// order is stable), so a tile whose first and last tokens are 127 apart is the
// consecutive rows row0 .. row0 + 127 of x and y.
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc.cuh"

namespace lora {

constexpr int kTM = LORA_TILE_M;  // 128

__device__ __forceinline__ void named_sync_epi() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier of the four epilogue warps that also ANDs `v` over their threads.
__device__ __forceinline__ bool named_and_epi(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// One long tile: rows p0 .. p0 + cnt - 1 of the segment order, all on adapter ad.
struct TileInfo {
  int ad, p0, cnt;
  int row0;  // token of the first row
  bool tma;  // 128 consecutive tokens and tensor maps available
};

__device__ __forceinline__ TileInfo load_tile(const int32_t* long_units, const int32_t* seg_adapter,
                                              const int32_t* indptr, const int32_t* perm, int tile, int use_tma) {
  TileInfo t;
  const int s = long_units[2 * tile], m0 = long_units[2 * tile + 1];
  t.ad = seg_adapter[s];
  t.p0 = indptr[s] + m0;
  t.cnt = min(kTM, indptr[s + 1] - t.p0);
  t.row0 = perm[t.p0];
  t.tma = use_tma && t.cnt == kTM && perm[t.p0 + kTM - 1] - t.row0 == kTM - 1;
  return t;
}

// Rank, every page-list slot and page of A_i and B_i, checked by one warp;
// returns 0 or LORA_DERR_* bits (the same in every lane).
__device__ __forceinline__ int check_adapter_warp(const DevView& v, const lora_adapter_desc_t& d, int lane) {
  if (d.rank < 1 || d.rank > v.max_rank || d.rank > LORA_MAX_RANK) return LORA_DERR_BAD_RANK;
  const long long na = ((long long)d.rank * v.d_in + (1LL << v.page_shift) - 1) >> v.page_shift;
  const long long nb = ((long long)d.rank * v.d_out + (1LL << v.page_shift) - 1) >> v.page_shift;
  int mine = 0;
  for (long long i = lane; i < na + nb; i += 32) {
    const long long slot = i < na ? d.a_page0 + i : d.b_page0 + (i - na);
    if (slot < 0 || slot >= v.n_page_list) {
      mine = 1;
    } else {
      const long long pg = v.page_list[slot];
      if (pg < 0 || pg >= v.n_pages) mine = 1;
    }
  }
  return __any_sync(0xffffffffu, mine) ? LORA_DERR_BAD_PAGE : 0;
}

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

constexpr int kSThreads = 224;  // warps 0-1 load (alternate units), warp 2 MMA, warps 3-6 epilogue
constexpr int kSRings = 2;      // one stage ring per loader warp
constexpr int kSStages = 3;     // stages per ring
constexpr int kSXBytes = kTM * 128;  // x tile: 128 rows x 64 bf16
constexpr int kSABytes = 64 * 128;   // A tile: up to 64 rank rows x 64 bf16
constexpr int kSStageBytes = kSXBytes + kSABytes;
constexpr int kSMaxChunks = 32;  // 64-column chunks per unit
constexpr int kRecSkip = 1, kRecEnd = 2;

// What a loader tells the MMA warp about the chunk in a stage.
struct SRec {
  int tile, q, r, rpad, c, nch, p0, cnt, flags;
};
// What the MMA warp tells the epilogue about the unit in an accumulator.
struct ARec {
  int tile, q, r, rpad, p0, cnt, flags;
};

constexpr size_t kSOffPg = (size_t)kSRings * kSStages * kSStageBytes;
constexpr size_t kSOffRec = kSOffPg + (size_t)kSRings * 64 * kSMaxChunks * 4;
constexpr size_t kSOffARec = kSOffRec + (size_t)kSRings * kSStages * 64;
constexpr size_t kSOffBars = kSOffARec + 2 * 64;
constexpr size_t kShrinkSmem = kSOffBars + 64 * 8 + 1024;  // + alignment slack

struct ShrinkArgs {
  CUtensorMap xmap;  // x as [T rows, d_in columns], 128 x 64 boxes, 128-byte swizzle
  const uint16_t* x;
  long long ldx;
  float* h;
  long long ldh;
  int h_by_token;  // h rows by token (caller's h) or by segment position (scratch)
  int use_tma;
  float* part;  // [ksplit][T][LORA_MAX_RANK] partial sums by segment position
  int32_t* tickets;
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

// Units of this CTA are w_k = blockIdx.x + k * gridDim.x, k = 0, 1, ...  Loader
// warp k % 2 stages unit k into ring k % 2, so one loader resolves its next
// unit's tile, adapter and pages while the other's unit streams.  Only the
// loaders read the segment and adapter tables: every stage carries a record of
// its chunk, and the MMA warp takes the rings in unit order (a unit's last chunk,
// or a skipped unit, hands over to the other ring) and passes each unit's
// record on to the epilogue with its accumulator.
__global__ void __launch_bounds__(kSThreads, 1) shrink_tc_kernel(const __grid_constant__ ShrinkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // stage records [ring * stages + stage] and accumulator records [2], 64-byte slots
  auto srec_at = [&](int s) { return reinterpret_cast<SRec*>(sm + kSOffRec + (size_t)s * 64); };
  auto arec_at = [&](int b) { return reinterpret_cast<ARec*>(sm + kSOffARec + (size_t)b * 64); };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSOffBars);
  uint64_t* full_tma = bars;                           // [ring][stage] 1 arrival (+ TMA bytes)
  uint64_t* full_cp = bars + kSRings * kSStages;       // [ring][stage] 32 loader lanes' copies landed
  uint64_t* empty = bars + 2 * kSRings * kSStages;     // [ring][stage] MMA done with the stage
  uint64_t* acc_full = bars + 3 * kSRings * kSStages;  // [2] MMAs of the unit done
  uint64_t* acc_empty = acc_full + 2;                  // [2] 4 epilogue warps done
  uint64_t* rec_full = acc_empty + 2;                  // [2] unit record written
  uint64_t* mma_done = rec_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  if (tid == 0) {
    for (int s = 0; s < kSRings * kSStages; ++s) {
      mbar_init(smem_u32(&full_tma[s]), 1);
      mbar_init(smem_u32(&full_cp[s]), 32);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
      mbar_init(smem_u32(&rec_full[b]), 1);
    }
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(smem_u32(tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_then_release();

  const int ks = a.ksplit;
  bool ok = true;

  if (warp < kSRings) {
    // ---------------- loaders ----------------
    const int ring = warp;
    const int n_work = a.meta[3] * ks;
    const int shift = v.page_shift;
    const long long pmask = (1LL << shift) - 1;
    uint8_t* rsm = sm + (size_t)ring * kSStages * kSStageBytes;
    int* pgtab = reinterpret_cast<int*>(sm + kSOffPg) + ring * 64 * kSMaxChunks;  // [64][kSMaxChunks]
    uint64_t* rf_tma = full_tma + ring * kSStages;
    uint64_t* rf_cp = full_cp + ring * kSStages;
    uint64_t* rempty = empty + ring * kSStages;
    if (lane == 0 && a.use_tma) prefetch_tensormap(&a.xmap);
    uint32_t g = 0;
    // next free stage of this ring (waits for the MMA warp to release it)
    auto take_stage = [&]() -> uint32_t {
      const uint32_t st = g % kSStages;
      if (g >= kSStages && !mbar_wait(smem_u32(&rempty[st]), ((g / kSStages) - 1) & 1)) ok = false;
      return st;
    };
    // a record with no data: every lane and the record's writer arrive by hand
    auto post_flag = [&](int flags) {
      const uint32_t st = take_stage();
      if (lane == 0) {
        srec_at(ring * kSStages + st)->flags = flags;
        mbar_arrive(smem_u32(&rf_tma[st]));
      }
      mbar_arrive(smem_u32(&rf_cp[st]));
      ++g;
    };
    for (int w = blockIdx.x + ring * gridDim.x; w < n_work && ok; w += kSRings * gridDim.x) {
      const int tile = w / ks, q = w - tile * ks;
      const TileInfo ti = load_tile(a.long_units, a.seg_adapter, a.indptr, a.perm, tile, a.use_tma);
      const lora_adapter_desc_t d = v.adapters[ti.ad];
      const int bad = check_adapter_warp(v, d, lane);
      if (bad) {
        if (lane == 0 && q == 0) report(a.err, bad);
        post_flag(kRecSkip);
        continue;
      }
      const int r = d.rank, rpad = (r + 15) & ~15;
      const int kbeg = q * a.klen, nch = (min(v.d_in, kbeg + a.klen) - kbeg) / 64;
      int toks[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = lane + 32 * i;
        toks[i] = (!ti.tma && m < ti.cnt) ? a.perm[ti.p0 + m] : -1;
      }
      __syncwarp();
      for (int i = lane; i < r * nch; i += 32) {
        const int j = i / nch, c = i - j * nch;
        const long long e = (long long)j * v.d_in + kbeg + 64 * c;
        pgtab[j * kSMaxChunks + c] = v.page_list[d.a_page0 + (e >> shift)];
      }
      __syncwarp();
      for (int c = 0; c < nch; ++c, ++g) {
        const uint32_t st = take_stage();
        const uint32_t xs = smem_u32(rsm + st * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
        const int kcol = kbeg + 64 * c;
        if (lane == 0) {
          SRec* rc = srec_at(ring * kSStages + st);
          rc->tile = tile;
          rc->q = q;
          rc->r = r;
          rc->rpad = rpad;
          rc->c = c;
          rc->nch = nch;
          rc->p0 = ti.p0;
          rc->cnt = ti.cnt;
          rc->flags = 0;
        }
        if (ti.tma) {
          if (lane == 0) {
            mbar_arrive_expect_tx(smem_u32(&rf_tma[st]), kSXBytes);
            tma_load_2d(xs, &a.xmap, kcol, ti.row0, smem_u32(&rf_tma[st]));
          }
        } else {
          if (lane == 0) mbar_arrive(smem_u32(&rf_tma[st]));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int m = lane + 32 * i;
            const uint16_t* src = a.x + (long long)(toks[i] < 0 ? 0 : toks[i]) * a.ldx + kcol;
#pragma unroll
            for (int p = 0; p < 8; ++p) cp_async16(xs + sw128_offset(m, p), src + 8 * p, toks[i] >= 0);
          }
        }
        for (int i = lane; i < rpad * 8; i += 32) {
          const int j = i >> 3, p = i & 7;
          const bool real = j < r;
          const long long e = real ? ((long long)j * v.d_in + kcol) : 0;
          const uint16_t* src =
              real ? v.pool + ((long long)pgtab[j * kSMaxChunks + c] << shift) + (e & pmask) + 8 * p : v.pool;
          cp_async16(as + sw128_offset(j, p), src, real);
        }
        cp_async_arrive_noinc(smem_u32(&rf_cp[st]));
      }
    }
    post_flag(kRecEnd);
    // nothing may still be landing in shared memory when the CTA ends
    cp_async_wait<0>();
    if (lane == 0) {
      drain_ring(rf_tma, g, kSStages);
      drain_ring(rf_cp, g, kSStages);
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
  } else if (warp == 2) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      uint32_t g0 = 0, g1 = 0, nunit = 0;  // stages taken per ring, units started
      int ring = 0;
      for (;;) {
        const uint32_t g = ring ? g1 : g0, st = g % kSStages, ph = (g / kSStages) & 1;
        const int s = ring * kSStages + st;
        if (!mbar_wait(smem_u32(&full_tma[s]), ph) || !mbar_wait(smem_u32(&full_cp[s]), ph)) {
          ok = false;
          break;
        }
        if (ring) ++g1; else ++g0;
        const SRec rc = *srec_at(s);
        if (rc.flags & kRecEnd) break;
        if (rc.flags & kRecSkip) {
          mbar_arrive(smem_u32(&empty[s]));
          ring ^= 1;
          continue;
        }
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
        const uint32_t xs = smem_u32(sm + (size_t)s * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
        const uint32_t idesc = idesc_bf16(kTM, rc.rpad, 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem + b * 64, sdesc_sw128(xs + 32 * kk, 16, 1024), sdesc_sw128(as + 32 * kk, 16, 1024), idesc,
                   (rc.c | kk) != 0);
        mma_commit(smem_u32(&empty[s]));
        if (rc.c == rc.nch - 1) {
          mma_commit(smem_u32(&acc_full[b]));
          ++nunit;
          ring ^= 1;
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
    // ---------------- epilogue: h or a partial H, then the tile's reduction ----------------
    const int etid = tid - 96;
    const int quarter = warp & 3;  // tensor-memory lanes this warp may read
    const int m = quarter * 32 + lane;
    for (uint32_t nunit = 0;; ++nunit) {
      const uint32_t b = nunit & 1, k = nunit >> 1;
      bool got = mbar_wait(smem_u32(&rec_full[b]), k & 1);
      if (ks > 1) got = named_and_epi(got);  // leave together: the reduction below uses barriers
      if (!got) {
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
      if (ks == 1) continue;
      __threadfence();
      ok = named_and_epi(ok);  // the same verdict in every epilogue thread before the next barrier
      if (etid == 0) *flag = atomicAdd(&a.tickets[ar.tile], 1) == ks - 1 ? 1 : 0;
      named_sync_epi();
      if (*flag) {  // the tile's last slice to finish: sum the partials in slice order
        __threadfence();
        if (mine) {
          float* hrow = a.h + (long long)(a.h_by_token ? a.perm[ar.p0 + m] : ar.p0 + m) * a.ldh;
          for (int j = 0; j < r; j += 4) {
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int qq = 0; qq < ks; ++qq) {
              const float4 p4 = __ldcg(
                  reinterpret_cast<const float4*>(a.part + ((long long)qq * a.T + ar.p0 + m) * LORA_MAX_RANK + j));
              s4.x += p4.x;
              s4.y += p4.y;
              s4.z += p4.z;
              s4.w += p4.w;
            }
            store_h4(hrow, j, r, s4.x, s4.y, s4.z, s4.w);
          }
        }
        if (etid == 0) a.tickets[ar.tile] = 0;  // ready for the next call on these segments
      }
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- expand_tc --

constexpr int kEThreads = 320;  // warp 0 loads, warp 1 MMA, warps 2-9 epilogue
constexpr int kEEpiWarps = 8;   // (tensor-memory lane quarter, 64-column half) each
constexpr int kENC = 128;       // output columns per unit
constexpr int kEStages = 4;
constexpr int kEYBytes = kTM * kENC * 2;  // y0 / y tile: 2 atoms of 128 rows x 64 columns
constexpr int kEAtom = kTM * 128;         // one 128 x 64 bf16 atom column
constexpr int kEBBytes = 64 * kENC * 2;   // B tile: up to 64 rank rows x 128 columns
constexpr int kEStageBytes = kEYBytes + kEBBytes;
constexpr int kRecTma = 4, kRecNewTile = 8;

// What the loader tells the MMA warp and the epilogue about the unit in a stage.
struct ERec {
  int tile, n0, r, rpad, p0, cnt, row0, flags;
  float scale;
};

constexpr size_t kEOffH = (size_t)kEStages * kEStageBytes;  // H hi, then lo: 2 x 16 KB
constexpr size_t kEOffPg = kEOffH + 2 * kTM * 128;
constexpr size_t kEOffRec = kEOffPg + 64 * 4;
constexpr size_t kEOffBars = kEOffRec + (size_t)kEStages * 64;
constexpr size_t kExpandSmem = kEOffBars + 32 * 8 + 1024;

struct ExpandArgs {
  CUtensorMap ymap;  // y as [T rows, d_out columns], 128 x 64 boxes, 128-byte swizzle
  uint16_t* y;
  long long ldy;
  const float* h;
  long long ldh;
  int h_by_token;
  int use_tma;
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* err;
};

// Units of this CTA are a contiguous range of (tile, column chunk), so
// consecutive units mostly share a tile and its H operand.  Only the loader
// reads the segment and adapter tables; every stage carries a record of its
// unit, and a record with the end flag closes the ring.
__global__ void __launch_bounds__(kEThreads, 1) expand_tc_kernel(const __grid_constant__ ExpandArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* hhi = sm + kEOffH;
  uint8_t* hlo = hhi + kTM * 128;
  int* pgb = reinterpret_cast<int*>(sm + kEOffPg);
  auto erec_at = [&](uint32_t st) { return reinterpret_cast<ERec*>(sm + kEOffRec + (size_t)st * 64); };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kEOffBars);
  uint64_t* full_tma = bars;                 // [stages] 1 arrival (+ TMA bytes of y0)
  uint64_t* full_cp = bars + kEStages;       // [stages] 32 loader lanes' copies landed
  uint64_t* empty = bars + 2 * kEStages;     // [stages] MMA commit + 8 epilogue warps
  uint64_t* acc_full = bars + 3 * kEStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2] 8 epilogue warps
  uint64_t* h_ready = acc_empty + 2;         // 256 epilogue threads per tile's H operand
  uint64_t* mma_done = h_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  if (tid == 0) {
    for (int s = 0; s < kEStages; ++s) {
      mbar_init(smem_u32(&full_tma[s]), 1);
      mbar_init(smem_u32(&full_cp[s]), 32);
      mbar_init(smem_u32(&empty[s]), 1 + kEEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kEEpiWarps);
    }
    mbar_init(smem_u32(h_ready), 32 * kEEpiWarps);
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_then_release();
  bool ok = true;

  if (warp == 0) {
    // ---------------- loader ----------------
    const int n_nc = v.d_out / kENC;
    const long long n_work = (long long)a.meta[3] * n_nc;
    const long long w0 = n_work * blockIdx.x / gridDim.x, w1 = n_work * (blockIdx.x + 1) / gridDim.x;
    const int shift = v.page_shift;
    const long long pmask = (1LL << shift) - 1;
    if (lane == 0 && a.use_tma) prefetch_tensormap(&a.ymap);
    uint32_t g = 0;
    int cur = -1, bad = 0, r = 0, rpad = 16;
    bool new_tile = false;
    TileInfo ti;
    lora_adapter_desc_t d;
    int toks[4];
    auto take_stage = [&]() -> uint32_t {
      const uint32_t st = g % kEStages;
      if (g >= kEStages && !mbar_wait(smem_u32(&empty[st]), ((g / kEStages) - 1) & 1)) ok = false;
      return st;
    };
    for (long long w = w0; w < w1 && ok; ++w) {
      const int tile = (int)(w / n_nc), n0 = (int)(w - (long long)tile * n_nc) * kENC;
      if (tile != cur) {
        cur = tile;
        ti = load_tile(a.long_units, a.seg_adapter, a.indptr, a.perm, tile, a.use_tma);
        d = v.adapters[ti.ad];
        bad = check_adapter_warp(v, d, lane);
        if (bad && lane == 0 && n0 == 0) report(a.err, bad);
        r = d.rank;
        rpad = (r + 15) & ~15;
        new_tile = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = lane + 32 * i;
          toks[i] = (!ti.tma && m < ti.cnt) ? a.perm[ti.p0 + m] : -1;
        }
      }
      if (bad) continue;
      __syncwarp();
      for (int j = lane; j < r; j += 32) pgb[j] = v.page_list[d.b_page0 + (((long long)j * v.d_out + n0) >> shift)];
      __syncwarp();
      const uint32_t st = take_stage();
      const uint32_t ys = smem_u32(sm + st * kEStageBytes);
      const uint32_t bs = ys + kEYBytes;
      if (lane == 0) {
        ERec* rc = erec_at(st);
        rc->tile = tile;
        rc->n0 = n0;
        rc->r = r;
        rc->rpad = rpad;
        rc->p0 = ti.p0;
        rc->cnt = ti.cnt;
        rc->row0 = ti.row0;
        rc->flags = (ti.tma ? kRecTma : 0) | (new_tile ? kRecNewTile : 0);
        rc->scale = d.scale;
      }
      new_tile = false;
      if (ti.tma) {
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&full_tma[st]), kEYBytes);
          tma_load_2d(ys, &a.ymap, n0, ti.row0, smem_u32(&full_tma[st]));
          tma_load_2d(ys + kEAtom, &a.ymap, n0 + 64, ti.row0, smem_u32(&full_tma[st]));
        }
      } else {
        if (lane == 0) mbar_arrive(smem_u32(&full_tma[st]));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (toks[i] < 0) continue;
          const int m = lane + 32 * i;
          const uint16_t* src = a.y + (long long)toks[i] * a.ldy + n0;
#pragma unroll
          for (int p = 0; p < 16; ++p) cp_async16(ys + (p >> 3) * kEAtom + sw128_offset(m, p & 7), src + 8 * p);
        }
      }
      // B rows: MN-major operand, 2 atoms of 64 columns, 8 rank rows per
      // 1024-byte group, 128-byte swizzle; zero beyond r.
      const int kg = rpad / 8;
      for (int i = lane; i < rpad * 16; i += 32) {
        const int j = i >> 4, p = i & 15;
        const bool real = j < r;
        const long long e = real ? ((long long)j * v.d_out + n0) : 0;
        const uint16_t* src = real ? v.pool + ((long long)pgb[j] << shift) + (e & pmask) + 8 * p : v.pool;
        cp_async16(bs + (uint32_t)((((p >> 3) * kg) + (j >> 3)) * 1024) + sw128_offset(j & 7, p & 7), src, real);
      }
      cp_async_arrive_noinc(smem_u32(&full_cp[st]));
      ++g;
    }
    {  // the end record
      const uint32_t st = take_stage();
      if (lane == 0) {
        erec_at(st)->flags = kRecEnd;
        mbar_arrive(smem_u32(&full_tma[st]));
      }
      mbar_arrive(smem_u32(&full_cp[st]));
      ++g;
    }
    cp_async_wait<0>();
    if (lane == 0) {
      drain_ring(full_tma, g, kEStages);
      drain_ring(full_cp, g, kEStages);
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      uint32_t g = 0, uc = 0, tc = 0;
      for (;; ++g) {
        const uint32_t st = g % kEStages, ph = (g / kEStages) & 1;
        if (!mbar_wait(smem_u32(&full_tma[st]), ph) || !mbar_wait(smem_u32(&full_cp[st]), ph)) {
          ok = false;
          break;
        }
        const ERec rc = *erec_at(st);
        if (rc.flags & kRecEnd) break;
        const uint32_t b = uc & 1, k = uc >> 1;
        if (rc.flags & kRecNewTile) {
          ++tc;
          if (!mbar_wait(smem_u32(h_ready), (tc - 1) & 1)) ok = false;
        }
        if (k >= 1 && !mbar_wait(smem_u32(&acc_empty[b]), (k - 1) & 1)) ok = false;
        fence_proxy_async_smem();  // asynchronous-copy writes, seen here, before the tensor cores read them
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kTM, 64, 1);
        const uint32_t bs = smem_u32(sm + st * kEStageBytes) + kEYBytes;
        const int kg = rc.rpad / 8;
        for (int na = 0; na < kENC / 64; ++na) {
          int first = 1;
          for (int part = 0; part < 2; ++part) {
            const uint32_t abase = smem_u32(part ? hlo : hhi);
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
  } else {
    // ---------------- epilogue: H operand per tile, y per unit ----------------
    const int quarter = warp & 3;      // tensor-memory lanes this warp may read
    const int half = (warp - 2) >> 2;  // 64-column half of the unit (one swizzle atom)
    const int m = quarter * 32 + lane;  // tile row
    int tok_m = -1;
    for (uint32_t g = 0, uc = 0;; ++g, ++uc) {
      const uint32_t st = g % kEStages, ph = (g / kEStages) & 1;
      if (!mbar_wait(smem_u32(&full_tma[st]), ph) || !mbar_wait(smem_u32(&full_cp[st]), ph)) {
        ok = false;
        break;
      }
      const ERec rc = *erec_at(st);
      if (rc.flags & kRecEnd) break;
      const bool mine = m < rc.cnt;
      if (rc.flags & kRecNewTile) {
        tok_m = !mine ? -1 : (rc.flags & kRecTma) ? rc.row0 + m : a.perm[rc.p0 + m];
        // s * h as two bf16 parts, K-major, 128-byte swizzle, one atom; zero
        // beyond r and beyond the tile's rows.  This thread builds 16-byte
        // chunks half * 4 .. half * 4 + 3 of row m.  The previous tile's MMAs
        // have completed: its last accumulator was read below.
        const float* hrow = a.h + (mine ? (a.h_by_token ? (long long)tok_m : (long long)(rc.p0 + m)) : 0) * a.ldh;
        for (int qq = half * 4; qq < min(rc.rpad / 8, half * 4 + 4); ++qq) {
          float hv[8];
#pragma unroll
          for (int e4 = 0; e4 < 2; ++e4) {
            const int j = qq * 8 + 4 * e4;
            if (mine && j + 3 < rc.r) {
              const float4 f = *reinterpret_cast<const float4*>(hrow + j);
              hv[4 * e4] = f.x;
              hv[4 * e4 + 1] = f.y;
              hv[4 * e4 + 2] = f.z;
              hv[4 * e4 + 3] = f.w;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) hv[4 * e4 + e] = (mine && j + e < rc.r) ? hrow[j + e] : 0.f;
            }
          }
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float s0 = rc.scale * hv[2 * e], s1 = rc.scale * hv[2 * e + 1];
            hi[e] = pack_bf16x2(s0, s1);
            lo[e] = pack_bf16x2(s0 - bf_lo(hi[e]), s1 - bf_hi(hi[e]));
          }
          *reinterpret_cast<uint4*>(hhi + sw128_offset(m, qq)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(hlo + sw128_offset(m, qq)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(h_ready));
      }
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
          const int sub = rr + (lane >> 3), mr = quarter * 32 + sub, p = lane & 7;
          const int tk = __shfl_sync(0xffffffffu, tok_m, sub);
          if (mr < rc.cnt)
            *reinterpret_cast<uint4*>(a.y + (long long)tk * a.ldy + rc.n0 + half * 64 + 8 * p) =
                *reinterpret_cast<const uint4*>(atom + sw128_offset(mr, p));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
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

// bf16 matrix [rows, cols] with a row stride of `ld` elements as a tensor map
// of box_rows x 64 boxes with 128-byte swizzle.  False when the driver offers
// no encoder or rejects the map; the kernels then copy every tile row by row.
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

// Slices of d_in per tile: about 512 columns each, at most LORA_KSPLIT_MAX.  A
// function of d_in alone, so a token's h does not depend on the rest of the batch.
void shrink_split(int d_in, int* ks, int* klen) {
  int k = d_in / 512;
  if (k < 1) k = 1;
  if (k > LORA_KSPLIT_MAX) k = LORA_KSPLIT_MAX;
  const int len = ((d_in + k - 1) / k + 63) / 64 * 64;
  *klen = len;
  *ks = (d_in + len - 1) / len;
}

}  // namespace

bool tc_shrink_ok(const lora_pool_view_t* v) {
  int ks, klen;
  shrink_split(v->d_in, &ks, &klen);
  return v->d_in % 64 == 0 && v->page_elems >= 128 && klen / 64 <= kSMaxChunks;
}

bool tc_expand_ok(const lora_pool_view_t* v) { return v->d_out % kENC == 0 && v->page_elems >= kENC; }

lora_status_t launch_shrink_tc(const void* x, long long ldx, float* h, long long ldh, int h_by_token,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  ShrinkArgs a;
  shrink_split(view->d_in, &a.ksplit, &a.klen);
  const long long upper = (long long)seg->max_long_units * a.ksplit;
  long long grid = sm_count();
  if (upper < grid) grid = upper;
  if (grid <= 0) return LORA_OK;
  a.use_tma = make_act_map(&a.xmap, x, seg->T, view->d_in, ldx, kTM) ? 1 : 0;
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.h = h;
  a.ldh = ldh;
  a.h_by_token = h_by_token;
  a.part = seg->k_partials;
  a.tickets = seg->tickets;
  a.T = seg->T;
  fill_common(&a, seg, view, err);
  if (ensure_smem_attr((const void*)shrink_tc_kernel, kShrinkSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)shrink_tc_kernel, dim3((unsigned)grid), dim3(kSThreads), kShrinkSmem, stream, 0,
                    &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status_t launch_expand_tc(const float* h, long long ldh, int h_by_token, void* y, long long ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  ExpandArgs a;
  const long long upper = (long long)seg->max_long_units * (view->d_out / kENC);
  long long grid = sm_count();
  if (upper < grid) grid = upper;
  if (grid <= 0) return LORA_OK;
  a.use_tma = make_act_map(&a.ymap, y, seg->T, view->d_out, ldy, kTM) ? 1 : 0;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.h_by_token = h_by_token;
  fill_common(&a, seg, view, err);
  if (ensure_smem_attr((const void*)expand_tc_kernel, kExpandSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)expand_tc_kernel, dim3((unsigned)grid), dim3(kEThreads), kExpandSmem, stream, 0,
                    &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
