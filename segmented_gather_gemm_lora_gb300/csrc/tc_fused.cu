// Fused tensor-core path for long segments: shrink, scale and expand of a
// 128-token tile in one kernel, the rank-r intermediate kept on chip.
//
// "Multi-LoRA serving: the single translator with a thousand glossaries",
// TL;DR (Y += sum_i X_i A_i B_i in a single pass) and section "SGMV: the kernel
// that holds it all up" (large segments through the tensor cores);
// "Multi-LoRA Serving in Production", section "Punica and Segmented Gather
// Matrix-Vector Multiplication (SGMV)" (a shrink stage to the rank-r
// intermediate, an expand stage that scales it and accumulates into the base
// output).
//
// Work decomposition.  A unit is one tile (up to 128 consecutive positions of
// one segment) of one projection.  A thread-block cluster of C CTAs takes a
// unit; C is the number of d_in slices the shrink splits a tile into (a
// function of d_in alone, at most four, the same slices the staged kernels of
// tc_long.cu use):
//   shrink   CTA c:  P_c[128, r] = X[128, slice c] . A_i[:, slice c]^T
//            (tcgen05.mma, M = 128, N = r padded to 16, accumulator in tensor
//            memory, 64 columns of d_in per stage);
//   exchange row m of every P_c goes to the CTA that owns row m (rows split
//            in C equal blocks) through distributed shared memory; the owner
//            sums the C partials in CTA order, scales by s_i, splits s_i h into
//            bf16 hi + lo parts and writes them into the H operand of every
//            CTA of the cluster;
//   expand   CTA c:  Y[128, slice c of d_out] = bf16(Y0 + H_hi . B_i + H_lo . B_i),
//            64 output columns per stage (M = 128, N = 64, K = r padded to 16).
// So h never leaves the chip, and x, y0 and y are each read or written once.
// The shrink-only form (the shrink stage of "Multi-LoRA Serving in
// Production", section "Punica and Segmented Gather Matrix-Vector
// Multiplication (SGMV)", alone) runs the same shrink and exchange, and the
// owner of each row also writes the row's unscaled h to global memory; no
// expand stage runs.
// Rows past a partial tile's end compute garbage that is never stored.
//
// Warp roles (10 warps).  Warp 0 resolves units (tile, adapter, page of each
// rank row's first element in this CTA's slices) into a 4-slot queue.  Warps
// 1-4 load: per stage one TMA tensor copy of the 128 x 64 activation box (x for
// the shrink, y0 for the expand) when the tile's tokens are consecutive, else
// 16-byte asynchronous copies of each token row, plus the adapter's rows of
// that stage (16-byte copies through the page table, zero past the rank).
// Warp 5 issues the MMAs.  Warps 6-13 run the epilogues in two groups of four
// (one warp per tensor-memory lane quarter): group 0 takes the shrink partial out
// of tensor memory, exchanges it and runs the owner's reduction; the two groups
// take alternate expand stages (each with its own accumulator), y = y0 +
// accumulator written back into the stage and stored by one TMA copy per warp.
#include <cudaTypedefs.h>

#include <cstring>

#include "internal.h"
#include "tc.cuh"

namespace lora {

constexpr int kFThreads = 448;
constexpr int kFEpiGroups = 2;
constexpr int kFWarpLoad0 = 1, kFLoad = 4, kFWarpMma = 5, kFWarpEpi0 = 6;
constexpr int kFLoadThreads = 32 * kFLoad;
constexpr int kFStages = 6;
constexpr int kFActBytes = kTM * 128;  // 128 rows x 64 bf16 (x or y0), 128-byte swizzle
constexpr int kFAdBytes = 64 * 128;    // up to 64 rank rows x 64 bf16 (A, K-major) or 64 columns (B, MN-major)
constexpr int kFStageBytes = kFActBytes + kFAdBytes;
constexpr int kFHBytes = 2 * kTM * 128;  // H operand: hi part, then lo part
constexpr int kFRecvBytes = kTM * LORA_MAX_RANK * 4;  // [C sources][128 / C rows][64] fp32
constexpr int kFSlots = 4;
constexpr int kFSlotBytes = 128 + kTM * 4 + 2 * LORA_MAX_RANK * 4;  // record, token rows, first pages

constexpr size_t kFOffH = (size_t)kFStages * kFStageBytes;
constexpr size_t kFOffRecv = kFOffH + kFHBytes;
constexpr size_t kFOffSlot = kFOffRecv + kFRecvBytes;
constexpr size_t kFOffBars = kFOffSlot + (size_t)kFSlots * kFSlotBytes;
constexpr int kFNBars = 2 * kFStages + 3 * kFSlots + 4 + 4 + 2 + 1 + 2 + 2;
// + tensor-memory slot, release counters, claim mailbox, alignment slack
constexpr size_t kFusedSmem = kFOffBars + kFNBars * 8 + 16 + 4 * kFStages + 16 + 1024;

constexpr int kFRecEnd = 1, kFRecTma = 2;

struct FUnit {  // scheduler -> loaders, MMA warp, epilogue
  int flags;
  int g;     // projection
  int p0;    // first position of the tile in segment order
  int cnt;   // tokens of the tile
  int row0;  // token of the first row (TMA tiles)
  int r, rpad;
  float scale;
  int k0, nk;  // this CTA's d_in slice: first column, 64-column chunks
  int n0, nn;  // this CTA's d_out slice: first column, 64-column chunks
  int a_page0, b_page0;
};
static_assert(sizeof(FUnit) <= 128, "unit record slot");

struct FProj {
  CUtensorMap xmap;    // x as [T rows, d_in columns], 64 x 128 boxes, 128-byte swizzle
  CUtensorMap ymap;    // y (y0) as [T rows, d_out columns], the same boxes
  CUtensorMap ystore;  // y as [T rows, d_out columns], 64 x 32 boxes (one epilogue warp's rows)
  const uint16_t* x;
  uint16_t* y;
  float* yf;  // non-null: fp32 output rows (y is then read only, for y0)
  float* h;   // non-null: h rows by token, unscaled, columns < r (the shrink-only form's output)
  long long ldx, ldy, ldyf, ldh;
  DevView v;
  int tma;  // every map valid
};

struct FusedArgs {
  FProj proj[kMaxFusedProj];
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* counter;  // unit claims; zero between calls (the last claim of a launch puts it back)
  int32_t* err;
  int n_proj;
  int klen;          // columns per d_in slice (a multiple of 64)
  int after_gather;  // launched right after this call's gather kernel (disjoint data): no wait at entry
  int shrink_only;   // the shrink-only form: h out, no expand
  long long probe;   // > 0: the timeout probe's wait limit in cycles (lora_debug_wait_probe)
};

__global__ void __launch_bounds__(kFThreads, 1) fused_tc_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto stage_at = [&](uint32_t st) { return sm + (size_t)st * kFStageBytes; };
  auto slot_at = [&](uint32_t q) { return sm + kFOffSlot + (size_t)q * kFSlotBytes; };
  uint8_t* hbuf = sm + kFOffH;
  float* recv = reinterpret_cast<float*>(sm + kFOffRecv);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kFOffBars);
  uint64_t* full = bars;                       // [stages] lead's expect_tx + 128 loader threads' copies
  uint64_t* empty = bars + kFStages;           // [stages] MMA commit (shrink) or the epilogue (expand)
  uint64_t* slot_full = bars + 2 * kFStages;   // [slots] 32 scheduler lanes
  uint64_t* slot_empty = slot_full + kFSlots;  // [slots] 4 loader + 1 MMA + 8 epilogue warps
  uint64_t* accs_full = slot_empty + kFSlots;  // [2] MMA commit: a unit's shrink partial
  uint64_t* accs_empty = accs_full + 2;        // [2] 4 epilogue warps
  uint64_t* acce_full = accs_empty + 2;        // [2] MMA commit: one expand stage
  uint64_t* acce_empty = acce_full + 2;        // [2] the 4 warps of epilogue group b
  uint64_t* recv_full = acce_empty + 2;        // this CTA's rows of every CTA's partial (bytes)
  uint64_t* h_full = recv_full + 1;            // the whole H operand (bytes)
  uint64_t* mma_done = h_full + 1;
  uint64_t* slot_taken = mma_done + 1;         // [slots] the loaders have read the unit's record
  uint64_t* claim_full = slot_taken + kFSlots;  // [2] CTA 0's scheduler posted a claimed unit here
  uint64_t* claim_empty = claim_full + 2;       // [2] (CTA 0 only) every CTA has read the claim
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(claim_empty + 2);
  int* rel_cnt = reinterpret_cast<int*>(tmem_slot + 4);  // [stages] epilogue warps done with an expand stage
  int* claim_val = rel_cnt + kFStages;                    // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
  const uint32_t cid = cluster_id_x(), ncl = ncluster_x();
  if (a.after_gather == 0) pdl_enter(false);  // otherwise the segments are complete already (see pdl_enter)
  if (a.meta[3] == 0) {  // no long tile: every CTA of every cluster leaves at once
    if (a.after_gather != 0) pdl_enter(true);
    pdl_exit(a.after_gather != 0);
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1 + kFLoadThreads);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int q = 0; q < kFSlots; ++q) {
      mbar_init(smem_u32(&slot_full[q]), 32);
      mbar_init(smem_u32(&slot_empty[q]), kFLoad + 1 + 4 * kFEpiGroups);
      mbar_init(smem_u32(&slot_taken[q]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&claim_full[b]), 1);
      mbar_init(smem_u32(&claim_empty[b]), ncta);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accs_full[b]), 1);
      mbar_init(smem_u32(&accs_empty[b]), 4);
      mbar_init(smem_u32(&acce_full[b]), 1);
      mbar_init(smem_u32(&acce_empty[b]), 4);
    }
    mbar_init(smem_u32(recv_full), 1);
    mbar_init(smem_u32(h_full), 1);
    mbar_init(smem_u32(mma_done), 1);
    for (int st = 0; st < kFStages; ++st) rel_cnt[st] = 0;
    fence_mbar_init();
  }
  if (warp == kFWarpMma) tmem_alloc(smem_u32(tmem_slot), 256);
  tc_fence_before();
  // every barrier of every CTA initialised (and tensor memory allocated) before
  // any peer writes into this CTA
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // shrink partials at columns 0 / 64, expand accumulators at 128 / 192
  if (a.after_gather != 0) pdl_enter(true);
  bool ok = true;
  if (a.probe > 0) {  // the timeout probe: every CTA takes the exit of a wait that ran out
    __shared__ uint64_t probe_bar;
    __shared__ int probe_ok;
    if (tid == 0) probe_ok = wait_probe(&probe_bar, a.probe) ? 1 : 0;
    __syncthreads();
    ok = probe_ok != 0;
  }
  const int R = kTM / (int)ncta;  // rows each CTA owns in the exchange

  if (warp == 0) {
    // ---------------- scheduler ----------------
    // Units: cluster cid takes unit cid first, then the units CTA 0 claims from
    // the counter (n_clusters + claim) and hands to every CTA of the cluster, so
    // clusters that start late, or draw small tiles, take more.  The next unit
    // is claimed once the loaders have taken the previous one, so that when the
    // units run out no cluster holds more than one in reserve.  Every cluster
    // over-claims the counter exactly once; the last claim of all puts it back
    // to zero for the next call.
    const int n_units = a.meta[3] * a.n_proj;
    const int n_dyn = max(0, n_units - (int)ncl);
    int claim = 0;      // CTA 0, lane 0: the counter's last answer
    bool over = false;  // CTA 0, lane 0: this cluster's over-claim is made
    uint32_t nclaim = 0;
    auto next_unit = [&]() -> int {
      const uint32_t qc = nclaim & 1;
      if (crank == 0) {
        int nu = 0;
        if (lane == 0) {
          if (nclaim >= 2 && !mbar_wait_cluster(smem_u32(&claim_empty[qc]), ((nclaim >> 1) - 1) & 1)) ok = false;
          claim = atomicAdd(a.counter, 1);
          if (claim < n_dyn) {
            nu = (int)ncl + claim;
          } else {
            nu = n_units;
            over = true;
          }
        }
        nu = __shfl_sync(0xffffffffu, nu, 0);
        __syncwarp();  // lane 0 saw every CTA done with this mailbox before any lane rewrites it
        if (lane < (int)ncta) {  // lane p hands the claim to CTA p
          st_dsmem_u32(mapa(smem_u32(&claim_val[qc]), (uint32_t)lane), (uint32_t)nu);
          mbar_arrive_cluster(mapa(smem_u32(&claim_full[qc]), (uint32_t)lane));
        }
      }
      if (!mbar_wait_cluster(smem_u32(&claim_full[qc]), (nclaim >> 1) & 1)) ok = false;
      const int v = claim_val[qc];
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa(smem_u32(&claim_empty[qc]), 0));
      ++nclaim;
      return v;
    };
    uint32_t np = 0;  // records posted
    for (int u = ok ? (int)cid : n_units, k = 0;; ++k) {  // after a failed wait: the end record only
      if (k > 0) {
        // the loaders have taken the last record posted before the next claim
        if (np > 0 && !mbar_wait(smem_u32(&slot_taken[(np - 1) % kFSlots]), ((np - 1) / kFSlots) & 1)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) break;
        u = next_unit();
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const bool end = u >= n_units;
      int g = 0;
      TileInfo ti{};
      lora_adapter_desc_t d{};
      if (!end) {
        const int tile = u / a.n_proj;
        g = u - tile * a.n_proj;
        const DevView& v = a.proj[g].v;
        ti = load_tile(a.long_units, a.seg_adapter, a.indptr, a.perm, tile, 0);
        d = adapter_desc(v, ti.ad);
        const int bad = check_adapter_warp(v, ti.ad, d, lane);
        if (bad) {  // every CTA of the cluster reaches the same verdict and skips the unit
          if (crank == 0 && lane == 0) report(a.err, bad);
          continue;
        }
      }
      const uint32_t q = np % kFSlots;
      if (np >= kFSlots && !mbar_wait(smem_u32(&slot_empty[q]), ((np / kFSlots) - 1) & 1)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) {  // a wait ran out: stop (warp-uniform)
        ok = false;
        break;
      }
      uint8_t* slot = slot_at(q);
      FUnit* fu = reinterpret_cast<FUnit*>(slot);
      if (end) {
        if (lane == 0) fu->flags = kFRecEnd;
        mbar_arrive(smem_u32(&slot_full[q]));
        break;
      }
      const FProj& P = a.proj[g];
      const DevView& v = P.v;
      // consecutive tokens: one TMA box per stage (rows past the tile are loaded, never stored)
      const int last = a.perm[ti.p0 + ti.cnt - 1];
      const bool tma = P.tma && last - ti.row0 == ti.cnt - 1;
      const int k0 = (int)crank * a.klen;
      const int nk = (min(v.d_in, k0 + a.klen) - k0) / 64;
      const int n_nc = v.d_out / 64;
      const int nc0 = (int)(((long long)n_nc * crank) / ncta);
      const int nc1 = a.shrink_only ? nc0 : (int)(((long long)n_nc * (crank + 1)) / ncta);
      if (lane == 0) {
        fu->flags = tma ? kFRecTma : 0;
        fu->g = g;
        fu->p0 = ti.p0;
        fu->cnt = ti.cnt;
        fu->row0 = ti.row0;
        fu->r = d.rank;
        fu->rpad = (d.rank + 15) & ~15;
        fu->scale = d.scale;
        fu->k0 = k0;
        fu->nk = nk;
        fu->n0 = nc0 * 64;
        fu->nn = nc1 - nc0;
        fu->a_page0 = d.a_page0;
        fu->b_page0 = d.b_page0;
      }
      int* rows = reinterpret_cast<int*>(slot + 128);
      int rv[kTM / 32];  // every lane's loads in flight before the stores
#pragma unroll
      for (int i = 0; i < kTM / 32; ++i) {
        const int m = lane + 32 * i;
        rv[i] = m >= ti.cnt ? -1 : tma ? ti.row0 + m : a.perm[ti.p0 + m];
      }
#pragma unroll
      for (int i = 0; i < kTM / 32; ++i) rows[lane + 32 * i] = rv[i];
      // physical page of each rank row's first element in this CTA's slices
      int* pa = rows + kTM;
      int* pb = pa + LORA_MAX_RANK;
      const int shift = v.page_shift;
      int pv[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = lane + 32 * i;
        pv[i] = j < d.rank ? v.page_list[d.a_page0 + (((long long)j * v.d_in + k0) >> shift)] : 0;
        pv[2 + i] = j < d.rank && nc1 > nc0  // a CTA without a d_out slice reads no B page
                        ? v.page_list[d.b_page0 + (((long long)j * v.d_out + nc0 * 64) >> shift)]
                        : 0;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        pa[lane + 32 * i] = pv[i];
        pb[lane + 32 * i] = pv[2 + i];
      }
      mbar_arrive(smem_u32(&slot_full[q]));  // each lane after its own writes
      ++np;
    }
    if (crank == 0 && lane == 0) {
      if (!over) claim = atomicAdd(a.counter, 1);  // no unit was claimed (cid >= n_units, or a wait ran out)
      // `claim` holds this cluster's over-claim now; the last of all resets the counter
      if (claim == n_dyn + (int)ncl - 1) *a.counter = 0;
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp < kFWarpMma) {
    // ---------------- loaders ----------------
    const int ltid = tid - 32 * kFWarpLoad0;  // 0..127: token row ltid; rank row ltid / 2, pieces 4 (ltid & 1) + 0..3
    const bool lead = ltid == 0;
    const int jr = ltid >> 1, p4 = (ltid & 1) * 4;
    uint32_t gs = 0;  // stages used
    // Every wait is followed by a warp vote, so a warp stops as a whole when one
    // of its lanes' waits ran out.
    auto take_stage = [&]() -> uint32_t {
      const uint32_t st = gs % kFStages;
      bool w = true;
      if (gs >= kFStages) w = mbar_wait(smem_u32(&empty[st]), ((gs / kFStages) - 1) & 1);
      if (!__all_sync(0xffffffffu, w)) ok = false;
      return st;
    };
    for (uint32_t np = 0; ok; ++np) {
      const uint32_t q = np % kFSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&slot_full[q]), (np / kFSlots) & 1))) {
        ok = false;
        break;
      }
      const uint8_t* slot = slot_at(q);
      const FUnit U = *reinterpret_cast<const FUnit*>(slot);
      if (U.flags & kFRecEnd) break;
      if (lead) mbar_arrive(smem_u32(&slot_taken[q]));
      const FProj& P = a.proj[U.g];
      const DevView& v = P.v;
      const bool tma = U.flags & kFRecTma;
      if (lead && tma) {
        prefetch_tensormap(&P.xmap);
        if (U.nn > 0) prefetch_tensormap(&P.ymap);
      }
      const int tok = reinterpret_cast<const int*>(slot + 128)[ltid];
      const int shift = v.page_shift;
      const long long pmask = (1LL << shift) - 1;
      const bool real = jr < U.r;
      // this thread's rank row: the page it is on (looked up again when a chunk crosses into the next)
      long long cur_idx = real ? (((long long)jr * v.d_in + U.k0) >> shift) : 0;
      long long cur_pg = real ? reinterpret_cast<const int*>(slot + 128 + kTM * 4)[jr] : 0;
      for (int c = 0; c < U.nk; ++c, ++gs) {
        const uint32_t st = take_stage();
        if (!ok) break;
        const uint32_t act = smem_u32(stage_at(st)), ad = act + kFActBytes;
        const uint32_t bar = smem_u32(&full[st]);
        const int kcol = U.k0 + 64 * c;
        if (lead) {
          mbar_arrive_expect_tx(bar, tma ? (uint32_t)kFActBytes : 0u);
          if (tma) tma_load_2d(act, &P.xmap, kcol, U.row0, bar);
        }
        if (!tma && tok >= 0) {
          const uint16_t* src = P.x + (long long)tok * P.ldx + kcol;
#pragma unroll
          for (int p = 0; p < 8; ++p) cp_async16(act + sw128_offset(ltid, p), src + 8 * p);
        }
        if (jr < U.rpad) {  // A_i rows, K-major: row jr, pieces p4 .. p4 + 3; zero past the rank
          const long long e = (long long)jr * v.d_in + kcol;
          if (real && (e >> shift) != cur_idx) {
            cur_idx = e >> shift;
            cur_pg = v.page_list[U.a_page0 + cur_idx];
          }
          const uint16_t* src = real ? v.pool + (cur_pg << shift) + (e & pmask) : v.pool;
#pragma unroll
          for (int p = 0; p < 4; ++p) cp_async16(ad + sw128_offset(jr, p4 + p), src + 8 * (p4 + p), real);
        }
        cp_async_arrive_noinc(bar);
      }
      cur_idx = real ? (((long long)jr * v.d_out + U.n0) >> shift) : 0;
      cur_pg = real ? reinterpret_cast<const int*>(slot + 128 + kTM * 4)[LORA_MAX_RANK + jr] : 0;
      for (int nc = 0; ok && nc < U.nn; ++nc, ++gs) {
        const uint32_t st = take_stage();
        if (!ok) break;
        const uint32_t act = smem_u32(stage_at(st)), ad = act + kFActBytes;
        const uint32_t bar = smem_u32(&full[st]);
        const int ncol = U.n0 + 64 * nc;
        if (lead) {
          mbar_arrive_expect_tx(bar, tma ? (uint32_t)kFActBytes : 0u);
          if (tma) tma_load_2d(act, &P.ymap, ncol, U.row0, bar);
        }
        if (!tma && tok >= 0) {
          const uint16_t* src = P.y + (long long)tok * P.ldy + ncol;
#pragma unroll
          for (int p = 0; p < 8; ++p) cp_async16(act + sw128_offset(ltid, p), src + 8 * p);
        }
        if (jr < U.rpad) {  // B_i rows, MN-major: 8-row groups of 1024 bytes, 128-byte swizzle; zero past the rank
          const long long e = (long long)jr * v.d_out + ncol;
          if (real && (e >> shift) != cur_idx) {
            cur_idx = e >> shift;
            cur_pg = v.page_list[U.b_page0 + cur_idx];
          }
          const uint16_t* src = real ? v.pool + (cur_pg << shift) + (e & pmask) : v.pool;
          const uint32_t rowbase = ad + (uint32_t)((jr >> 3) * 1024);
#pragma unroll
          for (int p = 0; p < 4; ++p) cp_async16(rowbase + sw128_offset(jr & 7, p4 + p), src + 8 * (p4 + p), real);
        }
        cp_async_arrive_noinc(bar);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&slot_empty[q]));
    }
    // nothing may still be landing in shared memory when the CTA ends
    cp_async_commit();
    cp_async_wait<0>();
    if (lead)
      for (uint32_t gg = gs > kFStages ? gs - kFStages : 0; gg < gs; ++gg)
        mbar_wait(smem_u32(&full[gg % kFStages]), (gg / kFStages) & 1);
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp == kFWarpMma) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      uint32_t gs = 0, ne = 0, nu = 0;
      bool issued = false;
      for (uint32_t np = 0; ok; ++np) {
        const uint32_t q = np % kFSlots;
        if (!mbar_wait(smem_u32(&slot_full[q]), (np / kFSlots) & 1)) {
          ok = false;
          break;
        }
        const FUnit U = *reinterpret_cast<const FUnit*>(slot_at(q));
        if (U.flags & kFRecEnd) break;
        nu = np + 1;
        const uint32_t ub = np & 1;
        if (np >= 2 && !mbar_wait(smem_u32(&accs_empty[ub]), ((np >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t idesc_s = idesc_bf16(kTM, U.rpad, 0);
        for (int c = 0; c < U.nk; ++c, ++gs) {
          const uint32_t st = gs % kFStages;
          if (!mbar_wait(smem_u32(&full[st]), (gs / kFStages) & 1)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // asynchronous-copy writes, seen here, before the tensor cores read them
          tc_fence_after();
          const uint32_t act = smem_u32(stage_at(st)), ad = act + kFActBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + ub * 64, sdesc_sw128(act + 32 * kk, 16, 1024), sdesc_sw128(ad + 32 * kk, 16, 1024),
                     idesc_s, (c | kk) != 0);
          issued = true;
          mma_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
        if (a.shrink_only) {
          // No expand: the previous unit's H only says that its owners are done
          // with their receive buffers, which this unit's partial is about to
          // refill; waited for after this unit's MMAs are issued.
          if (np >= 1 && !mbar_wait(smem_u32(h_full), (np - 1) & 1)) {
            ok = false;
            break;
          }
          mma_commit(smem_u32(&accs_full[ub]));
          mbar_arrive(smem_u32(&slot_empty[q]));
          continue;
        }
        mma_commit(smem_u32(&accs_full[ub]));
        // the H operand of this unit, written by the owners of its rows
        if (!mbar_wait(smem_u32(h_full), np & 1)) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t idesc_e = idesc_bf16(kTM, 64, 1);
        const uint32_t hhi = smem_u32(hbuf), hlo = hhi + kTM * 128;
        for (int nc = 0; nc < U.nn; ++nc, ++gs, ++ne) {
          const uint32_t st = gs % kFStages;
          const uint32_t eb = ne & 1;
          if (!mbar_wait(smem_u32(&full[st]), (gs / kFStages) & 1) ||
              (ne >= 2 && !mbar_wait(smem_u32(&acce_empty[eb]), ((ne >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t bs = smem_u32(stage_at(st)) + kFActBytes;
          int first = 1;
          for (int part = 0; part < 2; ++part) {
            const uint32_t abase = part ? hlo : hhi;
            for (int kk = 0; kk < U.rpad / 16; ++kk) {
              mma_bf16(tmem + 128 + eb * 64, sdesc_sw128(abase + 32 * kk, 16, 1024),
                       sdesc_sw128(bs + (uint32_t)kk * 2048, 0, 1024), idesc_e, first ? 0u : 1u);
              first = 0;
            }
          }
          mma_commit(smem_u32(&acce_full[eb]));
        }
        if (!ok) break;
        mbar_arrive(smem_u32(&slot_empty[q]));
      }
      // the last unit's H has landed here before the CTA can end (the peers' copies
      // into this CTA are complete)
      if (a.shrink_only && ok && nu > 0 && !mbar_wait(smem_u32(h_full), (nu - 1) & 1)) ok = false;
      if (issued) {  // every MMA of this CTA has completed before tensor memory is freed
        mma_commit(smem_u32(mma_done));
        mbar_wait(smem_u32(mma_done), 0);
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    const int grp = (warp - kFWarpEpi0) >> 2;  // group: 0 also runs the exchange
    const int quarter = warp & 3;              // tensor-memory lanes this warp may read
    const int m = quarter * 32 + lane;         // tile row
    const int et = tid - 32 * (kFWarpEpi0 + 4 * grp);  // 0..127 within the group
    uint32_t gs = 0, ne = 0;
    // Every wait is followed by a warp vote, so a warp stops as a whole when one
    // of its lanes' waits ran out; the epilogue warps meet at no blocking barrier
    // (an expand stage is released by whichever of its group's warps is last).
    auto waited = [&](bool w) {
      if (!__all_sync(0xffffffffu, w)) ok = false;
      return ok;
    };
    // A warp's stage whose TMA store may still be reading it: released once the
    // warp has issued its next store (or at the end of the unit).
    int pending = -1;
    auto release = [&](int st) {  // lane 0: this warp is done with stage st
      __threadfence_block();
      if (atomicAdd(&rel_cnt[st], 1) == 3) {
        rel_cnt[st] = 0;
        mbar_arrive(smem_u32(&empty[st]));
      }
    };
    auto flush = [&]() {  // lane 0
      if (pending >= 0) {
        bulk_wait_read0();
        release(pending);
        pending = -1;
      }
    };
    for (uint32_t np = 0; ok; ++np) {
      const uint32_t q = np % kFSlots;
      if (!waited(mbar_wait(smem_u32(&slot_full[q]), (np / kFSlots) & 1))) break;
      const uint8_t* slot = slot_at(q);
      const FUnit U = *reinterpret_cast<const FUnit*>(slot);
      if (U.flags & kFRecEnd) break;
      const FProj& P = a.proj[U.g];
      const int tok_m = reinterpret_cast<const int*>(slot + 128)[m];
      const int rpad = U.rpad;
      if (grp == 0) {
        // -- shrink partial: row m out of tensor memory, to the owner of row m
        const uint32_t ub = np & 1;
        if (!waited(mbar_wait(smem_u32(&accs_full[ub]), (np >> 1) & 1))) break;
        // This unit's exchange: the bytes of the partial rows this CTA owns, and of
        // the H operand.  Armed only now: the MMA warp has waited for the previous
        // unit's H before committing this unit's partial, so that phase is over.
        if (et == 0) {
          mbar_arrive_expect_tx(smem_u32(recv_full), (uint32_t)(ncta * R * rpad * 4));
          mbar_arrive_expect_tx(smem_u32(h_full), (uint32_t)(kTM * rpad * 4));
        }
        tc_fence_after();
        uint32_t pr[64];
        const uint32_t taddr = tmem + ub * 64 + ((uint32_t)(quarter * 32) << 16);
        tmem_ld32_nowait(taddr, pr);
        tmem_ld32_nowait(taddr + 32, pr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&accs_empty[ub]));
        {
          const uint32_t owner = (uint32_t)(m / R);
          const uint32_t dst = smem_u32(recv + ((size_t)crank * R + (m - (int)owner * R)) * LORA_MAX_RANK);
          const uint32_t rbar = mapa(smem_u32(recv_full), owner);
#pragma unroll
          for (int j = 0; j < LORA_MAX_RANK; j += 4)
            if (j < rpad)
              st_async_v4(mapa(dst + 4 * j, owner),
                          make_float4(__uint_as_float(pr[j]), __uint_as_float(pr[j + 1]),
                                      __uint_as_float(pr[j + 2]), __uint_as_float(pr[j + 3])),
                          rbar);
        }
        // -- owner: sum the partials of its rows in CTA order, scale, split, send H rows to every CTA
        if (!waited(mbar_wait(smem_u32(recv_full), np & 1))) break;
        const int ng = rpad / 8;  // 8-column groups of a row
        for (int gi = et; gi < R * ng; gi += 128) {
          const int rr = gi / ng, cg = gi - rr * ng;
          const int mm = (int)crank * R + rr;
          float sum[8];
          const float4* p0 = reinterpret_cast<const float4*>(recv + (size_t)rr * LORA_MAX_RANK + 8 * cg);
          float4 lo4 = p0[0], hi4 = p0[1];
          sum[0] = lo4.x; sum[1] = lo4.y; sum[2] = lo4.z; sum[3] = lo4.w;
          sum[4] = hi4.x; sum[5] = hi4.y; sum[6] = hi4.z; sum[7] = hi4.w;
          for (uint32_t c = 1; c < ncta; ++c) {
            const float4* pc =
                reinterpret_cast<const float4*>(recv + ((size_t)c * R + rr) * LORA_MAX_RANK + 8 * cg);
            lo4 = pc[0];
            hi4 = pc[1];
            sum[0] += lo4.x; sum[1] += lo4.y; sum[2] += lo4.z; sum[3] += lo4.w;
            sum[4] += hi4.x; sum[5] += hi4.y; sum[6] += hi4.z; sum[7] += hi4.w;
          }
          if (P.h != nullptr && mm < U.cnt) {  // the shrink-only form: row mm's h, unscaled, columns < r
            float* hrow = P.h + (long long)reinterpret_cast<const int*>(slot + 128)[mm] * P.ldh + 8 * cg;
            if (8 * cg + 8 <= U.r) {
              reinterpret_cast<float4*>(hrow)[0] = make_float4(sum[0], sum[1], sum[2], sum[3]);
              reinterpret_cast<float4*>(hrow)[1] = make_float4(sum[4], sum[5], sum[6], sum[7]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (8 * cg + e < U.r) hrow[e] = sum[e];
            }
          }
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * cg + 2 * e;
            const float s0 = j < U.r ? U.scale * sum[2 * e] : 0.f;
            const float s1 = j + 1 < U.r ? U.scale * sum[2 * e + 1] : 0.f;
            hv[e] = pack_bf16x2(s0, s1);
            lv[e] = pack_bf16x2(s0 - bf_lo(hv[e]), s1 - bf_hi(hv[e]));
          }
          const uint32_t hdst = smem_u32(hbuf) + sw128_offset(mm, cg);
          const float4 hq = make_float4(__uint_as_float(hv[0]), __uint_as_float(hv[1]), __uint_as_float(hv[2]),
                                        __uint_as_float(hv[3]));
          const float4 lq = make_float4(__uint_as_float(lv[0]), __uint_as_float(lv[1]), __uint_as_float(lv[2]),
                                        __uint_as_float(lv[3]));
          for (uint32_t c = 0; c < ncta; ++c) {
            const uint32_t hb = mapa(smem_u32(h_full), c);
            st_async_v4(mapa(hdst, c), hq, hb);
            st_async_v4(mapa(hdst + kTM * 128, c), lq, hb);
          }
        }
      }
      // -- expand stages of this group: y = y0 + accumulator
      gs += (uint32_t)U.nk;
      for (int nc = 0; nc < U.nn; ++nc, ++gs, ++ne) {
        const uint32_t eb = ne & 1;
        if ((int)eb != grp) continue;  // the other group's stage
        const uint32_t st = gs % kFStages;
        if (!waited(mbar_wait(smem_u32(&full[st]), (gs / kFStages) & 1) &&
                    mbar_wait(smem_u32(&acce_full[eb]), (ne >> 1) & 1)))
          break;
        tc_fence_after();
        uint32_t acc[64];
        const uint32_t ta = tmem + 128 + eb * 64 + ((uint32_t)(quarter * 32) << 16);
        tmem_ld32_nowait(ta, acc);
        tmem_ld32_nowait(ta + 32, acc + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&acce_empty[eb]));
        uint8_t* act = stage_at(st);
        const int ncol = U.n0 + 64 * nc;
        // a warp whose 32 rows are all in a tile of consecutive tokens stores them
        // with one TMA copy from the stage (the result overwrites the row's y0 there)
        const bool wstore = (U.flags & kFRecTma) && P.yf == nullptr && quarter * 32 + 31 < U.cnt;
        if (wstore) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint4* qp = reinterpret_cast<uint4*>(act + sw128_offset(m, cc));
            float y0[8];
            unpack8(*qp, y0);
            uint4 o;
            o.x = pack_bf16x2(y0[0] + __uint_as_float(acc[8 * cc]), y0[1] + __uint_as_float(acc[8 * cc + 1]));
            o.y = pack_bf16x2(y0[2] + __uint_as_float(acc[8 * cc + 2]), y0[3] + __uint_as_float(acc[8 * cc + 3]));
            o.z = pack_bf16x2(y0[4] + __uint_as_float(acc[8 * cc + 4]), y0[5] + __uint_as_float(acc[8 * cc + 5]));
            o.w = pack_bf16x2(y0[6] + __uint_as_float(acc[8 * cc + 6]), y0[7] + __uint_as_float(acc[8 * cc + 7]));
            *qp = o;
          }
          fence_proxy_async_smem();  // the rows, written here, before the TMA engine reads them
          __syncwarp();
          if (lane == 0) {
            if (ok) {
              tma_store_2d(&P.ystore, ncol, U.row0 + quarter * 32, smem_u32(act) + (uint32_t)(quarter * 32 * 128));
              bulk_commit();
            }
            // the previous store has read its stage once at most this one is pending
            if (pending >= 0) {
              asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
              release(pending);
            }
            pending = (int)st;
          }
        } else {
          if (ok && m < U.cnt) {
            if (P.yf != nullptr) {  // fp32 output (diagnostic form): the same sums, not rounded to bf16
              float* frow = P.yf + (long long)tok_m * P.ldyf + ncol;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                float y0[8];
                unpack8(*reinterpret_cast<const uint4*>(act + sw128_offset(m, cc)), y0);
                float4* o4 = reinterpret_cast<float4*>(frow + 8 * cc);
                o4[0] = make_float4(y0[0] + __uint_as_float(acc[8 * cc]), y0[1] + __uint_as_float(acc[8 * cc + 1]),
                                    y0[2] + __uint_as_float(acc[8 * cc + 2]), y0[3] + __uint_as_float(acc[8 * cc + 3]));
                o4[1] = make_float4(y0[4] + __uint_as_float(acc[8 * cc + 4]), y0[5] + __uint_as_float(acc[8 * cc + 5]),
                                    y0[6] + __uint_as_float(acc[8 * cc + 6]), y0[7] + __uint_as_float(acc[8 * cc + 7]));
              }
            } else {
              uint4* yrow = reinterpret_cast<uint4*>(P.y + (long long)tok_m * P.ldy + ncol);
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                float y0[8];
                unpack8(*reinterpret_cast<const uint4*>(act + sw128_offset(m, cc)), y0);
                uint4 o;
                o.x = pack_bf16x2(y0[0] + __uint_as_float(acc[8 * cc]), y0[1] + __uint_as_float(acc[8 * cc + 1]));
                o.y = pack_bf16x2(y0[2] + __uint_as_float(acc[8 * cc + 2]), y0[3] + __uint_as_float(acc[8 * cc + 3]));
                o.z = pack_bf16x2(y0[4] + __uint_as_float(acc[8 * cc + 4]), y0[5] + __uint_as_float(acc[8 * cc + 5]));
                o.w = pack_bf16x2(y0[6] + __uint_as_float(acc[8 * cc + 6]), y0[7] + __uint_as_float(acc[8 * cc + 7]));
                yrow[cc] = o;
              }
            }
          }
          __syncwarp();
          if (lane == 0) release((int)st);  // read its y0 rows: done with the stage
        }
      }
      // A stage held back for its store is released before the next unit: the
      // loaders may need it to bring in that unit's shrink stages.
      if (lane == 0) flush();
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&slot_empty[q]));
    }
    if (lane == 0) {
      flush();
      bulk_wait0();  // this warp's y stores are complete before the CTA ends
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  // no CTA leaves while a peer may still write into it or read its barriers
  cluster_sync();
  if (warp == kFWarpMma) tmem_dealloc(tmem, 256);
  pdl_exit(a.after_gather != 0);
}

// ---------------------------------------------------------------- launcher --

bool tc_fused_shrink_ok(const lora_pool_view_t* v) { return v->d_in % 64 == 0 && v->page_elems >= 64; }

bool tc_fused_ok(const lora_pool_view_t* v) {
  int ks, klen;
  shrink_split(v->d_in, &ks, &klen);
  return v->d_in % 64 == 0 && v->d_out % 64 == 0 && v->page_elems >= 64 && ks <= kMaxKSplit;
}

lora_status_t launch_fused_tc(int n_proj, const ProjCall* projs, const lora_segments_t* seg, int after_gather,
                              int32_t* err, cudaStream_t stream, int shrink_only) {
  if (n_proj < 1 || n_proj > kMaxFusedProj) return LORA_ERR_INVALID_ARG;
  FusedArgs a;
  memset(&a, 0, sizeof(a));
  int ks = 1, klen = 64;
  shrink_split(projs[0].view->d_in, &ks, &klen);
  for (int g = 0; g < n_proj; ++g) {
    const ProjCall& h = projs[g];
    FProj& P = a.proj[g];
    make_dev_view(h.view, &P.v);
    P.x = static_cast<const uint16_t*>(h.x);
    P.y = static_cast<uint16_t*>(h.y);
    P.yf = h.yf;
    P.h = h.h;
    P.ldx = h.ldx;
    P.ldy = h.ldy;
    P.ldyf = h.ldyf;
    P.ldh = h.ldh;
    P.tma = make_act_map(&P.xmap, h.x, seg->T, h.view->d_in, h.ldx, kTM) &&
                    (shrink_only || (make_act_map(&P.ymap, h.y, seg->T, h.view->d_out, h.ldy, kTM) &&
                                     make_act_map(&P.ystore, h.y, seg->T, h.view->d_out, h.ldy, 32)))
                ? 1
                : 0;
  }
  a.perm = seg->token_perm;
  a.indptr = seg->seg_indptr;
  a.seg_adapter = seg->seg_adapter;
  a.long_units = seg->long_units;
  a.meta = seg->meta;
  a.counter = seg->meta + 5;
  a.err = err;
  a.n_proj = n_proj;
  a.klen = klen;
  a.after_gather = after_gather;
  a.shrink_only = shrink_only;
  a.probe = wait_probe_cycles();
  const long long upper = (long long)seg->max_long_units * n_proj;
  if (upper <= 0) return LORA_OK;
  if (ensure_smem_attr((const void*)fused_tc_kernel, kFusedSmem) != cudaSuccess) return LORA_ERR_CUDA;
  const int cap = max_active_clusters((const void*)fused_tc_kernel, kFThreads, kFusedSmem, ks);
  const long long n_clusters = upper < cap ? upper : cap;
  return launch_pdl((const void*)fused_tc_kernel, dim3((unsigned)(n_clusters * ks)), dim3(kFThreads), kFusedSmem,
                    stream, ks, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
