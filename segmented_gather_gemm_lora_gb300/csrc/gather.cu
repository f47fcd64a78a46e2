// Gather path of the multi-adapter LoRA product on CUDA cores.
//
// "Multi-LoRA serving: the single translator with a thousand glossaries",
// section "SGMV: the kernel that holds it all up": small segments (one request
// per adapter) take a batched gather path.  This kernel is that path, for
// segments of at most LORA_SHORT_MAX_TOKENS tokens, for the one-token-per-
// request decode form (MBGMV in "Multi-LoRA Serving in Production", section
// "S-LoRA: MBGMV and MBGMM Kernels"), and for the shrink / expand stages alone.
//
// Work decomposition.  One thread-block cluster of CL CTAs (CL <= 8) takes one
// work unit (an adapter and its tokens, in groups of up to 4) at a time.  CTA c
// of the cluster owns the c-th slice of d_in for the shrink and the c-th slice
// of d_out for the expand, so every adapter byte and every activation byte is
// read once per unit:
//   shrink  partial_c[t, j] = sum_{k in slice c} x[t, k] * A_i[j, k]
//   reduce  h[t, j] = s_i * sum_c partial_c[t, j]   through distributed shared
//           memory, in fixed CTA order (deterministic; no float atomics)
//   expand  y[t, n] = bf16(y0[t, n] + sum_j h[t, j] * B_i[j, n]),  n in slice c
// The rank-r intermediate never leaves the chip.
//
// Warp roles.  Warp 9 of every CTA schedules: it claims units (from a counter,
// CTA 0 of a cluster claiming and handing the claim to its peers, when the
// segments give one; one-token units go round-robin), resolves each unit's
// tokens and adapter, checks every page slot of the adapter and caches its
// physical pages, up to three units ahead of the producers.  Warps 8, 10 and 11
// produce: they stage 16-row chunks of the adapter (1 KB row runs, translated
// through the page table, "Multi-LoRA Serving in Production", section "Unified
// Paged Memory"; one bulk copy per row run and page) with the unit's token rows
// for the same columns into a 4-stage ring, a stage's copies going round the
// three warps; every stage carries a record of what it holds.
// Warps 0-7 consume the ring.  Between a group's shrink and expand each CTA
// pushes its partial h into every peer's shared memory (asynchronous stores
// whose bytes complete on the peer's own mbarrier) and sums what it received
// in CTA order; the producer keeps streaming the expand rows meanwhile.
//
// Summation order.  Each rank row's shrink dot product over a sub-slice and
// each output's expand sum over a 16-row chunk are fixed functions of column
// and row positions, and partial results combine in sub-slice / chunk order.
// A token's result therefore depends neither on how many tokens share its unit
// nor on its adapter's rank: zero-padding an adapter or moving a token between
// units changes no bit of its output.
#include <algorithm>
#include <cstring>

#include "chunk_mma.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lora {

constexpr int kGCons = 8;            // consumer warps
constexpr int kGProd = kGCons;       // the first producer warp
constexpr int kGSched = kGCons + 1;  // the scheduler warp
constexpr int kGProd2 = kGCons + 2;  // the second producer warp
constexpr int kGProd3 = kGCons + 3;  // the third producer warp
constexpr int kGProds = 3;           // producer warps: a stage's copies go round them
constexpr int kGThreads = 32 * (kGCons + 4);
constexpr int kGConsThreads = 32 * kGCons;
constexpr int kMaxCluster = 8;
constexpr int kStages = 4;
constexpr int kStageBytes = (kChunkRows + kNT) * kRowStride;  // 20.3 KB
constexpr int kMaxPgSlots = 320;  // page-list slots of one adapter cached in shared memory
constexpr int kUSlots = 4;        // unit slots: the scheduler resolves up to three units ahead

enum GKind { kGShrink = 0, kGExpand = 1, kGReduce = 2, kGEnd = 3 };
enum GFlag {
  kFFirst = 1,   // shrink: first sub-slice of the row block; expand: first row block of the sub-slice
  kFLast = 2,    // shrink: last sub-slice of the row block (partials to the warp's h);
                 // expand: last row block of the sub-slice (adds y0, writes y; token rows staged)
  kFRed = 8,     // after this record: h of the group from the cluster's partials
  kFHLoad = 16,  // before this record: h of the group from the caller
  kFNoK = 32     // this CTA has no d_in slice (its partial is zero)
};

// What the producer tells the consumers about a stage.  The group's reduction
// rides on its last shrink chunk, so only a CTA without a d_in slice spends a
// stage on a record without data.
struct __align__(16) GRec {
  int kind;
  int ntok;   // tokens of the group
  int j0;     // first adapter row of the chunk
  int nrows;  // adapter rows of the chunk
  int nvec;   // 16-byte pieces per row of the sub-slice
  int col0;   // first column of the sub-slice
  int flags;  // GFlag bits
  int r;      // rank
  float sc;   // scale
  int g;      // projection
  int tok[kNT];
};
static_assert(sizeof(GRec) <= 64 && sizeof(GRec) % 16 == 0, "record slot, read as 16-byte pieces");

// A stage's record, by 16-byte shared-memory loads (one per piece, all in
// flight together) rather than one load per field.
__device__ __forceinline__ GRec load_rec(const GRec* p) {
  union {
    GRec r;
    uint4 v[sizeof(GRec) / 16];
  } u;
#pragma unroll
  for (int i = 0; i < (int)(sizeof(GRec) / 16); ++i) u.v[i] = reinterpret_cast<const uint4*>(p)[i];
  return u.r;
}

// What the scheduler tells the producer about a unit it has resolved: the
// adapter's rank, scale and page-list origin, the unit's tokens, and whether
// its page slots sit checked in the unit's page cache.
struct GUnit {
  int end;       // 1: no more units
  int r;         // rank
  float sc;      // scale
  int tb;        // first position of the unit in token order (segments)
  int cnt;       // tokens of the unit
  int na;        // page slots of A_i; B_i's follow them in the cache
  int cached;    // 1: every page slot of the adapter is in the cache
  int g;         // projection
  int tok[kNT];  // the first group's tokens
  long long a_page0, b_page0;
};
static_assert(sizeof(GUnit) <= 64, "unit slot");
static_assert(kSub / 64 <= kGCons, "one warp per block of 8 output vectors");

// One projection of the call: its activations and its view of the adapter pool.
struct GProj {
  const uint16_t* x;
  long long ldx;
  uint16_t* y;
  long long ldy;
  DevView v;
};

constexpr size_t kOffRec = (size_t)kStages * kStageBytes;
constexpr size_t kOffPw = kOffRec + (size_t)kStages * 64;                     // fp32 [kGCons][kNT][kHMax]
constexpr size_t kOffRecv = kOffPw + (size_t)kGCons * kNT * kHMax * sizeof(float);  // fp32 [2][kMaxCluster][kNT][kHMax]
constexpr size_t kOffHs = kOffRecv + 2 * (size_t)kMaxCluster * kNT * kHMax * sizeof(float);  // fp32 [kNT][kHMax]
constexpr size_t kOffPgt = kOffHs + kNT * kHMax * sizeof(float);          // int [kUSlots][kMaxPgSlots]
constexpr size_t kOffUnit = kOffPgt + kUSlots * kMaxPgSlots * sizeof(int);  // GUnit [kUSlots], 64-byte slots
constexpr size_t kOffClaim = kOffUnit + kUSlots * 64;                     // int [2]
constexpr size_t kOffCls = kOffClaim + 16;                                // uint32 [3][32] unit classes
constexpr size_t kOffProj = kOffCls + 3 * 32 * sizeof(uint32_t);        // GProj [kMaxFusedProj], 16-byte slots
constexpr size_t kOffBars = kOffProj + kMaxFusedProj * ((sizeof(GProj) + 15) / 16 * 16);
constexpr int kNBars = 2 * kStages + 2 + 2 + 2 + 2 * kUSlots + 1 + 1;
constexpr size_t kGatherSmem = kOffBars + kNBars * 8;
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(kGatherSmem <= 233472 / 2 - 1024, "two gather CTAs per SM");


struct GatherArgs {
  GProj proj[kMaxFusedProj];
  int n_proj;  // projections sharing the segments (apply mode); unit u is (u / n_proj, projection u % n_proj)
  float* h;    // shrink / expand modes (one projection)
  long long ldh;
  float* yf;  // non-null: fp32 output rows (y is then read only, for y0; one projection)
  long long ldyf;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* short_units;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* counter;  // unit claims (segments); zero between calls
  const int32_t* token_adapter;
  int T;
  int32_t* err;
  int mode;
  int src;
  int short_only;
  long long probe;  // > 0: the timeout probe's wait limit in cycles (lora_debug_wait_probe)
};

// The chunk arithmetic (chunk_mma.cuh) over a stage: adapter rows first, the
// group's token rows after the chunk's kChunkRows rows.
__device__ __forceinline__ void expand_chunk(uint16_t* ybase, long long ldy, float* yf, long long ldyf,
                                             uint32_t sbase, const uint8_t* sb, const float* hs, float* scr,
                                             float (&acc)[4][4], const GRec& rc, bool ok, int warp, int lane) {
  const int wsub = rc.nvec * 8;
  if (warp * 64 >= wsub) return;
  expand_mma(sbase, hs, rc.j0, rc.nrows, rc.ntok, wsub, (rc.flags & kFFirst) != 0, acc, warp, lane);
  if ((rc.flags & kFLast) && ok)
    expand_store(ybase, ldy, yf, ldyf, sb + kChunkRows * kRowStride, scr, acc, rc.ntok, rc.tok, rc.col0, wsub, warp,
                 lane);
}

__global__ void __launch_bounds__(kGThreads, 2) gather_kernel(const __grid_constant__ GatherArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  GRec* recs = reinterpret_cast<GRec*>(sm + kOffRec);  // 64-byte slots
  float* pw = reinterpret_cast<float*>(sm + kOffPw);  // each warp's partial h of the group
  float* recv = reinterpret_cast<float*>(sm + kOffRecv);  // the cluster's partials, by CTA
  float* hs = reinterpret_cast<float*>(sm + kOffHs);
  int* pgt = reinterpret_cast<int*>(sm + kOffPgt);
  GUnit* units = reinterpret_cast<GUnit*>(sm + kOffUnit);
  int* claim_val = reinterpret_cast<int*>(sm + kOffClaim);
  uint32_t* cls = reinterpret_cast<uint32_t*>(sm + kOffCls);  // CTA 0: claimable units by class
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  // The projections' parameters, copied once into shared memory: the loops
  // index them by the unit's projection, which kernel parameters serve slowly.
  GProj* projs = reinterpret_cast<GProj*>(sm + kOffProj);
  uint64_t* full = bars;                   // [stages] the record writer (+ the copies' bytes)
  uint64_t* empty = bars + kStages;        // [stages] 8 consumer warps
  uint64_t* recv_full = bars + 2 * kStages;  // [2] this CTA's arrival + every CTA's partial bytes
  uint64_t* claim_full = recv_full + 2;     // [2] CTA 0's scheduler
  uint64_t* claim_empty = claim_full + 2;  // [2] (CTA 0 only) one arrival per CTA
  uint64_t* unit_full = claim_empty + 2;   // [kUSlots] the scheduler
  uint64_t* unit_empty = unit_full + kUSlots;  // [kUSlots] the producers
  uint64_t* cons = unit_empty + kUSlots;   // 8 consumer warps, twice per group
  uint64_t* cls_ready = cons + 1;          // 8 consumer warps, once

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
  const uint32_t cid = cluster_id_x(), ncl = ncluster_x();
  const bool dynamic = a.src == kSrcSegments;
  const int G = a.n_proj;
  const bool reduce_h = a.mode != kModeExpand;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), kGProds);
      mbar_init(smem_u32(&empty[s]), kGCons);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&recv_full[b]), 1);
      mbar_init(smem_u32(&claim_full[b]), 1);
      mbar_init(smem_u32(&claim_empty[b]), ncta);
    }
    for (int b = 0; b < kUSlots; ++b) {
      mbar_init(smem_u32(&unit_full[b]), 1);
      mbar_init(smem_u32(&unit_empty[b]), kGProds);
    }
    mbar_init(smem_u32(cons), kGCons);
    mbar_init(smem_u32(cls_ready), kGCons);
    fence_mbar_init();
  }
  if (tid < 3 * 32) cls[tid] = 0u;
  if (tid < a.n_proj) projs[tid] = a.proj[tid];
  // every barrier of every CTA initialised before any peer arrives on it
  cluster_sync();
  pdl_wait_then_release();

  bool ok = true;
  if (a.probe > 0) {  // the timeout probe: every CTA takes the exit of a wait that ran out
    __shared__ uint64_t probe_bar;
    __shared__ int probe_ok;
    if (tid == 0) probe_ok = wait_probe(&probe_bar, a.probe) ? 1 : 0;
    __syncthreads();
    ok = probe_ok != 0;
  }
  const int n_short = a.src == kSrcSegments ? a.meta[2] : 0;
  // units of one projection (a segment's group of tokens, or a token), times the projections
  const int n_base = a.src == kSrcTokens ? a.T : a.meta[2] + (a.short_only ? 0 : a.meta[3]);
  const int n_units = n_base * G;
  if (n_units == 0) return;  // every CTA of every cluster leaves: nothing has touched a peer or the counter
  // When the same call's fused tensor-core kernel follows with long tiles to do,
  // half of the clusters take part and the others leave at once: their SMs go to
  // the fused kernel, which then runs beside this one instead of after it (the
  // two write disjoint rows).  Measured: the 13B forward 18.5 -> 17.6 ms, the
  // prefill call 64.7 -> 62.0 us.
  const bool beside_fused = a.short_only && a.src == kSrcSegments && a.meta[3] > 0;
  const int ncl_eff = beside_fused ? max(1, (int)ncl / 2) : (int)ncl;  // clusters that take part
  if ((int)cid >= ncl_eff) return;  // the whole cluster leaves: nothing has touched a peer
  const int n_dyn = max(0, n_units - ncl_eff);  // units claimed from the counter
  // Order of the claimed units: largest first.  A unit's time grows with its
  // adapter's row blocks, and a cluster that draws a large unit last keeps the
  // call waiting; so CTA 0's consumer warps, idle until the first chunk lands,
  // classify the claimable units (more than two row blocks, two, one) into bit
  // masks (word L holds units ncl + 32 L + b), and CTA 0's scheduler maps
  // counter value c to the c-th unit of that order (segment order within a
  // class).  Up to 1024 claimable units; beyond, segment order.
  const bool ordered = dynamic && crank == 0 && n_dyn <= 32 * 32;

  if (warp == kGSched) {
    // ---------------- scheduler ----------------
    // Claims a unit, resolves its segment, tokens and adapter, checks every
    // page slot of the adapter and caches the physical pages, up to three
    // units ahead of the producers.
    // Claims: unit cid first, then units ncl + counter, CTA 0 claiming for the
    // cluster.  Each cluster over-claims the counter exactly once; the last
    // claim of all puts it back to zero for the next call.  A unit is claimed
    // once the producers have started on the one three before it (kUSlots
    // unit slots), so that the resolution of small units (a chain of dependent
    // loads) hides behind the copies of the units between.  Measured on the
    // hetero up + down pair (µs), units claimed once the producers started on
    // the one 1 / 2 / 3 before: 123.5, 119.6, 116.2; a reserve cut back to one
    // unit once fewer than two per cluster remain took it back to 123.1, and
    // the 13B-shaped forward is fastest with three too.
    int u = (int)cid;
    int claim = 0;      // CTA 0, lane 0: the counter's last answer
    bool over = false;  // CTA 0, lane 0: this cluster's over-claim is made
    uint32_t nclaim = 0;
    uint32_t cmask[3] = {0u, 0u, 0u};  // CTA 0: this lane's units of each class
    int cpre[3] = {0, 0, 0};           // CTA 0: units of the class in lower lanes
    int ctot[3] = {0, 0, 0};           // CTA 0: units of the class
    auto classify = [&]() {  // the consumers' masks, then each class's prefix over the lanes
      if (!mbar_wait(smem_u32(cls_ready), 0)) ok = false;
#pragma unroll
      for (int c = 0; c < 3; ++c) cmask[c] = cls[c * 32 + lane];
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        const int n = __popc(cmask[c]);
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        cpre[c] = incl - n;
        ctot[c] = __shfl_sync(0xffffffffu, incl, 31);
      }
    };
    // the unit of the c-th claim, c < n_dyn (every lane of CTA 0's warp)
    auto ordered_unit = [&](int c) -> int {
      const int k = c < ctot[0] ? 0 : c < ctot[0] + ctot[1] ? 1 : 2;
      const int n = c - (k > 0 ? ctot[0] : 0) - (k > 1 ? ctot[1] : 0);
      const uint32_t m = k == 0 ? cmask[0] : k == 1 ? cmask[1] : cmask[2];
      const int pre = k == 0 ? cpre[0] : k == 1 ? cpre[1] : cpre[2];
      const uint32_t hit = __ballot_sync(0xffffffffu, pre <= n && n < pre + __popc(m));
      const int owner = __ffs(hit) - 1;
      uint32_t mm = m;  // the (n - pre)-th set bit of the owner's mask
      for (int j = 0; j < n - pre && j < 32; ++j) mm &= mm - 1;
      const int bit = __ffs(mm) - 1;
      return ncl_eff + 32 * owner + __shfl_sync(0xffffffffu, bit, owner);
    };
    auto next_unit = [&]() {
      if (!dynamic) {
        u += ncl_eff;
        return;
      }
      const int q = nclaim & 1;
      if (crank == 0) {
        if (ordered && nclaim == 0) classify();
        int nu = 0;
        if (lane == 0) {
          if (nclaim >= 2 && !mbar_wait_cluster(smem_u32(&claim_empty[q]), ((nclaim >> 1) - 1) & 1)) ok = false;
          claim = atomicAdd(a.counter, 1);
          if (claim < n_dyn) {
            nu = ncl_eff + claim;
          } else {
            nu = n_units;
            over = true;
          }
        }
        nu = __shfl_sync(0xffffffffu, nu, 0);
        if (ordered && nu < n_units) nu = ordered_unit(nu - ncl_eff);
        __syncwarp();  // lane 0 saw every CTA done with this slot before any lane rewrites it
        // lane p hands the claim to CTA p
        if (lane < (int)ncta) {
          st_dsmem_u32(mapa(smem_u32(&claim_val[q]), (uint32_t)lane), (uint32_t)nu);
          mbar_arrive_cluster(mapa(smem_u32(&claim_full[q]), (uint32_t)lane));
        }
      }
      if (!mbar_wait_cluster(smem_u32(&claim_full[q]), (nclaim >> 1) & 1)) ok = false;
      u = claim_val[q];
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa(smem_u32(&claim_empty[q]), 0));
      ++nclaim;
    };
    uint32_t nposted = 0;  // units handed to the producer
    // the slot of the next unit, once the producers are done with its last
    // use (they have then started on the unit after that one)
    auto take_slot = [&]() -> uint32_t {
      const uint32_t q = nposted % kUSlots;
      if (nposted >= kUSlots && !mbar_wait(smem_u32(&unit_empty[q]), ((nposted / kUSlots) - 1) & 1)) ok = false;
      return q;
    };
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t q = take_slot();
      if (k > 0) next_unit();
      if (u >= n_units) break;
      const int ub = u / G, g = u - ub * G;  // the unit of its projection, the projection
      const DevView& v = projs[g].v;
      const int shift = v.page_shift;
      int ad, tb = 0, cnt;
      if (a.src == kSrcTokens) {
        ad = a.token_adapter[ub];
        tb = ub;
        cnt = 1;
        if (ad == -1) continue;
        if (ad < -1 || ad >= v.n_adapters) {
          if (crank == 0 && lane == 0) report(a.err, LORA_DERR_BAD_ADAPTER);
          continue;
        }
      } else if (ub < n_short) {
        const int s = a.short_units[ub];
        ad = a.seg_adapter[s];
        tb = a.indptr[s];
        cnt = a.indptr[s + 1] - tb;
      } else {
        const int s = a.long_units[2 * (ub - n_short)];
        const int m0 = a.long_units[2 * (ub - n_short) + 1];
        ad = a.seg_adapter[s];
        tb = a.indptr[s] + m0;
        cnt = min(LORA_TILE_M, a.indptr[s + 1] - tb);
      }
      // The first group's tokens do not depend on the adapter: load them
      // alongside its descriptor.
      const int first_tok = lane < min(kNT, cnt) ? (a.src == kSrcTokens ? ub : a.perm[tb + lane]) : -1;
      if (ad < 0 || ad >= v.n_adapters) {  // segments built for more adapters than the view has
        if (crank == 0 && lane == 0) report(a.err, LORA_DERR_BAD_ADAPTER);
        continue;
      }
      const lora_adapter_desc_t d = adapter_desc(v, ad);
      if (d.rank < 1 || d.rank > v.max_rank || d.rank > kHMax) {
        if (crank == 0 && lane == 0) report(a.err, LORA_DERR_BAD_RANK);
        continue;
      }
      // Every CTA checks the whole adapter, so all reach the same verdict
      // without talking to each other; the same pass caches the physical
      // pages.  Each lane has up to 8 page-list reads in flight at once.
      const long long P = 1LL << shift;
      const long long na = ((long long)d.rank * v.d_in + P - 1) >> shift;
      const long long nb = ((long long)d.rank * v.d_out + P - 1) >> shift;
      const bool cached = na + nb <= kMaxPgSlots;
      int* pc = pgt + q * kMaxPgSlots;
      int mine = 0;
      for (long long i0 = 0; i0 < na + nb; i0 += 32 * 8) {
        int pv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const long long i = i0 + k * 32 + lane;
          const long long slot = i < na ? d.a_page0 + i : d.b_page0 + (i - na);
          pv[k] = 0;
          if (i < na + nb) pv[k] = (slot < 0 || slot >= v.n_page_list) ? -1 : v.page_list[slot];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const long long i = i0 + k * 32 + lane;
          if (i < na + nb) {
            if (pv[k] < 0 || pv[k] >= v.n_pages) mine = 1;
            if (cached) pc[i] = pv[k];
          }
        }
      }
      if (__any_sync(0xffffffffu, mine)) {
        if (crank == 0 && lane == 0) report(a.err, LORA_DERR_BAD_PAGE);
        continue;  // the slot stays free
      }
      GUnit un;
      un.end = 0;
      un.r = d.rank;
      un.sc = d.scale;
      un.tb = tb;
      un.cnt = cnt;
      un.na = (int)na;
      un.cached = cached ? 1 : 0;
      un.g = g;
#pragma unroll
      for (int t = 0; t < kNT; ++t) un.tok[t] = __shfl_sync(0xffffffffu, first_tok, t);
      un.a_page0 = d.a_page0;
      un.b_page0 = d.b_page0;
      __syncwarp();  // every lane's cache writes before the hand-over
      if (lane == 0) {
        units[q] = un;
        mbar_arrive(smem_u32(&unit_full[q]));
      }
      ++nposted;
    }
    if (dynamic && crank == 0 && lane == 0) {
      if (!over) claim = atomicAdd(a.counter, 1);  // no unit was claimed (cid >= n_units)
      // `claim` holds this cluster's over-claim now; the last of all resets the counter
      if (claim == n_dyn + ncl_eff - 1) *a.counter = 0;
    }
    {
      const uint32_t q = take_slot();
      if (lane == 0) {
        units[q].end = 1;
        mbar_arrive(smem_u32(&unit_full[q]));
      }
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else if (warp == kGProd || warp == kGProd2 || warp == kGProd3) {
    // ---------------- producers ----------------
    // The producer warps walk the same units and stages; a stage's copies
    // (adapter rows, then token rows) go round them, copy i to producer
    // i % kGProds, since one warp alone issues bulk copies too slowly to keep
    // the memory system busy.  Each arrives on the stage barrier with the bytes
    // of its own copies; producer 0 writes the stage's record.
    const int pi = warp == kGProd ? 0 : warp == kGProd2 ? 1 : 2;
    uint32_t g = 0;  // stages posted
    auto take_stage = [&]() -> uint32_t {
      const uint32_t st = g % kStages;
      if (g >= kStages && !mbar_wait(smem_u32(&empty[st]), ((g / kStages) - 1) & 1)) ok = false;
      return st;
    };
    // a record without data
    auto post_record = [&](const GRec& rc) {
      const uint32_t st = take_stage();
      if (lane == 0) {
        if (pi == 0) recs[st] = rc;
        mbar_arrive(smem_u32(&full[st]));
      }
      ++g;
    };
    for (uint32_t nu = 0; ok; ++nu) {
      const uint32_t q = nu % kUSlots;
      if (!mbar_wait(smem_u32(&unit_full[q]), (nu / kUSlots) & 1)) {
        ok = false;
        break;
      }
      const GUnit un = units[q];
      if (un.end) break;
      const GProj& P = projs[un.g];
      const DevView& v = P.v;
      const int shift = v.page_shift;
      const long long pmask = (1LL << shift) - 1;
      // this CTA's slices of d_in (shrink) and d_out (expand) for the unit's projection
      const int kc = ((v.d_in + (int)ncta - 1) / (int)ncta + 7) & ~7;
      const int nc = ((v.d_out + (int)ncta - 1) / (int)ncta + 7) & ~7;
      const int k0 = min(v.d_in, (int)crank * kc), k1 = min(v.d_in, k0 + kc);
      const int n0 = min(v.d_out, (int)crank * nc), n1 = min(v.d_out, n0 + nc);
      const int nks = (a.mode != kModeExpand && k1 > k0) ? (k1 - k0 + kSub - 1) / kSub : 0;
      const int nns = (a.mode != kModeShrink && n1 > n0) ? (n1 - n0 + kSub - 1) / kSub : 0;
      const int* pc = pgt + q * kMaxPgSlots;
      const int r = un.r, cnt = un.cnt;
      const long long na = un.na;
      const int njb = (r + kChunkRows - 1) / kChunkRows;
      for (int g0 = 0; g0 < cnt; g0 += kNT) {
        const int ntok = min(kNT, cnt - g0);
        const int mytok = g0 == 0 ? (lane < kNT ? units[q].tok[lane] : -1)
                                  : (lane < ntok ? a.perm[un.tb + g0 + lane] : -1);
        GRec rc{};
        rc.ntok = ntok;
        rc.r = r;
        rc.sc = un.sc;
        rc.g = un.g;
#pragma unroll
        for (int t = 0; t < kNT; ++t) rc.tok[t] = __shfl_sync(0xffffffffu, mytok, t);
        // One chunk: adapter rows [j0, j0 + nrows) of the sub-slice at col0,
        // with the group's x (shrink) or y0 (expand) rows of the same columns
        // when `tokens`.  Lane i copies row i as one bulk copy per page the
        // row run touches; the copies complete as transaction bytes on the
        // stage barrier.
        auto post_chunk = [&](int kind, int col0, int w, int j0, int nrows, bool tokens, int flags) {
          const uint32_t st = take_stage();
          const uint32_t sbase = smem_u32(sm + (size_t)st * kStageBytes);
          const uint32_t bar = smem_u32(&full[st]);
          const bool shrink = kind == kGShrink;
          const int ntr = tokens ? ntok : 0;
          const uint32_t rowb = (uint32_t)w * 2;
          const int ncopy = nrows + ntr;
          if (lane == 0) {
            if (pi == 0) {
              GRec r2 = rc;
              r2.kind = kind;
              r2.j0 = j0;
              r2.nrows = nrows;
              r2.nvec = w >> 3;
              r2.col0 = col0;
              r2.flags = flags;
              recs[st] = r2;
            }
            // copies pi, pi + kGProds, ...
            mbar_arrive_expect_tx(bar, (uint32_t)((ncopy + kGProds - 1 - pi) / kGProds) * rowb);
          }
          __syncwarp();
          const int idx = kGProds * lane + pi;  // this lane's copy of the stage
          const int tk = __shfl_sync(0xffffffffu, mytok, (idx - nrows) & (kNT - 1));
          if (idx < nrows) {
            const long long rowlen = shrink ? v.d_in : v.d_out;
            const long long page0 = shrink ? un.a_page0 : un.b_page0;
            const int pbase = shrink ? 0 : (int)na;
            long long e = (long long)(j0 + idx) * rowlen + col0;
            uint32_t dst = sbase + (uint32_t)(idx * kRowStride);
            for (int rem = w; rem > 0;) {
              const long long idx = e >> shift, off = e & pmask;
              const long long page = un.cached ? pc[pbase + idx] : v.page_list[page0 + idx];
              const int n = (int)min((long long)rem, (1LL << shift) - off);
              bulk_g2s(dst, v.pool + (page << shift) + off, (uint32_t)n * 2, bar);
              e += n;
              dst += (uint32_t)n * 2;
              rem -= n;
            }
          } else if (idx < ncopy) {
            const uint16_t* src = (shrink ? P.x + (long long)tk * P.ldx : P.y + (long long)tk * P.ldy) + col0;
            bulk_g2s(sbase + (uint32_t)((kChunkRows + idx - nrows) * kRowStride), src, rowb, bar);
          }
          ++g;
        };
        for (int jb = 0; jb < njb; ++jb) {
          for (int ks = 0; ks < nks; ++ks) {
            const int col0 = k0 + ks * kSub, w = min(kSub, k1 - col0);
            const int f = (ks == 0 ? kFFirst : 0) | (ks == nks - 1 ? kFLast : 0) |
                          (ks == nks - 1 && jb == njb - 1 ? kFRed : 0);
            post_chunk(kGShrink, col0, w, jb * kChunkRows, min(kChunkRows, r - jb * kChunkRows), true, f);
          }
        }
        if (reduce_h && nks == 0) {
          GRec red = rc;
          red.kind = kGReduce;
          red.flags = kFRed | kFNoK;
          post_record(red);
        }
        for (int ns = 0; ns < nns; ++ns) {
          const int col0 = n0 + ns * kSub, w = min(kSub, n1 - col0);
          for (int jb = 0; jb < njb; ++jb) {
            const bool last = jb == njb - 1;
            const int f = (jb == 0 ? kFFirst : 0) | (last ? kFLast : 0) | (!reduce_h && ns == 0 && jb == 0 ? kFHLoad : 0);
            post_chunk(kGExpand, col0, w, jb * kChunkRows, min(kChunkRows, r - jb * kChunkRows), last, f);
          }
        }
      }
      __syncwarp();  // every lane's last page-cache read is done
      if (lane == 0) mbar_arrive(smem_u32(&unit_empty[q]));
    }
    {
      GRec end{};
      end.kind = kGEnd;
      post_record(end);
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  } else {
    // ---------------- consumers ----------------
    const int ctid = tid;  // 0 .. 255
    float* const yf = a.yf;  // parameters the loop needs, read once up front
    const long long ldyf = a.ldyf;
    float* const hout = a.h;
    const long long ldh = a.ldh;
    const int mode = a.mode;
    uint32_t ngroup = 0, ncons = 0;
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};  // shrink: the lane's part of the row block's 16 x 8 tile
    float eacc[4][4];  // expand: the lane's parts of the warp's four 16 x 8 output tiles
#pragma unroll
    for (int i = 0; i < 4; ++i) eacc[i][0] = eacc[i][1] = eacc[i][2] = eacc[i][3] = 0.f;
    if (ordered) {  // classify the claimable units: four per thread, every load in flight
      int val[4];
      int gk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ctid + kGConsThreads * k, uu = ncl_eff + i;
        const int ub = uu / G;
        gk[k] = uu - ub * G;
        val[k] = i >= n_dyn ? -1 : ub < n_short ? a.short_units[ub] : a.long_units[2 * (ub - n_short)];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) val[k] = val[k] < 0 ? -1 : a.seg_adapter[val[k]];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const DevView& vk = projs[gk[k]].v;
        val[k] = val[k] < 0 || val[k] >= vk.n_adapters ? 0 : vk.adapters[val[k]].rank;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ctid + kGConsThreads * k;
        if (i < n_dyn) {
          const int nb = (val[k] + kChunkRows - 1) / kChunkRows;  // a bad adapter falls in the last class
          atomicOr(&cls[(nb > 2 ? 0 : nb == 2 ? 1 : 2) * 32 + (i >> 5)], 1u << (i & 31));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(cls_ready));
    }
    auto cons_sync = [&]() {  // the 8 consumer warps, bounded
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(cons));
      if (!mbar_wait(smem_u32(cons), ncons & 1)) ok = false;
      ++ncons;
    };
    for (uint32_t g = 0;; ++g) {
      const uint32_t st = g % kStages;
      if (!mbar_wait(smem_u32(&full[st]), (g / kStages) & 1)) {
        ok = false;
        break;
      }
      const GRec rc = load_rec(&recs[st]);  // in registers: every field is used below
      if (rc.kind == kGEnd) break;
      const uint8_t* sb = sm + (size_t)st * kStageBytes;
      const int b = ngroup & 1;
      if (rc.kind == kGShrink) {
        if (rc.flags & kFFirst) sacc[0] = sacc[1] = sacc[2] = sacc[3] = 0.f;
        shrink_chunk(smem_u32(sb), smem_u32(sb) + kChunkRows * kRowStride, rc.nvec * 8, rc.ntok, sacc, warp,
                     lane);
        if (rc.flags & kFLast) {  // the row block is done: the warp's partial of every row and token
          const int gr = lane >> 2, tq = lane & 3;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = gr + 8 * (e >> 1), t = 2 * tq + (e & 1);
            if (j < rc.nrows && t < rc.ntok) pw[(warp * kNT + t) * kHMax + rc.j0 + j] = sacc[e];
          }
        }
      }
      if (rc.flags & kFRed) {  // h of the group from the cluster's partials
        // Buffer b last held group ngroup - 2, which this CTA read before it
        // sent group ngroup - 1; no peer sends group ngroup before receiving that.
        cons_sync();  // every warp's partial is in, and every warp is done with the previous h
        const int q4 = (rc.r + 3) >> 2;  // 16-byte pieces of one token's partial
        const int nq = rc.ntok * q4;
        float* rb = recv + b * kMaxCluster * kNT * kHMax;
        const uint32_t bar = smem_u32(&recv_full[b]);
        if (ctid == 0) mbar_arrive_expect_tx(bar, (uint32_t)(ncta * nq * 16));
        if (ctid < nq) {
          // this CTA's partial (the warps' partials in warp order), pushed to
          // every CTA of the cluster, this one included
          const int t = ctid / q4, j = (ctid - t * q4) * 4;
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!(rc.flags & kFNoK)) {
#pragma unroll
            for (int w = 0; w < kGCons; ++w) {
              const float4 p = *reinterpret_cast<const float4*>(pw + (w * kNT + t) * kHMax + j);
              sum.x += p.x;
              sum.y += p.y;
              sum.z += p.z;
              sum.w += p.w;
            }
          }
          const uint32_t dst = smem_u32(rb + (crank * kNT + t) * kHMax + j);
          for (uint32_t c = 0; c < ncta; ++c) st_async_v4(mapa(dst, c), sum, mapa(bar, c));
        }
        if (!mbar_wait(bar, (ngroup >> 1) & 1)) ok = false;
        for (int i = ctid; i < rc.ntok * rc.r; i += kGConsThreads) {
          const int t = i / rc.r, j = i - t * rc.r;
          float sum = 0.f;  // in fixed CTA order
          for (uint32_t c = 0; c < ncta; ++c) sum += rb[(c * kNT + t) * kHMax + j];
          hs[t * kHMax + j] = mode == kModeApply ? rc.sc * sum : sum;
          // the unscaled h: the shrink's output, or, with an h array, the apply's intermediate too
          if ((mode == kModeShrink || (mode == kModeApply && hout != nullptr)) && ok && (uint32_t)t % ncta == crank)
            hout[(long long)recs[st].tok[t] * ldh + j] = sum;
        }
        cons_sync();  // h complete here
        ++ngroup;
      }
      if (rc.flags & kFHLoad) {  // h of the group from the caller
        cons_sync();  // every warp is done with the previous group's h
        for (int i = ctid; i < rc.ntok * rc.r; i += kGConsThreads) {
          const int t = i / rc.r, j = i - t * rc.r;
          hs[t * kHMax + j] = rc.sc * hout[(long long)recs[st].tok[t] * ldh + j];
        }
        cons_sync();
      }
      if (rc.kind == kGExpand)
        expand_chunk(projs[rc.g].y, projs[rc.g].ldy, yf, ldyf, smem_u32(sb), sb, hs, pw + warp * kNT * kHMax, eacc,
                     rc, ok, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    if (!ok && ctid == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  // No CTA may leave while a peer can still read its partials or arrive on
  // its barriers.
  cluster_sync();
}

// Cluster width.  CTA c of a cluster of w owns the c-th of w equal runs of
// d_in and of d_out, staged in kSub-column sub-slices, so a unit of one row
// block costs w * (sub-slices of a d_in run + of a d_out run) stages, and a
// stage costs the same hand-offs however few columns it carries.  The width is
// the one with the fewest stages per unit among w in [w0 / 2, w0], w0 the width
// whose runs are one sub-slice (at most kMaxCluster); ties go to the wider.
// For d = 5120 that is 5 CTAs of 1024 columns (8 CTAs of 640 would stage every
// row block as a 512- and a 128-column piece).
static int cluster_size_for(const lora_pool_view_t* const* views, int n) {
  int d = 0;
  for (int g = 0; g < n; ++g) d = std::max(d, std::max(views[g]->d_in, views[g]->d_out));
  const int w0 = std::min(std::max((d + kSub - 1) / kSub, 1), kMaxCluster);
  int best = w0;
  long long best_cost = -1;
  for (int w = w0; w >= std::max(1, w0 / 2); --w) {
    long long cost = 0;
    for (int g = 0; g < n; ++g) {
      const int kc = ((views[g]->d_in + w - 1) / w + 7) & ~7, nc = ((views[g]->d_out + w - 1) / w + 7) & ~7;
      cost += (long long)w * ((kc + kSub - 1) / kSub + (nc + kSub - 1) / kSub);
    }
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = w;
    }
  }
  return best;
}

lora_status_t launch_gather_multi(int mode, int src, int short_only, int n_proj, const ProjCall* projs, float* h,
                                  long long ldh, const lora_segments_t* seg, const int32_t* token_adapter, int T,
                                  int32_t* err, cudaStream_t stream) {
  if (n_proj < 1 || n_proj > kMaxFusedProj) return LORA_ERR_INVALID_ARG;
  GatherArgs a;
  memset(&a, 0, sizeof(a));
  const lora_pool_view_t* views[kMaxFusedProj];
  for (int g = 0; g < n_proj; ++g) {
    a.proj[g].x = static_cast<const uint16_t*>(projs[g].x);
    a.proj[g].ldx = projs[g].ldx;
    a.proj[g].y = static_cast<uint16_t*>(projs[g].y);
    a.proj[g].ldy = projs[g].ldy;
    make_dev_view(projs[g].view, &a.proj[g].v);
    views[g] = projs[g].view;
  }
  a.n_proj = n_proj;
  a.h = h;
  a.ldh = ldh;
  a.yf = projs[0].yf;
  a.ldyf = projs[0].ldyf;
  a.perm = seg ? seg->token_perm : nullptr;
  a.indptr = seg ? seg->seg_indptr : nullptr;
  a.seg_adapter = seg ? seg->seg_adapter : nullptr;
  a.short_units = seg ? seg->short_units : nullptr;
  a.long_units = seg ? seg->long_units : nullptr;
  a.meta = seg ? seg->meta : nullptr;
  a.counter = seg ? seg->meta + 7 : nullptr;
  a.token_adapter = token_adapter;
  a.T = T;
  a.err = err;
  a.mode = mode;
  a.src = src;
  a.short_only = short_only;
  a.probe = wait_probe_cycles();

  const int upper = (src == kSrcTokens ? T : seg->T + (short_only ? 0 : seg->max_long_units)) * n_proj;
  if (upper <= 0) return LORA_OK;
  if (ensure_smem_attr((const void*)gather_kernel, kGatherSmem) != cudaSuccess) return LORA_ERR_CUDA;
  // The widest cluster whose resident clusters take every unit at once
  // (halving from the width the slices want); if none does, the full width.
  const int cl0 = cluster_size_for(views, n_proj);
  int cl = cl0;
  for (int c = cl0; c >= 2; c /= 2) {
    if (upper <= max_active_clusters((const void*)gather_kernel, kGThreads, kGatherSmem, c)) {
      cl = c;
      break;
    }
  }
  const int cap = max_active_clusters((const void*)gather_kernel, kGThreads, kGatherSmem, cl);
  const int n_clusters = upper < cap ? upper : cap;
  return launch_pdl((const void*)gather_kernel, dim3((unsigned)(n_clusters * cl)), dim3(kGThreads), kGatherSmem,
                    stream, cl, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status_t launch_gather(int mode, int src, int short_only, const void* x, long long ldx, void* y, long long ldy,
                            float* h, long long ldh, const lora_segments_t* seg,
                            const int32_t* token_adapter, int T, const lora_pool_view_t* view,
                            int32_t* err, cudaStream_t stream, float* yf, long long ldyf) {
  const ProjCall p{x, ldx, y, ldy, yf, ldyf, view};
  return launch_gather_multi(mode, src, short_only, 1, &p, h, ldh, seg, token_adapter, T, err, stream);
}

}  // namespace lora

extern "C" int32_t lora_debug_gather_width(const lora_pool_view_t* views, int32_t n) {
  if (views == nullptr || n < 1 || n > lora::kMaxFusedProj) return -1;
  const lora_pool_view_t* v[lora::kMaxFusedProj];
  for (int g = 0; g < n; ++g) {
    if (views[g].d_in < 8 || views[g].d_out < 8) return -1;
    v[g] = &views[g];
  }
  return lora::cluster_size_for(v, n);
}

