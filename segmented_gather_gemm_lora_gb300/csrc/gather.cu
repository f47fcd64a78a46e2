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
// work unit (an adapter and up to 8 of its tokens) at a time.  CTA c of the
// cluster owns the c-th slice of d_in for the shrink and the c-th slice of
// d_out for the expand, so every adapter byte and every activation byte is
// read once per unit:
//   shrink  partial_c[t, j] = sum_{k in slice c} x[t, k] * A_i[j, k]
//   reduce  h[t, j] = s_i * sum_c partial_c[t, j]   through distributed shared
//           memory, in fixed CTA order (deterministic; no float atomics)
//   expand  y[t, n] = bf16(y0[t, n] + sum_j h[t, j] * B_i[j, n]),  n in slice c
// The rank-r intermediate never leaves the chip.
//
// Data movement.  Adapter rows (translated page by page through the page
// table, "Multi-LoRA Serving in Production", section "Unified Paged Memory")
// and token rows are staged in shared memory by 16-byte asynchronous copies
// from every thread into a ring of stages, each completed through an mbarrier;
// the expand's B and y0 chunks are issued before the shrink's arithmetic
// finishes, so both phases' bytes are in flight together.
#include "common.cuh"
#include "internal.h"

namespace lora {

constexpr int kGThreads = 256;
constexpr int kStages = 4;
constexpr int kStageBytes = 16384;
constexpr int kNT = LORA_SHORT_MAX_TOKENS;  // tokens per group
constexpr int kHMax = LORA_MAX_RANK;
constexpr int kMaxCluster = 8;

struct GatherArgs {
  const uint16_t* x;
  long long ldx;
  uint16_t* y;
  long long ldy;
  float* h;
  long long ldh;
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* short_units;
  const int32_t* long_units;
  const int32_t* meta;
  const int32_t* token_adapter;
  int T;
  int32_t* err;
  int mode;
  int src;
  int short_only;
};

constexpr size_t kOffBars = (size_t)kStages * kStageBytes;
constexpr size_t kOffHp = kOffBars + kStages * 8;
constexpr size_t kOffHs = kOffHp + 2 * kNT * kHMax * sizeof(float);
constexpr size_t kOffTok = kOffHs + kNT * kHMax * sizeof(float);
constexpr int kMaxPgSlots = 1024;  // page-list slots of one adapter cached in shared memory
constexpr size_t kOffPgt = kOffTok + kNT * sizeof(int) + 64;
constexpr size_t kGatherSmem = kOffPgt + kMaxPgSlots * sizeof(int);

// Elements per row of one stage: the stage holds up to max_rank adapter rows
// and up to kNT token rows.  A function of the view's max_rank alone, so a
// token's arithmetic depends neither on how many tokens share its unit nor on
// its adapter's rank (zero-padding an adapter does not change its result).
__device__ __forceinline__ int chunk_width(int r) {
  int w = ((kStageBytes / 2) / (r + kNT)) & ~7;
  return w < 8 ? 8 : w;
}

struct ChunkPlan {
  int r, ntok, nkc, nnc, wk, wn, k0, k1, n0, n1;
  int a_page0, b_page0;
  int na;          // page-list slots of A_i (B_i's follow in the cached table)
  const int* pgt;  // cached physical pages of A_i then B_i, or null
};

// Stage chunk c (shrink chunks first, then expand chunks) into `stage`: every
// thread of the CTA copies 16-byte pieces with cp.async (the load/store units
// issue these in parallel; one TMA bulk copy per row costs tens of
// nanoseconds of issue each, far too slow for rows of a few hundred bytes)
// and then arrives on `bar` when its own pieces have landed.
__device__ __forceinline__ void issue_chunk(const GatherArgs& a, const ChunkPlan& p, const int* tok,
                                            int c, uint8_t* stage, uint32_t bar, int tid) {
  const bool shrink = c < p.nkc;
  const int stride = shrink ? p.wk : p.wn;
  const int cols = shrink ? p.k0 + c * p.wk : p.n0 + (c - p.nkc) * p.wn;
  const int w = shrink ? min(p.wk, p.k1 - cols) : min(p.wn, p.n1 - cols);
  const long long rowlen = shrink ? a.v.d_in : a.v.d_out;
  const long long page0 = shrink ? p.a_page0 : p.b_page0;
  const uint16_t* act = shrink ? a.x : a.y;
  const long long ld = shrink ? a.ldx : a.ldy;
  const int shift = a.v.page_shift;
  const long long pmask = (1LL << shift) - 1;
  const uint32_t sbase = smem_u32(stage);
  const int nq = w >> 3;  // 16-byte pieces per row
  const int warp = tid >> 5, lane = tid & 31;
  for (int item = warp; item < p.r + p.ntok; item += kGThreads / 32) {
    const uint32_t drow = sbase + (uint32_t)(item * stride * 2);
    if (item < p.r) {
      const long long e0 = (long long)item * rowlen + cols;  // first element of the row piece
      for (int q = lane; q < nq; q += 32) {
        const long long e = e0 + 8 * q;
        const long long idx = e >> shift;
        const long long page = p.pgt ? p.pgt[(shrink ? 0 : p.na) + idx] : a.v.page_list[page0 + idx];
        const uint16_t* src = a.v.pool + (page << shift) + (e & pmask);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(drow + 16 * q), "l"(src) : "memory");
      }
    } else {
      const uint16_t* src0 = act + (long long)tok[item - p.r] * ld + cols;
      for (int q = lane; q < nq; q += 32)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(drow + 16 * q), "l"(src0 + 8 * q) : "memory");
    }
  }
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Partial shrink of one staged chunk for NT tokens: warp w takes rank rows
// j = w, w + 8, ...; its lanes take 8-element vectors of the chunk; the row's
// dot products with every token are reduced over the warp and added to the
// CTA's partial h.  Instantiated per token count so that a one-token decode
// unit executes only its own arithmetic.
template <int NT>
__device__ __forceinline__ void shrink_chunk(const uint8_t* sb, const ChunkPlan& p, int nvec, float* hpb, int warp,
                                             int lane) {
  for (int j = warp; j < p.r; j += kGThreads / 32) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    const uint4* arow = reinterpret_cast<const uint4*>(sb + (size_t)j * p.wk * 2);
    const uint4* xrow = reinterpret_cast<const uint4*>(sb + (size_t)p.r * p.wk * 2);
    const int xstride = p.wk / 8;  // uint4 per staged row
    for (int vv = lane; vv < nvec; vv += 32) {
      float af[8];
      unpack8(arow[vv], af);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float xf[8];
        unpack8(xrow[t * xstride + vv], xf);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t] = fmaf(af[q], xf[q], acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t) hpb[t * kHMax + j] += acc[t];
    }
  }
}

__global__ void __launch_bounds__(kGThreads, 3) gather_kernel(const __grid_constant__ GatherArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  float* hp = reinterpret_cast<float*>(sm + kOffHp);
  float* hs = reinterpret_cast<float*>(sm + kOffHs);
  int* tok = reinterpret_cast<int*>(sm + kOffTok);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
  const uint32_t cid = cluster_id_x(), ncl = ncluster_x();
  const DevView& v = a.v;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[s]), kGThreads);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait_then_release();

  // kSrcSegments walks the short units, then the long tiles, in one launch.
  const int n_short = a.src == kSrcSegments ? a.meta[2] : 0;
  const int n_units = a.src == kSrcTokens ? a.T : a.meta[2] + (a.short_only ? 0 : a.meta[3]);
  const int kc = ((v.d_in + (int)ncta - 1) / (int)ncta + 7) & ~7;
  const int nc = ((v.d_out + (int)ncta - 1) / (int)ncta + 7) & ~7;
  const int k0 = min(v.d_in, (int)crank * kc), k1 = min(v.d_in, k0 + kc);
  const int n0 = min(v.d_out, (int)crank * nc), n1 = min(v.d_out, n0 + nc);
  uint32_t parity = 0;  // bit s: parity of stage s's next phase
  int gbuf = 0;

  int* pgt = reinterpret_cast<int*>(sm + kOffPgt);
  for (int u = (int)cid; u < n_units; u += (int)ncl) {
    int ad, tb = 0, cnt;
    if (a.src == kSrcTokens) {
      ad = a.token_adapter[u];
      cnt = 1;
      if (ad == -1) continue;
      if (ad < -1 || ad >= v.n_adapters) {
        if (crank == 0 && tid == 0) report(a.err, LORA_DERR_BAD_ADAPTER);
        continue;
      }
    } else if (u < n_short) {
      const int s = a.short_units[u];
      ad = a.seg_adapter[s];
      tb = a.indptr[s];
      cnt = a.indptr[s + 1] - tb;
    } else {
      const int s = a.long_units[2 * (u - n_short)];
      const int m0 = a.long_units[2 * (u - n_short) + 1];
      ad = a.seg_adapter[s];
      tb = a.indptr[s] + m0;
      cnt = min(LORA_TILE_M, a.indptr[s + 1] - tb);
    }
    // The first group's token indices do not depend on the adapter: load them
    // alongside its descriptor.
    const int first_tok = tid < min(kNT, cnt) ? (a.src == kSrcTokens ? u : a.perm[tb + tid]) : -1;
    const lora_adapter_desc_t d = v.adapters[ad];
    // Every CTA checks the whole adapter, so all reach the same verdict without
    // talking to each other; the same pass caches the physical pages.
    int bad = 0;
    long long na = 0, nb = 0;
    bool cached = false;
    if (d.rank < 1 || d.rank > v.max_rank || d.rank > kHMax) {
      bad = LORA_DERR_BAD_RANK;
    } else {
      const long long P = 1LL << v.page_shift;
      na = ((long long)d.rank * v.d_in + P - 1) >> v.page_shift;
      nb = ((long long)d.rank * v.d_out + P - 1) >> v.page_shift;
      cached = na + nb <= kMaxPgSlots;
      int mine = 0;
      for (long long i = tid; i < na + nb; i += kGThreads) {
        const long long slot = i < na ? d.a_page0 + i : d.b_page0 + (i - na);
        long long pg = -1;
        if (slot < 0 || slot >= v.n_page_list) {
          mine = 1;
        } else {
          pg = v.page_list[slot];
          if (pg < 0 || pg >= v.n_pages) mine = 1;
        }
        if (cached) pgt[i] = (int)pg;
      }
      if (__syncthreads_or(mine)) bad = LORA_DERR_BAD_PAGE;
    }
    if (bad) {
      if (crank == 0 && tid == 0) report(a.err, bad);
      continue;
    }

    ChunkPlan p;
    p.r = d.rank;
    p.wk = chunk_width(v.max_rank);
    p.wn = p.wk;
    p.k0 = k0; p.k1 = k1; p.n0 = n0; p.n1 = n1;
    p.nkc = (a.mode != kModeExpand && k1 > k0) ? (k1 - k0 + p.wk - 1) / p.wk : 0;
    p.nnc = (a.mode != kModeShrink && n1 > n0) ? (n1 - n0 + p.wn - 1) / p.wn : 0;
    p.a_page0 = d.a_page0;
    p.b_page0 = d.b_page0;
    p.na = (int)na;
    p.pgt = cached ? pgt : nullptr;
    const float sc = d.scale;

    for (int g0 = 0; g0 < cnt; g0 += kNT) {
      p.ntok = min(kNT, cnt - g0);
      const int ntok = p.ntok;
      if (tid < ntok) tok[tid] = g0 == 0 ? first_tok : a.perm[tb + g0 + tid];
      float* hpb = hp + gbuf * kNT * kHMax;
      for (int i = tid; i < kNT * kHMax; i += kGThreads) hpb[i] = 0.f;
      __syncthreads();

      const int nch = p.nkc + p.nnc;
      for (int c = 0; c < min(kStages, nch); ++c)
        issue_chunk(a, p, tok, c, sm + (size_t)c * kStageBytes, smem_u32(&bars[c]), tid);
      bool ok = true;

      // ---- shrink: partial h over this CTA's d_in slice ----
      for (int c = 0; c < p.nkc; ++c) {
        const int st = c % kStages;
        if (!mbar_wait(smem_u32(&bars[st]), (parity >> st) & 1u)) ok = false;
        parity ^= 1u << st;
        const uint8_t* sb = sm + (size_t)st * kStageBytes;
        const int cols = p.k0 + c * p.wk;
        const int w = min(p.wk, p.k1 - cols);
        const int nvec = w >> 3;
        switch (ntok) {
          case 1: shrink_chunk<1>(sb, p, nvec, hpb, warp, lane); break;
          case 2: shrink_chunk<2>(sb, p, nvec, hpb, warp, lane); break;
          case 3: shrink_chunk<3>(sb, p, nvec, hpb, warp, lane); break;
          case 4: shrink_chunk<4>(sb, p, nvec, hpb, warp, lane); break;
          case 5: shrink_chunk<5>(sb, p, nvec, hpb, warp, lane); break;
          case 6: shrink_chunk<6>(sb, p, nvec, hpb, warp, lane); break;
          case 7: shrink_chunk<7>(sb, p, nvec, hpb, warp, lane); break;
          default: shrink_chunk<8>(sb, p, nvec, hpb, warp, lane); break;
        }
        __syncthreads();
        if (c + kStages < nch)
          issue_chunk(a, p, tok, c + kStages, sm + (size_t)st * kStageBytes, smem_u32(&bars[st]), tid);
      }

      // ---- h: cluster reduction (apply / shrink) or load (expand) ----
      if (a.mode != kModeExpand) {
        cluster_sync();
        const uint32_t hp_addr = smem_u32(hpb);
        for (int i = tid; i < ntok * p.r; i += kGThreads) {
          const int t = i / p.r, j = i - t * p.r;
          const uint32_t off = (uint32_t)((t * kHMax + j) * sizeof(float));
          // all peers' loads in flight first, then the sum in fixed CTA order
          float part[kMaxCluster];
#pragma unroll
          for (int c = 0; c < kMaxCluster; ++c)
            part[c] = (uint32_t)c < ncta ? ld_dsmem_f32(mapa(hp_addr + off, (uint32_t)c)) : 0.f;
          float sum = 0.f;
#pragma unroll
          for (int c = 0; c < kMaxCluster; ++c)
            if ((uint32_t)c < ncta) sum += part[c];
          hs[t * kHMax + j] = a.mode == kModeApply ? sc * sum : sum;
        }
        __syncthreads();
        if (a.mode == kModeShrink && ok) {
          for (int i = tid; i < ntok * p.r; i += kGThreads) {
            const int t = i / p.r, j = i - t * p.r;
            if ((uint32_t)t % ncta == crank) a.h[(long long)tok[t] * a.ldh + j] = hs[t * kHMax + j];
          }
        }
      } else {
        for (int i = tid; i < ntok * p.r; i += kGThreads) {
          const int t = i / p.r, j = i - t * p.r;
          hs[t * kHMax + j] = sc * a.h[(long long)tok[t] * a.ldh + j];
        }
        __syncthreads();
      }

      // ---- expand: y over this CTA's d_out slice ----
      for (int c = p.nkc; c < nch; ++c) {
        const int st = c % kStages;
        if (!mbar_wait(smem_u32(&bars[st]), (parity >> st) & 1u)) ok = false;
        parity ^= 1u << st;
        const uint8_t* sb = sm + (size_t)st * kStageBytes;
        const int cols = p.n0 + (c - p.nkc) * p.wn;
        const int w = min(p.wn, p.n1 - cols);
        const int nvec = w >> 3;
        // Eight consecutive lanes share one (token, 8-column vector); lane jq
        // sums rank rows j = jq, jq + 8, ... in ascending order and the eight
        // partial sums meet in a fixed butterfly.  The order depends neither on
        // the unit's token count nor on the adapter's rank.
        const int items = ntok * nvec * 8;
        for (int base = 0; base < items; base += kGThreads) {
          const int it = base + tid;
          const bool act = it < items;
          const int jq = it & 7, tv = it >> 3;
          const int t = act ? tv / nvec : 0, vv = act ? tv - t * nvec : 0;
          float o[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = 0.f;
          if (act) {
            for (int j = jq; j < p.r; j += 8) {
              const float hj = hs[t * kHMax + j];
              float bf[8];
              unpack8(reinterpret_cast<const uint4*>(sb + (size_t)j * p.wn * 2)[vv], bf);
#pragma unroll
              for (int q = 0; q < 8; ++q) o[q] = fmaf(hj, bf[q], o[q]);
            }
          }
#pragma unroll
          for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] += __shfl_xor_sync(0xffffffffu, o[q], m);
          }
          if (act && jq == 0 && ok) {
            float yf[8];
            unpack8(reinterpret_cast<const uint4*>(sb + (size_t)(p.r + t) * p.wn * 2)[vv], yf);
            uint4 out;
            out.x = pack_bf16x2(yf[0] + o[0], yf[1] + o[1]);
            out.y = pack_bf16x2(yf[2] + o[2], yf[3] + o[3]);
            out.z = pack_bf16x2(yf[4] + o[4], yf[5] + o[5]);
            out.w = pack_bf16x2(yf[6] + o[6], yf[7] + o[7]);
            *reinterpret_cast<uint4*>(a.y + (long long)tok[t] * a.ldy + cols + vv * 8) = out;
          }
        }
        __syncthreads();
        if (c + kStages < nch)
          issue_chunk(a, p, tok, c + kStages, sm + (size_t)st * kStageBytes, smem_u32(&bars[st]), tid);
      }
      if (!ok && tid == 0) report(a.err, LORA_DERR_TIMEOUT);
      gbuf ^= 1;
    }
  }
  // No CTA may leave while a peer can still read its partials.
  cluster_sync();
}

static int cluster_size_for(const lora_pool_view_t* view) {
  const int d = view->d_in > view->d_out ? view->d_in : view->d_out;
  int cl = (d + 511) / 512;
  if (cl < 1) cl = 1;
  if (cl > kMaxCluster) cl = kMaxCluster;
  return cl;
}

lora_status_t launch_gather(int mode, int src, int short_only, const void* x, long long ldx, void* y, long long ldy,
                            float* h, long long ldh, const lora_segments_t* seg,
                            const int32_t* token_adapter, int T, const lora_pool_view_t* view,
                            int32_t* err, cudaStream_t stream) {
  GatherArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  make_dev_view(view, &a.v);
  a.perm = seg ? seg->token_perm : nullptr;
  a.indptr = seg ? seg->seg_indptr : nullptr;
  a.seg_adapter = seg ? seg->seg_adapter : nullptr;
  a.short_units = seg ? seg->short_units : nullptr;
  a.long_units = seg ? seg->long_units : nullptr;
  a.meta = seg ? seg->meta : nullptr;
  a.token_adapter = token_adapter;
  a.T = T;
  a.err = err;
  a.mode = mode;
  a.src = src;
  a.short_only = short_only;

  const int upper = src == kSrcTokens ? T : seg->T + (short_only ? 0 : seg->max_long_units);
  if (upper <= 0) return LORA_OK;
  const int cl = cluster_size_for(view);
  int cap = sm_count() * 3 / cl;
  if (cap < 1) cap = 1;
  const int n_clusters = upper < cap ? upper : cap;

  if (ensure_smem_attr((const void*)gather_kernel, kGatherSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)gather_kernel, dim3((unsigned)(n_clusters * cl)), dim3(kGThreads), kGatherSmem,
                    stream, cl, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
