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
// work unit (an adapter and up to 8 of its tokens, in groups of 4) at a time.  CTA c of the
// cluster owns the c-th slice of d_in for the shrink and the c-th slice of
// d_out for the expand, so every adapter byte and every activation byte is
// read once per unit:
//   shrink  partial_c[t, j] = sum_{k in slice c} x[t, k] * A_i[j, k]
//   reduce  h[t, j] = s_i * sum_c partial_c[t, j]   through distributed shared
//           memory, in fixed CTA order (deterministic; no float atomics)
//   expand  y[t, n] = bf16(y0[t, n] + sum_j h[t, j] * B_i[j, n]),  n in slice c
// The rank-r intermediate never leaves the chip.
//
// Data movement.  A slice is cut into sub-slices of 512 columns and each
// sub-slice into chunks of 16 adapter rows, so every staged row is a 1 KB run
// (translated 16 bytes at a time through the page table, "Multi-LoRA Serving
// in Production", section "Unified Paged Memory"), staged together with the
// unit's token rows for the same columns.  Every thread copies 16-byte pieces
// with cp.async, one warp per row (512 bytes per instruction), into a ring of
// three stages, each completed through an mbarrier; expand chunks are issued
// as soon as stages free up, so the two phases' bytes overlap.  Rows of 1 KB are
// what keeps a streaming multiprocessor near its share of HBM bandwidth;
// rows of a few hundred bytes fall to a half or less.
//
// Summation order.  Each rank row's shrink dot product over a sub-slice and
// each output's expand sum over a 16-row chunk are fixed functions of column
// and row positions, and partial results combine in sub-slice / chunk order.
// A token's result therefore depends neither on how many tokens share its unit
// nor on its adapter's rank: zero-padding an adapter or moving a token between
// units changes no bit of its output.
#include "common.cuh"
#include "internal.h"

namespace lora {

constexpr int kGThreads = 256;
constexpr int kNT = 4;  // tokens per group (a unit of up to 8 tokens runs in two groups)
constexpr int kHMax = LORA_MAX_RANK;
constexpr int kMaxCluster = 8;
constexpr int kSub = 512;                      // columns per sub-slice (one 1 KB row)
constexpr int kChunkRows = 16;                 // adapter rows per chunk
constexpr int kRowBytes = kSub * 2;
constexpr int kStages = 3;
constexpr int kStageBytes = (kChunkRows + kNT) * kRowBytes;  // 20 KB
constexpr int kMaxPgSlots = 512;  // page-list slots of one adapter cached in shared memory

constexpr size_t kOffBars = (size_t)kStages * kStageBytes;
constexpr size_t kOffEacc = kOffBars + 64;                                  // fp32 [kNT][kSub]
constexpr size_t kOffHp = kOffEacc + (size_t)kNT * kSub * sizeof(float);    // fp32 [2][kNT][kHMax]
constexpr size_t kOffHs = kOffHp + 2 * kNT * kHMax * sizeof(float);         // fp32 [kNT][kHMax]
constexpr size_t kOffTok = kOffHs + kNT * kHMax * sizeof(float);
constexpr size_t kOffPgt = kOffTok + kNT * sizeof(int) + 32;
constexpr size_t kGatherSmem = kOffPgt + kMaxPgSlots * sizeof(int);

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

// One unit's chunk schedule: shrink chunks (sub-slice ks, row block jb) first,
// then expand chunks (sub-slice ns, row block jb).
struct ChunkPlan {
  int r, ntok, njb;  // rank, tokens, row blocks of kChunkRows
  int nks, nns;      // sub-slices of the d_in / d_out slices (0 if the phase is skipped)
  int k0, k1, n0, n1;
  int a_page0, b_page0;
  int na;            // page-list slots of A_i (B_i's follow in the cached table)
  const int* pgt;    // cached physical pages of A_i then B_i, or null
};

// Stage chunk c into `stage`: adapter rows [16 jb, 16 jb + 16) of the chunk's
// sub-slice at rows 0..15, then the unit's token rows (x for the shrink, y0
// for the expand) of the same columns at rows 16..23.  One warp per row,
// 16-byte pieces per lane; every thread then arrives on `bar` once its own
// pieces have landed.
__device__ __forceinline__ void issue_chunk(const GatherArgs& a, const ChunkPlan& p, const int* tok, int c,
                                            uint8_t* stage, uint32_t bar, int tid) {
  const int nsh = p.nks * p.njb;
  const bool shrink = c < nsh;
  const int cc = shrink ? c : c - nsh;
  const int sub = cc / p.njb, jb = cc - sub * p.njb;
  const int col0 = shrink ? p.k0 + sub * kSub : p.n0 + sub * kSub;
  const int w = shrink ? min(kSub, p.k1 - col0) : min(kSub, p.n1 - col0);
  const int j0 = jb * kChunkRows, nrows = min(kChunkRows, p.r - j0);
  const long long rowlen = shrink ? a.v.d_in : a.v.d_out;
  const long long page0 = shrink ? p.a_page0 : p.b_page0;
  const uint16_t* act = shrink ? a.x : a.y;
  const long long ld = shrink ? a.ldx : a.ldy;
  const int shift = a.v.page_shift;
  const long long pmask = (1LL << shift) - 1;
  const uint32_t sbase = smem_u32(stage);
  const int nq = w >> 3;  // 16-byte pieces per row
  const int warp = tid >> 5, lane = tid & 31;
  for (int item = warp; item < nrows + p.ntok; item += kGThreads / 32) {
    const bool adapter_row = item < nrows;
    const uint32_t drow = sbase + (uint32_t)((adapter_row ? item : kChunkRows + item - nrows) * kRowBytes);
    if (adapter_row) {
      const long long e0 = (long long)(j0 + item) * rowlen + col0;
      for (int q = lane; q < nq; q += 32) {
        const long long e = e0 + 8 * q;
        const long long idx = e >> shift;
        const long long page = p.pgt ? p.pgt[(shrink ? 0 : p.na) + idx] : a.v.page_list[page0 + idx];
        const uint16_t* src = a.v.pool + (page << shift) + (e & pmask);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(drow + 16 * q), "l"(src) : "memory");
      }
    } else {
      const uint16_t* src0 = act + (long long)tok[item - nrows] * ld + col0;
      for (int q = lane; q < nq; q += 32)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(drow + 16 * q), "l"(src0 + 8 * q) : "memory");
    }
  }
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Shrink of one staged chunk for NT tokens: warp w takes the chunk's rows w
// and w + 8 together (one unpack of each token vector serves both); its lanes
// take fixed 8-column vectors of the sub-slice; each row's dot product with
// every token is reduced over the warp and added to the CTA's partial h
// (sub-slices in order).  Instantiated per token count so that a one-token
// decode unit executes only its own arithmetic.
template <int NT>
__device__ __forceinline__ void shrink_chunk(const uint8_t* sb, int j0, int nrows, int nvec, float* hpb,
                                             int warp, int lane) {
  const uint4* xrow = reinterpret_cast<const uint4*>(sb + kChunkRows * kRowBytes);
  const int i0 = warp, i1 = warp + kGThreads / 32;  // the warp's two rows (16-row chunks)
  const bool has0 = i0 < nrows, has1 = i1 < nrows;
  if (!has0) return;
  float acc0[NT], acc1[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc0[t] = acc1[t] = 0.f;
  const uint4* arow0 = reinterpret_cast<const uint4*>(sb + i0 * kRowBytes);
  const uint4* arow1 = reinterpret_cast<const uint4*>(sb + (has1 ? i1 : i0) * kRowBytes);
  for (int vv = lane; vv < nvec; vv += 32) {
    float a0[8], a1[8];
    unpack8(arow0[vv], a0);
    unpack8(arow1[vv], a1);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float xf[8];
      unpack8(xrow[t * (kRowBytes / 16) + vv], xf);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        acc0[t] = fmaf(a0[q], xf[q], acc0[t]);
        acc1[t] = fmaf(a1[q], xf[q], acc1[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc0[t] += __shfl_xor_sync(0xffffffffu, acc0[t], o);
      acc1[t] += __shfl_xor_sync(0xffffffffu, acc1[t], o);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      hpb[t * kHMax + j0 + i0] += acc0[t];
      if (has1) hpb[t * kHMax + j0 + i1] += acc1[t];
    }
  }
}

// Expand of one staged chunk.  A warp takes one (token, block of 8 output
// vectors): lane = 8 g + u handles vector u of the block for the chunk's rows
// 4 g .. 4 g + 3 (ascending), so each group of 8 lanes reads 128 contiguous
// bytes of one row (no bank conflicts); the four row-quarter sums meet in a
// fixed two-step butterfly, and chunk sums accumulate in chunk order in eacc.
// The sub-slice's last chunk adds y0 and writes y.
__device__ __forceinline__ void expand_chunk(const GatherArgs& a, const uint8_t* sb, const float* hs, float* eacc,
                                             const int* tok, int ntok, int nvec, int j0, int nrows, bool first,
                                             bool last, int col0, bool ok, int warp, int lane) {
  const int nblk = (nvec + 7) >> 3;
  const int g = lane >> 3, u = lane & 7;
  for (int wi = warp; wi < ntok * nblk; wi += kGThreads / 32) {
    const int t = wi / nblk, vv = (wi - t * nblk) * 8 + u;
    const bool act = vv < nvec;
    float o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = 0.f;
    if (act) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * g + k;
        if (i < nrows) {
          const float hj = hs[t * kHMax + j0 + i];
          float bf[8];
          unpack8(reinterpret_cast<const uint4*>(sb + i * kRowBytes)[vv], bf);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = fmaf(hj, bf[q], o[q]);
        }
      }
    }
#pragma unroll
    for (int m = 8; m < 32; m <<= 1) {
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] += __shfl_xor_sync(0xffffffffu, o[q], m);
    }
    if (act && g == 0) {
      float4* ea = reinterpret_cast<float4*>(eacc + (t * kSub + vv * 8));
      if (!first) {
        const float4 e0 = ea[0], e1 = ea[1];
        o[0] = e0.x + o[0]; o[1] = e0.y + o[1]; o[2] = e0.z + o[2]; o[3] = e0.w + o[3];
        o[4] = e1.x + o[4]; o[5] = e1.y + o[5]; o[6] = e1.z + o[6]; o[7] = e1.w + o[7];
      }
      if (!last) {
        ea[0] = make_float4(o[0], o[1], o[2], o[3]);
        ea[1] = make_float4(o[4], o[5], o[6], o[7]);
      } else if (ok) {
        float yf[8];
        unpack8(reinterpret_cast<const uint4*>(sb + (kChunkRows + t) * kRowBytes)[vv], yf);
        uint4 out;
        out.x = pack_bf16x2(yf[0] + o[0], yf[1] + o[1]);
        out.y = pack_bf16x2(yf[2] + o[2], yf[3] + o[3]);
        out.z = pack_bf16x2(yf[4] + o[4], yf[5] + o[5]);
        out.w = pack_bf16x2(yf[6] + o[6], yf[7] + o[7]);
        *reinterpret_cast<uint4*>(a.y + (long long)tok[t] * a.ldy + col0 + vv * 8) = out;
      }
    }
  }
}

__global__ void __launch_bounds__(kGThreads, 3) gather_kernel(const __grid_constant__ GatherArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  float* eacc = reinterpret_cast<float*>(sm + kOffEacc);
  float* hp = reinterpret_cast<float*>(sm + kOffHp);
  float* hs = reinterpret_cast<float*>(sm + kOffHs);
  int* tok = reinterpret_cast<int*>(sm + kOffTok);
  int* pgt = reinterpret_cast<int*>(sm + kOffPgt);

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
    p.njb = (p.r + kChunkRows - 1) / kChunkRows;
    p.k0 = k0; p.k1 = k1; p.n0 = n0; p.n1 = n1;
    p.nks = (a.mode != kModeExpand && k1 > k0) ? (k1 - k0 + kSub - 1) / kSub : 0;
    p.nns = (a.mode != kModeShrink && n1 > n0) ? (n1 - n0 + kSub - 1) / kSub : 0;
    p.a_page0 = d.a_page0;
    p.b_page0 = d.b_page0;
    p.na = (int)na;
    p.pgt = cached ? pgt : nullptr;
    const float sc = d.scale;
    const int nsh = p.nks * p.njb;
    const int nch = nsh + p.nns * p.njb;

    for (int g0 = 0; g0 < cnt; g0 += kNT) {
      p.ntok = min(kNT, cnt - g0);
      const int ntok = p.ntok;
      if (tid < ntok) tok[tid] = g0 == 0 ? first_tok : a.perm[tb + g0 + tid];
      float* hpb = hp + gbuf * kNT * kHMax;
      for (int i = tid; i < kNT * kHMax; i += kGThreads) hpb[i] = 0.f;
      __syncthreads();

      for (int c = 0; c < min(kStages, nch); ++c)
        issue_chunk(a, p, tok, c, sm + (size_t)c * kStageBytes, smem_u32(&bars[c]), tid);
      bool ok = true;

      // ---- shrink: partial h over this CTA's d_in slice ----
      for (int c = 0; c < nsh; ++c) {
        const int st = c % kStages;
        if (!mbar_wait(smem_u32(&bars[st]), (parity >> st) & 1u)) ok = false;
        parity ^= 1u << st;
        const uint8_t* sb = sm + (size_t)st * kStageBytes;
        const int ks = c / p.njb, jb = c - ks * p.njb;
        const int nvec = min(kSub, p.k1 - (p.k0 + ks * kSub)) >> 3;
        const int j0 = jb * kChunkRows, nrows = min(kChunkRows, p.r - j0);
        switch (ntok) {
          case 1: shrink_chunk<1>(sb, j0, nrows, nvec, hpb, warp, lane); break;
          case 2: shrink_chunk<2>(sb, j0, nrows, nvec, hpb, warp, lane); break;
          case 3: shrink_chunk<3>(sb, j0, nrows, nvec, hpb, warp, lane); break;
          default: shrink_chunk<4>(sb, j0, nrows, nvec, hpb, warp, lane); break;
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
      for (int c = nsh; c < nch; ++c) {
        const int st = c % kStages;
        if (!mbar_wait(smem_u32(&bars[st]), (parity >> st) & 1u)) ok = false;
        parity ^= 1u << st;
        const uint8_t* sb = sm + (size_t)st * kStageBytes;
        const int ns = (c - nsh) / p.njb, jb = (c - nsh) - ns * p.njb;
        const int col0 = p.n0 + ns * kSub;
        const int nvec = min(kSub, p.n1 - col0) >> 3;
        const int j0 = jb * kChunkRows, nrows = min(kChunkRows, p.r - j0);
        expand_chunk(a, sb, hs, eacc, tok, ntok, nvec, j0, nrows, jb == 0, jb == p.njb - 1, col0, ok, warp, lane);
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
