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
// Two kernels:
//  shrink_tc  H[128, r] = X[128, d_in] . A_i^T.  A cluster of CL CTAs splits
//             d_in; each CTA streams 64-column chunks of the x tile and of A_i
//             (both K-major, 128-byte swizzle) through a 3-stage ring and
//             accumulates into tensor memory (M = 128, N = r padded to 16);
//             the partial H is reduced across the cluster through distributed
//             shared memory in fixed CTA order (deterministic) and written to h
//             (fp32, unscaled).
//  expand_tc  Y[128, n0:n0+128] = bf16(Y0 + (s_i H) . B_i[:, n0:n0+128]).
//             Work units are (tile, 128-column chunk), so the expand, which
//             carries two thirds of the bytes, spreads over every SM.  s_i H is
//             split into bf16 hi + lo parts (two MMAs accumulating into the
//             same fp32 tensor-memory columns), which keeps the rank-r
//             intermediate at about fp32 accuracy on bf16 tensor cores.  B_i
//             rows are MN-major operands (r_i rows of d_out contiguous
//             elements, as stored).  y0 rows arrive by 16-byte asynchronous
//             copies and y rows leave by coalesced 16-byte stores, both through
//             a padded staging tile in shared memory.
#include "internal.h"
#include "tc.cuh"

namespace lora {

constexpr int kTcThreads = 160;  // warps 0-3: loads + epilogue, warp 4: MMA issue
constexpr int kTM = LORA_TILE_M;  // 128
constexpr int kMaxClusterTc = 8;

// ---------------------------------------------------------------- shrink_tc --

constexpr int kSStages = 3;
constexpr int kSXBytes = kTM * 128;  // x tile: 128 rows x 64 bf16
constexpr int kSABytes = 64 * 128;   // A tile: up to 64 rank rows x 64 bf16
constexpr int kSStageBytes = kSXBytes + kSABytes;
constexpr int kSMaxChunks = 32;  // 64-column chunks per CTA
constexpr int kHPad = 68;        // fp32 row stride of the partial-H exchange buffer
constexpr size_t kSOffPages = (size_t)kSStages * kSStageBytes;
constexpr size_t kSOffTok = kSOffPages + 64 * kSMaxChunks * 4;
constexpr size_t kSOffBars = kSOffTok + kTM * 4;
constexpr size_t kShrinkSmem = kSOffBars + 16 * 8 + 1024;  // + alignment slack

struct TcArgs {
  const uint16_t* x;
  long long ldx;
  uint16_t* y;
  long long ldy;
  float* h;
  long long ldh;
  int h_by_token;  // h rows indexed by token (user h) or by segment position (scratch)
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* long_units;
  const int32_t* meta;
  int32_t* err;
};

// Validate adapter `ad` for use (rank, every page-list slot and page of A and
// B).  Returns 0 or LORA_DERR_* bits; all threads of the CTA get the verdict.
__device__ __forceinline__ int check_adapter(const DevView& v, int ad, lora_adapter_desc_t& d, int* flag) {
  d = v.adapters[ad];
  if (d.rank < 1 || d.rank > v.max_rank || d.rank > LORA_MAX_RANK) return LORA_DERR_BAD_RANK;
  const long long na = ((long long)d.rank * v.d_in + (1LL << v.page_shift) - 1) >> v.page_shift;
  const long long nb = ((long long)d.rank * v.d_out + (1LL << v.page_shift) - 1) >> v.page_shift;
  int mine = 0;
  for (long long i = threadIdx.x; i < na + nb; i += blockDim.x) {
    const long long slot = i < na ? d.a_page0 + i : d.b_page0 + (i - na);
    if (slot < 0 || slot >= v.n_page_list) {
      mine = 1;
    } else {
      const long long pg = v.page_list[slot];
      if (pg < 0 || pg >= v.n_pages) mine = 1;
    }
  }
  return __syncthreads_or(mine) ? LORA_DERR_BAD_PAGE : 0;
}

__global__ void __launch_bounds__(kTcThreads, 2) shrink_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  int* pgtab = reinterpret_cast<int*>(sm + kSOffPages);  // [64][kSMaxChunks] physical pages
  int* tok = reinterpret_cast<int*>(sm + kSOffTok);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSOffBars);
  uint64_t* full = bars;                  // [kSStages], 128 producer arrivals
  uint64_t* empty = bars + kSStages;      // [kSStages], one MMA commit
  uint64_t* acc_full = bars + 2 * kSStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kSStages + 2);
  float* hpart = reinterpret_cast<float*>(sm);  // aliases stages 0-1 once a tile's MMAs are done

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
  const uint32_t cid = cluster_id_x(), ncl = ncluster_x();

  if (tid == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(smem_u32(&full[s]), 128);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    fence_mbar_init();
  }
  if (warp == 4) tmem_alloc(smem_u32(tmem_slot), 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_then_release();

  // This CTA's slice of d_in, in whole 64-column chunks.
  const int kc = (((v.d_in + (int)ncta - 1) / (int)ncta) + 63) & ~63;
  const int k0 = min(v.d_in, (int)crank * kc);
  const int k1 = min(v.d_in, k0 + kc);
  const int nch = (k1 - k0) / 64;
  const int n_units = a.meta[3];
  uint32_t gchunk = 0;  // chunks streamed so far by this CTA (stage / phase bookkeeping)
  uint32_t nacc = 0;    // tiles accumulated so far
  bool ok = true;

  for (int u = (int)cid; u < n_units; u += (int)ncl) {
    const int s = a.long_units[2 * u], m0 = a.long_units[2 * u + 1];
    const int ad = a.seg_adapter[s];
    const int p0 = a.indptr[s] + m0;
    const int cnt = min(kTM, a.indptr[s + 1] - p0);
    if (tid < kTM) tok[tid] = tid < cnt ? a.perm[p0 + tid] : -1;
    lora_adapter_desc_t d;
    const int bad = check_adapter(v, ad, d, nullptr);  // includes a __syncthreads
    if (bad) {
      if (crank == 0 && tid == 0) report(a.err, bad);
      continue;  // the same verdict in every CTA of the cluster
    }
    const int r = d.rank;
    const int rpad = (r + 15) & ~15;
    // physical page of every (rank row, chunk) of this CTA's slice of A_i
    for (int i = tid; i < r * nch; i += kTcThreads) {
      const int j = i / nch, c = i - j * nch;
      const long long e = (long long)j * v.d_in + k0 + 64 * c;
      pgtab[j * kSMaxChunks + c] = v.page_list[d.a_page0 + (e >> v.page_shift)];
    }
    __syncthreads();

    if (warp < 4) {
      // ---- producers: cp.async 16-byte pieces into 128-byte-swizzled tiles ----
      const long long pmask = (1LL << v.page_shift) - 1;
      for (int c = 0; c < nch; ++c) {
        const uint32_t g = gchunk + c, st = g % kSStages, use = g / kSStages;
        if (use > 0 && !mbar_wait(smem_u32(&empty[st]), (use - 1) & 1)) ok = false;
        const uint32_t xs = smem_u32(sm + st * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
        const int kcol = k0 + 64 * c;
        for (int i = tid; i < kTM * 8; i += 128) {  // x: 128 rows x 8 pieces
          const int m = i >> 3, q = i & 7;
          const int t = tok[m];
          cp_async16(xs + sw128_offset(m, q), a.x + (long long)(t < 0 ? 0 : t) * a.ldx + kcol + 8 * q, t >= 0);
        }
        for (int i = tid; i < rpad * 8; i += 128) {  // A_i: rpad rows x 8 pieces, zero beyond r
          const int j = i >> 3, q = i & 7;
          const bool real = j < r;
          const long long e = real ? ((long long)j * v.d_in + kcol) : 0;
          const uint16_t* src = real ? v.pool + ((long long)pgtab[j * kSMaxChunks + c] << v.page_shift) + (e & pmask) + 8 * q
                                     : v.pool;
          cp_async16(as + sw128_offset(j, q), src, real);
        }
        cp_async_commit();
        if (c >= kSStages - 1) {
          cp_async_wait<kSStages - 1>();
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&full[(g - (kSStages - 1)) % kSStages]));
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (int c = max(0, nch - (kSStages - 1)); c < nch; ++c) mbar_arrive(smem_u32(&full[(gchunk + c) % kSStages]));
    } else if (lane == 0) {
      // ---- MMA issue: M = 128, N = rpad, K = 64 per chunk ----
      const uint32_t idesc = idesc_bf16(kTM, rpad, 0);
      for (int c = 0; c < nch; ++c) {
        const uint32_t g = gchunk + c, st = g % kSStages;
        if (!mbar_wait(smem_u32(&full[st]), (g / kSStages) & 1)) ok = false;
        tc_fence_after();
        const uint32_t xs = smem_u32(sm + st * kSStageBytes);
        const uint32_t as = xs + kSXBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, sdesc_sw128(xs + 32 * kk, 16, 1024), sdesc_sw128(as + 32 * kk, 16, 1024), idesc,
                   (c | kk) != 0);
        mma_commit(smem_u32(&empty[st]));
      }
      if (nch > 0) mma_commit(smem_u32(acc_full));
    }
    gchunk += nch;

    // ---- epilogue: partial H to shared memory, reduce across the cluster ----
    if (warp < 4) {
      const int m = warp * 32 + lane;
      if (nch > 0) {
        if (!mbar_wait(smem_u32(acc_full), nacc & 1)) ok = false;
        tc_fence_after();
        for (int c0 = 0; c0 < rpad; c0 += 16) {
          float vals[16];
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, vals);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(&hpart[m * kHPad + c0 + i]) = make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
        }
      } else {
        for (int c0 = 0; c0 < rpad; c0 += 4) *reinterpret_cast<float4*>(&hpart[m * kHPad + c0]) = make_float4(0, 0, 0, 0);
      }
      tc_fence_before();
    }
    if (nch > 0) ++nacc;
    cluster_sync();
    {
      // CTA crank reduces rows [rb0, rb1) over the cluster, in CTA order.
      const int rows_per = (kTM + (int)ncta - 1) / (int)ncta;
      const int rb0 = (int)crank * rows_per, rb1 = min(kTM, rb0 + rows_per);
      const int nq = rpad / 4;
      const uint32_t hbase = smem_u32(hpart);
      for (int i = tid; i < (rb1 - rb0) * nq; i += kTcThreads) {
        const int m = rb0 + i / nq, c4 = (i % nq) * 4;
        if (m >= cnt || c4 >= r) continue;
        const uint32_t off = (uint32_t)((m * kHPad + c4) * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t q = 0; q < ncta; ++q) {
          float4 p;
          asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
              : "=f"(p.x), "=f"(p.y), "=f"(p.z), "=f"(p.w)
              : "r"(mapa(hbase + off, q)));
          acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
        }
        if (ok) {
          const long long row = a.h_by_token ? tok[m] : p0 + m;
          float* dst = a.h + row * a.ldh + c4;
          const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
          for (int q = 0; q < 4 && c4 + q < r; ++q) dst[q] = vv[q];
        }
      }
    }
    cluster_sync();
  }
  if (!ok && tid == 0) report(a.err, LORA_DERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 4) tmem_dealloc(tmem, 64);
  cluster_sync();
}

// ---------------------------------------------------------------- expand_tc --

constexpr int kENC = 128;                    // output columns per work unit
constexpr int kEHBytes = kTM * 128;          // one H operand tile: 128 rows x 64 bf16
constexpr int kEBBytes = 64 * kENC * 2;      // B tile: up to 64 rank rows x 128 columns
constexpr int kEYRow = kENC * 2 + 16;        // padded staging row (bytes)
constexpr size_t kEOffHlo = kEHBytes;
constexpr size_t kEOffB = 2 * kEHBytes;
constexpr size_t kEOffY = kEOffB + kEBBytes;
constexpr size_t kEOffTok = kEOffY + (size_t)kTM * kEYRow;
constexpr size_t kEOffPg = kEOffTok + kTM * 4;
constexpr size_t kEOffBars = kEOffPg + 64 * 4;
constexpr size_t kExpandSmem = kEOffBars + 8 * 8 + 1024;

// Barrier among the 128 loader / epilogue threads (warps 0-3) only.
__device__ __forceinline__ void named_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kTcThreads, 2) expand_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* hhi = sm;
  uint8_t* hlo = sm + kEOffHlo;
  uint8_t* bt = sm + kEOffB;
  uint8_t* ys = sm + kEOffY;
  int* tok = reinterpret_cast<int*>(sm + kEOffTok);
  int* pgb = reinterpret_cast<int*>(sm + kEOffPg);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kEOffBars);
  uint64_t* bar_b = bars;       // 128 producer arrivals: B tile and H operand in place
  uint64_t* acc_full = bars + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  if (tid == 0) {
    mbar_init(smem_u32(bar_b), 128);
    mbar_init(smem_u32(acc_full), 1);
    fence_mbar_init();
  }
  if (warp == 4) tmem_alloc(smem_u32(tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_then_release();

  const int n_nc = v.d_out / kENC;
  const long long n_work = (long long)a.meta[3] * n_nc;
  const long long w0 = n_work * blockIdx.x / gridDim.x, w1 = n_work * (blockIdx.x + 1) / gridDim.x;
  int cur_tile = -1, r = 0, rpad = 16, cnt = 0, p0 = 0, tile_bad = 0;
  float sc = 0.f;
  lora_adapter_desc_t d;
  uint32_t nunit = 0;
  bool ok = true;
  const long long pmask = (1LL << v.page_shift) - 1;

  for (long long w = w0; w < w1; ++w) {
    const int tile = (int)(w / n_nc), ncc = (int)(w - (long long)tile * n_nc);
    const int n0 = ncc * kENC;
    if (tile != cur_tile) {
      cur_tile = tile;
      const int s = a.long_units[2 * tile], m0 = a.long_units[2 * tile + 1];
      const int ad = a.seg_adapter[s];
      p0 = a.indptr[s] + m0;
      cnt = min(kTM, a.indptr[s + 1] - p0);
      if (tid < kTM) tok[tid] = tid < cnt ? a.perm[p0 + tid] : -1;
      tile_bad = check_adapter(v, ad, d, nullptr);
      if (tile_bad) {
        if (tid == 0 && ncc == 0) report(a.err, tile_bad);
        continue;
      }
      r = d.rank;
      rpad = (r + 15) & ~15;
      sc = d.scale;
      // H operand, two bf16 parts of s * h: row m, rank column j (K-major,
      // 128-byte swizzle, one 64-column atom).  Zero beyond r and beyond cnt.
      if (warp < 4) {
        const int m = tid;
        const long long row = m < cnt ? (a.h_by_token ? tok[m] : p0 + m) : 0;
        for (int q = 0; q < rpad / 8; ++q) {
          float hv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = q * 8 + e;
            hv[e] = (m < cnt && j < r) ? sc * a.h[row * a.ldh + j] : 0.f;
          }
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = pack_bf16x2(hv[2 * e], hv[2 * e + 1]);
            lo[e] = pack_bf16x2(hv[2 * e] - bf_lo(hi[e]), hv[2 * e + 1] - bf_hi(hi[e]));
          }
          *reinterpret_cast<uint4*>(hhi + sw128_offset(m, q)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(hlo + sw128_offset(m, q)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();
      }
    } else if (tile_bad) {
      continue;
    }
    // physical page of each B row's 128-column chunk
    if (tid < r) {
      const long long e = (long long)tid * v.d_out + n0;
      pgb[tid] = v.page_list[d.b_page0 + (e >> v.page_shift)];
    }
    __syncthreads();

    if (warp < 4) {
      // y0 rows: 16-byte pieces, 16 consecutive threads per 256-byte row
      for (int i = tid; i < kTM * (kENC / 8); i += 128) {
        const int m = i / (kENC / 8), q = i % (kENC / 8);
        if (m < cnt)
          cp_async16(smem_u32(ys + m * kEYRow + q * 16), a.y + (long long)tok[m] * a.ldy + n0 + 8 * q);
      }
      // B rows: MN-major operand, 2 atoms of 64 columns, 8 rank rows per
      // 1024-byte group, 128-byte swizzle; zero beyond r.
      const int kg = rpad / 8;
      for (int i = tid; i < rpad * (kENC / 8); i += 128) {
        const int j = i / (kENC / 8), q16 = i % (kENC / 8);
        const int na = q16 >> 3, q = q16 & 7;
        const uint32_t dst = smem_u32(bt) + (uint32_t)((na * kg + (j >> 3)) * 1024) + sw128_offset(j & 7, q);
        const bool real = j < r;
        const long long e = real ? ((long long)j * v.d_out + n0) : 0;
        const uint16_t* src = real ? v.pool + ((long long)pgb[j] << v.page_shift) + (e & pmask) + 8 * q16 : v.pool;
        cp_async16(dst, src, real);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      named_sync_128();  // every loader's y0 pieces visible to every epilogue thread
      tc_fence_before();
      mbar_arrive(smem_u32(bar_b));
    } else if (lane == 0) {
      if (!mbar_wait(smem_u32(bar_b), nunit & 1)) ok = false;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kTM, 64, 1);
      const int kg = rpad / 8;
      for (int na = 0; na < kENC / 64; ++na) {
        const uint32_t bbase = smem_u32(bt) + (uint32_t)(na * kg * 1024);
        int first = 1;
        for (int part = 0; part < 2; ++part) {
          const uint32_t abase = smem_u32(part ? hlo : hhi);
          for (int ks = 0; ks < rpad / 16; ++ks) {
            mma_bf16(tmem + (uint32_t)(na * 64), sdesc_sw128(abase + 32 * ks, 16, 1024),
                     sdesc_sw128(bbase + (uint32_t)(ks * 2048), 0, 1024), idesc, first ? 0u : 1u);
            first = 0;
          }
        }
      }
      mma_commit(smem_u32(acc_full));
    }

    if (warp < 4) {
      const int m = tid;
      if (!mbar_wait(smem_u32(acc_full), nunit & 1)) ok = false;
      tc_fence_after();
      uint8_t* yrow = ys + m * kEYRow;
      for (int c0 = 0; c0 < kENC; c0 += 16) {
        float dv[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, dv);
        uint4* p = reinterpret_cast<uint4*>(yrow + c0 * 2);
        uint4 u0 = p[0], u1 = p[1];
        float y0[16];
        unpack8(u0, y0);
        unpack8(u1, y0 + 8);
        uint4 o0, o1;
        o0.x = pack_bf16x2(y0[0] + dv[0], y0[1] + dv[1]);
        o0.y = pack_bf16x2(y0[2] + dv[2], y0[3] + dv[3]);
        o0.z = pack_bf16x2(y0[4] + dv[4], y0[5] + dv[5]);
        o0.w = pack_bf16x2(y0[6] + dv[6], y0[7] + dv[7]);
        o1.x = pack_bf16x2(y0[8] + dv[8], y0[9] + dv[9]);
        o1.y = pack_bf16x2(y0[10] + dv[10], y0[11] + dv[11]);
        o1.z = pack_bf16x2(y0[12] + dv[12], y0[13] + dv[13]);
        o1.w = pack_bf16x2(y0[14] + dv[14], y0[15] + dv[15]);
        p[0] = o0;
        p[1] = o1;
      }
      tc_fence_before();
      named_sync_128();
      // y rows: 16 consecutive threads store one 256-byte row
      if (ok) {
        for (int i = tid; i < cnt * (kENC / 8); i += 128) {
          const int mm = i / (kENC / 8), q = i % (kENC / 8);
          *reinterpret_cast<uint4*>(a.y + (long long)tok[mm] * a.ldy + n0 + 8 * q) =
              *reinterpret_cast<const uint4*>(ys + mm * kEYRow + q * 16);
        }
      }
    }
    ++nunit;
    __syncthreads();
  }
  if (!ok && tid == 0) report(a.err, LORA_DERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 4) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- launchers --

bool tc_shrink_ok(const lora_pool_view_t* v) {
  const int cl = v->d_in >= 512 * kMaxClusterTc ? kMaxClusterTc : (v->d_in + 511) / 512;
  const int kc = (((v->d_in + cl - 1) / cl) + 63) & ~63;
  return v->d_in % 64 == 0 && v->page_elems >= 128 && kc / 64 <= kSMaxChunks;
}

bool tc_expand_ok(const lora_pool_view_t* v) { return v->d_out % kENC == 0 && v->page_elems >= kENC; }

static void fill_tc_args(TcArgs& a, const void* x, long long ldx, void* y, long long ldy, float* h, long long ldh,
                         int h_by_token, const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err) {
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.h_by_token = h_by_token;
  make_dev_view(view, &a.v);
  a.perm = seg->token_perm;
  a.indptr = seg->seg_indptr;
  a.seg_adapter = seg->seg_adapter;
  a.long_units = seg->long_units;
  a.meta = seg->meta;
  a.err = err;
}

lora_status_t launch_shrink_tc(const void* x, long long ldx, float* h, long long ldh, int h_by_token,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  TcArgs a;
  fill_tc_args(a, x, ldx, nullptr, 0, h, ldh, h_by_token, seg, view, err);
  const int cl = view->d_in >= 512 * kMaxClusterTc ? kMaxClusterTc : (view->d_in + 511) / 512;
  int cap = sm_count() * 2 / cl;
  if (cap < 1) cap = 1;
  const int n_clusters = seg->max_long_units < cap ? seg->max_long_units : cap;
  if (n_clusters <= 0) return LORA_OK;
  if (ensure_smem_attr((const void*)shrink_tc_kernel, kShrinkSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)shrink_tc_kernel, dim3((unsigned)(n_clusters * cl)), dim3(kTcThreads),
                    kShrinkSmem, stream, cl, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status_t launch_expand_tc(const float* h, long long ldh, int h_by_token, void* y, long long ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  TcArgs a;
  fill_tc_args(a, nullptr, 0, y, ldy, const_cast<float*>(h), ldh, h_by_token, seg, view, err);
  const long long upper = (long long)seg->max_long_units * (view->d_out / kENC);
  long long grid = sm_count() * 2;
  if (upper < grid) grid = upper;
  if (grid <= 0) return LORA_OK;
  if (ensure_smem_attr((const void*)expand_tc_kernel, kExpandSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)expand_tc_kernel, dim3((unsigned)grid), dim3(kTcThreads), kExpandSmem, stream,
                    0, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
