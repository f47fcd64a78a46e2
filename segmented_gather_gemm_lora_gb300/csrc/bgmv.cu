// Decode kernel: one token per thread-block cluster, for small adapters.
//
// "Multi-LoRA serving: the single translator with a thousand glossaries",
// section "SGMV: the kernel that holds it all up" (size-one segments take a
// batched gather path), and "Multi-LoRA Serving in Production", section
// "S-LoRA: MBGMV and MBGMM Kernels" (the decode form: every token gathers its
// own adapter, heterogeneous ranks unpadded).
//
// A decode call moves little (an adapter slice and a few KB of activations per
// CTA), so its time is a chain of latencies: the grid's start, the token's
// adapter id, its descriptor, its page list, the rows, the shrink, the cluster
// exchange, the expand.  This kernel shortens that chain and lets consecutive
// calls overlap:
//   - CTAs small enough (8 warps, about 38 KB of shared memory) that the next
//     call's CTAs are resident, with their set-up done, while this call runs;
//   - no record pipeline: a CTA holds its whole adapter slice, at most 16 rows,
//     so every copy is issued as soon as the page list is read, and B's rows
//     are prefetched into L2 then and copied into the same buffer once the
//     shrink is done with A's;
//   - the arithmetic of one token is a matrix-vector product, so it runs on the
//     CUDA cores (fp32 FMA, shuffle reductions), not the tensor cores;
//   - optionally (LORA_BGMV_STATIC_ADAPTERS) the adapter chain and A's copies
//     run before the kernel ahead of it on the stream has finished, and only
//     x, y0 and y wait for it.
//
// Work decomposition: the token's cluster has C CTAs, C = ceil(max(d_in,
// d_out) / 1024) (at most 8); CTA c owns slice c of d_in (shrink) and of d_out
// (expand), at most 1024 columns each (clusters of 8 CTAs of 512 columns
// measured 1-7 % slower for calls of 64-256 tokens, of 2 CTAs of 2048 columns
// slower still).  Each CTA pushes its partial h to every CTA of the cluster through
// distributed shared memory, and each adds the C partials in CTA order, so the
// result is deterministic and depends only on the token's row, its adapter and
// the projection's shape.  The sums are the exact fp32 ones (h not split into
// bf16 parts), so they differ from lora_apply's tensor-core sums by rounding
// only.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace lora {

namespace {

constexpr int kDHalves = 2;  // 512-column halves of a CTA's slice
constexpr int kDThreads = 128 * kDHalves;
constexpr int kDMaxRank = 16;    // the adapter's rows held at once
constexpr int kDMaxCols = 512 * kDHalves;   // columns of a CTA's slice of d_in or d_out
constexpr int kDRowStride = kDMaxCols * 2 + 16;  // bytes between staged rows
constexpr int kDMaxCluster = 8;
constexpr int kDMaxPg = 128;  // page-list slots of one adapter cached in shared memory (A's, then B's)
static_assert(kDMaxCols == 4 * kDThreads && kDMaxCols == 16 * 32 * kDHalves, "column ownership of the expand and the shrink");

// shared memory: adapter rows (A, then B) and the token's y0 row after them;
// the x row; page cache; this CTA's partial h; the cluster's partials; h; the
// verdict; four mbarriers
constexpr size_t kDOffBuf = 0;
constexpr size_t kDOffY0 = kDOffBuf + (size_t)kDMaxRank * kDRowStride;
constexpr size_t kDOffX = kDOffY0 + kDRowStride;
constexpr size_t kDOffPg = kDOffX + kDRowStride;
constexpr size_t kDOffPw = kDOffPg + kDMaxPg * sizeof(int);
constexpr size_t kDOffRecv = kDOffPw + kDHalves * kDMaxRank * sizeof(float);
constexpr size_t kDOffHs = kDOffRecv + kDMaxCluster * kDMaxRank * sizeof(float);
constexpr size_t kDOffInfo = kDOffHs + kDMaxRank * sizeof(float);
constexpr size_t kDOffBars = kDOffInfo + 8 * sizeof(int);
constexpr size_t kDSmem = kDOffBars + 4 * sizeof(uint64_t);
static_assert(kDOffY0 % 16 == 0 && kDOffX % 16 == 0 && kDOffBars % 8 == 0, "copy destinations and barriers");

struct BgmvArgs {
  const uint16_t* x;
  long long ldx;
  uint16_t* y;
  long long ldy;
  const int32_t* ids;
  DevView v;
  int32_t* err;
  int early;        // the adapter chain may run before the predecessor finishes
  long long probe;  // > 0: the timeout probe's wait limit in cycles
};

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// No release: nothing a peer reads is published through this barrier (the
// partials complete on mbarriers), so the arrive need not wait for this
// thread's stores to become visible.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Row j's part [e, e + w) of a paged matrix whose page-list slots (relative to
// the matrix's first) are cached in pg: one bulk copy per page the run touches,
// into dst, completing on bar; or, with bar == 0, an L2 prefetch of the same bytes.
__device__ __forceinline__ void copy_run(const DevView& v, const int* pg, long long e, int w, uint32_t dst,
                                         uint32_t bar) {
  const int shift = v.page_shift;
  const long long pmask = (1LL << shift) - 1;
  for (int rem = w; rem > 0;) {
    const long long off = e & pmask;
    const long long page = pg[e >> shift];
    const int n = (int)min((long long)rem, (1LL << shift) - off);
    const uint16_t* src = v.pool + (page << shift) + off;
    if (bar != 0u) bulk_g2s(dst, src, (uint32_t)n * 2, bar);
    else prefetch_l2(src, (uint32_t)n * 2);
    e += n;
    dst += (uint32_t)n * 2;
    rem -= n;
  }
}

__global__ void __launch_bounds__(kDThreads) bgmv_kernel(const __grid_constant__ BgmvArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* const buf = sm + kDOffBuf;
  const uint8_t* const y0row = sm + kDOffY0;
  int* const pg = reinterpret_cast<int*>(sm + kDOffPg);
  float* const pw = reinterpret_cast<float*>(sm + kDOffPw);
  float* const recv = reinterpret_cast<float*>(sm + kDOffRecv);
  float* const hs = reinterpret_cast<float*>(sm + kDOffHs);
  int* const info = reinterpret_cast<int*>(sm + kDOffInfo);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(sm + kDOffBars);
  const uint32_t bar_xy = smem_u32(&bars[0]);    // x and y0 rows
  const uint32_t bar_a = smem_u32(&bars[1]);     // A's rows
  const uint32_t bar_b = smem_u32(&bars[2]);     // B's rows
  const uint32_t bar_recv = smem_u32(&bars[3]);  // every CTA's partial h

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank(), C = cluster_nctarank();
  const int t = (int)cluster_id_x();  // the token
  const DevView& v = a.v;

  // this CTA's slices: C equal runs of d_in and of d_out, whole 16-byte pieces
  const int kc = ((v.d_in + (int)C - 1) / (int)C + 7) & ~7;
  const int nc = ((v.d_out + (int)C - 1) / (int)C + 7) & ~7;
  const int k0 = min(v.d_in, (int)crank * kc), k1 = min(v.d_in, k0 + kc);
  const int n0 = min(v.d_out, (int)crank * nc), n1 = min(v.d_out, n0 + nc);
  const int kw = k1 - k0, nw = n1 - n0;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    info[0] = 0;
    info[4] = 0;
  }
  // every barrier of every CTA initialised before any peer stores into it
  cluster_sync();
  bool ok = true;
  if (a.probe > 0) {  // the timeout probe: every CTA takes the exit of a wait that ran out
    __shared__ uint64_t probe_bar;
    __shared__ int probe_ok;
    if (tid == 0) probe_ok = wait_probe(&probe_bar, a.probe) ? 1 : 0;
    __syncthreads();
    ok = probe_ok != 0;
  }


  if (!a.early) grid_wait();
  if (warp == 0 && ok) {
    // The token's adapter: descriptor and every page slot, checked by every CTA
    // (so all reach the same verdict without talking), then A's rows of this
    // CTA's slice and an L2 prefetch of B's.  Global loads through L2 only.
    const int ad = __ldcg(a.ids + t);
    int bits = 0, active = 0, r = 0, na = 0;
    float sc = 0.f;
    if (ad < -1 || ad >= v.n_adapters) {
      bits = LORA_DERR_BAD_ADAPTER;
    } else if (ad >= 0) {
      // four 4-byte loads, in flight together (the descriptor array is only
      // 4-byte aligned by its type)
      const int* dp = reinterpret_cast<const int*>(v.adapters + ad);
      const int d0 = __ldcg(dp), d1 = __ldcg(dp + 1), d2 = __ldcg(dp + 2), d3 = __ldcg(dp + 3);
      r = d0;
      sc = __int_as_float(d1);
      const long long pa = v.swap_ab ? d3 : d2, pb = v.swap_ab ? d2 : d3;
      if (r < 1 || r > v.max_rank || r > kDMaxRank) {
        bits = LORA_DERR_BAD_RANK;
      } else {
        const long long P = 1LL << v.page_shift;
        na = (int)(((long long)r * v.d_in + P - 1) >> v.page_shift);
        const int nb = (int)(((long long)r * v.d_out + P - 1) >> v.page_shift);
        int mine = 0;
        for (int i = lane; i < na + nb; i += 32) {  // na + nb <= kDMaxPg (the host checked max_rank)
          const long long slot = i < na ? pa + i : pb + (i - na);
          const int p = (slot < 0 || slot >= v.n_page_list) ? -1 : __ldcg(v.page_list + slot);
          if (p < 0 || p >= v.n_pages) mine = 1;
          pg[i] = p;
        }
        if (__any_sync(0xffffffffu, mine)) bits = LORA_DERR_BAD_PAGE;
        else active = 1;
      }
    }
    if (lane == 0) info[4] = crank == 0 ? bits : 0;  // reported once the predecessor has finished
    __syncwarp();  // the page cache, written by every lane, before any lane reads it
    if (active) {
      if (lane == 0) mbar_arrive_expect_tx(bar_a, (uint32_t)(r * kw * 2));
      __syncwarp();
      if (lane < r && kw > 0)
        copy_run(v, pg, (long long)lane * v.d_in + k0, kw, smem_u32(buf + lane * kDRowStride), bar_a);
      if (lane < r && nw > 0) copy_run(v, pg + na, (long long)lane * v.d_out + n0, nw, 0u, 0u);
    }
    if (lane == 0) {
      info[0] = active;
      info[1] = r;
      info[2] = __float_as_int(sc);
      info[3] = na;
    }
  }
  if (a.early) grid_wait();
  grid_release();
  if (tid == 0 && ok && info[4] != 0) report(a.err, info[4]);
  if (warp == 1 && lane == 0 && ok) {  // the token's x and y0 slices; they do not depend on the adapter
    mbar_arrive_expect_tx(bar_xy, (uint32_t)((kw + nw) * 2));
    if (kw > 0) bulk_g2s(smem_u32(sm + kDOffX), a.x + (long long)t * a.ldx + k0, (uint32_t)kw * 2, bar_xy);
    if (nw > 0) bulk_g2s(smem_u32(y0row), a.y + (long long)t * a.ldy + n0, (uint32_t)nw * 2, bar_xy);
  }
  __syncthreads();
  const bool xy_issued = ok;
  const bool active = ok && info[0] != 0;
  bool b_issued = false;
  const int r = info[1];
  if (active) {
    const float sc = __int_as_float(info[2]);
    const int na = info[3];
    ok = __syncthreads_and(mbar_wait(bar_a, 0) && mbar_wait(bar_xy, 0)) != 0;
    if (ok) {
      // Shrink on the CUDA cores (one token: a matrix-vector product): warp w owns
      // rows w % 4 + 4 i of half w / 4 of the slice (512 columns); lane l the
      // 16-byte pieces at columns 8 l and 256 + 8 l of the half.  Each lane sums
      // its 16 products in column order, then a fixed butterfly of shuffles adds
      // the lanes; the halves' partials are added in order before the exchange.
      const int rw = warp & 3, hf = warp >> 2;
      float xv[2][8];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int c = 512 * hf + 8 * lane + 256 * p;
        if (c < kw) {
          unpack8(*reinterpret_cast<const uint4*>(sm + kDOffX + 2 * c), xv[p]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[p][e] = 0.f;
        }
      }
      // the warp's four rows side by side, so that their loads, products and
      // shuffles overlap
      constexpr int kRows = kDMaxRank / 4;
      float sr[kRows];
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int j = rw + 4 * i;
        sr[i] = 0.f;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const int c = 512 * hf + 8 * lane + 256 * p;
          if (j < r && c < kw) {
            float av[8];
            unpack8(*reinterpret_cast<const uint4*>(buf + j * kDRowStride + 2 * c), av);
#pragma unroll
            for (int e = 0; e < 8; ++e) sr[i] = fmaf(av[e], xv[p][e], sr[i]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < kRows; ++i) sr[i] += __shfl_xor_sync(0xffffffffu, sr[i], o);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
          if (rw + 4 * i < r) pw[hf * kDMaxRank + rw + 4 * i] = sr[i];
      }
    }
    __syncthreads();  // every block's partial is in; A's rows are free
    if (ok && warp == 1) {  // B's rows into the same buffer (mostly from L2 by now), beside warp 0's sends
      if (lane == 0) mbar_arrive_expect_tx(bar_b, (uint32_t)(r * nw * 2));
      __syncwarp();
      if (lane < r && nw > 0)
        copy_run(v, pg + na, (long long)lane * v.d_out + n0, nw, smem_u32(buf + lane * kDRowStride), bar_b);
    }
    b_issued = ok;
    // this CTA's partial (the blocks' partials in block order), pushed to every
    // CTA of the cluster, this one included; summed there in CTA order
    const int q4 = (r + 3) >> 2;
    if (ok && tid == 0) mbar_arrive_expect_tx(bar_recv, C * (uint32_t)q4 * 16u);
    if (ok && tid < q4) {
      float4 part = *reinterpret_cast<const float4*>(pw + 4 * tid);
      for (int hh = 1; hh < kDHalves; ++hh) {  // the halves' partials in order
        const float4 p2 = *reinterpret_cast<const float4*>(pw + hh * kDMaxRank + 4 * tid);
        part.x += p2.x; part.y += p2.y; part.z += p2.z; part.w += p2.w;
      }
      const uint32_t dst = smem_u32(recv + crank * kDMaxRank + 4 * tid);
      for (uint32_t c = 0; c < C; ++c) st_async_v4(mapa(dst, c), part, mapa(bar_recv, c));
    }
    bool got = true;
    if (ok && tid < r) {
      got = mbar_wait(bar_recv, 0);
      float s = 0.f;
      for (uint32_t c = 0; c < C; ++c) s += recv[c * kDMaxRank + tid];
      hs[tid] = sc * s;
    }
    ok = __syncthreads_and(ok && got) != 0;
  }
  // Every partial this CTA receives has landed (or it gave up): peers may leave
  // once all have arrived here.
  cluster_arrive();
  if (active && ok) {
    ok = __syncthreads_and(mbar_wait(bar_b, 0)) != 0;
    const int c = 4 * tid;
    if (ok && c < nw) {
      // Expand on the CUDA cores: thread i owns columns 4 i .. 4 i + 3 of the
      // slice and adds h_j B_i[j, n] over the rows in order, then y0.
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kDMaxRank; ++j) {
        if (j < r) {
          const uint2 bv = *reinterpret_cast<const uint2*>(buf + j * kDRowStride + 2 * c);
          const float hj = hs[j];
          acc[0] = fmaf(hj, bf_lo(bv.x), acc[0]);
          acc[1] = fmaf(hj, bf_hi(bv.x), acc[1]);
          acc[2] = fmaf(hj, bf_lo(bv.y), acc[2]);
          acc[3] = fmaf(hj, bf_hi(bv.y), acc[3]);
        }
      }
      const uint2 y0 = *reinterpret_cast<const uint2*>(y0row + 2 * c);
      uint2 out;
      out.x = pack_bf16x2(bf_lo(y0.x) + acc[0], bf_hi(y0.x) + acc[1]);
      out.y = pack_bf16x2(bf_lo(y0.y) + acc[2], bf_hi(y0.y) + acc[3]);
      *reinterpret_cast<uint2*>(a.y + (long long)t * a.ldy + n0 + c) = out;
    }
  }
  if (!ok) {
    // A wait ran out: no output was written.  Copies still in flight into this
    // CTA's shared memory get a second bounded wait before it leaves.
    if (tid == 0) {
      if (xy_issued) mbar_wait(bar_xy, 0);
      if (active) mbar_wait(bar_a, 0);
      if (b_issued) mbar_wait(bar_b, 0);
      report(a.err, LORA_DERR_TIMEOUT);
    }
  }
  cluster_wait();
}

// Cluster width of the decode kernel for a view: one CTA per kDMaxCols columns
// of the wider side, at most eight.
int slice_width(const lora_pool_view_t* v) {
  const int d = std::max(v->d_in, v->d_out);
  return std::min(std::max((d + kDMaxCols - 1) / kDMaxCols, 1), kDMaxCluster);
}

}  // namespace

bool bgmv_decode_ok(const lora_pool_view_t* v, int T) {
  if (T < 1 || T > (1 << 20) || v->max_rank > kDMaxRank) return false;
  const int C = slice_width(v);
  const int kc = ((v->d_in + C - 1) / C + 7) & ~7, nc = ((v->d_out + C - 1) / C + 7) & ~7;
  if (kc > kDMaxCols || nc > kDMaxCols) return false;
  const long long P = v->page_elems;
  const long long na = ((long long)v->max_rank * v->d_in + P - 1) / P;
  const long long nb = ((long long)v->max_rank * v->d_out + P - 1) / P;
  return na + nb <= kDMaxPg;
}

lora_status_t launch_bgmv(const void* x, long long ldx, void* y, long long ldy, const int32_t* ids, int T,
                          const lora_pool_view_t* view, int early, int32_t* err, cudaStream_t stream) {
  BgmvArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.ids = ids;
  make_dev_view(view, &a.v);
  a.err = err;
  a.early = early;
  a.probe = wait_probe_cycles();
  const int C = slice_width(view);
  if (ensure_smem_attr((const void*)bgmv_kernel, kDSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)bgmv_kernel, dim3((unsigned)(T * C)), dim3(kDThreads), kDSmem, stream, C, &a) ==
                 cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
