// Backward pass of the multi-adapter LoRA product, for training the adapters.
//
// "QLoRA and multi-LoRA at the limit on small models", section "The bare
// mechanism: LoRA, and why you can train on a 4-bit base": the base W is
// frozen and gets no gradient; only the adapter's A and B are trainable, and
// the gradient flows through the adapter alone.  Differentiating
//     y[t] = y0[t] + s_i (x[t] A_i^T) B_i
// token by token, with dy = dL/dy:
//     h[t]      = x[t] A_i^T                  (shrink of x over A_i)
//     u[t]      = dy[t] B_i^T                 (shrink of dy over B_i)
//     dB_i     += s_i sum_{t in i} h[t]^T dy[t]
//     dA_i     += s_i sum_{t in i} u[t]^T x[t]
//     dx[t]    += s_i u[t] A_i                (expand of u over A_i)
// The two shrinks and the expand are the forward kernels, the second shrink and
// the expand on transposed views of the adapters; this file holds the
// gradient kernel and the entry point.
//
// Gradient kernel.  A unit is (segment, matrix, 128-column block): the block's
// columns of dB_i (a slice of d_out) or of dA_i (a slice of d_in), for all the
// adapter's r_i rows.  Its CTA walks the segment's tokens 16 at a time: the 16
// token rows of dy (or x) for the block's columns and of h (or u) go to shared
// memory (h and u as bf16 hi + lo parts), and each of the 8 warps accumulates
// its 16 columns x r_i rows with mma.sync m16n8k16 (the contraction runs over
// the tokens).  At the end each element of the block is added once into the
// gradient pool, at its pool position, by one atomic add: with GROUP segments
// an adapter has one segment, so a call's sums are deterministic.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kBThreads = 256;
constexpr int kBCols = 128;              // gradient columns per unit
constexpr int kBTok = 16;                // tokens per step (the mma k dimension)
constexpr int kBStages = 4;              // steps in flight
constexpr int kBQStride = kBCols * 2 + 16;   // bytes per staged dy / x row (padded: conflict-free ldmatrix)
constexpr int kBPStride = kBTok * 2 + 16;  // bytes per staged rank row of h / u (16 tokens, bf16, padded)

struct GradArgs {
  const uint16_t* x;
  long long ldx;
  const uint16_t* dy;
  long long lddy;
  const float* h;
  const float* u;
  long long ldh;
  float* grad;
  DevView v;
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* meta;
  int32_t* err;
};

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kBThreads) grad_kernel(const __grid_constant__ GradArgs a) {
  // a ring of kBStages steps: each holds 16 token rows of dy (or x) for the block's
  // columns and the same tokens' h (or u) rows as fp32; the step being computed
  // has its h / u converted into bf16 hi + lo parts, transposed, in phi / plo
  __shared__ __align__(128) uint8_t qs[kBStages][kBTok * kBQStride];
  __shared__ __align__(16) float hraw[kBStages][kBTok][LORA_MAX_RANK];
  __shared__ __align__(128) uint8_t phi[LORA_MAX_RANK * kBPStride];  // h or u transposed [rank row][token], bf16 hi
  __shared__ __align__(128) uint8_t plo[LORA_MAX_RANK * kBPStride];  // lo part
  __shared__ int info[6];  // p0, count, rank, skip, a_page0 / b_page0 of the unit's matrix, scale bits
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DevView& v = a.v;
  pdl_wait_then_release();
  const int nbB = (v.d_out + kBCols - 1) / kBCols, nbA = (v.d_in + kBCols - 1) / kBCols;
  const int per_seg = nbB + nbA;
  const long long n_units = (long long)a.meta[0] * per_seg;
  const int shift = v.page_shift;
  const long long pmask = (1LL << shift) - 1;
  for (long long w = blockIdx.x; w < n_units; w += gridDim.x) {
    const int s = (int)(w / per_seg), b = (int)(w - (long long)s * per_seg);
    const bool isB = b < nbB;
    const int col0 = (isB ? b : b - nbB) * kBCols;
    const int d = isB ? v.d_out : v.d_in;
    if (warp == 0) {
      const int ad = a.seg_adapter[s];
      const lora_adapter_desc_t dsc = adapter_desc(v, ad);
      const int bad = check_adapter_warp(v, ad, dsc, lane);
      if (lane == 0) {
        if (bad && b == 0) report(a.err, bad);
        info[0] = a.indptr[s];
        info[1] = a.indptr[s + 1] - info[0];
        info[2] = dsc.rank;
        info[3] = bad;
        info[4] = isB ? dsc.b_page0 : dsc.a_page0;
        info[5] = __float_as_int(dsc.scale);
      }
    }
    __syncthreads();
    const int p0 = info[0], count = info[1], r = info[2], skip = info[3], page0 = info[4];
    const float scale = __int_as_float(info[5]);
    if (skip) {
      __syncthreads();
      continue;
    }
    const int rpad = (r + 7) & ~7;  // rows of the output, in n8 tiles
    const float* P = isB ? a.h : a.u;
    const uint16_t* Q = isB ? a.dy : a.x;
    const long long ldq = isB ? a.lddy : a.ldx;
    const int nsteps = (count + kBTok - 1) / kBTok;
    // step i's copies: row tid / 16 of its 16 tokens, 16-byte piece tid % 16 of the
    // block's columns and of the token's h / u row (zero past the rank or the tokens)
    auto load_step = [&](int i) {
      if (i < nsteps) {
        const int st = i % kBStages;
        const int tr = tid >> 4, pc = tid & 15;
        const int t0 = i * kBTok;
        const int tok = t0 + tr < count ? a.perm[p0 + t0 + tr] : -1;
        const int c = col0 + 8 * pc;
        const bool valid = tok >= 0 && c < d;  // d % 8 == 0: a piece is all in or all out
        cp_async16(smem_u32(&qs[st][tr * kBQStride + pc * 16]), valid ? Q + (long long)tok * ldq + c : Q, valid);
        const bool hv = tok >= 0 && 4 * pc < r;
        cp_async16(smem_u32(&hraw[st][tr][4 * pc]), hv ? P + (long long)tok * a.ldh + 4 * pc : P, hv);
      }
      cp_async_commit();  // one group per step, empty past the end, so the waits count evenly
    };
    float acc[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) acc[jt][0] = acc[jt][1] = acc[jt][2] = acc[jt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kBStages - 1; ++i) load_step(i);
    for (int i = 0; i < nsteps; ++i) {
      cp_async_wait<kBStages - 2>();  // this thread's copies of step i have landed
      __syncthreads();                // everyone's; the stage of step i - 1 and phi / plo are free
      load_step(i + kBStages - 1);
      const int st = i % kBStages;
      {  // h / u of step i: rank row j + e, token tr, as bf16 hi + lo (columns past r are zero)
        const int tr = tid >> 4, j = 4 * (tid & 15);
        const float4 f = *reinterpret_cast<const float4*>(&hraw[st][tr][j]);
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float val = j + e < r ? fv[e] : 0.f;
          const __nv_bfloat16 hi = __float2bfloat16_rn(val);
          const __nv_bfloat16 lo = __float2bfloat16_rn(val - __bfloat162float(hi));
          *reinterpret_cast<__nv_bfloat16*>(phi + (j + e) * kBPStride + tr * 2) = hi;
          *reinterpret_cast<__nv_bfloat16*>(plo + (j + e) * kBPStride + tr * 2) = lo;
        }
      }
      __syncthreads();
      // warp w: columns 16 w .. 16 w + 15 of the block (A operand: the staged rows
      // transposed, k = token); the rank rows 8 at a time (B operand: h / u)
      if (col0 + 16 * warp < d) {
        const int trow = (lane & 7) + 8 * (lane >> 4), tcol = 16 * warp + 8 * ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(smem_u32(&qs[st][trow * kBQStride + tcol * 2]), a0, a1, a2, a3);
        // B operand: rank rows 8 jt .. 8 jt + 7 of the transposed h / u, tokens 0-7
        // (lanes 0-7) and 8-15 (lanes 8-15)
        const int prow = lane & 7, pcol = 16 * ((lane >> 3) & 1);
#pragma unroll
        for (int jt = 0; jt < 8; ++jt) {
          if (8 * jt >= rpad) break;
          uint32_t b0, b1;
          ldsm_x2(smem_u32(phi + (8 * jt + prow) * kBPStride + pcol), b0, b1);
          mma_m16n8k16(acc[jt], a0, a1, a2, a3, b0, b1);
          ldsm_x2(smem_u32(plo + (8 * jt + prow) * kBPStride + pcol), b0, b1);
          mma_m16n8k16(acc[jt], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // every copy of this unit landed and every warp is done with the ring
    // acc[jt]: columns 16 w + lane / 4 (+ 8), rank rows 8 jt + 2 (lane % 4) (+ 1)
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
      if (8 * jt >= rpad) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = col0 + 16 * warp + g + 8 * (e >> 1), j = 8 * jt + 2 * q + (e & 1);
        if (j < r && col < d) {
          const long long el = (long long)j * d + col;
          const long long pg = v.page_list[page0 + (el >> shift)];
          atomicAdd(a.grad + (pg << shift) + (el & pmask), scale * acc[jt][e]);
        }
      }
    }
  }
}

}  // namespace

lora_status_t launch_grad(const void* x, long long ldx, const void* dy, long long lddy, const float* h,
                          const float* u, long long ldh, float* grad_pool, const lora_segments_t* seg,
                          const lora_pool_view_t* view, int32_t* err, cudaStream_t stream) {
  GradArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.dy = static_cast<const uint16_t*>(dy);
  a.lddy = lddy;
  a.h = h;
  a.u = u;
  a.ldh = ldh;
  a.grad = grad_pool;
  make_dev_view(view, &a.v);
  a.perm = seg->token_perm;
  a.indptr = seg->seg_indptr;
  a.seg_adapter = seg->seg_adapter;
  a.meta = seg->meta;
  a.err = err;
  const long long per_seg = (view->d_out + kBCols - 1) / kBCols + (view->d_in + kBCols - 1) / kBCols;
  long long grid = (long long)sm_count() * 8;
  grid = std::min(grid, std::max(1LL, (long long)seg->T * per_seg));
  return launch_pdl((const void*)grad_kernel, dim3((unsigned)grid), dim3(kBThreads), 0, stream, 0, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
