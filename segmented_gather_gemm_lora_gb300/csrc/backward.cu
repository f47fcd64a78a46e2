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
// The shrinks and the expand are the forward kernels: h by the shrink path; u
// and dx in one pass of the apply path over transposed views of the adapters
// (x = dy, y = dx, B_i as the shrink's matrix and A_i as the expand's), which
// also writes its intermediate u; this file holds the gradient kernel.
//
// Gradient kernel.  A unit is (segment, matrix, 128-column block): the block's
// columns of dB_i (a slice of d_out) or of dA_i (a slice of d_in), for all the
// adapter's r_i rows.  Its CTA walks the segment's tokens 32 at a time through
// a five-step ring: the token rows of dy (or x) for the block's columns and of
// h (or u) arrive in shared memory by asynchronous copies, their token indices
// five steps earlier; each step's h / u is converted once, a step ahead, into
// bf16 hi + lo parts, transposed; and each of the 8 warps accumulates its 16
// columns x r_i rows with mma.sync m16n8k16 (the contraction runs over the
// tokens, 16 per MMA).  At the end each element of the block is added once into the
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
constexpr int kBTok = 16;                // tokens per MMA (its k dimension)
constexpr int kBStepTok = 32;            // tokens per step
constexpr int kBStages = 5;              // steps in the ring
constexpr int kBTokRing = 2 * kBStages;  // token-index slots: step m's indices arrive kBStages steps ahead
constexpr int kBQStride = kBCols * 2 + 16;    // bytes per staged dy / x row (padded: conflict-free ldmatrix)
constexpr int kBHStride = LORA_MAX_RANK + 4;  // floats per staged h / u row (padded: conflict-free fragments)
constexpr size_t kBOffH = (size_t)kBStages * kBStepTok * kBQStride;
constexpr size_t kBOffTok = kBOffH + (size_t)kBStages * kBStepTok * kBHStride * sizeof(float);
constexpr int kBPStride = kBStepTok * 2 + 16;   // bytes per row of the transposed h / u (padded: conflict-free ldmatrix)
constexpr int kBPPart = LORA_MAX_RANK * kBPStride;  // the hi part, then the lo part
constexpr size_t kBOffP = kBOffTok + (size_t)kBTokRing * kBStepTok * sizeof(int);
constexpr size_t kBSmem = kBOffP + 2 * 2 * (size_t)kBPPart;  // two steps' transposed h / u
static_assert(kBOffH % 16 == 0 && (kBHStride * 4) % 16 == 0, "16-byte copy destinations");
static_assert(kBStepTok * 16 == 2 * kBThreads, "two 16-byte pieces of a row per thread and step");

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

// 4-byte global -> shared copy (LSU async copy, through L1)
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

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
  // a ring of kBStages steps: each holds 32 token rows of dy (or x) for the block's
  // columns and the same tokens' h (or u) rows as fp32; and the steps' token indices
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* const qs = sm;                                        // [stage][token][kBQStride bytes]
  float* const hraw = reinterpret_cast<float*>(sm + kBOffH);     // [stage][token][kBHStride]
  int* const tokring = reinterpret_cast<int*>(sm + kBOffTok);    // [slot][token]
  uint8_t* const pbuf = sm + kBOffP;  // [step & 1][hi, lo][rank row][token] bf16
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
    const int nsteps = (count + kBStepTok - 1) / kBStepTok;
    // Step m's token indices go to their ring slot by asynchronous copies, kBStages
    // steps before the step's own copies need them, so no copy waits on an index load.
    auto load_idx = [&](int m, int e) {
      const int ti = m * kBStepTok + e;
      if (ti < count) cp_async4(smem_u32(&tokring[(m % kBTokRing) * kBStepTok + e]), a.perm + p0 + ti);
    };
    // step i's copies: rows tr and tr + 16 of its 32 tokens, 16-byte piece pc of the
    // block's columns and of the token's h / u row (zero past the rank or the
    // tokens; pieces past the rank rounded up to 8 are not read); with them, in the
    // same group, the indices of step i + kBStages
    auto load_step = [&](int i) {
      if (i < nsteps) {
        const int st = i % kBStages;
        const int pc = tid & 15;
        const int c = col0 + 8 * pc;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int tr = (tid >> 4) + 16 * h2;
          const int t = i * kBStepTok + tr;
          const int tok = t < count ? tokring[(i % kBTokRing) * kBStepTok + tr] : -1;
          const bool valid = tok >= 0 && c < d;  // d % 8 == 0: a piece is all in or all out
          cp_async16(smem_u32(qs + ((size_t)st * kBStepTok + tr) * kBQStride + pc * 16),
                     valid ? Q + (long long)tok * ldq + c : Q, valid);
          if (4 * pc < rpad) {
            const bool hv = tok >= 0 && 4 * pc < r;
            cp_async16(smem_u32(hraw + ((size_t)st * kBStepTok + tr) * kBHStride + 4 * pc),
                       hv ? P + (long long)tok * a.ldh + 4 * pc : P, hv);
          }
        }
      }
      if (tid < kBStepTok && i + kBStages < nsteps) load_idx(i + kBStages, tid);
      cp_async_commit();  // one group per step, empty past the end, so the waits count evenly
    };
    if (tid < kBStages * kBStepTok && tid / kBStepTok < nsteps) load_idx(tid / kBStepTok, tid % kBStepTok);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();  // the first kBStages steps' indices
    // step m's h / u as bf16 hi + lo parts, transposed (rank row, token), into
    // buffer m & 1: thread (token pair tid % 16, rank rows 4 (tid / 16) ..), once
    // for all the warps
    auto convert = [&](int m) {
      const int cst = m % kBStages, tp = tid & 15, q4 = tid >> 4;
      if (4 * q4 < rpad) {
        const float* hp = hraw + ((size_t)cst * kBStepTok + 2 * tp) * kBHStride + 4 * q4;
        const float4 f0 = *reinterpret_cast<const float4*>(hp);
        const float4 f1 = *reinterpret_cast<const float4*>(hp + kBHStride);
        const float v0[4] = {f0.x, f0.y, f0.z, f0.w}, v1[4] = {f1.x, f1.y, f1.z, f1.w};
        uint8_t* ph = pbuf + (size_t)(m & 1) * 2 * kBPPart + (size_t)(4 * q4) * kBPStride + 4 * tp;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t hi = pack_bf16x2(v0[e], v1[e]);
          const uint32_t lo = pack_bf16x2(v0[e] - bf_lo(hi), v1[e] - bf_hi(hi));
          *reinterpret_cast<uint32_t*>(ph + e * kBPStride) = hi;
          *reinterpret_cast<uint32_t*>(ph + kBPPart + e * kBPStride) = lo;
        }
      }
    };
    float acc[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) acc[jt][0] = acc[jt][1] = acc[jt][2] = acc[jt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kBStages - 1; ++i) load_step(i);
    cp_async_wait<kBStages - 2>();  // step 0's copies
    __syncthreads();
    convert(0);
    const int g = lane >> 2, q = lane & 3;
    for (int i = 0; i < nsteps; ++i) {
      cp_async_wait<kBStages - 3>();  // this thread's copies of step i + 1, and the indices up to step i + kBStages + 1
      __syncthreads();                // everyone's; step i's parts are converted; the stage of step i - 1 is free
      load_step(i + kBStages - 1);
      if (i + 1 < nsteps) convert(i + 1);
      const int st = i % kBStages;
      // warp w: columns 16 w .. 16 w + 15 of the block (A operand: the staged rows
      // transposed, k = token); the rank rows 8 at a time (B operand: h / u, as
      // bf16 hi and lo parts, two MMAs each); 16 tokens per MMA, in token order
      if (col0 + 16 * warp < d) {
#pragma unroll
        for (int ks = 0; ks < kBStepTok / kBTok; ++ks) {
          if (i * kBStepTok + ks * kBTok >= count) break;  // nothing but zero rows left
          const int trow = ks * kBTok + (lane & 7) + 8 * (lane >> 4), tcol = 16 * warp + 8 * ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(smem_u32(qs + ((size_t)st * kBStepTok + trow) * kBQStride + tcol * 2), a0, a1, a2, a3);
          // B operand: rank rows 8 jt .. 8 jt + 7 of the transposed h / u, the MMA's
          // tokens 0-7 (lanes 0-7) and 8-15 (lanes 8-15)
          const uint32_t pb = smem_u32(pbuf + (size_t)(i & 1) * 2 * kBPPart) + (uint32_t)((lane & 7) * kBPStride +
                                                                                       32 * ks + 16 * ((lane >> 3) & 1));
#pragma unroll
          for (int jt = 0; jt < 8; ++jt) {
            if (8 * jt >= rpad) break;
            uint32_t bh0, bh1, bl0, bl1;
            ldsm_x2(pb + 8 * jt * kBPStride, bh0, bh1);
            ldsm_x2(pb + kBPPart + 8 * jt * kBPStride, bl0, bl1);
            mma_m16n8k16(acc[jt], a0, a1, a2, a3, bh0, bh1);
            mma_m16n8k16(acc[jt], a0, a1, a2, a3, bl0, bl1);
          }
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // every copy of this unit landed and every warp is done with the ring
    // acc[jt]: columns 16 w + lane / 4 (+ 8), rank rows 8 jt + 2 (lane % 4) (+ 1)
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
  if (ensure_smem_attr((const void*)grad_kernel, kBSmem) != cudaSuccess) return LORA_ERR_CUDA;
  return launch_pdl((const void*)grad_kernel, dim3((unsigned)grid), dim3(kBThreads), kBSmem, stream, 0, &a) ==
                 cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
