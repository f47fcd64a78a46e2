// Chunk arithmetic of the gather kernel: warp-level tensor-core tiles over
// staged adapter rows.
//
// "Multi-LoRA Serving in Production", sections "Shrink Stage" and "Expand
// Stage": the shrink contracts a token row with the adapter's rows, the expand
// multiplies the scaled rank-r intermediate by B_i and adds it to the base
// output.  Both run here on mma.sync m16n8k16 (bf16 operands, fp32
// accumulators): one instruction is 2048 multiply-adds, where a CUDA-core loop
// spends an instruction or more per adapter element.  Operands come from the
// staged rows with ldmatrix.
//
// Staging layout shared by every caller: adapter rows and token rows are
// kRowStride bytes apart (1 KB of a 512-column sub-slice plus 16 bytes, so that
// the eight rows one ldmatrix reads fall in eight different bank groups).  A
// sub-slice is split into 64-column blocks; block b's arithmetic is a fixed
// sequence of MMAs, so any kernel that runs the same blocks over the same
// sub-slices and adds the blocks' partials in block order gets the same bits.
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kNT = 4;  // tokens per group
constexpr int kHMax = LORA_MAX_RANK;
constexpr int kSub = 512;       // columns per sub-slice (one 1 KB row)
constexpr int kChunkRows = 16;  // adapter rows per chunk
constexpr int kRowBytes = kSub * 2;
constexpr int kRowStride = kRowBytes + 16;
constexpr int kSubBlocks = kSub / 64;  // 64-column blocks of a sub-slice

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
// d (16 x 8 fp32, row-major over lanes) += a (16 x 16 bf16) . b (16 x 8 bf16)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shrink of one staged chunk over 64-column block `blk` of a sub-slice of width
// wsub: D[j, t] += sum_k A_i[j0 + j, k] x[t, k], k in the block, as four k16
// steps in column order.  arows: shared-memory address of the chunk's first
// adapter row; xrows: of the group's first token row.  d is the lane's part of
// the 16 x 8 tile: rows (lane / 4, lane / 4 + 8), tokens (2 (lane % 4),
// 2 (lane % 4) + 1).  Rows past the chunk and tokens past the group give entries
// nobody reads; columns past the sub-slice are masked to zero in both operands.
// Each entry is a fixed function of its own adapter row and token row.
__device__ __forceinline__ void shrink_chunk(uint32_t arows, uint32_t xrows, int wsub, int ntok, float (&d)[4],
                                             int blk, int lane) {
  const int kw = blk * 64;
  if (kw >= wsub) return;
  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
  const int xrow = min(lane & 7, ntok - 1), xcol = ((lane >> 3) & 1) * 8;
  const uint32_t abase = arows + (uint32_t)(arow * kRowStride + (kw + acol) * 2);
  const uint32_t xbase = xrows + (uint32_t)(xrow * kRowStride + (kw + xcol) * 2);
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int k0 = kw + 16 * st;
    if (k0 >= wsub) break;
    uint32_t a0, a1, a2, a3, b0, b1;
    ldsm_x4(abase + 32 * st, a0, a1, a2, a3);
    ldsm_x2(xbase + 32 * st, b0, b1);
    if (k0 + 8 >= wsub) a2 = a3 = b1 = 0u;  // columns k0 + 8 .. k0 + 15 lie past the sub-slice
    mma16816(d, a0, a1, a2, a3, b0, b1);
  }
}

// Expand of one staged chunk over 64-column block `blk`: Y[n, t] += sum_j
// B_i[j0 + j, n] h[t, j0 + j] over the chunk's nrows rows (four n16 tiles; acc[i]
// is the lane's part of tile i: columns 16 i + lane / 4 (+ 8), tokens
// 2 (lane % 4) (+ 1)).  brows: shared-memory address of the chunk's first B row;
// hs: the group's scaled h, [kNT][kHMax] fp32.  h enters as bf16 hi + lo parts
// (two MMAs per tile, hi first), which keeps the intermediate at about fp32
// accuracy.  Rows past the chunk are masked to zero in both operands.
__device__ __forceinline__ void expand_mma(uint32_t brows, const float* hs, int j0, int nrows, int ntok, int wsub,
                                           bool first, float (&acc)[4][4], int blk, int lane) {
  const int nw = blk * 64;
  if (first) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  }
  const int g = lane >> 2, t = lane & 3;
  // h fragment of token g: rows 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1) of the chunk
  uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
  if (g < ntok) {
    const float* hrow = hs + g * kHMax + j0;
    float hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 2 * t + (e & 1) + 8 * (e >> 1);
      hv[e] = j < nrows ? hrow[j] : 0.f;
    }
    bh0 = pack_bf16x2(hv[0], hv[1]);
    bh1 = pack_bf16x2(hv[2], hv[3]);
    bl0 = pack_bf16x2(hv[0] - bf_lo(bh0), hv[1] - bf_hi(bh0));
    bl1 = pack_bf16x2(hv[2] - bf_lo(bh1), hv[3] - bf_hi(bh1));
  }
  // rows of the lane's A entries: 2t, 2t + 1 (a0, a1) and 2t + 8, 2t + 9 (a2, a3)
  const uint32_t m01 = (2 * t < nrows ? 0x0000ffffu : 0u) | (2 * t + 1 < nrows ? 0xffff0000u : 0u);
  const uint32_t m23 = (2 * t + 8 < nrows ? 0x0000ffffu : 0u) | (2 * t + 9 < nrows ? 0xffff0000u : 0u);
  const int jrow = (lane & 7) + 8 * (lane >> 4), ncol = 8 * ((lane >> 3) & 1);
  const uint32_t bbase = brows + (uint32_t)(jrow * kRowStride + (nw + ncol) * 2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (nw + 16 * i >= wsub) break;
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(bbase + 32 * i, a0, a1, a2, a3);
    a0 &= m01;
    a1 &= m01;
    a2 &= m23;
    a3 &= m23;
    mma16816(acc[i], a0, a1, a2, a3, bh0, bh1);
    mma16816(acc[i], a0, a1, a2, a3, bl0, bl1);
  }
}

// The block's outputs: y[tok[t], col0 + n] = bf16(y0 + acc) (or the fp32 sum into
// yf), n in the block.  y0rows: the group's first staged y0 row (rows kRowStride
// apart, columns of the sub-slice); scr: the warp's scratch, [kNT][64] fp32.  The
// lane's accumulator entries go through the scratch so that each lane then
// writes two adjacent columns of every token.
__device__ __forceinline__ void expand_store(uint16_t* ybase, long long ldy, float* yf, long long ldyf,
                                             const uint8_t* y0rows, float* scr, const float (&acc)[4][4], int ntok,
                                             const int (&tok)[kNT], int col0, int wsub, int blk, int lane) {
  const int nw = blk * 64;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tk = 2 * t + (e & 1), nn = 16 * i + g + 8 * (e >> 1);
      if (tk < ntok) scr[tk * 64 + nn] = acc[i][e];
    }
  __syncwarp();
  const int c2 = nw + 2 * lane;
  if (c2 < wsub) {
#pragma unroll
    for (int tk = 0; tk < kNT; ++tk) {
      if (tk >= ntok) break;
      const uint32_t y0 = *reinterpret_cast<const uint32_t*>(y0rows + tk * kRowStride + 2 * c2);
      const float v0 = scr[tk * 64 + 2 * lane], v1 = scr[tk * 64 + 2 * lane + 1];
      if (yf != nullptr)  // fp32 output (diagnostic form): the same sums, not rounded to bf16
        *reinterpret_cast<float2*>(yf + (long long)tok[tk] * ldyf + col0 + c2) =
            make_float2(bf_lo(y0) + v0, bf_hi(y0) + v1);
      else
        *reinterpret_cast<uint32_t*>(ybase + (long long)tok[tk] * ldy + col0 + c2) =
            pack_bf16x2(bf_lo(y0) + v0, bf_hi(y0) + v1);
    }
  }
  __syncwarp();
}

}  // namespace lora
