// The base projection with the adapters' correction in its epilogue.
//
// "Multi-LoRA Serving: Many Adapters on One GPU", section "How batching across
// adapters works": the whole batch shares one base product x W0 and each token
// adds its own adapter's term; "Multi-LoRA Serving in Production", section
// "Mathematical Formulation and the Batching Challenge": y = x W0 + (alpha/r)
// (x A) B.  Here the adapter term is added to the base product's accumulator
// before y is written, so y is written once and never read:
//     y[t, n] = bf16( sum_k x[t,k] W0[n,k]  +  s_i sum_j h[t,j] B_i[j,n] ),
// with h[t, j] = x[t] . A_i[j] computed beforehand by the shrink stage (by
// token, fp32) and s_i the token's scale (0 when the token has no usable
// adapter, which then gets the base product alone).
//
// Base product: a persistent tcgen05 GEMM over 128 x 256 output tiles, tiles
// taken in order (m = tile / n_tiles_n, n = tile % n_tiles_n) so that a wave of
// CTAs shares W0's tiles in L2 and x streams once.  Warp 0 loads: per 64-column
// K step one TMA box of x (128 x 64) and one of W0 (256 x 64), both with the
// 128-byte swizzle, into a 4-stage ring.  Warp 1 issues tcgen05.mma (M = 128,
// N = 256, bf16, fp32 accumulator in tensor memory), alternating two
// accumulators so that a tile's epilogue overlaps the next tile's MMAs.
// Warps 2-17 run the epilogue, one tile row and a quarter of the tile's
// columns per thread (the tensor-memory lane quarter of its warp): 32 columns
// at a time from tensor memory, plus the
// row's adapter term on the CUDA cores (fp32 FMA over the rank in order, from
// B_i's rows for the tile staged once per adapter in shared memory), rounded
// once to bf16 and stored.
#include <cudaTypedefs.h>

#include <cstring>

#include "internal.h"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kBStages = 4;
constexpr int kBEpiWarps = 16;  // four per tensor-memory lane quarter, one per quarter of the tile's columns
constexpr int kBEpiThreads = 32 * kBEpiWarps;
constexpr int kBThreads = 64 + kBEpiThreads;  // warp 0 TMA, warp 1 MMA, warps 2-17 epilogue
constexpr int kBEpiChunks = kBN / 32 / (kBEpiWarps / 4);  // 32-column chunks per epilogue warp
constexpr int kBABytes = kBM * kBK * 2;
constexpr int kBBBytes = kBN * kBK * 2;
constexpr int kBStageBytes = kBABytes + kBBBytes;  // 48 KB
constexpr size_t kBOffBars = (size_t)kBStages * kBStageBytes;
constexpr int kBNBars = 2 * kBStages + 2 + 2 + 1;
constexpr size_t kBOffB = (kBOffBars + kBNBars * 8 + 16 + 15) / 16 * 16;  // an adapter's B rows for the tile: [64][kBN] bf16
constexpr size_t kBOffCtl = kBOffB + (size_t)LORA_MAX_RANK * kBN * 2;  // round control: 4 ints + [128] row adapters
constexpr size_t kBSmem = kBOffCtl + (4 + kBM) * 4 + 1024;          // + 1024-byte alignment
static_assert(kBOffB % 16 == 0, "16-byte staging stores");
static_assert(kBSmem <= 232448, "shared memory of one CTA");

struct BaseArgs {
  CUtensorMap xmap;  // x [T, d_in], boxes of 128 rows x 64 columns
  CUtensorMap wmap;  // W0 [d_out, d_in], boxes of 256 rows x 64 columns
  uint16_t* y;
  long long ldy;
  const float* h;  // [T, ldh]: h[t, j] = x[t] . A_i[j] for tokens with a usable adapter
  long long ldh;
  const float* tscale;  // [T]: s_i for tokens with a usable adapter, else 0 (only read for ids >= 0)
  const int32_t* ids;
  DevView v;
  int T;
  int n_m, n_n, nk;
  int32_t* err;
  long long probe;
};

// The epilogue warps (512 threads) meet at named barrier 1; the other warps
// never use it.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// true in every epilogue thread iff `p` holds in all of them (a barrier too)
__device__ __forceinline__ bool epi_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, o;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred o, 1, 512, q;\n\t"
      "selp.u32 %0, 1, 0, o;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kBThreads, 1) base_gemm_kernel(const __grid_constant__ BaseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBOffBars);
  uint64_t* full = bars;                    // [stages] TMA bytes
  uint64_t* empty = bars + kBStages;        // [stages] MMA commit
  uint64_t* acc_full = empty + kBStages;    // [2] MMA commit: a tile's accumulator is complete
  uint64_t* acc_empty = acc_full + 2;       // [2] the 16 epilogue warps
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kBEpiWarps);
    }
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 2 * kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_then_release();
  bool ok = true;
  if (a.probe > 0) {  // the timeout probe: every CTA takes the exit of a wait that ran out
    __shared__ uint64_t probe_bar;
    __shared__ int probe_ok;
    if (tid == 0) probe_ok = wait_probe(&probe_bar, a.probe) ? 1 : 0;
    __syncthreads();
    ok = probe_ok != 0;
  }
  const int n_tiles = a.n_m * a.n_n;

  if (warp == 0) {
    // ---------------- TMA loads ----------------
    if (lane == 0 && ok) {
      prefetch_tensormap(&a.xmap);
      prefetch_tensormap(&a.wmap);
      uint32_t g = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m = tile / a.n_n, n = tile - m * a.n_n;
        for (int kb = 0; kb < a.nk; ++kb, ++g) {
          const uint32_t st = g % kBStages;
          if (g >= kBStages && !mbar_wait(smem_u32(&empty[st]), ((g / kBStages) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t dst = smem_u32(sm + (size_t)st * kBStageBytes);
          mbar_arrive_expect_tx(smem_u32(&full[st]), kBStageBytes);
          tma_load_2d(dst, &a.xmap, kb * kBK, m * kBM, smem_u32(&full[st]));
          tma_load_2d(dst + kBABytes, &a.wmap, kb * kBK, n * kBN, smem_u32(&full[st]));
        }
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0 && ok) {
      const uint32_t idesc = idesc_bf16(kBM, kBN, 0);
      uint32_t g = 0, lt = 0;
      bool issued = false;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
        const uint32_t ab = lt & 1;
        if (lt >= 2 && !mbar_wait(smem_u32(&acc_empty[ab]), ((lt >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < a.nk; ++kb, ++g) {
          const uint32_t st = g % kBStages;
          if (!mbar_wait(smem_u32(&full[st]), (g / kBStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t as = smem_u32(sm + (size_t)st * kBStageBytes), bs = as + kBABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(tmem + ab * kBN, sdesc_sw128(as + 32 * kk, 16, 1024), sdesc_sw128(bs + 32 * kk, 16, 1024), idesc,
                     (kb | kk) != 0);
          issued = true;
          mma_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&acc_full[ab]));
      }
      if (issued) {  // every MMA has completed before tensor memory is freed
        mma_commit(smem_u32(mma_done));
        mbar_wait(smem_u32(mma_done), 0);
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    // Per tile, in rounds: round 0 stores the rows without an adapter term; each
    // later round takes the adapter of the lowest row not yet stored, stages its
    // B_i[0 .. r)[n-tile] in shared memory (every epilogue thread copies 16-byte
    // pieces through the page table), and the rows of that adapter add their
    // term from it and store.  A tile of one request's tokens takes one or two
    // rounds; each round reads every column of the accumulator once per warp.
    const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
    const int row = quarter * 32 + lane;
    const int part = (warp - 2) >> 2;  // the tile's columns [64 part, 64 part + 64)
    const int et = tid - 64;           // 0..511
    const DevView& v = a.v;
    const int shift = v.page_shift;
    const long long pmask = (1LL << shift) - 1;
    uint16_t* bs = reinterpret_cast<uint16_t*>(sm + kBOffB);
    int* cand = reinterpret_cast<int*>(sm + kBOffCtl);  // [0] lowest row left; [1] its adapter, [2] rank, [3] b_page0
    int* row_ad = cand + 4;                             // [128] each row's adapter (-1: none)
    uint32_t lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
      const int m = tile / a.n_n, n = tile - m * a.n_n;
      const uint32_t ab = lt & 1;
      // the epilogue warps leave together when a wait ran out (they meet at named barriers)
      if (!epi_all(mbar_wait(smem_u32(&acc_full[ab]), (lt >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t = m * kBM + row;
      int ad = -1;
      float s = 0.f;
      if (t < a.T) {
        const int id = a.ids[t];
        if (id >= 0 && id < v.n_adapters) {
          s = a.tscale[t];
          if (s != 0.f) ad = id;
        }
      }
      row_ad[row] = ad;
      const float* hrow = a.h + (long long)(t < a.T ? t : 0) * a.ldh;
      const int n_base = n * kBN;
      const int wt = min(kBN, v.d_out - n_base);  // columns of this tile, a multiple of 8
      bool done = t >= a.T;
      for (int round = 0;; ++round) {
        int cur = -1, r = 0;
        if (round > 0) {
          if (et == 0) cand[0] = 0x7fffffff;
          epi_bar();
          if (!done) atomicMin(&cand[0], row);
          epi_bar();
          const int first = cand[0];
          if (first == 0x7fffffff) break;  // every row stored
          cur = row_ad[first];
          if (et == 0) {
            const lora_adapter_desc_t d = adapter_desc(v, cur);
            cand[2] = d.rank;
            cand[3] = d.b_page0;
          }
          epi_bar();
          r = cand[2];
          const long long b0 = cand[3];
          // stage B_cur[j][n_base .. n_base + wt) as [r][kBN] bf16
          const int pieces = r * (kBN / 8);
          for (int p0 = et; p0 < pieces; p0 += 4 * kBEpiThreads) {
            long long pg[4];
            long long el[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int p = p0 + kBEpiThreads * u;
              const int j = p / (kBN / 8), q = p - j * (kBN / 8);
              el[u] = (long long)j * v.d_out + n_base + 8 * q;
              pg[u] = (p < pieces && 8 * q < wt) ? v.page_list[b0 + (el[u] >> shift)] : -1;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int p = p0 + kBEpiThreads * u;
              if (pg[u] >= 0) {
                const int j = p / (kBN / 8), q = p - j * (kBN / 8);
                *reinterpret_cast<uint4*>(bs + j * kBN + 8 * q) =
                    __ldg(reinterpret_cast<const uint4*>(v.pool + (pg[u] << shift) + (el[u] & pmask)));
              }
            }
          }
          epi_bar();
        }
        const bool mine = !done && (round == 0 ? ad < 0 : ad == cur);
        for (int c = kBEpiChunks * part; c < kBEpiChunks * (part + 1); ++c) {
          __syncwarp();  // the warp converged for the collective load
          uint32_t raw[32];
          tmem_ld32_nowait(tmem + ab * kBN + c * 32 + ((uint32_t)(quarter * 32) << 16), raw);
          tmem_wait_ld();
          const int n0 = n_base + c * 32;
          if (mine && n0 < v.d_out) {
            float o[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __uint_as_float(raw[q]);
            const int w = min(32, v.d_out - n0);
            for (int j = 0; j < r; ++j) {
              const float hj = s * hrow[j];
              const uint16_t* brow = bs + j * kBN + c * 32;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (8 * q < w) {
                  float bv[8];
                  unpack8(*reinterpret_cast<const uint4*>(brow + 8 * q), bv);
#pragma unroll
                  for (int e8 = 0; e8 < 8; ++e8) o[8 * q + e8] = fmaf(hj, bv[e8], o[8 * q + e8]);
                }
              }
            }
            uint4* dst = reinterpret_cast<uint4*>(a.y + (long long)t * a.ldy + n0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (8 * q < w) {
                uint4 pk;
                pk.x = pack_bf16x2(o[8 * q + 0], o[8 * q + 1]);
                pk.y = pack_bf16x2(o[8 * q + 2], o[8 * q + 3]);
                pk.z = pack_bf16x2(o[8 * q + 4], o[8 * q + 5]);
                pk.w = pack_bf16x2(o[8 * q + 6], o[8 * q + 7]);
                dst[q] = pk;
              }
            }
          }
        }
        done = done || mine;
        epi_bar();  // the staged rows are free for the next round
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

// Per-token scale for the base kernel: s_i for every token of a segment whose
// adapter passes the checks (id, rank, every page of A_i and B_i) -- the same
// checks the shrink makes before it writes a token's h -- and 0 (set before
// this kernel) for every other token.  One warp per segment.
struct ScaleArgs {
  const int32_t* perm;
  const int32_t* indptr;
  const int32_t* seg_adapter;
  const int32_t* meta;
  float* tscale;
  DevView v;
  int32_t* err;
};

__global__ void __launch_bounds__(256) token_scale_kernel(const __grid_constant__ ScaleArgs a) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int w0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  const int n_segs = a.meta[0];
  for (int sg = w0; sg < n_segs; sg += nw) {
    const int ad = a.seg_adapter[sg];
    const lora_adapter_desc_t d = adapter_desc(a.v, ad);
    const int bad = check_adapter_warp(a.v, ad, d, lane);
    if (bad && lane == 0) report(a.err, bad);
    const float s = bad ? 0.f : d.scale;
    for (int p = a.indptr[sg] + lane; p < a.indptr[sg + 1]; p += 32) a.tscale[a.perm[p]] = s;
  }
}

}  // namespace

bool base_gemm_ok(const lora_pool_view_t* v) { return v->page_elems >= 32 && v->max_rank <= LORA_MAX_RANK; }

lora_status_t launch_base_gemm(const void* x, long long ldx, const void* w0, long long ldw, void* y, long long ldy,
                               const float* h, long long ldh, float* tscale, const int32_t* ids, int T,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream) {
  // per-token scales from the segments
  {
    ScaleArgs s;
    memset(&s, 0, sizeof(s));
    s.perm = seg->token_perm;
    s.indptr = seg->seg_indptr;
    s.seg_adapter = seg->seg_adapter;
    s.meta = seg->meta;
    s.tscale = tscale;
    make_dev_view(view, &s.v);
    s.err = err;
    if (cudaMemsetAsync(tscale, 0, (size_t)T * sizeof(float), stream) != cudaSuccess) return LORA_ERR_CUDA;
    const int blocks = std::max(1, std::min(sm_count() * 4, (T + 7) / 8));
    if (launch_pdl((const void*)token_scale_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 0, &s) !=
        cudaSuccess)
      return LORA_ERR_CUDA;
  }
  BaseArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_act_map(&a.xmap, x, T, view->d_in, ldx, kBM)) return LORA_ERR_UNSUPPORTED;
  if (!make_act_map(&a.wmap, w0, view->d_out, view->d_in, ldw, kBN)) return LORA_ERR_UNSUPPORTED;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.tscale = tscale;
  a.ids = ids;
  make_dev_view(view, &a.v);
  a.T = T;
  a.n_m = (T + kBM - 1) / kBM;
  a.n_n = (view->d_out + kBN - 1) / kBN;
  a.nk = (view->d_in + kBK - 1) / kBK;
  a.err = err;
  a.probe = wait_probe_cycles();
  if (ensure_smem_attr((const void*)base_gemm_kernel, kBSmem) != cudaSuccess) return LORA_ERR_CUDA;
  const long long tiles = (long long)a.n_m * a.n_n;
  const int grid = (int)std::min<long long>(tiles, sm_count());
  return launch_pdl((const void*)base_gemm_kernel, dim3((unsigned)grid), dim3(kBThreads), kBSmem, stream, 0, &a) ==
                 cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
