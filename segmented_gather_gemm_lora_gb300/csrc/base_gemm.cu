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
// token, fp32) and s_i the adapter's scale; a token without a usable adapter
// (id -1, or an adapter that fails the shrink's checks of id, rank and every
// page) gets the base product alone.
//
// Base product: a persistent tcgen05 GEMM over 128 x 256 output tiles.  A
// cluster of two CTAs takes the tiles (m, n) and (m + 1, n) together, pairs
// taken in order (m / 2 major, n minor) so that a wave of clusters shares W0's
// tiles in L2 and x streams once.  Warp 0 loads, per 64-column K step, its own
// TMA box of x (128 x 64) and one half (128 x 64) of the W0 box the two tiles
// share, multicast into both CTAs, all with the 128-byte swizzle, into a
// 4-stage ring: each CTA then reads two thirds of the bytes a CTA loading its
// own W0 box would.  A stage is free again once both CTAs' MMAs have read it
// (each MMA warp's commit arrives in both CTAs).  Warp 1 issues tcgen05.mma
// (M = 128, N = 256, bf16, fp32 accumulator in tensor memory), alternating two
// accumulators so that a tile's epilogue overlaps the next tile's MMAs.
//
// Adapter term: on the tensor cores, into the same accumulator, after the tile's
// K loop.  The tile's rows fall into runs of one adapter (rows without a usable
// adapter in none); each run's adapter contributes ceil(r / 16) blocks of 16
// rank rows, and a round takes two blocks:
//     D += H . Bk,  H[m, k] = s_t h[t, j(k)] if row m is in block k's run, else 0,
//                   Bk[k, n] = B_i(k)[j(k), n],  k < 32,
// with H as bf16 hi and lo parts (one 128-byte row: hi in K 0..31, lo in K
// 32..63, four K-16 MMAs per N-64 block) so that the intermediate keeps about
// fp32 accuracy.  Warps 2-17 (the epilogue) build each round's H and B in
// shared memory while the MMA warp runs the tile's K loop, then, once the
// accumulator is complete, read it 32 columns at a time (each warp a quarter of
// the tile's columns in its tensor-memory lane quarter), round once to bf16 and
// store.
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
constexpr int kBRoundK = 32;  // rank rows of one adapter-term round (two 16-row blocks)
constexpr size_t kBOffH = (size_t)kBStages * kBStageBytes;        // H: [128 rows][hi K 0..31 | lo K 0..31], 128-byte swizzle
constexpr size_t kBOffD = kBOffH + (size_t)kBM * 128;             // B rows: [4 N-blocks][32 K rows][64 bf16], 128-byte swizzle
constexpr size_t kBOffBars = kBOffD + (size_t)(kBN / 64) * kBRoundK * 128;
constexpr int kBNBars = 2 * kBStages + 2 + 2 + 2 + 1;
// control: row runs [128], run adapters [128], run scales [128], the round's blocks [2][4], the MMA's
// round words [2], runs in the tile, tensor-memory slot
constexpr size_t kBOffCtl = (kBOffBars + kBNBars * 8 + 15) / 16 * 16;
constexpr size_t kBSmem = kBOffCtl + (3 * kBM + 8 + 2 + 1 + 1) * 4 + 1024;  // + 1024-byte alignment
static_assert(kBOffH % 1024 == 0 && kBOffD % 1024 == 0, "swizzle atoms");
static_assert(kBSmem <= 232448, "shared memory of one CTA");

struct BaseArgs {
  CUtensorMap xmap;  // x [T, d_in], boxes of 128 rows x 64 columns
  CUtensorMap wmap;  // W0 [d_out, d_in], boxes of 128 rows x 64 columns (half a tile's W0 box)
  uint16_t* y;
  long long ldy;
  const float* h;  // [T, ldh]: h[t, j] = x[t] . A_i[j] for tokens with a usable adapter
  long long ldh;
  const int32_t* ids;
  DevView v;
  int T;
  int n_m, n_n, nk;
  int n_pairs;  // (m / 2, n) pairs of tiles
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
  uint64_t* delta_full = acc_empty + 2;     // [1] the epilogue: a round's H and B are staged
  uint64_t* delta_empty = delta_full + 1;   // [1] MMA commit: the round's MMAs have read them
  uint64_t* mma_done = delta_empty + 1;
  int* row_run = reinterpret_cast<int*>(sm + kBOffCtl);  // [128] the row's run in the tile (-1: none)
  int* run_ad = row_run + kBM;                            // [128] each run's adapter (-1: it failed the checks)
  float* run_s = reinterpret_cast<float*>(run_ad + kBM);  // [128] each run's scale
  int* rblk = reinterpret_cast<int*>(run_s + kBM);        // [2][4] the round's blocks: run, j0, rank, b_page0
  int* rmma = rblk + 8;                                   // [2] blocks in the round, last round of the tile
  int* nruns = rmma + 2;                                  // runs in the tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(nruns + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const uint32_t crank = cluster_ctarank(), cid = cluster_id_x(), ncl = ncluster_x();
  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 2);  // both CTAs' MMA commits
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kBEpiWarps);
    }
    mbar_init(smem_u32(delta_full), 1);
    mbar_init(smem_u32(delta_empty), 1);
    mbar_init(smem_u32(mma_done), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 2 * kBN);
  tc_fence_before();
  // every barrier of both CTAs initialised before the peer's copies or commits reach it
  cluster_sync();
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
  // this CTA's tiles: (2 (p / n_n) + crank, p % n_n) for the cluster's pairs p
  const uint32_t hbuf = smem_u32(sm + kBOffH), dbuf = smem_u32(sm + kBOffD);

  if (warp == 0) {
    // ---------------- TMA loads ----------------
    if (lane == 0 && ok) {
      prefetch_tensormap(&a.xmap);
      prefetch_tensormap(&a.wmap);
      uint32_t g = 0;
      for (int p = (int)cid; p < a.n_pairs && ok; p += (int)ncl) {
        const int m = 2 * (p / a.n_n) + (int)crank, n = p % a.n_n;
        for (int kb = 0; kb < a.nk; ++kb, ++g) {
          const uint32_t st = g % kBStages;
          if (g >= kBStages && !mbar_wait(smem_u32(&empty[st]), ((g / kBStages) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t dst = smem_u32(sm + (size_t)st * kBStageBytes);
          // this CTA's x box, then its half of the shared W0 box into both CTAs
          // (the peer's half lands here too, on the same barrier)
          mbar_arrive_expect_tx(smem_u32(&full[st]), kBStageBytes);
          tma_load_2d(dst, &a.xmap, kb * kBK, m * kBM, smem_u32(&full[st]));
          tma_load_2d_mc(dst + kBABytes + crank * (kBBBytes / 2), &a.wmap, kb * kBK, n * kBN + (int)crank * (kBN / 2),
                         smem_u32(&full[st]), (uint16_t)3u);
        }
      }
      if (!ok) report(a.err, LORA_DERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    if (lane == 0 && ok) {
      const uint32_t idesc = idesc_bf16(kBM, kBN, 0);
      const uint32_t idesc_d = idesc_bf16(kBM, 64, 1);  // the adapter term: N = 64 per block, B MN-major
      uint32_t g = 0, lt = 0, rd = 0;
      bool issued = false;
      for (int p = (int)cid; p < a.n_pairs && ok; p += (int)ncl, ++lt) {
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
          mma_commit_mc(smem_u32(&empty[st]), (uint16_t)3u);  // the stage is free in both CTAs once both read it
        }
        if (!ok) break;
        // the adapter term, a round at a time (a tile without one has one empty round)
        for (bool last = false; !last; ++rd) {
          if (!mbar_wait(smem_u32(delta_full), rd & 1)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // the epilogue's shared-memory writes, seen here, before the tensor cores read them
          tc_fence_after();
          const int nblk = rmma[0];
          last = rmma[1] != 0;
          // H's K slices: hi of blocks 0, 1, then lo of blocks 0, 1
          for (int kk = 0; kk < 4; ++kk) {
            const int bk = kk & 1;
            if (bk >= nblk) continue;
#pragma unroll
            for (int nb = 0; nb < kBN / 64; ++nb)
              mma_bf16(tmem + ab * kBN + nb * 64, sdesc_sw128(hbuf + 32 * kk, 16, 1024),
                       sdesc_sw128(dbuf + nb * (kBRoundK * 128) + bk * 2048, 0, 1024), idesc_d, 1u);
          }
          mma_commit(smem_u32(delta_empty));
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
    // Per tile: its rows' runs of one adapter; the adapter term's rounds staged
    // (H and B in shared memory), each once the MMA warp is done with the last;
    // then the accumulator rounded to bf16 and stored.
    const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
    const int row = quarter * 32 + lane;
    const int part = (warp - 2) >> 2;  // the tile's columns [64 part, 64 part + 64); H chunks part, part + 4
    const int et = tid - 64;           // 0..511
    const DevView& v = a.v;
    const int shift = v.page_shift;
    uint32_t lt = 0, rd = 0;
    for (int p = (int)cid; p < a.n_pairs; p += (int)ncl, ++lt) {
      const int m = 2 * (p / a.n_n) + (int)crank, n = p % a.n_n;
      const uint32_t ab = lt & 1;
      const int t = m * kBM + row;
      const int n_base = n * kBN;
      int ad = -1;
      if (t < a.T) {
        const int id = a.ids[t];
        if (id >= 0 && id < v.n_adapters) ad = id;
      }
      if (part == 0) row_run[row] = ad;
      epi_bar();
      if (warp == 2) {  // runs: a row starts one when its adapter differs from the row before
        int a0[kBM / 32], ap[kBM / 32];
#pragma unroll
        for (int i = 0; i < kBM / 32; ++i) {  // every row read before any is overwritten
          const int rr = 32 * i + lane;
          a0[i] = row_run[rr];
          ap[i] = rr > 0 ? row_run[rr - 1] : -1;
        }
        __syncwarp();
        int base = 0;
#pragma unroll
        for (int i = 0; i < kBM / 32; ++i) {
          const bool head = a0[i] >= 0 && a0[i] != ap[i];
          const uint32_t hm = __ballot_sync(0xffffffffu, head);
          const int k = base + __popc(hm & ((2u << lane) - 1u)) - 1;  // heads up to this row, less one
          if (head) run_ad[k] = a0[i];
          row_run[32 * i + lane] = a0[i] >= 0 ? k : -1;
          base += __popc(hm);
        }
        if (lane == 0) *nruns = base;
      }
      epi_bar();
      const int n_runs = *nruns;
      // each run's adapter checked as the shrink checks it (id, rank, every page),
      // the sixteen warps taking the runs in turn; a run that fails adds nothing
      for (int k = warp - 2; k < n_runs; k += kBEpiWarps) {
        const int rad = run_ad[k];
        const lora_adapter_desc_t dk = adapter_desc(v, rad);
        const int bad = check_adapter_warp(v, rad, dk, lane);
        __syncwarp();
        if (lane == 0) {
          run_s[k] = dk.scale;
          if (bad) run_ad[k] = -1;
        }
      }
      epi_bar();
      int my_run = row_run[row];
      if (my_run >= 0 && run_ad[my_run] < 0) my_run = -1;
      const float s = my_run >= 0 ? run_s[my_run] : 0.f;
      const float* hrow = a.h + (long long)(t < a.T ? t : 0) * a.ldh;
      // rounds: two 16-row blocks each, walking the runs that passed in order
      int cur_run = 0, cur_j0 = 0, cur_r = 0, cur_bp = 0;  // thread 0's cursor
      if (et == 0) {
        while (cur_run < n_runs && run_ad[cur_run] < 0) ++cur_run;
        if (cur_run < n_runs) {
          const lora_adapter_desc_t d0 = adapter_desc(v, run_ad[cur_run]);
          cur_r = d0.rank;
          cur_bp = d0.b_page0;
        }
      }
      for (bool last = false; !last; ++rd) {
        // the MMA warp is done with the previous round's H and B
        if (!epi_all(rd == 0 || mbar_wait(smem_u32(delta_empty), (rd - 1) & 1))) {
          ok = false;
          break;
        }
        if (et == 0) {
          int nb = 0;
          for (int b = 0; b < 2; ++b) {
            if (cur_run < n_runs) {
              rblk[4 * b] = cur_run;
              rblk[4 * b + 1] = cur_j0;
              rblk[4 * b + 2] = cur_r;
              rblk[4 * b + 3] = cur_bp;
              ++nb;
              cur_j0 += 16;
              if (cur_j0 >= cur_r) {
                cur_j0 = 0;
                ++cur_run;
                while (cur_run < n_runs && run_ad[cur_run] < 0) ++cur_run;
                if (cur_run < n_runs) {
                  const lora_adapter_desc_t d1 = adapter_desc(v, run_ad[cur_run]);
                  cur_r = d1.rank;
                  cur_bp = d1.b_page0;
                }
              }
            } else {
              rblk[4 * b] = -1;
            }
          }
          rmma[0] = nb;
          rmma[1] = cur_run >= n_runs ? 1 : 0;
        }
        epi_bar();
        last = rmma[1] != 0;
        // H: this thread's row, chunk pair `part` (K 8 part .. 8 part + 7 of block part / 2)
        if (rmma[0] > 0) {
          const int bk = part >> 1;
          const int brun = rblk[4 * bk], j = rblk[4 * bk + 1] + 8 * (part & 1), br = rblk[4 * bk + 2];
          float hv[8];
          if (brun >= 0 && my_run == brun && j < br) {
            const float4 h0 = *reinterpret_cast<const float4*>(hrow + j);
            const float4 h1 = *reinterpret_cast<const float4*>(hrow + j + 4);
            hv[0] = h0.x; hv[1] = h0.y; hv[2] = h0.z; hv[3] = h0.w;
            hv[4] = h1.x; hv[5] = h1.y; hv[6] = h1.z; hv[7] = h1.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = j + e < br ? s * hv[e] : 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = 0.f;
          }
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = pack_bf16x2(hv[2 * e], hv[2 * e + 1]);
            lo[e] = pack_bf16x2(hv[2 * e] - bf_lo(hi[e]), hv[2 * e + 1] - bf_hi(hi[e]));
          }
          *reinterpret_cast<uint4*>(sm + kBOffH + sw128_offset(row, part)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm + kBOffH + sw128_offset(row, part + 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // B: rows k of the round (block k / 16, rank row j0 + k % 16) for the tile's
        // 256 columns, 16-byte pieces through the page table, zero past the rank,
        // past d_out or without a block
#pragma unroll
        for (int u = 0; u < (kBRoundK * kBN / 8) / kBEpiThreads; ++u) {
          const int pc = et + kBEpiThreads * u;
          const int k = pc / (kBN / 8), q = pc - k * (kBN / 8);
          const int bk = k >> 4;
          const int brun = rblk[4 * bk], j = rblk[4 * bk + 1] + (k & 15), br = rblk[4 * bk + 2];
          const int col = n_base + 8 * q;
          const bool valid = brun >= 0 && j < br && col < v.d_out;
          const uint16_t* src = v.pool;
          if (valid) {
            const long long el = (long long)j * v.d_out + col;
            src = v.pool + ((long long)v.page_list[rblk[4 * bk + 3] + (el >> shift)] << shift) + (el & ((1LL << shift) - 1));
          }
          if (rmma[0] > 0) cp_async16(dbuf + (uint32_t)((q >> 3) * (kBRoundK * 128)) + sw128_offset(k, q & 7), src, valid);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();  // this thread's writes, before the tensor cores read them
        epi_bar();
        if (et == 0) mbar_arrive(smem_u32(delta_full));
      }
      if (!ok) break;
      // the accumulator: base product + adapter term
      if (!epi_all(mbar_wait(smem_u32(&acc_full[ab]), (lt >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool store = t < a.T;
      for (int c = kBEpiChunks * part; c < kBEpiChunks * (part + 1); ++c) {
        uint32_t raw[32];
        tmem_ld32_nowait(tmem + ab * kBN + c * 32 + ((uint32_t)(quarter * 32) << 16), raw);
        tmem_wait_ld();
        const int n0 = n_base + c * 32;
        if (store && n0 < v.d_out) {
          const int w = min(32, v.d_out - n0);
          uint4* dst = reinterpret_cast<uint4*>(a.y + (long long)t * a.ldy + n0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (8 * q < w) {
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(raw[8 * q + 0]), __uint_as_float(raw[8 * q + 1]));
              pk.y = pack_bf16x2(__uint_as_float(raw[8 * q + 2]), __uint_as_float(raw[8 * q + 3]));
              pk.z = pack_bf16x2(__uint_as_float(raw[8 * q + 4]), __uint_as_float(raw[8 * q + 5]));
              pk.w = pack_bf16x2(__uint_as_float(raw[8 * q + 6]), __uint_as_float(raw[8 * q + 7]));
              dst[q] = pk;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
    }
    if (!ok && lane == 0) report(a.err, LORA_DERR_TIMEOUT);
  }
  tc_fence_before();
  // neither CTA leaves while the peer may still copy into it or arrive on its barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

}  // namespace

bool base_gemm_ok(const lora_pool_view_t* v) { return v->page_elems >= 32 && v->max_rank <= LORA_MAX_RANK; }

lora_status_t launch_base_gemm(const void* x, long long ldx, const void* w0, long long ldw, void* y, long long ldy,
                               const float* h, long long ldh, const int32_t* ids, int T, const lora_pool_view_t* view,
                               int32_t* err, cudaStream_t stream) {
  BaseArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_act_map(&a.xmap, x, T, view->d_in, ldx, kBM)) return LORA_ERR_UNSUPPORTED;
  if (!make_act_map(&a.wmap, w0, view->d_out, view->d_in, ldw, kBN / 2)) return LORA_ERR_UNSUPPORTED;
  a.y = static_cast<uint16_t*>(y);
  a.ldy = ldy;
  a.h = h;
  a.ldh = ldh;
  a.ids = ids;
  make_dev_view(view, &a.v);
  a.T = T;
  a.n_m = (T + kBM - 1) / kBM;
  a.n_n = (view->d_out + kBN - 1) / kBN;
  a.nk = (view->d_in + kBK - 1) / kBK;
  a.n_pairs = (a.n_m + 1) / 2 * a.n_n;
  a.err = err;
  a.probe = wait_probe_cycles();
  if (ensure_smem_attr((const void*)base_gemm_kernel, kBSmem) != cudaSuccess) return LORA_ERR_CUDA;
  const int cap = max_active_clusters((const void*)base_gemm_kernel, kBThreads, kBSmem, 2);
  const int clusters = (int)std::min<long long>(a.n_pairs, std::max(1, cap));
  return launch_pdl((const void*)base_gemm_kernel, dim3((unsigned)(2 * clusters)), dim3(kBThreads), kBSmem, stream, 2,
                    &a) ==
                 cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
