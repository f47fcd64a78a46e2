// Segment construction: group a batch's tokens by adapter id.
//
// "Multi-LoRA serving: the single translator with a thousand glossaries",
// section "SGMV: the kernel that holds it all up": SGMV groups the batch's
// tokens by adapter (it segments them) -- GROUP mode: one segment per adapter
// id, ascending id, tokens ascending inside a segment (a stable counting sort).
// "Multi-LoRA Serving in Production", section "Punica and Segmented Gather
// Matrix-Vector Multiplication (SGMV)": contiguous segments whose tokens share
// one adapter id -- CONTIGUOUS mode: one segment per maximal run.
//
// One CTA of 1024 threads does the whole job (the batch is at most a few
// thousand tokens):
//   1. run-length pass: maximal runs of equal, valid ids (block-wide scan of
//      run heads); serving batches are runs (a prefill request is one run), so
//      the sort below works on runs, not tokens;
//   2. GROUP: per-adapter token counts (shared-memory atomics on run lengths,
//      an exact integer sum), exclusive scan -> segment starts; one warp then
//      walks the runs in order and hands each its position inside its
//      adapter's segment (warp match + in-order prefix), which keeps the sort
//      stable;  CONTIGUOUS: segments are the runs, starts by a scan;
//   3. scatter of token indices to their positions;
//   4. the work lists of the compute kernels (segments of at most
//      LORA_SHORT_MAX_TOKENS tokens; LORA_TILE_M-token tiles of longer ones).
// Everything is integer arithmetic with a fixed order: the output is
// bit-exact and deterministic.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace lora {

constexpr int kSegThreads = 1024;

// Exclusive scan over the CTA; *total receives the sum.  ws: 33 ints of smem.
__device__ __forceinline__ int block_scan_ex(int v, int* total, int* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    ws[lane] = wi - w;
    if (lane == 31) ws[32] = wi;
  }
  __syncthreads();
  int ex = ws[warp] + incl - v;
  *total = ws[32];
  __syncthreads();
  return ex;
}

struct SegKernelArgs {
  const int32_t* ids;
  int T;
  int n_adapters;
  int mode;
  int runs_in_smem;
  int32_t* perm;
  int32_t* indptr;
  int32_t* seg_adapter;
  int32_t* meta;
  int32_t* short_units;
  int32_t* long_units;
  int32_t* scratch;  // global run arrays when they do not fit in shared memory
  int32_t* err;
};

__global__ void __launch_bounds__(kSegThreads, 1) segments_kernel(const __grid_constant__ SegKernelArgs a) {
  extern __shared__ __align__(16) int dyn[];
  __shared__ int ws[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, NA = a.n_adapters;

  int* counts = dyn;  // [NA] (GROUP)
  int* runs = a.runs_in_smem ? dyn + ((a.mode == LORA_SEG_GROUP ? NA : 0) + 3) / 4 * 4 : a.scratch;
  int* run_start = runs;
  int* run_end = runs + T;
  int* run_id = runs + 2 * T;
  int* run_pos = runs + 3 * T;

  // 1. runs of equal valid ids.
  int bad = 0, R = 0;
  for (int base = 0; base < T; base += kSegThreads) {
    const int t = base + tid;
    const int id = t < T ? a.ids[t] : -1;
    const bool valid = t < T && id >= 0 && id < NA;
    if (t < T && (id < -1 || id >= NA)) bad = 1;
    const int prev = (t > 0 && t < T) ? a.ids[t - 1] : INT_MIN;
    const int next = (t + 1 < T) ? a.ids[t + 1] : INT_MIN;
    const bool head = valid && (t == 0 || prev != id);
    const bool tail = valid && (t == T - 1 || next != id);
    int total;
    const int ex = block_scan_ex(head ? 1 : 0, &total, ws);
    const int rho = R + ex + (head ? 1 : 0) - 1;
    if (head) {
      run_start[rho] = t;
      run_id[rho] = id;
    }
    if (tail) run_end[rho] = t + 1;
    R += total;
  }
  __syncthreads();

  // 2. segment starts and every run's position.
  int n_segs = 0, n_tok = 0;
  if (a.mode == LORA_SEG_GROUP) {
    for (int i = tid; i < NA; i += kSegThreads) counts[i] = 0;
    __syncthreads();
    for (int rho = tid; rho < R; rho += kSegThreads)
      atomicAdd(&counts[run_id[rho]], run_end[rho] - run_start[rho]);
    __syncthreads();
    for (int base = 0; base < NA; base += kSegThreads) {
      const int ad = base + tid;
      const int c = ad < NA ? counts[ad] : 0;
      const int ne = c > 0 ? 1 : 0;
      int tc, tn;
      const int exc = block_scan_ex(c, &tc, ws);
      const int exn = block_scan_ex(ne, &tn, ws);
      if (ne) {
        a.indptr[n_segs + exn] = n_tok + exc;
        a.seg_adapter[n_segs + exn] = ad;
      }
      if (ad < NA) counts[ad] = n_tok + exc;  // becomes the adapter's fill cursor
      n_tok += tc;
      n_segs += tn;
    }
    __syncthreads();
    if (warp == 0) {  // stable: runs take their places in token order
      for (int base = 0; base < R; base += 32) {
        const int rho = base + lane;
        const bool act = rho < R;
        const int ad = act ? run_id[rho] : -(lane + 2);
        const int len = act ? run_end[rho] - run_start[rho] : 0;
        const unsigned peers = __match_any_sync(0xffffffffu, ad);
        int pre = 0, tot = 0;
        for (int i = 0; i < 32; ++i) {
          const int li = __shfl_sync(0xffffffffu, len, i);
          if ((peers >> i) & 1u) {
            tot += li;
            if (i < lane) pre += li;
          }
        }
        const int cur = act ? counts[ad] : 0;
        __syncwarp();
        if (act) run_pos[rho] = cur + pre;
        if (act && lane == __ffs(peers) - 1) counts[ad] = cur + tot;
        __syncwarp();
      }
    }
  } else {
    for (int base = 0; base < R; base += kSegThreads) {
      const int rho = base + tid;
      const int len = rho < R ? run_end[rho] - run_start[rho] : 0;
      int tot;
      const int ex = block_scan_ex(len, &tot, ws);
      if (rho < R) {
        a.indptr[rho] = n_tok + ex;
        a.seg_adapter[rho] = run_id[rho];
        run_pos[rho] = n_tok + ex;
      }
      n_tok += tot;
    }
    n_segs = R;
  }
  if (tid == 0) a.indptr[n_segs] = n_tok;
  __syncthreads();

  // 3. token indices to their positions.
  int rbase = 0;
  for (int base = 0; base < T; base += kSegThreads) {
    const int t = base + tid;
    const int id = t < T ? a.ids[t] : -1;
    const bool valid = t < T && id >= 0 && id < NA;
    const int prev = (t > 0 && t < T) ? a.ids[t - 1] : INT_MIN;
    const bool head = valid && (t == 0 || prev != id);
    int total;
    const int ex = block_scan_ex(head ? 1 : 0, &total, ws);
    if (valid) {
      const int rho = rbase + ex + (head ? 1 : 0) - 1;
      a.perm[run_pos[rho] + (t - run_start[rho])] = t;
    }
    rbase += total;
  }
  __syncthreads();

  // 4. work lists.
  int ns = 0, nl = 0;
  for (int base = 0; base < n_segs; base += kSegThreads) {
    const int s = base + tid;
    const bool act = s < n_segs;
    const int len = act ? a.indptr[s + 1] - a.indptr[s] : 0;
    const int sh = (act && len <= LORA_SHORT_MAX_TOKENS) ? 1 : 0;
    const int tiles = (act && !sh) ? (len + LORA_TILE_M - 1) / LORA_TILE_M : 0;
    int ts, tl;
    const int exs = block_scan_ex(sh, &ts, ws);
    const int exl = block_scan_ex(tiles, &tl, ws);
    if (sh) a.short_units[ns + exs] = s;
    for (int i = 0; i < tiles; ++i) {
      a.long_units[2 * (nl + exl + i)] = s;
      a.long_units[2 * (nl + exl + i) + 1] = i * LORA_TILE_M;
    }
    ns += ts;
    nl += tl;
  }
  if (tid == 0) {
    a.meta[0] = n_segs;
    a.meta[1] = n_tok;
    a.meta[2] = ns;
    a.meta[3] = nl;
    a.meta[4] = R;
    a.meta[5] = 0;
    a.meta[6] = 0;
    a.meta[7] = 0;
  }
  if (__syncthreads_or(bad) && tid == 0) report(a.err, LORA_DERR_BAD_ADAPTER);
}

lora_status_t launch_segments(const int32_t* ids, int T, int n_adapters, int mode,
                              const lora_segments_t* seg, int32_t* err, cudaStream_t stream) {
  const size_t counts_bytes = mode == LORA_SEG_GROUP ? ((size_t)n_adapters + 3) / 4 * 16 : 0;
  const size_t runs_bytes = (size_t)4 * T * sizeof(int);
  const size_t smem_cap = 200 * 1024;
  int runs_in_smem = counts_bytes + runs_bytes <= smem_cap ? 1 : 0;
  const size_t dyn = counts_bytes + (runs_in_smem ? runs_bytes : 0);
  if (dyn > smem_cap) return LORA_ERR_UNSUPPORTED;
  if (ensure_smem_attr((const void*)segments_kernel, dyn) != cudaSuccess) return LORA_ERR_CUDA;
  SegKernelArgs a;
  a.ids = ids;
  a.T = T;
  a.n_adapters = n_adapters;
  a.mode = mode;
  a.runs_in_smem = runs_in_smem;
  a.perm = seg->token_perm;
  a.indptr = seg->seg_indptr;
  a.seg_adapter = seg->seg_adapter;
  a.meta = seg->meta;
  a.short_units = seg->short_units;
  a.long_units = seg->long_units;
  a.scratch = seg->scratch;
  a.err = err;
  segments_kernel<<<1, kSegThreads, dyn, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace lora
