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
// One CTA does the whole job (a batch is at most some thousands of tokens),
// sized to the batch so that its barriers stay cheap for small decode batches.
// Each thread owns a span of up to 12 consecutive tokens, loaded with all its
// loads in flight at once:
//   1. run-length pass: maximal runs of equal, valid ids; one block scan of the
//      per-thread run counts numbers the runs.  Serving batches are runs (a
//      prefill request is one run), so the grouping below works on runs;
//   2. GROUP: per-adapter token counts (shared-memory atomics on run lengths,
//      an exact integer sum); one block scan over adapters gives segment
//      starts, segment numbers and both work lists at once; one warp then walks
//      the runs in token order and hands each its place inside its adapter's
//      segment (warp match + in-order prefix), which keeps the grouping
//      stable.  CONTIGUOUS: segments are the runs, one scan over runs;
//   3. scatter of token indices to their positions;
//   work lists: segments of at most LORA_SHORT_MAX_TOKENS tokens are short
//   units; longer ones are cut into LORA_TILE_M-token tiles.
// Everything is integer arithmetic with a fixed order: the output is
// bit-exact and deterministic.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace lora {

constexpr int kSpan = 12;          // tokens per thread per pass (three 16-byte loads; 16 measured ~2 us slower on prefill)
constexpr int kSegMaxThreads = 1024;

// Exclusive scan of one counter over the CTA; *total receives the sum.  ws: 33
// ints of shared memory.
__device__ __forceinline__ int block_scan1(int v, int* total, int* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += a;
  }
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += a;
    }
    ws[lane] = wi - w;
    if (lane == 31) ws[32] = wi;
  }
  __syncthreads();
  const int base = ws[warp];
  *total = ws[32];
  __syncthreads();
  return base + inc - v;
}

// Exclusive scan of four counters at once over the CTA; *total receives the
// sums.  ws: 33 int4 of shared memory.
__device__ __forceinline__ int4 block_scan4(int4 v, int4* total, int4* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc.x, o), b = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int c = __shfl_up_sync(0xffffffffu, inc.z, o), d = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) { inc.x += a; inc.y += b; inc.z += c; inc.w += d; }
  }
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int4 w = lane < nw ? ws[lane] : make_int4(0, 0, 0, 0);
    int4 wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, wi.x, o), b = __shfl_up_sync(0xffffffffu, wi.y, o);
      const int c = __shfl_up_sync(0xffffffffu, wi.z, o), d = __shfl_up_sync(0xffffffffu, wi.w, o);
      if (lane >= o) { wi.x += a; wi.y += b; wi.z += c; wi.w += d; }
    }
    ws[lane] = make_int4(wi.x - w.x, wi.y - w.y, wi.z - w.z, wi.w - w.w);
    if (lane == 31) ws[32] = wi;
  }
  __syncthreads();
  const int4 base = ws[warp];
  *total = ws[32];
  __syncthreads();
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z, base.w + inc.w - v.w);
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

// Short / long classification of a segment of `len` tokens: (short, tiles).
__device__ __forceinline__ int2 unit_counts(int len) {
  if (len <= 0) return make_int2(0, 0);
  if (len <= LORA_SHORT_MAX_TOKENS) return make_int2(1, 0);
  return make_int2(0, (len + LORA_TILE_M - 1) / LORA_TILE_M);
}

__device__ __forceinline__ void emit_units(const SegKernelArgs& a, int s, int2 uc, int short_at, int long_at) {
  if (uc.x) a.short_units[short_at] = s;
  for (int i = 0; i < uc.y; ++i) {
    a.long_units[2 * (long_at + i)] = s;
    a.long_units[2 * (long_at + i) + 1] = i * LORA_TILE_M;
  }
}

__global__ void __launch_bounds__(kSegMaxThreads, 1) segments_kernel(const __grid_constant__ SegKernelArgs a) {
  extern __shared__ __align__(16) int dyn[];
  __shared__ int4 ws[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int T = a.T, NA = a.n_adapters;
  pdl_wait_then_release();

  int* counts = dyn;  // [NA] (GROUP)
  int* runs = a.runs_in_smem ? dyn + ((a.mode == LORA_SEG_GROUP ? NA : 0) + 3) / 4 * 4 : a.scratch;
  int* run_start = runs;
  int* run_end = runs + T;
  int* run_id = runs + 2 * T;
  int* run_pos = runs + 3 * T;
  const int per_pass = nthr * kSpan;
  const bool ids_vec = (reinterpret_cast<uintptr_t>(a.ids) & 15) == 0;  // spans start at multiples of 16 ids

  // 1. runs of equal valid ids.  A batch that fits one pass keeps its ids, its
  // predecessor id and its run numbering for step 3.
  const bool one_pass = T <= per_pass;
  int keep_v[kSpan], keep_prev = INT_MIN, keep_ex = 0;
  int bad = 0, R = 0;
  for (int base = 0; base < T; base += per_pass) {
    const int t0 = base + tid * kSpan;
    int v[kSpan];
    if (ids_vec && t0 + kSpan <= T) {  // a whole span: four 16-byte loads
#pragma unroll
      for (int q = 0; q < kSpan / 4; ++q) {
        const int4 w = reinterpret_cast<const int4*>(a.ids + t0)[q];
        v[4 * q] = w.x;
        v[4 * q + 1] = w.y;
        v[4 * q + 2] = w.z;
        v[4 * q + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kSpan; ++k) v[k] = (t0 + k < T) ? a.ids[t0 + k] : INT_MIN;
    }
    const int prev = (t0 > 0 && t0 < T) ? a.ids[t0 - 1] : INT_MIN;
    const int next = (t0 + kSpan < T) ? a.ids[t0 + kSpan] : INT_MIN;
    int heads = 0;
#pragma unroll
    for (int k = 0; k < kSpan; ++k) {
      const bool valid = v[k] >= 0 && v[k] < NA;
      if (t0 + k < T && (v[k] < -1 || v[k] >= NA)) bad = 1;
      const int before = k == 0 ? prev : v[k - 1];
      heads += (valid && before != v[k]) ? 1 : 0;
    }
    int tot;
    const int ex = block_scan1(heads, &tot, reinterpret_cast<int*>(ws));
    if (one_pass) {
#pragma unroll
      for (int k = 0; k < kSpan; ++k) keep_v[k] = v[k];
      keep_prev = prev;
      keep_ex = ex;
    }
    int rho = R + ex - 1;
#pragma unroll
    for (int k = 0; k < kSpan; ++k) {
      const bool valid = v[k] >= 0 && v[k] < NA;
      const int before = k == 0 ? prev : v[k - 1];
      const int after = k == kSpan - 1 ? next : v[k + 1];
      if (valid && before != v[k]) {
        ++rho;
        run_start[rho] = t0 + k;
        run_id[rho] = v[k];
      }
      if (valid && after != v[k]) run_end[rho] = t0 + k + 1;
    }
    R += tot;
  }
  __syncthreads();

  // 2. segments, their starts and the work lists; every run's position.
  int n_segs = 0, n_tok = 0, n_short = 0, n_long = 0;
  if (a.mode == LORA_SEG_GROUP) {
    for (int i = tid; i < NA; i += nthr) counts[i] = 0;
    __syncthreads();
    for (int rho = tid; rho < R; rho += nthr) atomicAdd(&counts[run_id[rho]], run_end[rho] - run_start[rho]);
    __syncthreads();
    for (int base = 0; base < NA; base += nthr) {
      const int ad = base + tid;
      const int c = ad < NA ? counts[ad] : 0;
      const int2 uc = unit_counts(c);
      int4 tot;
      const int4 ex = block_scan4(make_int4(c, c > 0 ? 1 : 0, uc.x, uc.y), &tot, ws);
      if (c > 0) {
        const int sidx = n_segs + ex.y;
        a.indptr[sidx] = n_tok + ex.x;
        a.seg_adapter[sidx] = ad;
        emit_units(a, sidx, uc, n_short + ex.z, n_long + ex.w);
      }
      if (ad < NA) counts[ad] = n_tok + ex.x;  // becomes the adapter's fill cursor
      n_tok += tot.x;
      n_segs += tot.y;
      n_short += tot.z;
      n_long += tot.w;
    }
    __syncthreads();
    if (warp == 0) {  // stable: runs take their places in token order
      for (int base = 0; base < R; base += 32) {
        const int rho = base + lane;
        const bool act = rho < R;
        const int ad = act ? run_id[rho] : -(lane + 2);
        const unsigned peers = __match_any_sync(0xffffffffu, ad);
        // lengths of this batch's runs with the same adapter: earlier ones and all
        // (a run's peers are few: each adapter's runs inside 32 consecutive runs)
        int pre = 0, tot = 0;
        for (unsigned m = act ? peers : 0u; m != 0; m &= m - 1) {  // an inactive lane's only peer is itself
          const int i = __ffs(m) - 1;
          const int li = run_end[base + i] - run_start[base + i];
          tot += li;
          if (i < lane) pre += li;
        }
        const int cur = act ? counts[ad] : 0;
        __syncwarp();
        if (act) run_pos[rho] = cur + pre;
        if (act && lane == __ffs(peers) - 1) counts[ad] = cur + tot;
        __syncwarp();
      }
    }
  } else {
    for (int base = 0; base < R; base += nthr) {
      const int rho = base + tid;
      const int len = rho < R ? run_end[rho] - run_start[rho] : 0;
      const int2 uc = unit_counts(len);
      int4 tot;
      const int4 ex = block_scan4(make_int4(len, 0, uc.x, uc.y), &tot, ws);
      if (rho < R) {
        a.indptr[rho] = n_tok + ex.x;
        a.seg_adapter[rho] = run_id[rho];
        run_pos[rho] = n_tok + ex.x;
        emit_units(a, rho, uc, n_short + ex.z, n_long + ex.w);
      }
      n_tok += tot.x;
      n_short += tot.z;
      n_long += tot.w;
    }
    n_segs = R;
  }
  if (tid == 0) a.indptr[n_segs] = n_tok;
  __syncthreads();

  // 3. token indices to their positions (the runs are renumbered exactly as in 1).
  // With the runs in shared memory, the positions are staged there (over the run
  // ends, which step 2 was the last to read) and leave in coalesced 16-byte stores.
  int* stage = a.runs_in_smem ? run_end : nullptr;
  // Maximal runs with every token valid keep token order: the identity.
  const bool identity = a.mode == LORA_SEG_CONTIGUOUS && n_tok == T;
  if (identity) {
    const int n4 = (reinterpret_cast<uintptr_t>(a.perm) & 15) == 0 ? T / 4 : 0;
    for (int i = tid; i < n4; i += nthr) reinterpret_cast<int4*>(a.perm)[i] = make_int4(4 * i, 4 * i + 1, 4 * i + 2, 4 * i + 3);
    for (int i = 4 * n4 + tid; i < T; i += nthr) a.perm[i] = i;
  }
  int rbase = 0;
  for (int base = identity ? T : 0; base < T; base += per_pass) {
    const int t0 = base + tid * kSpan;
    int v[kSpan];
    int prev, exx, totx;
    if (one_pass) {
#pragma unroll
      for (int k = 0; k < kSpan; ++k) v[k] = keep_v[k];
      prev = keep_prev;
      exx = keep_ex;
      totx = R;
    } else {
#pragma unroll
      for (int k = 0; k < kSpan; ++k) v[k] = (t0 + k < T) ? a.ids[t0 + k] : INT_MIN;
      prev = (t0 > 0 && t0 < T) ? a.ids[t0 - 1] : INT_MIN;
      int heads = 0;
#pragma unroll
      for (int k = 0; k < kSpan; ++k) {
        const int before = k == 0 ? prev : v[k - 1];
        heads += (v[k] >= 0 && v[k] < NA && before != v[k]) ? 1 : 0;
      }
      int tot;
      exx = block_scan1(heads, &tot, reinterpret_cast<int*>(ws));
      totx = tot;
    }
    int rho = rbase + exx - 1;
    int pos = 0;
#pragma unroll
    for (int k = 0; k < kSpan; ++k) {
      const bool valid = v[k] >= 0 && v[k] < NA;
      const int before = k == 0 ? prev : v[k - 1];
      if (valid && before != v[k]) {
        ++rho;
        pos = run_pos[rho];
      } else if (valid && k == 0) {
        pos = run_pos[rho] + (t0 - run_start[rho]);  // a run that began in an earlier span
      }
      if (valid) {
        if (stage) stage[pos++] = t0 + k;
        else a.perm[pos++] = t0 + k;
      }
    }
    rbase += totx;
  }
  if (stage && !identity) {
    __syncthreads();
    const int n4 = (reinterpret_cast<uintptr_t>(a.perm) & 15) == 0 ? n_tok / 4 : 0;  // carved buffers are aligned
    for (int i = tid; i < n4; i += nthr)
      reinterpret_cast<int4*>(a.perm)[i] = make_int4(stage[4 * i], stage[4 * i + 1], stage[4 * i + 2], stage[4 * i + 3]);
    for (int i = 4 * n4 + tid; i < n_tok; i += nthr) a.perm[i] = stage[i];
  }

  if (tid == 0) {
    a.meta[0] = n_segs;
    a.meta[1] = n_tok;
    a.meta[2] = n_short;
    a.meta[3] = n_long;
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
  // Enough threads for the token spans and for one pass over the adapters.
  int want = (T + kSpan - 1) / kSpan;
  if (mode == LORA_SEG_GROUP && n_adapters > want) want = n_adapters;
  int nthr = (want + 31) / 32 * 32;
  if (nthr < 64) nthr = 64;
  if (nthr > kSegMaxThreads) nthr = kSegMaxThreads;
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
  return launch_pdl((const void*)segments_kernel, dim3(1), dim3(nthr), dyn, stream, 0, &a) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

}  // namespace lora
