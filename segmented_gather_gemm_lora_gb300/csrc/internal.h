// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_sgmv.h"

namespace lora {

struct DevView;

// Raise a kernel's dynamic shared-memory limit on the current device (once per
// device and size).
cudaError_t ensure_smem_attr(const void* func, size_t bytes);

// Launch `func` (whose only parameter is the struct at `args`) with a cluster
// of `cluster_x` CTAs (0 = launched without clusters) and programmatic stream serialization,
// so it may start while its predecessor in the stream finishes; the kernel
// itself waits for the predecessor before touching global memory.
cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster_x,
                       void* args);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Clusters of `cluster_x` CTAs of `func` (block threads, smem dynamic bytes,
// its shared-memory attribute already raised) that the current device holds
// at once (cached).
int max_active_clusters(const void* func, int block, size_t smem, int cluster_x);

// Fill a DevView from a validated host view.
void make_dev_view(const lora_pool_view_t* v, DevView* out);

// While one of these lives on a host thread, the views that thread's launches
// build see every adapter transposed: B_i in the role of A_i and A_i in the
// role of B_i (the backward pass runs the shrink over B_i and the expand over
// A_i); the host view given to them has d_in and d_out exchanged to match.
struct TransposedViews {
  TransposedViews();
  ~TransposedViews();
};

// The checks every compute call makes on a view (LORA_OK if it passes).
lora_status_t validate_view(const lora_pool_view_t* v);

// Count one kernel launch made without launch_pdl (lora_launch_count).
void count_launch();

// The wait limit, in cycles, of the timeout probe lora_debug_wait_probe armed
// (0: no probe).  The compute kernels pass it to their CTAs.
long long wait_probe_cycles();

lora_status_t launch_segments(const int32_t* ids, int T, int n_adapters, int mode,
                              const lora_segments_t* seg, int32_t* err, cudaStream_t stream);

// One projection of a call: its activations, optional fp32 output and view.
constexpr int kMaxFusedProj = LORA_MAX_PROJ;
struct ProjCall {
  const void* x;
  long long ldx;
  void* y;  // bf16 y, updated in place (or only read, for y0, when yf is set)
  long long ldy;
  float* yf;  // optional fp32 output
  long long ldyf;
  const lora_pool_view_t* view;
  float* h = nullptr;  // non-null: the fused kernel also writes h rows by token, unscaled
  long long ldh = 0;   // (its only output in the shrink-only form)
};

enum GatherMode { kModeApply = 0, kModeShrink = 1, kModeExpand = 2 };
enum GatherSrc { kSrcSegments = 0, kSrcTokens = 1 };

// CUDA-core gather kernel over the segments' work lists (short units, then
// long tiles unless short_only, when the tensor-core kernels take them) or over
// one-token units.
// The gather kernel over n_proj projections that share the segments (apply
// mode): a unit is (segment or token, projection), projections fastest.  h, and
// projs[0].yf, only with one projection.
lora_status_t launch_gather_multi(int mode, int src, int short_only, int n_proj, const ProjCall* projs, float* h,
                                  long long ldh, const lora_segments_t* seg, const int32_t* token_adapter, int T,
                                  int32_t* err, cudaStream_t stream);

// yf (apply mode only): when non-null, outputs go to yf as fp32 [T, ldyf] and y
// is only read (for y0).
lora_status_t launch_gather(int mode, int src, int short_only, const void* x, long long ldx, void* y,
                            long long ldy, float* h, long long ldh, const lora_segments_t* seg,
                            const int32_t* token_adapter, int T, const lora_pool_view_t* view,
                            int32_t* err, cudaStream_t stream, float* yf = nullptr, long long ldyf = 0);

// Decode kernel (bgmv.cu): one token per cluster, small CTAs, for views with
// max_rank <= 16 whose slices fit one 512-column sub-slice (d_in, d_out <=
// 4096) and whose adapters span at most 128 page-list slots.  early: read the
// ids and the pool before the predecessor grid finishes (LORA_BGMV_STATIC_ADAPTERS).
bool bgmv_decode_ok(const lora_pool_view_t* v, int T);
lora_status_t launch_bgmv(const void* x, long long ldx, void* y, long long ldy, const int32_t* ids, int T,
                          const lora_pool_view_t* view, int early, int32_t* err, cudaStream_t stream);

// Base projection with the adapter term (base_gemm.cu): the tcgen05 GEMM
// y = x W0^T + s_i h[t] B_i for tokens whose adapter passes the shrink's
// checks.  h: [T, ldh] by token, as the shrink writes it; ids: the tokens'
// adapters.
bool base_gemm_ok(const lora_pool_view_t* v);
lora_status_t launch_base_gemm(const void* x, long long ldx, const void* w0, long long ldw, void* y, long long ldy,
                               const float* h, long long ldh, const int32_t* ids, int T, const lora_pool_view_t* view,
                               int32_t* err, cudaStream_t stream);

// Slices of d_in the tensor-core shrink splits a tile into (ks, each of klen
// columns, a multiple of 64; the last may be shorter): about 512 columns each,
// at most kMaxKSplit.  A function of d_in alone, so a token's h does not depend
// on the rest of the batch; the staged and the fused tensor-core paths use the
// same slices and so compute the same h bit for bit.
constexpr int kMaxKSplit = 4;
void shrink_split(int d_in, int* ks, int* klen);

// Gradients of adapters' A and B from a batch's segments (backward.cu):
// dB_i += s_i h^T dy and dA_i += s_i u^T x over each segment's tokens, added
// into grad_pool at the elements' pool positions.  h and u by token, fp32.
lora_status_t launch_grad(const void* x, long long ldx, const void* dy, long long lddy, const float* h,
                          const float* u, long long ldh, float* grad_pool, const lora_segments_t* seg,
                          const lora_pool_view_t* view, int32_t* err, cudaStream_t stream);

// Tensor-core path for long tiles.  Eligibility: d_in % 64 == 0 (shrink),
// d_out % 128 == 0 (expand), pages of at least 128 elements.
bool tc_shrink_ok(const lora_pool_view_t* v);
bool tc_expand_ok(const lora_pool_view_t* v);
// Fused tensor-core path (tc_fused.cu): shrink, exchange of the intermediate
// between the CTAs of a cluster and expand of each long tile in one kernel, for
// up to kMaxFusedProj projections that share the segments and d_in.
// Eligibility: d_in % 64 == 0, d_out % 64 == 0.  With projs[g].h set the kernel
// also writes each long tile's h rows (unscaled, by token); with shrink_only it
// writes them and runs no expand (eligibility then: d_in % 64 == 0).
bool tc_fused_ok(const lora_pool_view_t* v);
bool tc_fused_shrink_ok(const lora_pool_view_t* v);
lora_status_t launch_fused_tc(int n_proj, const ProjCall* projs, const lora_segments_t* seg, int after_gather,
                              int32_t* err, cudaStream_t stream, int shrink_only = 0);

// lora_apply through the staged tensor-core kernels (shrink_tc, reduce_partials,
// expand_tc) with the intermediate in seg->h_scratch; arguments checked as for
// lora_apply.  Same results as lora_apply, bit for bit.
lora_status_t apply_staged(const void* x, long long ldx, void* y, long long ldy, const lora_segments_t* seg,
                           const lora_pool_view_t* view, int32_t* err, cudaStream_t stream);

// after_gather: the gather kernel of the same call was launched just before
// (the two touch disjoint data), so this grid need not wait for it.
lora_status_t launch_shrink_tc(const void* x, long long ldx, float* h, long long ldh, int h_by_token, int after_gather,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream);
// after_gather: as for launch_shrink_tc; only in expand-only calls (lora_apply's
// expand reads the h its shrink wrote and waits).
// yf: as for launch_gather.
lora_status_t launch_expand_tc(const float* h, long long ldh, int h_by_token, int after_gather, void* y, long long ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* err,
                               cudaStream_t stream, float* yf = nullptr, long long ldyf = 0);

}  // namespace lora
