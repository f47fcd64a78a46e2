// lora_apply_fixed_scratch: lora_apply whose scratch lives in the library.
//
// The staged tensor-core path of lora_apply (a shrink grid, then an expand
// grid) keeps the rank-r intermediate of long segments in global memory
// between the two, in seg->h_scratch, memory the caller sized and allocated.
// Some callers can neither size nor request such a workspace: their device
// memory is planned once, at start-up, by a host runtime that hands the
// library only the activation, weight and segment buffers, and they cannot
// call cudaMalloc afterwards.  For them this entry point runs that staged path
// with the intermediate in a fixed-size array that is part of the library's
// own device image: it is created when the library is loaded onto a GPU and
// stays there until the process exits.  Nothing is allocated per call.  The
// result equals lora_apply's bit for bit (the staged and fused tensor-core
// kernels split and sum the same way).
#include "internal.h"

namespace {

// Scratch for LORA_FIXED_SCRATCH_MAX_TOKENS tokens x LORA_MAX_RANK fp32 values
// (4 MiB).  In host code `g_fixed_h` only stands in for the symbol: its device
// address comes from cudaGetSymbolAddress on the current device.
static __device__ __align__(256) float g_fixed_h[(size_t)LORA_FIXED_SCRATCH_MAX_TOKENS * LORA_MAX_RANK];

// Device address of g_fixed_h on the current device and context.  Looked up on
// every call (a host-side query, no device work): a cached address could be
// stale after a device reset or under another context.
lora_status_t fixed_scratch_address(float** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fixed_h) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return LORA_ERR_CUDA;
  }
  *out = static_cast<float*>(p);
  return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_apply_fixed_scratch(const void* x, int64_t ldx, void* y, int64_t ldy,
                                                   const lora_segments_t* seg, const lora_pool_view_t* view,
                                                   int32_t* dev_err, lora_stream_t stream) {
  if (seg == nullptr) return LORA_ERR_INVALID_ARG;
  if (seg->T > LORA_FIXED_SCRATCH_MAX_TOKENS) return LORA_ERR_UNSUPPORTED;
  float* h = nullptr;
  const lora_status_t st = fixed_scratch_address(&h);
  if (st != LORA_OK) return st;
  // Same arguments and results as lora_apply, through the staged kernels, which
  // keep the intermediate in global memory between the shrink and the expand:
  // here in the library's array instead of the caller's h_scratch.
  lora_segments_t local = *seg;
  local.h_scratch = h;
  return lora::apply_staged(x, ldx, y, ldy, &local, view, dev_err, (cudaStream_t)stream);
}
