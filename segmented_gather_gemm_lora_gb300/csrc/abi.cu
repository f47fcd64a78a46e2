// C ABI entry points: host-side argument checks, then launches on the caller's
// stream.  Nothing here allocates device memory or synchronises.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lora {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }

int log2i(long long v) {
  int s = 0;
  while ((1LL << s) < v) ++s;
  return s;
}

lora_status_t check_view(const lora_pool_view_t* v) {
  if (v == nullptr) return LORA_ERR_INVALID_ARG;
  if (v->pool == nullptr || v->page_list == nullptr || v->adapters == nullptr) return LORA_ERR_INVALID_ARG;
  if (!aligned16(v->pool)) return LORA_ERR_INVALID_ARG;
  if (v->n_pages < 1 || v->n_page_list < 1 || v->n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (v->page_elems < 8 || v->page_elems % 8 != 0) return LORA_ERR_INVALID_ARG;
  if (!is_pow2(v->page_elems) || v->page_elems < 64 || v->page_elems > (1 << 30)) return LORA_ERR_UNSUPPORTED;
  if (v->d_in < 8 || v->d_out < 8 || v->d_in % 8 != 0 || v->d_out % 8 != 0) return LORA_ERR_INVALID_ARG;
  if (v->max_rank < 1) return LORA_ERR_INVALID_ARG;
  if (v->max_rank > LORA_MAX_RANK) return LORA_ERR_UNSUPPORTED;
  if (v->n_pages > (1LL << 40) / v->page_elems) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

lora_status_t check_seg(const lora_segments_t* s) {
  if (s == nullptr) return LORA_ERR_INVALID_ARG;
  if (s->T < 0) return LORA_ERR_INVALID_ARG;
  if (s->T == 0) return LORA_OK;
  if (!s->token_perm || !s->seg_indptr || !s->seg_adapter || !s->meta || !s->short_units ||
      !s->long_units || !s->scratch || !s->h_scratch || !s->k_partials)
    return LORA_ERR_INVALID_ARG;
  const long long need = (long long)s->T / LORA_TILE_M + (long long)s->T / (LORA_SHORT_MAX_TOKENS + 1) + 1;
  if (s->max_long_units < need) return LORA_ERR_WORKSPACE;
  return LORA_OK;
}

// An activation matrix [T, ld] of bf16 with `width` used columns.
lora_status_t check_act(const void* p, long long ld, int width, int T) {
  if (T == 0) return LORA_OK;
  if (p == nullptr || !aligned16(p)) return LORA_ERR_INVALID_ARG;
  if (ld < width || ld % 8 != 0) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

bool overlap(const void* a, long long abytes, const void* b, long long bbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t ensure_smem_attr(const void* func, size_t bytes) {
  // A few kernels, each raised once per device to its largest request.
  static std::atomic<size_t> cache[8][kMaxDevices];
  static std::atomic<const void*> funcs[8];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  int slot = -1;
  for (int i = 0; i < 8; ++i) {
    const void* f = funcs[i].load();
    if (f == func) { slot = i; break; }
    if (f == nullptr) {
      const void* expected = nullptr;
      if (funcs[i].compare_exchange_strong(expected, func) || expected == func) { slot = i; break; }
    }
  }
  if (slot >= 0 && cache[slot][dev].load() >= bytes) return cudaSuccess;
  // Raised even below 48 KB: the default limit covers dynamic and static shared
  // memory together, so a kernel with static shared memory of its own needs the
  // attribute for a dynamic size just under 48 KB too.
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && slot >= 0) {
    size_t cur = cache[slot][dev].load();
    while (cur < bytes && !cache[slot][dev].compare_exchange_weak(cur, bytes)) {}
  }
  return e;
}

std::atomic<uint64_t> g_launches{0};
std::atomic<long long> g_wait_probe{0};

long long wait_probe_cycles() { return g_wait_probe.load(std::memory_order_relaxed); }

int max_active_clusters(const void* func, int block, size_t smem, int cluster_x) {
  struct Entry {
    int dev;
    const void* func;
    int block;
    size_t smem;
    int cluster_x;
    int n;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cache = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i) {
    const Entry& e = cache[i];
    if (e.dev == dev && e.func == func && e.block == block && e.smem == smem && e.cluster_x == cluster_x) return e.n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster_x);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cluster_x;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  if (n_cache < 32) cache[n_cache++] = Entry{dev, func, block, smem, cluster_x, n};
  return n;
}

cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster_x,
                       void* args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x >= 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  void* params[1] = {args};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, func, params);
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices) {
    int c = g_sm_count[dev].load();
    if (c > 0) return c;
  }
  int c = 1;
  if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1) c = 1;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(c);
  return c;
}

lora_status_t validate_view(const lora_pool_view_t* v) { return check_view(v); }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

thread_local bool t_transposed = false;

TransposedViews::TransposedViews() { t_transposed = true; }
TransposedViews::~TransposedViews() { t_transposed = false; }

void make_dev_view(const lora_pool_view_t* v, DevView* out) {
  out->swap_ab = t_transposed ? 1 : 0;
  out->pool = static_cast<const uint16_t*>(v->pool);
  out->page_list = v->page_list;
  out->adapters = v->adapters;
  out->n_pages = v->n_pages;
  out->n_page_list = v->n_page_list;
  out->n_adapters = v->n_adapters;
  out->page_shift = log2i(v->page_elems);
  out->max_rank = v->max_rank;
  out->d_in = v->d_in;
  out->d_out = v->d_out;
}

}  // namespace lora

using namespace lora;

extern "C" {

int32_t lora_abi_version(void) { return LORA_ABI_VERSION; }

const char* lora_status_string(lora_status_t s) {
  switch (s) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID_ARG: return "invalid argument";
    case LORA_ERR_UNSUPPORTED: return "unsupported by this build";
    case LORA_ERR_CUDA: return "CUDA runtime error";
    case LORA_ERR_WORKSPACE: return "segment buffer or adapter pool too small";
    default: return "unknown status";
  }
}

int64_t lora_pool_pages_needed(int32_t rank, int32_t d_in, int32_t d_out, int32_t page_elems) {
  if (rank < 0 || d_in < 0 || d_out < 0 || page_elems < 1) return -1;
  const int64_t a = (int64_t)rank * d_in, b = (int64_t)rank * d_out;
  return (a + page_elems - 1) / page_elems + (b + page_elems - 1) / page_elems;
}

static size_t seg_layout(int32_t T, size_t* off) {
  // token_perm, seg_indptr, seg_adapter, meta, short_units, long_units, scratch, h_scratch,
  // k_partials
  const size_t t = (size_t)(T > 0 ? T : 0);
  const size_t n_long = t / LORA_TILE_M + t / (LORA_SHORT_MAX_TOKENS + 1) + 1;
  const size_t sizes[9] = {t, t + 1, t, 8, t, 2 * n_long, 4 * t + 8, t * LORA_MAX_RANK,
                           (size_t)LORA_KSPLIT_MAX * t * LORA_MAX_RANK};
  size_t cur = 0;
  for (int i = 0; i < 9; ++i) {
    if (off) off[i] = cur;
    cur = align_up(cur + sizes[i] * sizeof(int32_t), 16);
  }
  return cur;
}

size_t lora_segments_buffer_bytes(int32_t T) {
  if (T < 0) return 0;
  return seg_layout(T, nullptr);
}

lora_status_t lora_segments_carve(void* buf, size_t bytes, int32_t T, lora_segments_t* out) {
  if (out == nullptr || T < 0) return LORA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (buf == nullptr || !aligned16(buf)) return LORA_ERR_INVALID_ARG;
  size_t off[9];
  const size_t need = seg_layout(T, off);
  if (bytes < need) return LORA_ERR_WORKSPACE;
  char* b = static_cast<char*>(buf);
  out->T = T;
  out->max_long_units = (int32_t)(T / LORA_TILE_M + T / (LORA_SHORT_MAX_TOKENS + 1) + 1);
  out->token_perm = reinterpret_cast<int32_t*>(b + off[0]);
  out->seg_indptr = reinterpret_cast<int32_t*>(b + off[1]);
  out->seg_adapter = reinterpret_cast<int32_t*>(b + off[2]);
  out->meta = reinterpret_cast<int32_t*>(b + off[3]);
  out->short_units = reinterpret_cast<int32_t*>(b + off[4]);
  out->long_units = reinterpret_cast<int32_t*>(b + off[5]);
  out->scratch = reinterpret_cast<int32_t*>(b + off[6]);
  out->h_scratch = reinterpret_cast<float*>(b + off[7]);
  out->k_partials = reinterpret_cast<float*>(b + off[8]);
  return LORA_OK;
}

lora_status_t lora_segments_build(const int32_t* token_adapter, int32_t T, int32_t n_adapters,
                                  int32_t mode, const lora_segments_t* seg, int32_t* dev_err,
                                  lora_stream_t stream) {
  if (seg == nullptr || T < 0 || T != seg->T) return LORA_ERR_INVALID_ARG;
  if (mode != LORA_SEG_GROUP && mode != LORA_SEG_CONTIGUOUS) return LORA_ERR_INVALID_ARG;
  if (n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (n_adapters > LORA_MAX_ADAPTERS) return LORA_ERR_UNSUPPORTED;
  if (seg->meta == nullptr || seg->seg_indptr == nullptr) return LORA_ERR_INVALID_ARG;
  if (T > 0 && token_adapter == nullptr) return LORA_ERR_INVALID_ARG;
  lora_status_t st = check_seg(seg);
  if (st != LORA_OK) return st;
  return launch_segments(token_adapter, T, n_adapters, mode, seg, dev_err, (cudaStream_t)stream);
}

static lora_status_t run_segmented(int mode, const void* x, long long ldx, void* y, long long ldy,
                                   float* h, long long ldh, const lora_segments_t* seg,
                                   const lora_pool_view_t* view, int32_t* dev_err, cudaStream_t s,
                                   float* yf = nullptr, long long ldyf = 0, bool staged = false) {
  // Long tiles go to the tensor-core kernels when the shapes allow it: the fused
  // kernel for lora_apply, the staged ones for the separate stages.
  // A shrink alone goes to the fused kernel's shrink-only form when it can (its
  // cluster sums the d_in slices on chip), else to the staged shrink.
  bool tc;
  const bool fused_shrink = mode == kModeShrink && tc_fused_shrink_ok(view);
  if (mode == kModeApply) tc = staged ? tc_shrink_ok(view) && tc_expand_ok(view) : tc_fused_ok(view);
  else if (mode == kModeShrink) tc = fused_shrink || tc_shrink_ok(view);
  else tc = tc_expand_ok(view);
  lora_status_t st = launch_gather(mode, kSrcSegments, tc ? 1 : 0, x, ldx, y, ldy, h, ldh, seg, nullptr, 0, view,
                                   dev_err, s, yf, ldyf);
  if (st != LORA_OK || !tc) return st;
  // the gather kernel was launched iff the buffer has tokens (its short-only bound is T)
  const int after_gather = seg->T > 0 ? 1 : 0;
  if (mode == kModeApply && !staged) {
    ProjCall p{x, ldx, y, ldy, yf, ldyf, view};
    p.h = h;  // with an h array, the apply writes its intermediate there too
    p.ldh = ldh;
    return launch_fused_tc(1, &p, seg, after_gather, dev_err, s);
  }
  if (mode == kModeApply) {
    st = launch_shrink_tc(x, ldx, seg->h_scratch, LORA_MAX_RANK, 0, after_gather, seg, view, dev_err, s);
    if (st != LORA_OK) return st;
    return launch_expand_tc(seg->h_scratch, LORA_MAX_RANK, 0, 0, y, ldy, seg, view, dev_err, s, yf, ldyf);
  }
  if (fused_shrink) {
    ProjCall p{x, ldx, nullptr, 0, nullptr, 0, view};
    p.h = h;
    p.ldh = ldh;
    return launch_fused_tc(1, &p, seg, after_gather, dev_err, s, 1);
  }
  if (mode == kModeShrink) return launch_shrink_tc(x, ldx, h, ldh, 1, after_gather, seg, view, dev_err, s);
  return launch_expand_tc(h, ldh, 1, after_gather, y, ldy, seg, view, dev_err, s);
}

// The checks of lora_apply.
static lora_status_t check_apply(const void* x, long long ldx, void* y, long long ldy, const lora_segments_t* seg,
                                 const lora_pool_view_t* view) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if ((st = check_act(y, ldy, view->d_out, T)) != LORA_OK) return st;
  if (T > 0 && overlap(x, (long long)T * ldx * 2, y, (long long)T * ldy * 2)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status_t lora_sgmv_shrink(const void* x, int64_t ldx, float* h, int64_t ldh,
                               const lora_segments_t* seg, const lora_pool_view_t* view,
                               int32_t* dev_err, lora_stream_t stream) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if (T > 0 && (h == nullptr || !aligned16(h) || ldh < view->max_rank || ldh % 4 != 0)) return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  return run_segmented(kModeShrink, x, ldx, nullptr, 0, h, ldh, seg, view, dev_err, (cudaStream_t)stream);
}

lora_status_t lora_sgmv_expand(const float* h, int64_t ldh, void* y, int64_t ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view,
                               int32_t* dev_err, lora_stream_t stream) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(y, ldy, view->d_out, T)) != LORA_OK) return st;
  if (T > 0 && (h == nullptr || !aligned16(h) || ldh < view->max_rank || ldh % 4 != 0)) return LORA_ERR_INVALID_ARG;
  if (T > 0 && overlap(h, (long long)T * ldh * 4, y, (long long)T * ldy * 2)) return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  return run_segmented(kModeExpand, nullptr, 0, y, ldy, const_cast<float*>(h), ldh, seg, view, dev_err,
                       (cudaStream_t)stream);
}

lora_status_t lora_apply(const void* x, int64_t ldx, void* y, int64_t ldy, const lora_segments_t* seg,
                         const lora_pool_view_t* view, int32_t* dev_err, lora_stream_t stream) {
  const lora_status_t st = check_apply(x, ldx, y, ldy, seg, view);
  if (st != LORA_OK || seg->T == 0) return st;
  return run_segmented(kModeApply, x, ldx, y, ldy, nullptr, 0, seg, view, dev_err, (cudaStream_t)stream);
}

lora_status_t lora_apply_multi(const lora_proj_t* projs, int32_t n_proj, const lora_segments_t* seg,
                               int32_t* dev_err, lora_stream_t stream) {
  if (projs == nullptr || n_proj < 1) return LORA_ERR_INVALID_ARG;
  if (n_proj > LORA_MAX_PROJ) return LORA_ERR_UNSUPPORTED;
  lora_status_t st = check_seg(seg);
  if (st != LORA_OK) return st;
  const int T = seg->T;
  ProjCall calls[LORA_MAX_PROJ];
  bool tc = true;
  for (int g = 0; g < n_proj; ++g) {
    const lora_proj_t& p = projs[g];
    if ((st = check_view(&p.view)) != LORA_OK) return st;
    if (p.view.d_in != projs[0].view.d_in) return LORA_ERR_INVALID_ARG;
    if ((st = check_act(p.x, p.ldx, p.view.d_in, T)) != LORA_OK) return st;
    if ((st = check_act(p.y, p.ldy, p.view.d_out, T)) != LORA_OK) return st;
    calls[g] = ProjCall{p.x, p.ldx, p.y, p.ldy, nullptr, 0, &p.view};
    tc = tc && tc_fused_ok(&p.view);
  }
  if (T == 0) return LORA_OK;
  for (int g = 0; g < n_proj; ++g)  // no output overlaps an input or another output
    for (int k = 0; k < n_proj; ++k) {
      const lora_proj_t &pg = projs[g], &pk = projs[k];
      if (overlap(pg.y, (long long)T * pg.ldy * 2, pk.x, (long long)T * pk.ldx * 2)) return LORA_ERR_INVALID_ARG;
      if (k != g && overlap(pg.y, (long long)T * pg.ldy * 2, pk.y, (long long)T * pk.ldy * 2))
        return LORA_ERR_INVALID_ARG;
    }
  const cudaStream_t s = (cudaStream_t)stream;
  st = launch_gather_multi(kModeApply, kSrcSegments, tc ? 1 : 0, n_proj, calls, nullptr, 0, seg, nullptr, 0,
                           dev_err, s);
  if (st != LORA_OK || !tc) return st;
  return launch_fused_tc(n_proj, calls, seg, 1, dev_err, s);
}

lora_status_t lora_apply_f32y(const void* x, int64_t ldx, const void* y0, int64_t ldy0, float* yf, int64_t ldyf,
                              const lora_segments_t* seg, const lora_pool_view_t* view, int32_t* dev_err,
                              lora_stream_t stream) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if ((st = check_act(y0, ldy0, view->d_out, T)) != LORA_OK) return st;
  if (T > 0 && (yf == nullptr || !aligned16(yf) || ldyf < view->d_out || ldyf % 4 != 0)) return LORA_ERR_INVALID_ARG;
  if (T > 0 && (overlap(yf, (long long)T * ldyf * 4, x, (long long)T * ldx * 2) ||
                overlap(yf, (long long)T * ldyf * 4, y0, (long long)T * ldy0 * 2)))
    return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  return run_segmented(kModeApply, x, ldx, const_cast<void*>(y0), ldy0, nullptr, 0, seg, view, dev_err,
                       (cudaStream_t)stream, yf, ldyf);
}

lora_status_t lora_sgmv_backward(const void* x, int64_t ldx, const void* dy, int64_t lddy, void* dx, int64_t lddx,
                                 float* grad_pool, float* hu, int64_t ldh, const lora_segments_t* seg,
                                 const lora_pool_view_t* view, int32_t* dev_err, lora_stream_t stream) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if ((st = check_act(dy, lddy, view->d_out, T)) != LORA_OK) return st;
  if (dx != nullptr && (st = check_act(dx, lddx, view->d_in, T)) != LORA_OK) return st;
  if (T == 0) return LORA_OK;
  if (grad_pool == nullptr || !aligned16(grad_pool)) return LORA_ERR_INVALID_ARG;
  if (hu == nullptr || !aligned16(hu) || ldh < view->max_rank || ldh % 4 != 0) return LORA_ERR_INVALID_ARG;
  const long long hu_bytes = 2LL * T * ldh * 4, g_bytes = view->n_pages * (long long)view->page_elems * 4;
  if (overlap(hu, hu_bytes, x, (long long)T * ldx * 2) || overlap(hu, hu_bytes, dy, (long long)T * lddy * 2) ||
      overlap(grad_pool, g_bytes, hu, hu_bytes) || overlap(grad_pool, g_bytes, x, (long long)T * ldx * 2) ||
      overlap(grad_pool, g_bytes, dy, (long long)T * lddy * 2))
    return LORA_ERR_INVALID_ARG;
  if (dx != nullptr && (overlap(dx, (long long)T * lddx * 2, x, (long long)T * ldx * 2) ||
                        overlap(dx, (long long)T * lddx * 2, dy, (long long)T * lddy * 2) ||
                        overlap(dx, (long long)T * lddx * 2, hu, hu_bytes) ||
                        overlap(dx, (long long)T * lddx * 2, grad_pool, g_bytes)))
    return LORA_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  float* h = hu;
  float* u = hu + (long long)T * ldh;
  // h = x A_i^T
  if ((st = run_segmented(kModeShrink, x, ldx, nullptr, 0, h, ldh, seg, view, dev_err, s)) != LORA_OK) return st;
  lora_pool_view_t vt = *view;  // the adapters transposed: B_i as the shrink's matrix, A_i as the expand's
  std::swap(vt.d_in, vt.d_out);
  {
    TransposedViews transposed;
    // u = dy B_i^T, and with dx, dx += s_i u A_i in the same pass: lora_apply over
    // the transposed adapters (x = dy, y = dx), writing its intermediate u
    st = dx == nullptr ? run_segmented(kModeShrink, dy, lddy, nullptr, 0, u, ldh, seg, &vt, dev_err, s)
                       : run_segmented(kModeApply, dy, lddy, dx, lddx, u, ldh, seg, &vt, dev_err, s);
    if (st != LORA_OK) return st;
  }
  return launch_grad(x, ldx, dy, lddy, h, u, ldh, grad_pool, seg, view, dev_err, s);
}

lora_status_t lora_base_apply(const void* x, int64_t ldx, const void* w0, int64_t ldw, void* y, int64_t ldy,
                              const int32_t* token_adapter, const lora_segments_t* seg,
                              const lora_pool_view_t* view, int32_t* dev_err, lora_stream_t stream) {
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if ((st = check_seg(seg)) != LORA_OK) return st;
  const int T = seg->T;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if ((st = check_act(y, ldy, view->d_out, T)) != LORA_OK) return st;
  if (T > 0 && token_adapter == nullptr) return LORA_ERR_INVALID_ARG;
  if (w0 == nullptr || !aligned16(w0) || ldw < view->d_in || ldw % 8 != 0) return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  if (overlap(x, (long long)T * ldx * 2, y, (long long)T * ldy * 2) ||
      overlap(w0, (long long)view->d_out * ldw * 2, y, (long long)T * ldy * 2))
    return LORA_ERR_INVALID_ARG;
  if (!base_gemm_ok(view)) return LORA_ERR_UNSUPPORTED;
  const cudaStream_t s = (cudaStream_t)stream;
  st = run_segmented(kModeShrink, x, ldx, nullptr, 0, seg->h_scratch, LORA_MAX_RANK, seg, view, dev_err, s);
  if (st != LORA_OK) return st;
  return launch_base_gemm(x, ldx, w0, ldw, y, ldy, seg->h_scratch, LORA_MAX_RANK, token_adapter, T, view, dev_err, s);
}

lora_status_t lora_bgmv(const void* x, int64_t ldx, void* y, int64_t ldy, const int32_t* token_adapter,
                        int32_t T, const lora_pool_view_t* view, int32_t* dev_err, lora_stream_t stream) {
  return lora_bgmv_ex(x, ldx, y, ldy, token_adapter, T, view, 0u, dev_err, stream);
}

lora_status_t lora_bgmv_ex(const void* x, int64_t ldx, void* y, int64_t ldy, const int32_t* token_adapter,
                           int32_t T, const lora_pool_view_t* view, uint32_t flags, int32_t* dev_err,
                           lora_stream_t stream) {
  if (flags & ~LORA_BGMV_STATIC_ADAPTERS) return LORA_ERR_INVALID_ARG;
  lora_status_t st = check_view(view);
  if (st != LORA_OK) return st;
  if (T < 0) return LORA_ERR_INVALID_ARG;
  if ((st = check_act(x, ldx, view->d_in, T)) != LORA_OK) return st;
  if ((st = check_act(y, ldy, view->d_out, T)) != LORA_OK) return st;
  if (T > 0 && token_adapter == nullptr) return LORA_ERR_INVALID_ARG;
  if (T > 0 && overlap(x, (long long)T * ldx * 2, y, (long long)T * ldy * 2)) return LORA_ERR_INVALID_ARG;
  if (T == 0) return LORA_OK;
  if (bgmv_decode_ok(view, T))
    return launch_bgmv(x, ldx, y, ldy, token_adapter, T, view, (flags & LORA_BGMV_STATIC_ADAPTERS) ? 1 : 0, dev_err,
                       (cudaStream_t)stream);
  return launch_gather(kModeApply, kSrcTokens, 0, x, ldx, y, ldy, nullptr, 0, nullptr, token_adapter, T, view,
                       dev_err, (cudaStream_t)stream);
}

}  // extern "C"

extern "C" uint64_t lora_launch_count(void) { return lora::g_launches.load(std::memory_order_relaxed); }

extern "C" void lora_debug_wait_probe(int64_t cycles) {
  lora::g_wait_probe.store(cycles > 0 ? (long long)cycles : 0, std::memory_order_relaxed);
}

namespace lora {

// Defined here, outside the C linkage block, so it can reach run_segmented.
lora_status_t apply_staged(const void* x, long long ldx, void* y, long long ldy, const lora_segments_t* seg,
                           const lora_pool_view_t* view, int32_t* err, cudaStream_t stream) {
  const lora_status_t st = check_apply(x, ldx, y, ldy, seg, view);
  if (st != LORA_OK || seg->T == 0) return st;
  return run_segmented(kModeApply, x, ldx, y, ldy, nullptr, 0, seg, view, err, stream, nullptr, 0, true);
}

}  // namespace lora

