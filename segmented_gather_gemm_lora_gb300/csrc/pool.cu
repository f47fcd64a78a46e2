// Residency of adapters in one projection's paged pool: a host-side manager of
// free pages, resident adapters, their order of last use and their pins, and
// the device work of a load or an eviction (copies from host memory, page-list
// and descriptor writes).
//
// "Multi-LoRA Serving in Production", sections "Unified Paged Memory" (pages
// handed out and taken back on demand, no contiguous space needed), "Tiered
// Storage Hierarchy and Asynchronous Streaming" (an adapter copied from host
// memory on a copy stream while the GPU computes) and "Eviction and
// Replacement Policies" (least recently used first; pinned adapters stay).
//
// Free pages are a bitmap scanned lowest page first, so a fresh or lightly
// used pool hands out runs of consecutive pages and a load needs few, large
// copies.  Resident adapters form a doubly linked list in order of last use.
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"
#include "lora_pool.h"

struct lora_pool_mgr {
  int64_t n_pages;
  int32_t page_elems, n_adapters, max_rank, d_in, d_out;
  int64_t slots_per;            // page-list slots owned by each adapter id
  int64_t n_free;               // free pages
  size_t hint;                  // no free page in a bitmap word below this one
  std::vector<uint64_t> used;   // bit p of the bitmap: page p in use
  std::vector<int32_t> rank;    // resident rank, 0 = not resident
  std::vector<int32_t> pins;    // pin counts
  std::vector<std::vector<int32_t>> pages;  // a resident adapter's pages: A's, then B's
  std::vector<int32_t> prev, next;          // list of resident adapters, least recent first
  int32_t head = -1, tail = -1;
  lora_pool_stats_t stats{};    // resident and pinned are counted when asked for
  // Set when zeroing an evicted adapter's descriptor failed to launch: the device
  // may still address pages the host now counts as free, so every later call
  // that hands out or frees pages returns LORA_ERR_CUDA.
  bool broken = false;
  mutable std::mutex mu;
};

namespace lora {
namespace {

constexpr int kMetaSlots = 512;  // page-list slots one metadata launch writes
constexpr int kMetaDescs = 48;   // descriptors one metadata launch writes

struct PoolMetaArgs {
  int32_t* page_list;
  lora_adapter_desc_t* adapters;
  int32_t slot0;
  int32_t n_slots;
  int32_t n_desc;
  int32_t pad;
  int32_t slots[kMetaSlots];
  int32_t desc_id[kMetaDescs];
  lora_adapter_desc_t desc[kMetaDescs];
};
static_assert(sizeof(PoolMetaArgs) <= 4096, "kernel parameters stay within 4 KB");

// page_list[slot0 + i] = slots[i]; adapters[desc_id[i]] = desc[i].  The host
// has checked every index against the view.  Launched without programmatic
// serialization: it starts only after every earlier kernel on the stream has
// finished, so none of them can see a half-written pool.
__global__ void pool_meta_kernel(const __grid_constant__ PoolMetaArgs a) {
  for (int i = threadIdx.x; i < a.n_slots; i += blockDim.x) a.page_list[a.slot0 + i] = a.slots[i];
  for (int i = threadIdx.x; i < a.n_desc; i += blockDim.x) a.adapters[a.desc_id[i]] = a.desc[i];
}

cudaError_t launch_meta(PoolMetaArgs* a, cudaStream_t stream) {
  void* params[1] = {a};
  const cudaError_t e = cudaLaunchKernel((const void*)pool_meta_kernel, dim3(1), dim3(256), params, 0, stream);
  if (e == cudaSuccess) count_launch();
  return e;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t pages_a(const lora_pool_mgr* m, int r) { return ceil_div((int64_t)r * m->d_in, m->page_elems); }
int64_t pages_b(const lora_pool_mgr* m, int r) { return ceil_div((int64_t)r * m->d_out, m->page_elems); }

void lru_unlink(lora_pool_mgr* m, int a) {
  const int p = m->prev[a], n = m->next[a];
  if (p >= 0) m->next[p] = n; else m->head = n;
  if (n >= 0) m->prev[n] = p; else m->tail = p;
  m->prev[a] = m->next[a] = -1;
}

void lru_push_back(lora_pool_mgr* m, int a) {
  m->prev[a] = m->tail;
  m->next[a] = -1;
  if (m->tail >= 0) m->next[m->tail] = a; else m->head = a;
  m->tail = a;
}

// The n lowest free pages, in increasing order, marked used.  The caller has
// checked that n pages are free.
void take_pages(lora_pool_mgr* m, int64_t n, std::vector<int32_t>* out) {
  out->clear();
  out->reserve((size_t)n);
  size_t w = m->hint;
  while ((int64_t)out->size() < n) {
    uint64_t free_bits = ~m->used[w];
    while (free_bits != 0 && (int64_t)out->size() < n) {
      const int b = __builtin_ctzll(free_bits);
      free_bits &= free_bits - 1;
      m->used[w] |= 1ull << b;
      out->push_back((int32_t)(w * 64 + b));
    }
    if (free_bits == 0) ++w;  // the word is full now
  }
  m->hint = w;
  m->n_free -= n;
}

void give_pages(lora_pool_mgr* m, const std::vector<int32_t>& pg) {
  for (const int32_t p : pg) {
    const size_t w = (size_t)p / 64;
    m->used[w] &= ~(1ull << (p % 64));
    if (w < m->hint) m->hint = w;
  }
  m->n_free += (int64_t)pg.size();
}

void release_locked(lora_pool_mgr* m, int a) {
  give_pages(m, m->pages[a]);
  m->pages[a].clear();
  m->pages[a].shrink_to_fit();
  m->rank[a] = 0;
  lru_unlink(m, a);
}

// Plan, check, then commit (nothing changes on an error).  *fresh = false when
// the adapter was already resident with this rank (only its last use moves).
lora_status_t reserve_locked(lora_pool_mgr* m, int a, int r, std::vector<int32_t>* evicted, bool* fresh) {
  evicted->clear();
  *fresh = false;
  if (a < 0 || a >= m->n_adapters || r < 1 || r > m->max_rank) return LORA_ERR_INVALID_ARG;
  if (m->rank[a] == r) {
    lru_unlink(m, a);
    lru_push_back(m, a);
    ++m->stats.hits;
    return LORA_OK;
  }
  const bool again = m->rank[a] != 0;  // resident with another rank: released first
  if (again && m->pins[a] > 0) return LORA_ERR_INVALID_ARG;
  const int64_t need = pages_a(m, r) + pages_b(m, r);
  int64_t avail = m->n_free + (again ? (int64_t)m->pages[a].size() : 0);
  if (again) evicted->push_back(a);
  for (int e = m->head; e >= 0 && avail < need; e = m->next[e]) {
    if (e == a || m->pins[e] > 0) continue;
    avail += (int64_t)m->pages[e].size();
    evicted->push_back(e);
  }
  if (avail < need) {
    evicted->clear();
    ++m->stats.refused;
    return LORA_ERR_WORKSPACE;
  }
  for (const int e : *evicted) release_locked(m, e);
  take_pages(m, need, &m->pages[a]);
  m->rank[a] = r;
  lru_push_back(m, a);
  ++m->stats.loads;
  m->stats.evictions += (int64_t)evicted->size();
  m->stats.pages_loaded += need;
  *fresh = true;
  return LORA_OK;
}

lora_status_t check_mgr_view(const lora_pool_mgr* m, const lora_pool_view_t* v) {
  const lora_status_t st = validate_view(v);
  if (st != LORA_OK) return st;
  if (v->page_elems != m->page_elems || v->n_pages != m->n_pages || v->n_adapters != m->n_adapters ||
      v->max_rank != m->max_rank || v->d_in != m->d_in || v->d_out != m->d_out ||
      v->n_page_list < (int64_t)m->n_adapters * m->slots_per)
    return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

// Descriptors of `ids` set to rank 0, in launches of kMetaDescs.
cudaError_t zero_descs(const std::vector<int32_t>& ids, const lora_pool_view_t* v, cudaStream_t stream) {
  for (size_t i0 = 0; i0 < ids.size(); i0 += kMetaDescs) {
    PoolMetaArgs a{};
    a.page_list = const_cast<int32_t*>(v->page_list);
    a.adapters = const_cast<lora_adapter_desc_t*>(v->adapters);
    a.n_desc = (int32_t)std::min(ids.size() - i0, (size_t)kMetaDescs);
    for (int k = 0; k < a.n_desc; ++k) a.desc_id[k] = ids[i0 + k];  // desc[k] stays all zero
    const cudaError_t e = launch_meta(&a, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// One copy per run of consecutive pages of one matrix of `elems` elements.
cudaError_t copy_matrix(const lora_pool_mgr* m, const int32_t* pg, int64_t npg, int64_t elems, const uint16_t* src,
                        const lora_pool_view_t* v, cudaStream_t stream) {
  const int64_t P = m->page_elems;
  uint16_t* pool = static_cast<uint16_t*>(const_cast<void*>(v->pool));
  for (int64_t k0 = 0; k0 < npg;) {
    int64_t k1 = k0 + 1;
    while (k1 < npg && pg[k1] == pg[k1 - 1] + 1) ++k1;
    const int64_t n = std::min((k1 - k0) * P, elems - k0 * P);
    const cudaError_t e = cudaMemcpyAsync(pool + (int64_t)pg[k0] * P, src + k0 * P, (size_t)n * 2,
                                          cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    k0 = k1;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" {

lora_status_t lora_pool_mgr_create(int64_t n_pages, int32_t page_elems, int32_t n_adapters, int32_t max_rank,
                                   int32_t d_in, int32_t d_out, lora_pool_mgr_t** out) {
  if (out == nullptr) return LORA_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_pages < 1 || n_pages > (int64_t)INT32_MAX || page_elems < 64 || (page_elems & (page_elems - 1)) != 0 ||
      page_elems > (1 << 30) || n_pages > (1LL << 40) / page_elems)
    return LORA_ERR_INVALID_ARG;
  if (n_adapters < 1 || n_adapters > LORA_MAX_ADAPTERS || max_rank < 1 || max_rank > LORA_MAX_RANK)
    return LORA_ERR_INVALID_ARG;
  if (d_in < 8 || d_out < 8 || d_in % 8 != 0 || d_out % 8 != 0) return LORA_ERR_INVALID_ARG;
  lora_pool_mgr* m = new (std::nothrow) lora_pool_mgr;
  if (m == nullptr) return LORA_ERR_INVALID_ARG;
  m->n_pages = n_pages;
  m->page_elems = page_elems;
  m->n_adapters = n_adapters;
  m->max_rank = max_rank;
  m->d_in = d_in;
  m->d_out = d_out;
  m->slots_per = pages_a(m, max_rank) + pages_b(m, max_rank);
  if ((int64_t)n_adapters * m->slots_per > (int64_t)INT32_MAX) {  // slots are int32 in the descriptors
    delete m;
    return LORA_ERR_INVALID_ARG;
  }
  m->n_free = n_pages;
  m->hint = 0;
  const size_t words = (size_t)ceil_div(n_pages, 64);
  try {
    m->used.assign(words, 0ull);
    m->rank.assign((size_t)n_adapters, 0);
    m->pins.assign((size_t)n_adapters, 0);
    m->pages.resize((size_t)n_adapters);
    m->prev.assign((size_t)n_adapters, -1);
    m->next.assign((size_t)n_adapters, -1);
  } catch (const std::bad_alloc&) {  // no exception crosses the C ABI
    delete m;
    return LORA_ERR_INVALID_ARG;
  }
  if (n_pages % 64 != 0) m->used[words - 1] = ~0ull << (n_pages % 64);  // beyond the pool: never free
  *out = m;
  return LORA_OK;
}

void lora_pool_mgr_destroy(lora_pool_mgr_t* mgr) { delete mgr; }

int64_t lora_pool_mgr_page_list_len(const lora_pool_mgr_t* mgr) {
  return mgr == nullptr ? -1 : (int64_t)mgr->n_adapters * mgr->slots_per;
}

int64_t lora_pool_mgr_free_pages(const lora_pool_mgr_t* mgr) {
  if (mgr == nullptr) return -1;
  std::lock_guard<std::mutex> lock(mgr->mu);
  return mgr->n_free;
}

int32_t lora_pool_resident_rank(const lora_pool_mgr_t* mgr, int32_t adapter) {
  if (mgr == nullptr || adapter < 0 || adapter >= mgr->n_adapters) return -1;
  std::lock_guard<std::mutex> lock(mgr->mu);
  return mgr->rank[adapter];
}

lora_status_t lora_pool_mgr_stats(const lora_pool_mgr_t* mgr, lora_pool_stats_t* out) {
  if (mgr == nullptr || out == nullptr) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mgr->mu);
  *out = mgr->stats;
  out->resident = 0;
  out->pinned = 0;
  for (int32_t a = 0; a < mgr->n_adapters; ++a) {
    out->resident += mgr->rank[a] != 0 ? 1 : 0;
    out->pinned += mgr->pins[a] > 0 ? 1 : 0;
  }
  return LORA_OK;
}

lora_status_t lora_pool_pin(lora_pool_mgr_t* mgr, int32_t adapter) {
  if (mgr == nullptr || adapter < 0 || adapter >= mgr->n_adapters) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->rank[adapter] == 0 || mgr->pins[adapter] == INT32_MAX) return LORA_ERR_INVALID_ARG;
  ++mgr->pins[adapter];
  return LORA_OK;
}

lora_status_t lora_pool_unpin(lora_pool_mgr_t* mgr, int32_t adapter) {
  if (mgr == nullptr || adapter < 0 || adapter >= mgr->n_adapters) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->pins[adapter] <= 0) return LORA_ERR_INVALID_ARG;
  --mgr->pins[adapter];
  return LORA_OK;
}

lora_status_t lora_pool_mgr_reserve(lora_pool_mgr_t* mgr, int32_t adapter, int32_t rank, int32_t* pages_out,
                                    int32_t pages_cap, int32_t* n_pages_out, int32_t* evicted_out,
                                    int32_t evicted_cap, int32_t* n_evicted_out) {
  if (mgr == nullptr || n_pages_out == nullptr || n_evicted_out == nullptr) return LORA_ERR_INVALID_ARG;
  if (pages_out == nullptr || pages_cap < mgr->slots_per) return LORA_ERR_INVALID_ARG;
  if (evicted_out == nullptr || evicted_cap < mgr->n_adapters) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->broken) return LORA_ERR_CUDA;
  std::vector<int32_t> evicted;
  bool fresh = false;
  const lora_status_t st = reserve_locked(mgr, adapter, rank, &evicted, &fresh);
  if (st != LORA_OK) return st;
  const std::vector<int32_t>& pg = mgr->pages[adapter];
  *n_pages_out = fresh ? (int32_t)pg.size() : 0;
  if (fresh)
    for (size_t i = 0; i < pg.size(); ++i) pages_out[i] = pg[i];
  *n_evicted_out = (int32_t)evicted.size();
  for (size_t i = 0; i < evicted.size(); ++i) evicted_out[i] = evicted[i];
  return LORA_OK;
}

lora_status_t lora_pool_mgr_release(lora_pool_mgr_t* mgr, int32_t adapter) {
  if (mgr == nullptr || adapter < 0 || adapter >= mgr->n_adapters) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->broken) return LORA_ERR_CUDA;
  if (mgr->rank[adapter] == 0) return LORA_OK;
  if (mgr->pins[adapter] > 0) return LORA_ERR_INVALID_ARG;
  release_locked(mgr, adapter);
  return LORA_OK;
}

lora_status_t lora_pool_load(lora_pool_mgr_t* mgr, int32_t adapter, int32_t rank, float scale, const void* host_A,
                             const void* host_B, const lora_pool_view_t* view, lora_stream_t stream) {
  if (mgr == nullptr || host_A == nullptr || host_B == nullptr) return LORA_ERR_INVALID_ARG;
  lora_status_t st = check_mgr_view(mgr, view);
  if (st != LORA_OK) return st;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->broken) return LORA_ERR_CUDA;
  std::vector<int32_t> evicted;
  bool fresh = false;
  st = reserve_locked(mgr, adapter, rank, &evicted, &fresh);
  if (st != LORA_OK || !fresh) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t na = pages_a(mgr, rank), nb = pages_b(mgr, rank);
  const std::vector<int32_t>& pg = mgr->pages[adapter];
  cudaError_t e = zero_descs(evicted, view, s);
  if (e != cudaSuccess) {
    // The evicted adapters' pages are free on the host but their descriptors may
    // still point at them on the device: nothing may hand those pages out again.
    mgr->broken = true;
    return LORA_ERR_CUDA;
  }
  if (e == cudaSuccess)
    e = copy_matrix(mgr, pg.data(), na, (int64_t)rank * mgr->d_in, static_cast<const uint16_t*>(host_A), view, s);
  if (e == cudaSuccess)
    e = copy_matrix(mgr, pg.data() + na, nb, (int64_t)rank * mgr->d_out, static_cast<const uint16_t*>(host_B), view,
                    s);
  const int64_t slot0 = (int64_t)adapter * mgr->slots_per;
  for (int64_t c0 = 0; e == cudaSuccess && c0 < na + nb; c0 += kMetaSlots) {
    PoolMetaArgs a{};
    a.page_list = const_cast<int32_t*>(view->page_list);
    a.adapters = const_cast<lora_adapter_desc_t*>(view->adapters);
    a.slot0 = (int32_t)(slot0 + c0);
    a.n_slots = (int32_t)std::min<int64_t>(na + nb - c0, kMetaSlots);
    for (int k = 0; k < a.n_slots; ++k) a.slots[k] = pg[(size_t)(c0 + k)];
    if (c0 + kMetaSlots >= na + nb) {  // the last launch also publishes the descriptor
      a.n_desc = 1;
      a.desc_id[0] = adapter;
      a.desc[0].rank = rank;
      a.desc[0].scale = scale;
      a.desc[0].a_page0 = (int32_t)slot0;
      a.desc[0].b_page0 = (int32_t)(slot0 + na);
    }
    e = launch_meta(&a, s);
  }
  if (e != cudaSuccess) {
    release_locked(mgr, adapter);
    return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

lora_status_t lora_pool_evict(lora_pool_mgr_t* mgr, int32_t adapter, const lora_pool_view_t* view,
                              lora_stream_t stream) {
  if (mgr == nullptr || adapter < 0 || adapter >= mgr->n_adapters) return LORA_ERR_INVALID_ARG;
  lora_status_t st = check_mgr_view(mgr, view);
  if (st != LORA_OK) return st;
  std::lock_guard<std::mutex> lock(mgr->mu);
  if (mgr->broken) return LORA_ERR_CUDA;
  if (mgr->rank[adapter] == 0) return LORA_OK;
  if (mgr->pins[adapter] > 0) return LORA_ERR_INVALID_ARG;
  release_locked(mgr, adapter);
  if (zero_descs(std::vector<int32_t>{adapter}, view, (cudaStream_t)stream) != cudaSuccess) {
    mgr->broken = true;  // as in lora_pool_load: the device may still address the freed pages
    return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

}  // extern "C"
