/*
 * lora_pool.h -- residency of adapters in one projection's paged pool.
 *
 * The compute calls of lora_sgmv.h read adapters through a lora_pool_view_t:
 * physical pages of page_elems bf16 elements, a page list mapping slots to
 * pages, and one descriptor per adapter id.  This part keeps that pool filled
 * on demand, as "Multi-LoRA Serving in Production" describes it:
 *   - section "Unified Paged Memory": pages are handed out and taken back as
 *     adapters come and go, with no need for contiguous space;
 *   - section "Tiered Storage Hierarchy and Asynchronous Streaming": an adapter
 *     not in HBM is copied from (pinned) host memory on a copy stream while the
 *     GPU computes;
 *   - section "Eviction and Replacement Policies": when pages run out, the
 *     least recently used adapter is evicted; pinned adapters stay resident.
 * ("Multi-LoRA Serving: Many Adapters on One GPU", section "Swap latency and
 * cache policy", gives the host-memory tier and its copy-time floor.)
 *
 * A manager (lora_pool_mgr_t) is a host object that the caller creates for one
 * projection's pool and destroys.  It records which physical pages are free,
 * which adapters are resident with which pages, their order of last use and
 * their pin counts.  It allocates no device memory: the caller allocates the
 * view's pool (n_pages * page_elems bf16), its page list
 * (lora_pool_mgr_page_list_len int32 slots) and its descriptors (n_adapters,
 * zero-filled: every adapter starts not resident), and passes the view to the
 * calls that touch the device.  Each adapter id owns a fixed range of
 * slots_per_adapter page-list slots, starting at adapter * slots_per_adapter,
 * with slots_per_adapter = ceil(max_rank * d_in / page_elems) +
 * ceil(max_rank * d_out / page_elems); a resident adapter of rank r uses the
 * first ceil(r * d_in / page_elems) of them for A and the next
 * ceil(r * d_out / page_elems) for B.
 *
 * Ordering.  lora_pool_load and lora_pool_evict enqueue their device work on
 * the given stream and return without synchronising: the copies and the page
 * list and descriptor writes run in stream order, after every kernel enqueued
 * earlier on that stream.  Kernels on another stream see a load only once that
 * stream waits for it (an event).  Pages are reused as soon as an adapter is
 * evicted, so an adapter that a kernel on another stream may still read must be
 * pinned (lora_pool_pin) until that kernel has finished.  Host memory given to
 * lora_pool_load must stay unchanged until its copies have run; pinned host
 * memory (cudaHostAlloc / cudaHostRegister) makes them asynchronous.  A
 * manager may be used from several host threads (every call locks it).
 */
#ifndef LORA_POOL_H
#define LORA_POOL_H

#include "lora_sgmv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_pool_mgr lora_pool_mgr_t;

/**
 * A manager for a pool of n_pages pages of page_elems elements (a power of two,
 * >= 64) holding adapters 0 .. n_adapters - 1 (<= LORA_MAX_ADAPTERS) of ranks
 * 1 .. max_rank (<= LORA_MAX_RANK) for a projection d_in -> d_out (multiples of
 * 8).  Every page starts free and every adapter not resident.  Host only.
 * Returns LORA_ERR_INVALID_ARG on bad geometry or a null out.
 */
lora_status_t lora_pool_mgr_create(int64_t n_pages, int32_t page_elems, int32_t n_adapters,
                                   int32_t max_rank, int32_t d_in, int32_t d_out,
                                   lora_pool_mgr_t** out);
void lora_pool_mgr_destroy(lora_pool_mgr_t* mgr);

/** Page-list slots the view needs: n_adapters * slots_per_adapter (-1 if mgr is null). */
int64_t lora_pool_mgr_page_list_len(const lora_pool_mgr_t* mgr);
/** Pages currently free (-1 if mgr is null). */
int64_t lora_pool_mgr_free_pages(const lora_pool_mgr_t* mgr);
/** Rank of a resident adapter, 0 if it is not resident, -1 on a bad argument. */
int32_t lora_pool_resident_rank(const lora_pool_mgr_t* mgr, int32_t adapter);

/** Counters of a manager since its creation (host only). */
typedef struct {
  int64_t hits;         /* reserves of an adapter already resident with that rank */
  int64_t loads;        /* reserves that handed out pages */
  int64_t refused;      /* reserves refused for want of unpinned pages (LORA_ERR_WORKSPACE) */
  int64_t evictions;    /* adapters released to make room, their own release on a rank change included */
  int64_t pages_loaded; /* pages handed out by those loads */
  int32_t resident;     /* adapters resident now */
  int32_t pinned;       /* of which pinned */
} lora_pool_stats_t;

/** Fill *out (LORA_ERR_INVALID_ARG if mgr or out is null). */
lora_status_t lora_pool_mgr_stats(const lora_pool_mgr_t* mgr, lora_pool_stats_t* out);

/** Pin counts: a pinned adapter (count > 0) is never evicted.  lora_pool_pin
 *  needs a resident adapter; lora_pool_unpin one with a count above zero
 *  (LORA_ERR_INVALID_ARG otherwise). */
lora_status_t lora_pool_pin(lora_pool_mgr_t* mgr, int32_t adapter);
lora_status_t lora_pool_unpin(lora_pool_mgr_t* mgr, int32_t adapter);

/**
 * The host-side step of lora_pool_load, exported for callers that fill pages
 * themselves.  Host only.
 *
 * If the adapter is resident with this rank, it becomes the most recently used
 * and *n_pages_out = 0, *n_evicted_out = 0.  Otherwise (not resident, or
 * resident with another rank and not pinned, in which case its pages are
 * released first) it takes ceil(rank * d_in / page_elems) +
 * ceil(rank * d_out / page_elems) free pages, lowest page numbers first (A's
 * pages, then B's, in logical order, into pages_out), evicting the least
 * recently used unpinned adapters (into evicted_out, in eviction order, after
 * the adapter itself when its rank changed) until enough pages are free, and
 * becomes resident and the most recently used.
 * Nothing changes if the pages cannot be found: LORA_ERR_WORKSPACE when even
 * evicting every unpinned adapter would not free enough, LORA_ERR_INVALID_ARG
 * for a bad id or rank, a pinned adapter of another rank, or capacities below
 * slots_per_adapter (pages_cap) or n_adapters (evicted_cap).
 *
 * A caller that uses it directly must then, in stream order: set the evicted
 * adapters' descriptors to rank 0, copy A and B into the returned pages, write
 * them into the adapter's page-list slots, and write its descriptor
 * {rank, scale, adapter * slots_per_adapter, that + ceil(rank * d_in / page_elems)}.
 */
lora_status_t lora_pool_mgr_reserve(lora_pool_mgr_t* mgr, int32_t adapter, int32_t rank,
                                    int32_t* pages_out, int32_t pages_cap, int32_t* n_pages_out,
                                    int32_t* evicted_out, int32_t evicted_cap,
                                    int32_t* n_evicted_out);

/** The host-side step of lora_pool_evict: the adapter's pages become free and
 *  it is no longer resident.  LORA_ERR_INVALID_ARG if it is pinned or the id is
 *  bad; LORA_OK (nothing to do) if it is not resident.  Host only. */
lora_status_t lora_pool_mgr_release(lora_pool_mgr_t* mgr, int32_t adapter);

/**
 * Make adapter `adapter` resident with rank `rank` and scale `scale`
 * (s = alpha / r, stored as given): lora_pool_mgr_reserve, then on `stream`:
 * the evicted adapters' descriptors set to rank 0, A (host bf16, rank rows x
 * d_in, row-major) and B (host bf16, rank rows x d_out) copied into the new
 * pages (one copy per run of consecutive pages), the page-list slots and the
 * descriptor written (one small kernel).  An adapter already resident with
 * this rank is only marked most recently used: nothing is copied and its
 * scale is kept (evict it first to change its weights or scale).
 *
 * view must describe the manager's pool: the same page_elems, n_pages,
 * n_adapters, max_rank, d_in and d_out, n_page_list >= the manager's
 * page_list_len, non-null device pointers (its pool, page list and adapters are
 * written, though the view declares them const).  Errors as
 * lora_pool_mgr_reserve, plus LORA_ERR_INVALID_ARG for a mismatched view or a
 * null host pointer and LORA_ERR_CUDA if a copy or the launch fails (the
 * adapter is then not resident).  If the kernel that zeroes the evicted
 * adapters' descriptors fails to launch, the device may still address pages
 * the manager now counts as free; the manager then refuses every later
 * lora_pool_mgr_reserve, lora_pool_mgr_release, lora_pool_load and
 * lora_pool_evict with LORA_ERR_CUDA (destroy it and rebuild the pool).
 */
lora_status_t lora_pool_load(lora_pool_mgr_t* mgr, int32_t adapter, int32_t rank, float scale,
                             const void* host_A, const void* host_B, const lora_pool_view_t* view,
                             lora_stream_t stream);

/** lora_pool_mgr_release, then the adapter's descriptor set to rank 0 on
 *  `stream` (one small kernel).  Errors as lora_pool_mgr_release and
 *  lora_pool_load; a failed launch of that kernel leaves the manager refusing
 *  later calls, as in lora_pool_load. */
lora_status_t lora_pool_evict(lora_pool_mgr_t* mgr, int32_t adapter, const lora_pool_view_t* view,
                              lora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_POOL_H */
