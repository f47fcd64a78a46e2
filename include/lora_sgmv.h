/*
 * lora_sgmv.h -- C ABI of the GB300 (sm_103a) multi-adapter LoRA library.
 *
 * The library computes, for a batch of T token rows that each carry their own
 * adapter i = a(t),
 *
 *     y[t, :] = y0[t, :] + s_i * (x[t, :] . A_i) . B_i,     s_i = alpha_i / r_i,
 *
 * in place in the caller's base output y (which holds y0 = x . W0 on entry).
 * The per-token form is the one of "Multi-LoRA serving: the single translator
 * with a thousand glossaries", section "SGMV: the kernel that holds it all up"
 * (y_t = W x_t + B_a(t) A_a(t) x_t for every t in the batch); the row-vector
 * orientation and the alpha/r scale are those of "Multi-LoRA Serving in
 * Production", section "Mathematical Formulation and the Batching Challenge"
 * (y = x W0 + (alpha/r) (x A) B, A in R^{d_in x r}, B in R^{r x d_out}).
 *
 * Data types: x, y and the adapter pool are bf16 (passed as void*, 2 bytes per
 * element, round-to-nearest-even on output); the rank-r intermediate h and the
 * scales are fp32; products accumulate in fp32.
 *
 * Storage of one adapter i of rank r_i for a projection d_in -> d_out:
 *   A_i: r_i rows x d_in elements, row-major (row j = column j of the math A_i);
 *   B_i: r_i rows x d_out elements, row-major (the math B_i as is).
 * Both live in a paged pool ("Multi-LoRA Serving in Production", section
 * "Unified Paged Memory": adapter matrices sliced into fixed-size pages, a
 * software page table mapping them to non-contiguous physical frames):
 * logical element e of a matrix whose first page-list slot is page0 lives at
 *     pool[page_list[page0 + e / page_elems] * page_elems + e % page_elems].
 * Low ranks are not padded: an adapter holds ceil(r_i * d / page_elems) pages
 * per matrix, only the last one partly used.
 *
 * Ownership and threading.  The caller owns every buffer (x, y, h, pool, page
 * list, descriptors, segment buffer, error word); all device buffers are plain
 * device pointers from any allocator.  The library allocates no device memory,
 * keeps no per-call state (the pool managers of lora_pool.h are host objects
 * the caller creates and destroys), and its entry points may be called from
 * several host threads.  Every compute entry point is asynchronous on the given CUDA
 * stream (NULL = the legacy default stream) and does not synchronise.
 *
 * Errors.  Argument errors found on the host are returned before anything is
 * launched.  A failed launch returns LORA_ERR_CUDA.  Errors that only the
 * device can see (an adapter id outside [-1, n_adapters), a rank outside
 * [1, max_rank], a page-list slot or page outside the pool, a wait that ran
 * out) OR a LORA_DERR_* bit into *dev_err (a device int32 the caller zeroes
 * and reads after its own synchronisation); the affected tokens' outputs are
 * left as they were, every other token is still computed.
 */
#ifndef LORA_SGMV_H
#define LORA_SGMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/** A CUDA stream (cudaStream_t); NULL means the legacy default stream. */
typedef struct CUstream_st* lora_stream_t;

typedef int32_t lora_status_t;
#define LORA_OK 0
#define LORA_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad size or stride, aliasing */
#define LORA_ERR_UNSUPPORTED (-2) /* valid but outside what this build handles */
#define LORA_ERR_CUDA (-3)        /* a CUDA runtime call or launch failed */
#define LORA_ERR_WORKSPACE (-4)   /* the segment buffer or the adapter pool is too small */

/* Bits OR-ed into the caller's device error word. */
#define LORA_DERR_BAD_ADAPTER 1 /* adapter id outside [-1, n_adapters) */
#define LORA_DERR_BAD_PAGE 2    /* page-list slot or physical page outside the pool */
#define LORA_DERR_BAD_RANK 4    /* adapter rank outside [1, max_rank] */
#define LORA_DERR_TIMEOUT 8     /* a bounded wait inside a kernel ran out */

/** Highest adapter rank this build supports (LORA_ERR_UNSUPPORTED above). */
#define LORA_MAX_RANK 64
/** Largest adapter count lora_segments_build accepts. */
#define LORA_MAX_ADAPTERS 32768
/** Segments of at most this many tokens take the gather path of lora_apply /
 *  lora_sgmv_*; longer ones are cut into tiles of LORA_TILE_M tokens for the
 *  tensor-core path ("Multi-LoRA serving: ...", section "SGMV: the kernel that
 *  holds it all up": large segments through tensor cores, small ones through a
 *  batched gather path).  Chosen by measurement: with 64 segments of L tokens
 *  (rank 16, 4096 -> 4096) the two paths take equal time near L = 24-28. */
#define LORA_SHORT_MAX_TOKENS 24
#define LORA_TILE_M 128

/** Segmentation modes of lora_segments_build. */
#define LORA_SEG_GROUP 0      /* one segment per adapter id, ascending id, tokens ascending */
#define LORA_SEG_CONTIGUOUS 1 /* one segment per maximal run of equal ids, in token order */

/** One adapter of one projection (16 bytes, device array of n_adapters). */
typedef struct {
  int32_t rank;    /* r_i; 0 marks an adapter that is not resident */
  float scale;     /* s_i = alpha_i / r_i, applied as given (never derived from rank) */
  int32_t a_page0; /* page-list slot of A_i's first page */
  int32_t b_page0; /* page-list slot of B_i's first page */
} lora_adapter_desc_t;

/** One projection's view of the paged adapter pool (host struct, device pointers). */
typedef struct {
  const void* pool;                    /* device bf16 [n_pages * page_elems], 16-byte aligned */
  int64_t n_pages;                     /* physical pages in the pool */
  const int32_t* page_list;            /* device int32 [n_page_list]: slot -> physical page */
  int64_t n_page_list;                 /* slots in page_list */
  const lora_adapter_desc_t* adapters; /* device [n_adapters] */
  int32_t n_adapters;
  int32_t page_elems; /* elements per page: a power of two, >= 64 */
  int32_t max_rank;   /* largest rank any call may meet, 1 .. LORA_MAX_RANK */
  int32_t d_in;       /* projection input width, a multiple of 8 */
  int32_t d_out;      /* projection output width, a multiple of 8 */
} lora_pool_view_t;

/**
 * Segments of one batch, laid out by lora_segments_carve in one caller-owned
 * device buffer.  Filled by lora_segments_build; read by the compute calls.
 * token_perm lists the segments' tokens in segment order; segment s covers
 * token_perm[seg_indptr[s] .. seg_indptr[s+1]) and uses adapter seg_adapter[s].
 * meta[0] = number of segments, meta[1] = tokens placed, meta[2] = short work
 * units, meta[3] = long work units, meta[4] = runs of equal ids, meta[5],
 * meta[6] and meta[7] = work counters of the tensor-core shrink, the tensor-core
 * expand and the gather kernel (zeroed by lora_segments_build, left at zero by
 * every call).  short_units lists the segments of at most
 * LORA_SHORT_MAX_TOKENS tokens; long_units lists (segment, offset) pairs, one
 * per LORA_TILE_M-token tile of every longer segment, both in segment order.
 * scratch belongs to lora_segments_build; h_scratch, k_partials and the work
 * counters to the compute calls, so calls that share a segment buffer
 * must be ordered on one stream.
 */
typedef struct {
  int32_t T;              /* tokens the buffer was carved for */
  int32_t max_long_units; /* capacity of long_units (pairs) */
  int32_t* token_perm;    /* [T] */
  int32_t* seg_indptr;    /* [T + 1] */
  int32_t* seg_adapter;   /* [T] */
  int32_t* meta;          /* [8] */
  int32_t* short_units;   /* [T] */
  int32_t* long_units;    /* [2 * max_long_units] */
  int32_t* scratch;       /* [4 * T + 8]: run starts, run ends, run ids, run positions */
  float* h_scratch;       /* [T * LORA_MAX_RANK]: the rank-r intermediate of tokens on
                             the staged tensor-core path (lora_apply_fixed_scratch uses
                             its own array instead), by segment position */
  float* k_partials;      /* [LORA_KSPLIT_MAX * T * LORA_MAX_RANK]: partial shrink sums of
                             the staged tensor-core path (lora_sgmv_shrink,
                             lora_sgmv_backward, lora_apply_fixed_scratch), one slab
                             per slice of d_in */
} lora_segments_t;

/** Slices of d_in the tensor-core shrink splits a tile into, at most. */
#define LORA_KSPLIT_MAX 8

/** Bytes of the device buffer lora_segments_carve needs for T tokens (T >= 0). */
size_t lora_segments_buffer_bytes(int32_t T);

/**
 * Point the arrays of *out into a caller-owned device buffer (no device access).
 * buf must be 16-byte aligned and hold lora_segments_buffer_bytes(T) bytes.
 * Returns LORA_ERR_WORKSPACE if it is too small, LORA_ERR_INVALID_ARG on a
 * null or misaligned pointer or T < 0.
 */
lora_status_t lora_segments_carve(void* buf, size_t bytes, int32_t T, lora_segments_t* out);

/**
 * Group the batch's tokens by adapter ("Multi-LoRA serving: ...", section
 * "SGMV: the kernel that holds it all up": SGMV segments the batch's tokens by
 * adapter; "Multi-LoRA Serving in Production", section "Punica and Segmented
 * Gather Matrix-Vector Multiplication (SGMV)": contiguous segments whose tokens
 * share an adapter id).  token_adapter: device int32 [T], -1 = no adapter.
 * mode: LORA_SEG_GROUP or LORA_SEG_CONTIGUOUS.  Tokens with id -1 belong to no
 * segment; ids outside [-1, n_adapters) set LORA_DERR_BAD_ADAPTER and are
 * dropped.  1 <= n_adapters <= LORA_MAX_ADAPTERS.  Output is bit-exact and
 * deterministic.  T = 0 is a no-op that still writes empty segments.
 */
lora_status_t lora_segments_build(const int32_t* token_adapter, int32_t T, int32_t n_adapters,
                                  int32_t mode, const lora_segments_t* seg, int32_t* dev_err,
                                  lora_stream_t stream);

/**
 * Shrink stage ("Multi-LoRA Serving in Production", section "Punica and
 * Segmented Gather Matrix-Vector Multiplication (SGMV)", "Shrink Stage"):
 *     h[t, j] = sum_k x[t, k] * A_i[j, k]     for j < r_i, unscaled,
 * for every token of the segments.  x: device bf16 [T, ldx] (ldx >= d_in,
 * ldx % 8 == 0, 16-byte aligned).  h: device fp32 [T, ldh], ldh >= max_rank,
 * ldh % 4 == 0, 16-byte aligned; columns >= r_i and rows of tokens in no
 * segment are not written.
 */
lora_status_t lora_sgmv_shrink(const void* x, int64_t ldx, float* h, int64_t ldh,
                               const lora_segments_t* seg, const lora_pool_view_t* view,
                               int32_t* dev_err, lora_stream_t stream);

/**
 * Expand stage (same section, "Expand Stage"): scale and accumulate into the
 * base output,
 *     y[t, n] = bf16( y[t, n] + sum_j (s_i * h[t, j]) * B_i[j, n] ).
 * h: device fp32 [T, ldh] as written by lora_sgmv_shrink.  y: device bf16
 * [T, ldy] in place (ldy >= d_out, ldy % 8 == 0, 16-byte aligned).
 */
lora_status_t lora_sgmv_expand(const float* h, int64_t ldh, void* y, int64_t ldy,
                               const lora_segments_t* seg, const lora_pool_view_t* view,
                               int32_t* dev_err, lora_stream_t stream);

/**
 * Fused shrink -> scale -> expand over the segments; h never leaves the chip
 * ("Multi-LoRA serving: ...", TL;DR: Y += sum_i X_i A_i B_i in a single pass):
 * short segments run on the gather kernel, the 128-token tiles of long ones on
 * the fused tensor-core kernel, which exchanges h between the CTAs of a cluster
 * through distributed shared memory.  It uses the segment buffer's index
 * arrays and work counter, not h_scratch or k_partials.
 *     y[t, n] = bf16( y[t, n] + sum_j (s_i * sum_k x[t,k] A_i[j,k]) * B_i[j, n] ).
 * x must not overlap y.
 */
lora_status_t lora_apply(const void* x, int64_t ldx, void* y, int64_t ldy,
                         const lora_segments_t* seg, const lora_pool_view_t* view,
                         int32_t* dev_err, lora_stream_t stream);

/** Projections one lora_apply_multi call takes, at most. */
#define LORA_MAX_PROJ 4

/** One projection of a lora_apply_multi call (host struct, device pointers). */
typedef struct {
  const void* x;          /* device bf16 [T, ldx]; may be shared with other projections */
  int64_t ldx;
  void* y;                /* device bf16 [T, ldy], updated in place */
  int64_t ldy;
  lora_pool_view_t view;  /* the projection's adapters */
} lora_proj_t;

/**
 * Several projections of one layer that share a batch in one grouped call:
 * the q, k and v projections of attention (one input x), or the gate and up
 * projections of an MLP ("Multi-LoRA Serving in Production", section "Ragged
 * Batching and FlashInfer Grouped GEMM": the adapters of every projection in a
 * single fused invocation).  The result is that of n_proj lora_apply calls,
 * one per projection, on the same segments: bit for bit for tokens on the
 * tensor-core path; tokens of short segments may be summed in another order,
 * within the stated tolerance, when the grouped call gives the gather kernel
 * narrower clusters.  The work units of all projections share each launch, a
 * tile's units for every projection side by side, so x rows that several
 * projections read come from DRAM once.
 * 1 <= n_proj <= LORA_MAX_PROJ.  Every view must have the same d_in; each
 * projection's x and y as for lora_apply; no y may overlap another y or any x.
 */
lora_status_t lora_apply_multi(const lora_proj_t* projs, int32_t n_proj, const lora_segments_t* seg,
                               int32_t* dev_err, lora_stream_t stream);

/**
 * lora_apply with an fp32 output, for checking accuracy: the same kernels and
 * the same sums, but the result float(y0[t, n]) + delta is written as fp32
 * into yf instead of being rounded to bf16 in place, so a comparison against
 * an exact reference sees the accumulation error alone (the bf16 rounding of
 * the output, half an ulp, hides it otherwise; "Multi-LoRA Serving in
 * Production", section "Mathematical Formulation and the Batching Challenge",
 * defines the result this approximates).
 *     yf[t, n] = float(y0[t, n]) + sum_j (s_i * sum_k x[t,k] A_i[j,k]) * B_i[j, n].
 * y0: device bf16 [T, ldy0], read only.  yf: device fp32 [T, ldyf], ldyf >=
 * d_out, ldyf % 4 == 0, 16-byte aligned, overlapping neither x nor y0; rows of
 * tokens in no segment (and of tokens whose adapter is flagged on the device)
 * and columns >= d_out are not written.
 */
lora_status_t lora_apply_f32y(const void* x, int64_t ldx, const void* y0, int64_t ldy0, float* yf,
                              int64_t ldyf, const lora_segments_t* seg, const lora_pool_view_t* view,
                              int32_t* dev_err, lora_stream_t stream);

/**
 * Backward pass, for training the adapters: the base stays frozen and gets no
 * gradient; only A_i and B_i do, and the adapter is the only path the
 * gradient flows through ("QLoRA and multi-LoRA at the limit on small
 * models", section "The bare mechanism: LoRA, and why you can train on a
 * 4-bit base").  Given the forward's input x and dy = dL/dy, for every token
 * t of the segments, with i = its adapter:
 *     h[t] = x[t] A_i^T,  u[t] = dy[t] B_i^T                 (fp32, into hu)
 *     dB_i += s_i sum_t h[t]^T dy[t],  dA_i += s_i sum_t u[t]^T x[t]
 *     dx[t] = bf16(dx[t] + s_i u[t] A_i)                      (if dx != NULL)
 * x: bf16 [T, ldx]; dy: bf16 [T, lddy] (lddy >= d_out); dx: bf16 [T, lddx],
 * updated in place, or NULL.  grad_pool: device fp32 [n_pages * page_elems],
 * the same page layout as view->pool: the gradient of the weight at pool
 * position q is added into grad_pool[q] (zero it to start; calls accumulate,
 * as gradient accumulation over micro-batches does).  hu: device fp32
 * workspace [2 * T * ldh] (h rows, then u rows, by token), ldh >= max_rank,
 * ldh % 4 == 0.  With GROUP segments each adapter's gradient elements receive
 * one addition per call, in a fixed order; with CONTIGUOUS segments an adapter
 * that has several segments receives one per segment, in any order.  x, dy,
 * dx, hu and grad_pool must not overlap.  Device errors as lora_apply: the
 * affected tokens add nothing to any gradient and leave their dx rows alone.
 */
lora_status_t lora_sgmv_backward(const void* x, int64_t ldx, const void* dy, int64_t lddy, void* dx,
                                 int64_t lddx, float* grad_pool, float* hu, int64_t ldh,
                                 const lora_segments_t* seg, const lora_pool_view_t* view,
                                 int32_t* dev_err, lora_stream_t stream);

/**
 * The base projection with the adapter term added before y is written
 * ("Multi-LoRA Serving: Many Adapters on One GPU", section "How batching
 * across adapters works": one base product shared by the batch plus each
 * token's own adapter term):
 *     y[t, n] = bf16( sum_k x[t,k] W0[n,k] + s_i sum_j (x[t] . A_i[j]) B_i[j,n] )
 * for every token t < T; tokens with id -1, or with an adapter that fails the
 * checks (their error bits OR into *dev_err), get the base term alone.  y is
 * written once and never read (it may hold anything before the call).
 * x: device bf16 [T, ldx]; w0: device bf16 [d_out, ldw] (row n holds output
 * n's weights over the d_in inputs, the layout of a linear layer's weight),
 * ldw >= d_in, ldw % 8 == 0, 16-byte aligned; y: device bf16 [T, ldy];
 * token_adapter: the device int32 [T] ids that seg was built from, with
 * n_adapters = view->n_adapters.  The call runs the shrink stage into
 * seg->h_scratch (by token), so calls sharing a segment buffer must be
 * ordered on one stream.
 * y must not overlap x, w0 or the segment buffer.  The base product runs on
 * the tensor cores through TMA tensor maps: LORA_ERR_UNSUPPORTED when the
 * driver offers no tensor-map encoder.
 */
lora_status_t lora_base_apply(const void* x, int64_t ldx, const void* w0, int64_t ldw, void* y, int64_t ldy,
                              const int32_t* token_adapter, const lora_segments_t* seg,
                              const lora_pool_view_t* view, int32_t* dev_err, lora_stream_t stream);

/**
 * Decode form without segments: each token t gathers its own adapter
 * token_adapter[t] (device int32 [T], -1 = no adapter), one token per request
 * (the batched gather path for size-1 segments of "Multi-LoRA serving: ...",
 * section "SGMV: the kernel that holds it all up"; MBGMV in "Multi-LoRA
 * Serving in Production", section "S-LoRA: MBGMV and MBGMM Kernels").
 * Same result as lora_apply up to rounding.  Views with max_rank <= 16,
 * d_in, d_out <= 8192 and at most 128 page-list slots per adapter run on a
 * decode kernel of small CTAs with fp32 CUDA-core arithmetic, where a token's
 * output depends only on its own row, its adapter and the projection's shape
 * (not on the rest of the batch); other views run on lora_apply's gather
 * kernel.
 */
lora_status_t lora_bgmv(const void* x, int64_t ldx, void* y, int64_t ldy,
                        const int32_t* token_adapter, int32_t T, const lora_pool_view_t* view,
                        int32_t* dev_err, lora_stream_t stream);

/* lora_bgmv_ex flags. */
/* token_adapter and the adapter pool (descriptors, page list, pages) were
 * final before the kernel enqueued just ahead of this call on the stream
 * started: nothing that kernel does writes them.  The call may then read them,
 * and stage the adapters' rows, while that kernel is still running; x and y
 * are still touched only after it has finished.  Host copies into those
 * buffers, and kernels followed by at least one other kernel before the call,
 * satisfy this; a lora_pool_load on the same stream directly ahead of the call
 * does not (put the load on its own stream and wait for it with an event). */
#define LORA_BGMV_STATIC_ADAPTERS 1u

/**
 * lora_bgmv with flags (LORA_BGMV_STATIC_ADAPTERS, or 0 for lora_bgmv's
 * behaviour).  Other bits: LORA_ERR_INVALID_ARG.  The flag takes effect on
 * the decode kernel (the views lora_bgmv runs there); the gather kernel
 * ignores it.
 */
lora_status_t lora_bgmv_ex(const void* x, int64_t ldx, void* y, int64_t ldy,
                           const int32_t* token_adapter, int32_t T, const lora_pool_view_t* view,
                           uint32_t flags, int32_t* dev_err, lora_stream_t stream);

/**
 * lora_apply for callers that cannot allocate device memory.  (The pages have
 * no counterpart: this is a deployment convenience of this library.)
 *
 * It computes lora_apply's result, bit for bit, through the staged
 * tensor-core kernels (a shrink grid, then an expand grid), which keep the
 * rank-r intermediate of long segments in global memory between the two: in
 * seg->h_scratch when the caller runs those stages itself.  Callers whose
 * device memory is planned once by a host runtime, and who can therefore
 * neither size nor request an extra workspace per call, use this entry point:
 * the intermediate goes to a fixed array of LORA_FIXED_SCRATCH_MAX_TOKENS x
 * LORA_MAX_RANK fp32 values (4 MiB) that is part of the library's device image
 * (every GPU that loads the library holds it until the process exits).  It
 * allocates nothing.
 *
 * Arguments, results and errors are those of lora_apply.  Only seg->h_scratch
 * moves into the library's array (it is not read and may be NULL); every other
 * array of the segment buffer, k_partials (the tensor-core path's partial
 * sums, LORA_KSPLIT_MAX x T x LORA_MAX_RANK fp32) included, is still the
 * caller's, carved as for lora_apply.  Returns LORA_ERR_UNSUPPORTED if seg->T
 * exceeds LORA_FIXED_SCRATCH_MAX_TOKENS.  Each call looks up the array's
 * device address on the current device (a host query; the first call on a
 * device may also load the library's device code there, so make it before any
 * stream capture).  Every call shares the one array: calls that may run at the
 * same time on the GPU (other streams, other host threads) race on it and must
 * be serialised by the caller.  The array keeps the last call's contents;
 * nothing in it needs to start at zero, because every value a call reads was
 * written earlier in the same call.
 */
#define LORA_FIXED_SCRATCH_MAX_TOKENS 16384
lora_status_t lora_apply_fixed_scratch(const void* x, int64_t ldx, void* y, int64_t ldy,
                                       const lora_segments_t* seg, const lora_pool_view_t* view,
                                       int32_t* dev_err, lora_stream_t stream);

/**
 * Kernels this library has launched in this process so far, on every device
 * and stream (a host-side count, incremented at each launch; a launch recorded
 * into a CUDA graph counts once, when it is recorded).  Diagnostic only: lets a
 * caller check how many kernels one call issues.
 */
uint64_t lora_launch_count(void);

/**
 * Test-only: exercises the kernels' timeout path without any fault.  With
 * cycles > 0, every CTA of every compute kernel launched afterwards (in this
 * process, on any stream) first waits, for at most `cycles` clock cycles, on a
 * barrier of its own that nothing ever arrives on, then takes the exit of a
 * wait that ran out: it ORs LORA_DERR_TIMEOUT into the error word, writes no
 * output and returns.  cycles <= 0 disarms the probe.  Not for production use:
 * while armed, every compute call fails this way.  (No passage of the pages;
 * the bounded waits themselves are this library's failure detection.)
 */
void lora_debug_wait_probe(int64_t cycles);

/**
 * Test-only, host only (no device work): the thread-block cluster width the
 * gather kernel is given for a call over the n projections `views` (1 <= n <=
 * LORA_MAX_PROJ; only d_in and d_out are read), before the launcher narrows it
 * by halves to fit every unit of the call in the resident clusters at once.
 * CTA c of a cluster of w owns the c-th of w equal column runs of d_in and of
 * d_out, staged 512 columns at a time; the width is the one with the fewest
 * stages per unit among w0 / 2 .. w0 (w0 = ceil(max(d_in, d_out) / 512), at
 * most 8), ties to the wider.  Returns -1 for a null pointer, n out of range or
 * a dimension below 8.  (No passage of the pages: a work decomposition of this
 * library.)
 */
int32_t lora_debug_gather_width(const lora_pool_view_t* views, int32_t n);

/**
 * Pages one adapter of rank r occupies in a pool of page_elems-element pages:
 * ceil(r * d_in / page_elems) + ceil(r * d_out / page_elems) (bytes per matrix
 * pair (d_in * r + r * d_out) * 2 before rounding to pages: "Multi-LoRA
 * serving: ...", section "The maths that matters").  Returns -1 on bad input.
 */
int64_t lora_pool_pages_needed(int32_t rank, int32_t d_in, int32_t d_out, int32_t page_elems);

/** Static, human-readable text for a status code. */
const char* lora_status_string(lora_status_t status);

/** ABI version of this header (bumped on any incompatible change). */
#define LORA_ABI_VERSION 1
int32_t lora_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_SGMV_H */
