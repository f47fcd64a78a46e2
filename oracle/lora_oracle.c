/*
 * lora_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * multi-adapter LoRA path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg call it; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * Everything is computed in IEEE double from the exact bf16 input bits.
 *
 * What it computes, and where the pages define it:
 *
 *  - oracle_adapter_bytes: bytes of one adapted matrix pair,
 *    (d_in * r + r * d_out) * b  ("Multi-LoRA serving: the single translator
 *    with a thousand glossaries", section "The maths that matters",
 *    memory-per-adapter formula and the Llama-3-70B table).
 *  - oracle_pages_needed: pages an adapter occupies in a paged pool: each of
 *    A and B is sliced into fixed-size pages ("Multi-LoRA Serving in
 *    Production", section "Unified Paged Memory").
 *  - oracle_segments_build: grouping of the batch's tokens by adapter
 *    ("Multi-LoRA serving: ...", section "SGMV: the kernel that holds it all
 *    up") -- GROUP mode -- or into contiguous runs that share one adapter id
 *    ("Multi-LoRA Serving in Production", section "Punica and Segmented
 *    Gather Matrix-Vector Multiplication (SGMV)") -- CONTIGUOUS mode.
 *  - oracle_work_lists: the per-segment work units derived from the segments
 *    (a deterministic function of the segments and two dispatch constants).
 *  - oracle_lora_apply: y = x W0 + (alpha/r) (x A) B per token, with x W0
 *    given as y0 ("Multi-LoRA Serving in Production", section "Mathematical
 *    Formulation and the Batching Challenge"; per-token adapter a(t) as in
 *    "Multi-LoRA serving: ...", section "SGMV: the kernel that holds it all
 *    up").  Adapter elements are read through the page table.
 *  - oracle_shrink / oracle_expand: the two stages of that product
 *    ("Multi-LoRA Serving in Production", "Shrink Stage" / "Expand Stage").
 *  - oracle_base_apply: the base projection x W0 with that product added in
 *    the same pass ("Multi-LoRA Serving: Many Adapters on One GPU", section
 *    "How batching across adapters works").
 *  - oracle_lora_backward: the gradients of that product for training the
 *    adapters; the base is frozen and receives none, only A and B do ("QLoRA
 *    and multi-LoRA at the limit on small models", section "The bare
 *    mechanism: LoRA, and why you can train on a 4-bit base").
 *  - oracle_bf16_rne: rounding of a double to the nearest bf16, ties to even.
 *
 * Conventions (the readings this oracle takes where the pages are silent):
 *  - A_i is stored as r_i rows of d_in elements (row j = column j of the
 *    d_in x r_i matrix A_i); B_i as r_i rows of d_out elements.
 *  - logical element e of a matrix whose first page-list slot is page0 is at
 *    pool[page_list[page0 + e / P] * P + e % P].
 *  - adapter id -1 means "no adapter": the token keeps y0.  Ids outside
 *    [-1, n_adapters), ranks outside [1, max_rank] and page ids outside the
 *    pool mark an error bit and the token keeps y0.
 *  - scale s_i is given per adapter (alpha_i / r_i), never derived from r_i.
 *
 * Parity pins: every function here is checked in tests/test_oracle_pins.py
 * against the pages' worked numbers, closed forms, library matmuls and
 * invariants (merged weight, B = 0, zero padding, segment order).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_ERR_BAD_ADAPTER 1
#define ORC_ERR_BAD_PAGE 2
#define ORC_ERR_BAD_RANK 4

typedef struct {
    int32_t rank;
    float scale;
    int32_t a_page0;
    int32_t b_page0;
} orc_desc_t;

/* ---------------------------------------------------------------- sizing -- */

int64_t oracle_adapter_bytes(int64_t rank, int64_t d_in, int64_t d_out, int64_t bytes_per_param)
{
    return (d_in * rank + rank * d_out) * bytes_per_param;
}

int64_t oracle_pages_needed(int64_t rank, int64_t d_in, int64_t d_out, int64_t page_elems)
{
    int64_t a = rank * d_in, b = rank * d_out;
    return (a + page_elems - 1) / page_elems + (b + page_elems - 1) / page_elems;
}

/* ----------------------------------------------------------- bf16 values -- */

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Nearest bf16 to v, ties to even (bf16: 8 significant bits, fp32 exponent range). */
uint16_t oracle_bf16_rne(double v)
{
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    if (isinf(v)) return v > 0 ? 0x7F80 : 0xFF80;
    int e;
    (void)frexp(v, &e);              /* |v| = m * 2^e, m in [0.5, 1) */
    int lead = e - 1;                /* |v| in [2^lead, 2^(lead+1)) */
    if (lead < -126) lead = -126;    /* subnormal range: fixed quantum 2^-133 */
    double q = ldexp(1.0, lead - 7); /* spacing of bf16 values around v */
    double r = nearbyint(v / q) * q; /* default rounding mode: ties to even */
    if (fabs(r) >= ldexp(1.0, 128)) return v > 0 ? 0x7F80 : 0xFF80;
    float f = (float)r;              /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

void oracle_bf16_rne_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(v[i]);
}

/* ------------------------------------------------------- page translation -- */

typedef struct {
    const uint16_t* pool;
    int64_t n_pages;
    int64_t page_elems;
    const int32_t* page_list;
    int64_t n_page_list;
} orc_pool_t;

/* Element e of the matrix whose pages start at slot page0.  Returns 0 and sets
 * *bad on an out-of-range page-list slot or physical page. */
static double pool_elem(const orc_pool_t* p, int64_t page0, int64_t e, int* bad)
{
    int64_t slot = page0 + e / p->page_elems;
    if (slot < 0 || slot >= p->n_page_list) { *bad = 1; return 0.0; }
    int64_t page = p->page_list[slot];
    if (page < 0 || page >= p->n_pages) { *bad = 1; return 0.0; }
    return oracle_bf16_to_double(p->pool[page * p->page_elems + e % p->page_elems]);
}

/* Copy out logical matrix rows x cols (row-major) whose pages start at page0. */
int oracle_unpack_matrix(const uint16_t* pool, int64_t n_pages, int64_t page_elems,
                         const int32_t* page_list, int64_t n_page_list,
                         int64_t page0, int64_t rows, int64_t cols, uint16_t* out)
{
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    for (int64_t e = 0; e < rows * cols; ++e) {
        int64_t slot = page0 + e / page_elems;
        if (slot < 0 || slot >= n_page_list) return ORC_ERR_BAD_PAGE;
        int64_t page = page_list[slot];
        if (page < 0 || page >= n_pages) return ORC_ERR_BAD_PAGE;
        out[e] = p.pool[page * page_elems + e % page_elems];
    }
    return 0;
}

/* Check one adapter for use by a token: returns 0 if usable, else error bits. */
static int adapter_check(const orc_desc_t* d, int32_t max_rank, const orc_pool_t* p,
                         int64_t d_in, int64_t d_out)
{
    if (d->rank < 1 || d->rank > max_rank) return ORC_ERR_BAD_RANK;
    int64_t na = (d->rank * d_in + p->page_elems - 1) / p->page_elems;
    int64_t nb = (d->rank * d_out + p->page_elems - 1) / p->page_elems;
    for (int64_t s = 0; s < na; ++s) {
        int64_t slot = d->a_page0 + s;
        if (slot < 0 || slot >= p->n_page_list) return ORC_ERR_BAD_PAGE;
        if (p->page_list[slot] < 0 || p->page_list[slot] >= p->n_pages) return ORC_ERR_BAD_PAGE;
    }
    for (int64_t s = 0; s < nb; ++s) {
        int64_t slot = d->b_page0 + s;
        if (slot < 0 || slot >= p->n_page_list) return ORC_ERR_BAD_PAGE;
        if (p->page_list[slot] < 0 || p->page_list[slot] >= p->n_pages) return ORC_ERR_BAD_PAGE;
    }
    return 0;
}

/* --------------------------------------------------------- the LoRA delta -- */

/*
 * For every token t with adapter i = ids[t] in [0, n_adapters):
 *     h_j    = sum_k x[t,k] * A_i[j,k]                       (j < r_i)
 *     y[t,n] = y0[t,n] + s_i * sum_j h_j * B_i[j,n]
 * Other tokens: y[t,n] = y0[t,n].  y is double [T, d_out] (dense).
 * Returns the OR of the error bits met.
 */
int oracle_lora_apply(const uint16_t* x, int64_t ldx, const uint16_t* y0, int64_t ldy0,
                      double* y, int64_t T, const int32_t* ids,
                      const uint16_t* pool, int64_t n_pages, int64_t page_elems,
                      const int32_t* page_list, int64_t n_page_list,
                      const void* adapters, int32_t n_adapters, int32_t max_rank,
                      int64_t d_in, int64_t d_out)
{
    const orc_desc_t* desc = (const orc_desc_t*)adapters;
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    int err = 0;
    double h[256];
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < d_out; ++n) y[t * d_out + n] = oracle_bf16_to_double(y0[t * ldy0 + n]);
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }
        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);
        if (bad || desc[i].rank > 256) { err |= bad ? bad : ORC_ERR_BAD_RANK; continue; }
        int64_t r = desc[i].rank;
        double s = (double)desc[i].scale;
        int oob = 0;
        for (int64_t j = 0; j < r; ++j) {            /* shrink: x . A_i (d_in -> r) */
            double acc = 0.0;
            for (int64_t k = 0; k < d_in; ++k)
                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);
            h[j] = acc;
        }
        for (int64_t n = 0; n < d_out; ++n) {        /* expand: h . B_i (r -> d_out) */
            double acc = 0.0;
            for (int64_t j = 0; j < r; ++j)
                acc += h[j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);
            y[t * d_out + n] += s * acc;
        }
    }
    return err;
}

/*
 * Shrink stage alone: h[t, j] = sum_k x[t,k] * A_i[j,k] for j < r_i (no scale);
 * h is double [T, ldh]; rows of tokens without a usable adapter are left as given.
 */
int oracle_shrink(const uint16_t* x, int64_t ldx, double* h, int64_t ldh, int64_t T,
                  const int32_t* ids, const uint16_t* pool, int64_t n_pages, int64_t page_elems,
                  const int32_t* page_list, int64_t n_page_list, const void* adapters,
                  int32_t n_adapters, int32_t max_rank, int64_t d_in, int64_t d_out)
{
    const orc_desc_t* desc = (const orc_desc_t*)adapters;
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    int err = 0;
    for (int64_t t = 0; t < T; ++t) {
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }
        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);
        if (bad) { err |= bad; continue; }
        int oob = 0;
        for (int64_t j = 0; j < desc[i].rank; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < d_in; ++k)
                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);
            h[t * ldh + j] = acc;
        }
    }
    return err;
}

/*
 * Expand stage alone: y[t,n] = y0[t,n] + s_i * sum_j h[t,j] * B_i[j,n], with h
 * given as fp32 values; y is double [T, d_out].
 */
int oracle_expand(const float* hin, int64_t ldh, const uint16_t* y0, int64_t ldy0, double* y,
                  int64_t T, const int32_t* ids, const uint16_t* pool, int64_t n_pages,
                  int64_t page_elems, const int32_t* page_list, int64_t n_page_list,
                  const void* adapters, int32_t n_adapters, int32_t max_rank,
                  int64_t d_in, int64_t d_out)
{
    const orc_desc_t* desc = (const orc_desc_t*)adapters;
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    int err = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < d_out; ++n) y[t * d_out + n] = oracle_bf16_to_double(y0[t * ldy0 + n]);
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }
        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);
        if (bad) { err |= bad; continue; }
        double s = (double)desc[i].scale;
        int oob = 0;
        for (int64_t n = 0; n < d_out; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < desc[i].rank; ++j)
                acc += (double)hin[t * ldh + j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);
            y[t * d_out + n] += s * acc;
        }
    }
    return err;
}

/* ------------------------------------------- base projection and delta -- */

/*
 * The base projection with every token's adapter term in the same pass
 * ("Multi-LoRA Serving: Many Adapters on One GPU", section "How batching
 * across adapters works": one base product shared by the whole batch plus each
 * token's own adapter term; "Multi-LoRA Serving in Production", section
 * "Mathematical Formulation and the Batching Challenge": y = x W0 + (alpha/r)
 * (x A) B):
 *     base     = sum_k x[t,k] * W0[n,k]
 *     h_j      = sum_k x[t,k] * A_i[j,k]                     (j < r_i)
 *     y[t,n]   = base + s_i * sum_j h_j * B_i[j,n]
 * W0 is bf16 [d_out, ldw]: row n holds output n's weights over the d_in inputs.
 * Tokens with id -1, and tokens whose adapter fails the checks (their error
 * bits are returned), get the base term alone.  y is double [T, d_out].
 */
int oracle_base_apply(const uint16_t* x, int64_t ldx, const uint16_t* w0, int64_t ldw, double* y,
                      int64_t T, const int32_t* ids, const uint16_t* pool, int64_t n_pages,
                      int64_t page_elems, const int32_t* page_list, int64_t n_page_list,
                      const void* adapters, int32_t n_adapters, int32_t max_rank,
                      int64_t d_in, int64_t d_out)
{
    const orc_desc_t* desc = (const orc_desc_t*)adapters;
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    int err = 0;
    double hv[256];
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < d_out; ++n) {        /* the shared base product */
            double base = 0.0;
            for (int64_t k = 0; k < d_in; ++k)
                base += oracle_bf16_to_double(x[t * ldx + k]) * oracle_bf16_to_double(w0[n * ldw + k]);
            y[t * d_out + n] = base;
        }
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }
        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);
        if (bad || desc[i].rank > 256) { err |= bad ? bad : ORC_ERR_BAD_RANK; continue; }
        int64_t r = desc[i].rank;
        double s = (double)desc[i].scale;
        int oob = 0;
        for (int64_t j = 0; j < r; ++j) {            /* the token's shrink over A_i */
            double acc = 0.0;
            for (int64_t k = 0; k < d_in; ++k)
                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);
            hv[j] = acc;
        }
        for (int64_t n = 0; n < d_out; ++n) {        /* its expand over B_i, onto the base */
            double term = 0.0;
            for (int64_t j = 0; j < r; ++j)
                term += hv[j] * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);
            y[t * d_out + n] += s * term;
        }
    }
    return err;
}

/* -------------------------------------------------------- the gradients -- */

/* Position of logical element e of the matrix whose pages start at page0, in
 * the pool's layout (the gradient arrays share it); -1 if out of range. */
static int64_t pool_pos(const orc_pool_t* p, int64_t page0, int64_t e)
{
    int64_t slot = page0 + e / p->page_elems;
    if (slot < 0 || slot >= p->n_page_list) return -1;
    int64_t page = p->page_list[slot];
    if (page < 0 || page >= p->n_pages) return -1;
    return page * p->page_elems + e % p->page_elems;
}

/*
 * Gradients of a loss L through the LoRA delta, given g = dL/dy (bf16).  The
 * base W0 is frozen and gets no gradient; only the adapters' A and B are
 * trainable, and the adapter path is the only one the gradient flows through.
 * Differentiating y[t,n] = y0[t,n] + s_i sum_j (sum_k x[t,k] A_i[j,k]) B_i[j,n]
 * token by token, for every token t with a usable adapter i:
 *     h_j        = sum_k x[t,k] A_i[j,k]
 *     u_j        = sum_n g[t,n] B_i[j,n]
 *     dB_i[j,n] += s_i h_j g[t,n]
 *     dA_i[j,k] += s_i u_j x[t,k]
 *     dx[t,k]    = s_i sum_j u_j A_i[j,k]
 * Other tokens: dx[t,k] = 0 and no gradient.  dA_i and dB_i are added (in
 * token order) into grad, a double array laid out like the pool: the gradient
 * of the element at pool position q is grad[q].  dx is double [T, d_in].
 * Returns the OR of the error bits met (as oracle_lora_apply).
 */
int oracle_lora_backward(const uint16_t* x, int64_t ldx, const uint16_t* g, int64_t ldg,
                         double* dx, double* grad, int64_t T, const int32_t* ids,
                         const uint16_t* pool, int64_t n_pages, int64_t page_elems,
                         const int32_t* page_list, int64_t n_page_list,
                         const void* adapters, int32_t n_adapters, int32_t max_rank,
                         int64_t d_in, int64_t d_out)
{
    const orc_desc_t* desc = (const orc_desc_t*)adapters;
    orc_pool_t p = {pool, n_pages, page_elems, page_list, n_page_list};
    int err = 0;
    double h[256], u[256];
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < d_in; ++k) dx[t * d_in + k] = 0.0;
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_adapters) { err |= ORC_ERR_BAD_ADAPTER; continue; }
        int bad = adapter_check(&desc[i], max_rank, &p, d_in, d_out);
        if (bad || desc[i].rank > 256) { err |= bad ? bad : ORC_ERR_BAD_RANK; continue; }
        int64_t r = desc[i].rank;
        double s = (double)desc[i].scale;
        int oob = 0;
        for (int64_t j = 0; j < r; ++j) {            /* h = x . A_i^T */
            double acc = 0.0;
            for (int64_t k = 0; k < d_in; ++k)
                acc += oracle_bf16_to_double(x[t * ldx + k]) * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);
            h[j] = acc;
        }
        for (int64_t j = 0; j < r; ++j) {            /* u = g . B_i^T */
            double acc = 0.0;
            for (int64_t n = 0; n < d_out; ++n)
                acc += oracle_bf16_to_double(g[t * ldg + n]) * pool_elem(&p, desc[i].b_page0, j * d_out + n, &oob);
            u[j] = acc;
        }
        for (int64_t j = 0; j < r; ++j) {            /* dB_i += s h g^T */
            for (int64_t n = 0; n < d_out; ++n)
                grad[pool_pos(&p, desc[i].b_page0, j * d_out + n)] += s * h[j] * oracle_bf16_to_double(g[t * ldg + n]);
        }
        for (int64_t j = 0; j < r; ++j) {            /* dA_i += s u x^T */
            for (int64_t k = 0; k < d_in; ++k)
                grad[pool_pos(&p, desc[i].a_page0, j * d_in + k)] += s * u[j] * oracle_bf16_to_double(x[t * ldx + k]);
        }
        for (int64_t k = 0; k < d_in; ++k) {         /* dx = s u . A_i */
            double acc = 0.0;
            for (int64_t j = 0; j < r; ++j) acc += u[j] * pool_elem(&p, desc[i].a_page0, j * d_in + k, &oob);
            dx[t * d_in + k] = s * acc;
        }
    }
    return err;
}

/* ------------------------------------------------------------ segmenting -- */

/*
 * GROUP (mode 0): one segment per adapter id that occurs, in ascending id;
 *   inside a segment, tokens in ascending original index.
 * CONTIGUOUS (mode 1): one segment per maximal run of consecutive tokens that
 *   share one id, in token order.
 * Tokens with id -1 (and invalid ids, which also set an error bit) belong to no
 * segment.  perm lists the segments' tokens in segment order; indptr[s] ..
 * indptr[s+1] is segment s's range of perm; seg_adapter[s] its adapter.
 * Returns the number of segments; *n_tokens receives the number of tokens
 * placed and *err the error bits.
 */
int32_t oracle_segments_build(const int32_t* ids, int32_t T, int32_t n_adapters, int32_t mode,
                              int32_t* perm, int32_t* indptr, int32_t* seg_adapter,
                              int32_t* n_tokens, int32_t* err)
{
    int32_t nseg = 0, placed = 0;
    *err = 0;
    for (int32_t t = 0; t < T; ++t)
        if (ids[t] < -1 || ids[t] >= n_adapters) *err |= ORC_ERR_BAD_ADAPTER;
    indptr[0] = 0;
    if (mode == 0) {
        for (int32_t a = 0; a < n_adapters; ++a) {      /* ascending adapter id */
            int32_t start = placed;
            for (int32_t t = 0; t < T; ++t)              /* ascending token index */
                if (ids[t] == a) perm[placed++] = t;
            if (placed > start) {
                seg_adapter[nseg] = a;
                indptr[++nseg] = placed;
            }
        }
    } else {
        int32_t t = 0;
        while (t < T) {
            int32_t a = ids[t];
            if (a < 0 || a >= n_adapters) { ++t; continue; }
            while (t < T && ids[t] == a) perm[placed++] = t++;
            seg_adapter[nseg] = a;
            indptr[++nseg] = placed;
        }
    }
    *n_tokens = placed;
    return nseg;
}

/*
 * Work units derived from the segments: a segment of at most short_max tokens
 * is one short unit (its segment index); a longer segment is cut into tiles of
 * tile_m tokens, one long unit (segment index, offset in the segment) each.
 * Both lists are in segment order.  counts[0] = short units, counts[1] = long.
 */
void oracle_work_lists(const int32_t* indptr, int32_t n_segs, int32_t short_max, int32_t tile_m,
                       int32_t* short_units, int32_t* long_units, int32_t* counts)
{
    int32_t ns = 0, nl = 0;
    for (int32_t s = 0; s < n_segs; ++s) {
        int32_t len = indptr[s + 1] - indptr[s];
        if (len <= short_max) {
            short_units[ns++] = s;
        } else {
            for (int32_t m0 = 0; m0 < len; m0 += tile_m) {
                long_units[2 * nl] = s;
                long_units[2 * nl + 1] = m0;
                ++nl;
            }
        }
    }
    counts[0] = ns;
    counts[1] = nl;
}
