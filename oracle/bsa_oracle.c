/*
 * bsa_oracle.c -- plain fp64 CPU oracle for block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * called by the tests, by the package's smoke check and by the benchmark's
 * CPU-baseline leg.  The product path (the CUDA library) never links, loads
 * or calls it, and this file includes nothing from the product path.
 *
 * What it computes, with the passage each part follows:
 *
 *  - orc_pattern_allows / orc_pattern_csr: the block mask of a pattern,
 *    brute-forced over every (query block, key block) pair.  Sliding window
 *    ("Mask[i][j] = 1 if |i - j| <= W", "Flash MSA Sparse Attention vs Full
 *    Attention", section "The Mechanics"), global tokens that "attend to
 *    everything and are attended by everything" (same page, "Sparse Patterns
 *    Beyond Sliding Windows", "Global Tokens"), causal "key <= query" (same page,
 *    the mask in the flash_sparse_attention pseudocode), block granularity and
 *    per-row lists of active key blocks ("How Do Sparse Attention Kernels Work
 *    in GPU Clusters?", section "How Does Flash-MSA Sparse Attention Work?",
 *    steps 1-3).
 *
 *  - orc_pattern_ex_allows / orc_pattern_ex_csr: the same brute force for
 *    patterns of dilated windows ("Dilated Sliding Window": windows of
 *    growing dilation), a stride ("Strided Patterns": keys sampled at a fixed
 *    interval, in phase with the query block) and global blocks, both in
 *    "Flash MSA Sparse Attention vs Full Attention", section "Sparse Patterns
 *    Beyond Sliding Windows"; per-head assignment is done by the caller.
 *
 *  - orc_attention_rows: exact masked softmax attention
 *    softmax(Q K^T / sqrt(d_k)) V restricted to the allowed (query, key)
 *    pairs ("Flash MSA Sparse Attention vs Full Attention", section "The
 *    Mechanics", the Attention(Q, K, V) formula; the naive masked form in
 *    "Sparse Attention Kernels vs Full Attention Performance", section "How
 *    Sparse Attention Kernels Actually Speed Up Inference").  The block mask
 *    is taken from a CSR as a SET (order and multiplicity ignored), expanded
 *    to tokens, and causal drops key token > query token -- except in a row
 *    flagged as a global query row of a causal model, which attends to every
 *    listed key token ("Global Tokens": they "attend to everything").
 *    FlashAttention tiling is exact, so the tiled kernel must reach this
 *    result up to rounding.  LSE = m + ln(sum exp(s - m)) of the scaled
 *    logits.
 *
 *  - orc_attention_backward: gradients of sum(dO * O) for the same masked
 *    attention, by the chain rule through the softmax, fp64 on fp64 inputs.
 *    Training differentiates through the sparse mask, which must be kept or
 *    rebuilt for the backward pass ("How Do Sparse Attention Kernels Work in
 *    GPU Clusters?", FAQ on training versus inference).
 *
 *  - orc_block_means / orc_block_scores / orc_topk_csr: content-based block
 *    selection: mean-pool Q and K per block (the pooled routing features of
 *    "The Only Guide You Need for Sparse Attention Kernels", section
 *    "Flash-MSA", taken per block), score every (query block, key block)
 *    pair by the dot product of the pooled vectors, keep the top-k key
 *    blocks ("the model predicts importance scores and picks top-k", "How Do
 *    Sparse Attention Kernels Work in GPU Clusters?", section "What Exactly
 *    Is a Sparse Attention Kernel?") plus the diagonal block.  The pages fix
 *    no arithmetic order; the selection is an integer decision, so both
 *    sides take it in fp32 with one stated order:
 *      pooled[d]  = (pairwise tree sum over the block's tokens, fp32) * (1/bs)
 *                   tree: level 1 adds tokens (0,1),(2,3),..., level 2 adds
 *                   neighbouring level-1 sums, ... down to one value;
 *      score(i,j) = a0 + a1, a_c = fp32 chain of fused multiply-adds
 *                   a_c <- fma(q[d], k[d], a_c) over d == c (mod 2), increasing
 *                   d, from 0 (each step rounded once: C fmaf);
 *      order      = score descending, ties to the smaller key block index.
 *    This file must be compiled with -ffp-contract=off.
 *
 * Parity pins live in tests/ (closed forms, invariants, library routines,
 * brute force on tiny inputs); the oracle is checked by them, never by the
 * CUDA path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- helpers */

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------- pattern -> mask */

typedef struct {
    int32_t n_blocks;
    int32_t window_left;
    int32_t window_right;
    int32_t causal;
    int32_t n_global;
    const int32_t *global_blocks; /* n_global entries */
    int32_t global_rows_attend_all;
    int32_t global_rows_noncausal;  /* global query rows take no causal cut */
} orc_pattern;

static int is_global(const orc_pattern *p, int32_t x)
{
    for (int32_t g = 0; g < p->n_global; ++g)
        if (p->global_blocks[g] == x) return 1;
    return 0;
}

/* Does query block i attend to key block j under pattern p?  A global query
 * row "attends to everything" ("Flash MSA Sparse Attention vs Full
 * Attention", "Sparse Patterns Beyond Sliding Windows", "Global Tokens"):
 * with global_rows_noncausal that holds even in a causal model, so such a
 * row is decided before the causal cut. */
int orc_pattern_allows(const orc_pattern *p, int32_t i, int32_t j)
{
    if (i < 0 || i >= p->n_blocks || j < 0 || j >= p->n_blocks) return 0;
    if (p->global_rows_attend_all && p->global_rows_noncausal && is_global(p, i)) return 1;
    if (p->causal && j > i) return 0;               /* key after query */
    if (p->global_rows_attend_all && is_global(p, i)) return 1; /* global query row */
    if (j >= i - p->window_left && j <= i + p->window_right) return 1; /* window */
    if (is_global(p, j)) return 1;                  /* global key block */
    return 0;
}

/* CSR of one (batch, head): row_ptr[n_blocks + 1]; col_idx may be NULL to
 * count only.  Rows list key blocks in ascending order.  Returns nnz. */
int64_t orc_pattern_csr(const orc_pattern *p, int32_t *row_ptr, int32_t *col_idx)
{
    int64_t nnz = 0;
    if (row_ptr) row_ptr[0] = 0;
    for (int32_t i = 0; i < p->n_blocks; ++i) {
        for (int32_t j = 0; j < p->n_blocks; ++j) {
            if (orc_pattern_allows(p, i, j)) {
                if (col_idx) col_idx[nnz] = j;
                ++nnz;
            }
        }
        if (row_ptr) row_ptr[i + 1] = (int32_t)nnz;
    }
    return nnz;
}

/* ----------------------------------------- dilated and strided patterns */

typedef struct {
    int32_t n_blocks;
    int32_t causal;
    int32_t n_windows;              /* 0..4 */
    int32_t window_left[4];
    int32_t window_right[4];
    int32_t window_dilation[4];     /* >= 1 */
    int32_t stride;                 /* 0 = none */
    int32_t n_global;
    const int32_t *global_blocks;
    int32_t global_rows_attend_all;
} orc_pattern_ex;

static int is_global_ex(const orc_pattern_ex *p, int32_t x)
{
    for (int32_t g = 0; g < p->n_global; ++g)
        if (p->global_blocks[g] == x) return 1;
    return 0;
}

/* Does query block i attend to key block j?  Window w holds the key blocks
 * i + dilation * t, -left <= t <= right (several windows of growing
 * dilation: "Flash MSA Sparse Attention vs Full Attention", section "Sparse
 * Patterns Beyond Sliding Windows", "Dilated Sliding Window"); the stride
 * holds the key blocks whose distance to i is a multiple of it (same
 * section, "Strided Patterns"); global blocks and causal as in
 * orc_pattern_allows. */
int orc_pattern_ex_allows(const orc_pattern_ex *p, int32_t i, int32_t j)
{
    if (i < 0 || i >= p->n_blocks || j < 0 || j >= p->n_blocks) return 0;
    if (p->causal && j > i) return 0;
    if (p->global_rows_attend_all && is_global_ex(p, i)) return 1;
    const int64_t delta = (int64_t)j - i;
    for (int32_t w = 0; w < p->n_windows; ++w) {
        const int64_t d = p->window_dilation[w];
        if (delta % d == 0 && delta >= -(int64_t)p->window_left[w] * d &&
            delta <= (int64_t)p->window_right[w] * d)
            return 1;
    }
    if (p->stride > 0 && delta % p->stride == 0) return 1;
    if (is_global_ex(p, j)) return 1;
    return 0;
}

/* CSR of one head under an orc_pattern_ex, brute force as orc_pattern_csr. */
int64_t orc_pattern_ex_csr(const orc_pattern_ex *p, int32_t *row_ptr, int32_t *col_idx)
{
    int64_t nnz = 0;
    if (row_ptr) row_ptr[0] = 0;
    for (int32_t i = 0; i < p->n_blocks; ++i) {
        for (int32_t j = 0; j < p->n_blocks; ++j) {
            if (orc_pattern_ex_allows(p, i, j)) {
                if (col_idx) col_idx[nnz] = j;
                ++nnz;
            }
        }
        if (row_ptr) row_ptr[i + 1] = (int32_t)nnz;
    }
    return nnz;
}

/* ------------------------------------------------------------- attention */

/*
 * Exact masked attention for a list of query rows.
 *   q, k, v     bf16 bit patterns, [BH, N, D] contiguous (BH = B*H)
 *   row_ptr     [BH*nb + 1], col_idx: CSR over rows r = bh*nb + i (nb = N/block)
 *   row_flags   optional [BH*nb]: bit 0 set = that CSR row takes no causal cut
 *               (a global query row of a causal model)
 *   rows        n_rows flat row ids bh*N + t
 *   out         [n_rows, D] fp64;  lse [n_rows] fp64 (-inf for an empty row)
 *   nkeys_out   optional [n_rows]: number of allowed key tokens per row
 */
void orc_attention_rows(int32_t BH, int32_t N, int32_t D, int32_t block,
                        const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *row_ptr, const int32_t *col_idx,
                        const uint8_t *row_flags,
                        double scale, int32_t causal,
                        int64_t n_rows, const int64_t *rows,
                        double *out, double *lse, int64_t *nkeys_out)
{
    const int32_t nb = N / block;
#pragma omp parallel
    {
        unsigned char *allowed = (unsigned char *)malloc((size_t)nb);
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < n_rows; ++n) {
            const int64_t flat = rows[n];
            const int32_t bh = (int32_t)(flat / N);
            const int32_t t = (int32_t)(flat % N);
            const int32_t i = t / block;
            const int64_t r = (int64_t)bh * nb + i;
            const int32_t row_causal = causal && !(row_flags && (row_flags[r] & 1));
            /* 1. block mask of this row, as a set */
            memset(allowed, 0, (size_t)nb);
            for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
                const int32_t j = col_idx[e];
                if (j >= 0 && j < nb) allowed[j] = 1;
            }
            /* 2. token mask + 3. logits */
            const uint16_t *qrow = q + ((int64_t)bh * N + t) * D;
            for (int32_t d = 0; d < D; ++d) qd[d] = bf16_to_f64(qrow[d]);
            int32_t cnt = 0;
            for (int32_t j = 0; j < nb; ++j) {
                if (!allowed[j]) continue;
                for (int32_t kk = j * block; kk < (j + 1) * block; ++kk) {
                    if (row_causal && kk > t) continue;
                    const uint16_t *krow = k + ((int64_t)bh * N + kk) * D;
                    double dot = 0.0;
                    for (int32_t d = 0; d < D; ++d) dot += qd[d] * bf16_to_f64(krow[d]);
                    s[cnt] = scale * dot;
                    key[cnt] = kk;
                    ++cnt;
                }
            }
            if (nkeys_out) nkeys_out[n] = cnt;
            double *o = out + n * (int64_t)D;
            if (cnt == 0) {
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                lse[n] = -INFINITY;
                continue;
            }
            /* 4. normalise */
            double m = s[0];
            for (int32_t c = 1; c < cnt; ++c) if (s[c] > m) m = s[c];
            double l = 0.0;
            for (int32_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int32_t c = 0; c < cnt; ++c) {
                const double p = exp(s[c] - m);
                l += p;
                const uint16_t *vrow = v + ((int64_t)bh * N + key[c]) * D;
                for (int32_t d = 0; d < D; ++d) acc[d] += p * bf16_to_f64(vrow[d]);
            }
            for (int32_t d = 0; d < D; ++d) o[d] = acc[d] / l;
            lse[n] = m + log(l);
        }
        free(allowed); free(s); free(key); free(qd); free(acc);
    }
}

/* ------------------------------------------------------------- backward */

/*
 * One query row of the backward: the allowed key tokens of row (bh, t)
 * (block mask as a set, expanded to tokens, causal k <= t), their softmax
 * weights p, dp = dO_t . V_k, Dt = sum_k p dp, and ds = p (dp - Dt), all fp64.
 * Returns the number of allowed keys; key[] ascending.
 */
static int32_t bwd_query_row(int32_t N, int32_t D, int32_t block, const double *q, const double *k,
                             const double *v, const double *dout, const int32_t *row_ptr,
                             const int32_t *col_idx, const uint8_t *row_flags, double scale,
                             int32_t causal_all, int32_t bh, int32_t t,
                             unsigned char *allowed, int32_t *key, double *p, double *ds)
{
    const int32_t nb = N / block;
    const int32_t i = t / block;
    const int64_t r = (int64_t)bh * nb + i;
    /* a flagged row (bit 0) takes no causal cut */
    const int32_t causal = causal_all && !(row_flags && (row_flags[r] & 1));
    memset(allowed, 0, (size_t)nb);
    for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
        const int32_t j = col_idx[e];
        if (j >= 0 && j < nb) allowed[j] = 1;
    }
    const double *qt = q + ((int64_t)bh * N + t) * D;
    const double *dot = dout + ((int64_t)bh * N + t) * D;
    int32_t n = 0;
    double m = -INFINITY;
    for (int32_t j = 0; j < nb; ++j) {
        if (!allowed[j]) continue;
        for (int32_t x = 0; x < block; ++x) {
            const int32_t kk = j * block + x;
            if (causal && kk > t) break;
            const double *kr = k + ((int64_t)bh * N + kk) * D;
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) acc += qt[d] * kr[d];
            key[n] = kk;
            p[n] = acc * scale;
            if (p[n] > m) m = p[n];
            ++n;
        }
    }
    double l = 0.0;
    for (int32_t a = 0; a < n; ++a) {
        p[a] = exp(p[a] - m);
        l += p[a];
    }
    double Dt = 0.0;
    for (int32_t a = 0; a < n; ++a) {
        p[a] /= l;
        const double *vr = v + ((int64_t)bh * N + key[a]) * D;
        double dp = 0.0;
        for (int32_t d = 0; d < D; ++d) dp += dot[d] * vr[d];
        ds[a] = dp;
        Dt += p[a] * dp;
    }
    for (int32_t a = 0; a < n; ++a) ds[a] = p[a] * (ds[a] - Dt);
    return n;
}

/*
 * Gradients of L = sum(dO * O) for the masked attention of orc_attention_rows,
 * by the chain rule through the softmax: dP = dO V^T, dS = P o (dP -
 * rowsum(P o dP)), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO; fp64.
 *   q, k, v, dout  fp64 [BH, N, D]
 *   dq     [n_q][D] for query rows qrows (flat bh*N + t)
 *   dk, dv [n_k][D] for key rows krows (flat bh*N + t), summed over every
 *          query row that attends the key
 *   row_flags  optional [BH*nb]: bit 0 set = that CSR row takes no causal cut
 *          (as in orc_attention_rows)
 * A row with no allowed key has zero gradients.
 */
void orc_attention_backward(int32_t BH, int32_t N, int32_t D, int32_t block,
                            const double *q, const double *k, const double *v, const double *dout,
                            const int32_t *row_ptr, const int32_t *col_idx, const uint8_t *row_flags,
                            double scale, int32_t causal,
                            int64_t n_q, const int64_t *qrows, double *dq,
                            int64_t n_k, const int64_t *krows, double *dk, double *dv)
{
    const int32_t nb = N / block;
    (void)BH;
#pragma omp parallel
    {
        unsigned char *allowed = (unsigned char *)malloc((size_t)nb);
        int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        double *ds = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t n = 0; n < n_q; ++n) {
            const int32_t bh = (int32_t)(qrows[n] / N), t = (int32_t)(qrows[n] % N);
            const int32_t cnt = bwd_query_row(N, D, block, q, k, v, dout, row_ptr, col_idx, row_flags, scale,
                                              causal, bh, t, allowed, key, p, ds);
            double *o = dq + n * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int32_t a = 0; a < cnt; ++a) {
                const double *kr = k + ((int64_t)bh * N + key[a]) * D;
                for (int32_t d = 0; d < D; ++d) o[d] += scale * ds[a] * kr[d];
            }
        }
        /* key rows: one group per (bh, key block); every query row that sees
         * the block is computed once per group and adds into each requested
         * key of the block it sees */
#pragma omp for schedule(dynamic, 1)
        for (int64_t g = 0; g < n_k; ++g) {
            const int32_t bh = (int32_t)(krows[g] / N), jb = (int32_t)(krows[g] % N) / block;
            int first = 1;
            for (int64_t h = 0; h < g; ++h)
                if (krows[h] / N == bh && (int32_t)(krows[h] % N) / block == jb) first = 0;
            if (!first) continue;  /* the group was handled at its first member */
            for (int64_t n = g; n < n_k; ++n)
                if (krows[n] / N == bh && (int32_t)(krows[n] % N) / block == jb)
                    for (int32_t d = 0; d < D; ++d) dk[n * D + d] = dv[n * D + d] = 0.0;
            for (int32_t i = 0; i < nb; ++i) {
                const int64_t r = (int64_t)bh * nb + i;
                int has = 0;
                for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) has |= (col_idx[e] == jb);
                if (!has) continue;
                for (int32_t x = 0; x < block; ++x) {
                    const int32_t t = i * block + x;
                    const int32_t cnt = bwd_query_row(N, D, block, q, k, v, dout, row_ptr, col_idx, row_flags,
                                                      scale, causal, bh, t, allowed, key, p, ds);
                    const double *qt = q + ((int64_t)bh * N + t) * D;
                    const double *dot = dout + ((int64_t)bh * N + t) * D;
                    for (int64_t n = g; n < n_k; ++n) {
                        if (krows[n] / N != bh || (int32_t)(krows[n] % N) / block != jb) continue;
                        const int32_t tk = (int32_t)(krows[n] % N);
                        int32_t lo = 0, hi = cnt;  /* key[] ascending: binary search */
                        while (lo < hi) {
                            const int32_t mid = (lo + hi) / 2;
                            if (key[mid] < tk) lo = mid + 1; else hi = mid;
                        }
                        if (lo == cnt || key[lo] != tk) continue;
                        for (int32_t d = 0; d < D; ++d) {
                            dk[n * D + d] += scale * ds[lo] * qt[d];
                            dv[n * D + d] += p[lo] * dot[d];
                        }
                    }
                }
            }
        }
        free(allowed);
        free(key);
        free(p);
        free(ds);
    }
}

/* ------------------------------------------------ content-based top-k */

/* Block means of x [BH, N, D] (bf16 bits) -> out [BH, nb, D] fp32.
 * block must be a power of two <= 4096. */
void orc_block_means(int32_t BH, int32_t N, int32_t D, int32_t block,
                     const uint16_t *x, float *out)
{
    const int32_t nb = N / block;
    const float inv = 1.0f / (float)block; /* exact: block is a power of two */
#pragma omp parallel
    {
        float *buf = (float *)malloc(sizeof(float) * (size_t)block);
#pragma omp for collapse(2) schedule(static)
        for (int32_t bh = 0; bh < BH; ++bh) {
            for (int32_t i = 0; i < nb; ++i) {
                for (int32_t d = 0; d < D; ++d) {
                    for (int32_t t = 0; t < block; ++t)
                        buf[t] = bf16_to_f32(x[((int64_t)bh * N + (int64_t)i * block + t) * D + d]);
                    for (int32_t w = block / 2; w >= 1; w /= 2)
                        for (int32_t t = 0; t < w; ++t) buf[t] = buf[2 * t] + buf[2 * t + 1];
                    out[((int64_t)bh * nb + i) * D + d] = buf[0] * inv;
                }
            }
        }
        free(buf);
    }
}

/* Block scores: scores[bh][i][j] = pooled_q[bh][i] . pooled_k[bh][j] in the
 * stated fp32 order (two fused multiply-add chains over even and odd d).  D
 * must be even. */
void orc_block_scores(int32_t BH, int32_t nb, int32_t D,
                      const float *qbar, const float *kbar, float *scores)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int32_t bh = 0; bh < BH; ++bh) {
        for (int32_t i = 0; i < nb; ++i) {
            const float *qi = qbar + ((int64_t)bh * nb + i) * D;
            for (int32_t j = 0; j < nb; ++j) {
                const float *kj = kbar + ((int64_t)bh * nb + j) * D;
                float a0 = 0.0f, a1 = 0.0f;
                for (int32_t d = 0; d + 1 < D; d += 2) {
                    a0 = fmaf(qi[d], kj[d], a0);
                    a1 = fmaf(qi[d + 1], kj[d + 1], a1);
                }
                scores[((int64_t)bh * nb + i) * nb + j] = a0 + a1;
            }
        }
    }
}

/* Is (s1, j1) ahead of (s2, j2) in the selection order? */
static int ahead(float s1, int32_t j1, float s2, int32_t j2)
{
    return (s1 > s2) || (s1 == s2 && j1 < j2);
}

/* Top-k selection over scores [BH, nb, nb] -> CSR over rows r = bh*nb + i.
 * Each row keeps its topk best key blocks, adds the diagonal when asked and
 * absent, and is written in ascending key order.  row_ptr [BH*nb + 1];
 * col_idx may be NULL (count only).  Returns nnz. */
int64_t orc_topk_csr(int32_t BH, int32_t nb, const float *scores, int32_t topk,
                     int32_t include_diag, int32_t *row_ptr, int32_t *col_idx)
{
    const int64_t R = (int64_t)BH * nb;
    int32_t *len = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)R * (size_t)(topk + 1));
#pragma omp parallel
    {
        int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            const int32_t i = (int32_t)(r % nb);
            const float *s = scores + r * nb;
            /* partial selection sort: the topk first positions of the order */
            for (int32_t j = 0; j < nb; ++j) idx[j] = j;
            for (int32_t a = 0; a < topk; ++a) {
                int32_t best = a;
                for (int32_t b = a + 1; b < nb; ++b)
                    if (ahead(s[idx[b]], idx[b], s[idx[best]], idx[best])) best = b;
                const int32_t tmp = idx[a]; idx[a] = idx[best]; idx[best] = tmp;
            }
            int32_t *out = sel + r * (topk + 1);
            int32_t n = 0, has_diag = 0;
            for (int32_t a = 0; a < topk; ++a) {
                out[n++] = idx[a];
                if (idx[a] == i) has_diag = 1;
            }
            if (include_diag && !has_diag) out[n++] = i;
            /* ascending order (insertion sort on <= topk+1 entries) */
            for (int32_t a = 1; a < n; ++a) {
                const int32_t x = out[a];
                int32_t b = a - 1;
                while (b >= 0 && out[b] > x) { out[b + 1] = out[b]; --b; }
                out[b + 1] = x;
            }
            len[r] = n;
        }
        free(idx);
    }
    int64_t nnz = 0;
    if (row_ptr) row_ptr[0] = 0;
    for (int64_t r = 0; r < R; ++r) {
        if (col_idx)
            for (int32_t a = 0; a < len[r]; ++a) col_idx[nnz + a] = sel[r * (topk + 1) + a];
        nnz += len[r];
        if (row_ptr) row_ptr[r + 1] = (int32_t)nnz;
    }
    free(len);
    free(sel);
    return nnz;
}
