/*
 * bsa.h -- C ABI of libbsa.so: block-sparse FlashAttention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The method (what every entry point below serves): attention
 * softmax(Q K^T * scale) V evaluated only on the (query block, key block)
 * pairs a block mask allows, tile by tile with an online softmax, never
 * materialising the score matrix.  Sources:
 *   - "How Do Sparse Attention Kernels Work in GPU Clusters? A 2026 Field
 *     Guide", section "How Does Flash-MSA Sparse Attention Work?": split the
 *     sequence into blocks, a (N_blocks x N_blocks) block mask, load only the
 *     active key/value blocks, FlashAttention tiling over them, online
 *     softmax, write the output;
 *   - "Flash MSA Sparse Attention vs Full Attention: What Actually Works in
 *     Production", section "The Mechanics": the attention formula, the
 *     sliding window, causal masking and the online-softmax recurrence;
 *     section "Sparse Patterns Beyond Sliding Windows": global tokens;
 *   - "Flash MSA Sparse Attention Kernels Explained", section "The
 *     Architecture of Flash MSA Sparse Attention Kernels": inputs
 *     (batch, heads, seq_len, d_head) and a list of block indices per row.
 *
 * Conventions for every entry point:
 *   - Tensors are device pointers into the caller's memory; the library
 *     never frees or retains them.  Q, K, V and O are bf16, contiguous
 *     [B, H, N, D]; LSE is fp32 [B, H, N].  16-byte aligned.
 *   - N must be a multiple of the block size: pad variable-length sequences
 *     up to it ("The Only Guide You Need for Sparse Attention Kernels in
 *     Long-Context LLMs", FAQ "How do I handle variable-length sequences?").
 *   - The block mask is a CSR over rows r = (b * H + h) * nb + i, nb = N /
 *     block: key blocks of row r are col_idx[row_ptr[r] .. row_ptr[r+1]-1].
 *     Entries in a row must be distinct; their order is free (the result does
 *     not depend on it).  row_ptr[0] == 0.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  None blocks the host except
 *     bsa_device_error and a workspace resize (first call, or a larger
 *     problem than any before on this device).
 *   - Every entry point returns a bsa_status and never aborts the process.
 *     Invalid arguments are rejected on the host before any launch.
 *   - The library owns one lazily grown workspace per device (schedule
 *     permutation, work counter, top-k buffers, error word).  Calls that use
 *     it must not overlap on the GPU (use one stream, or synchronise);
 *     bsa_release_workspace frees it.
 */
#ifndef BSA_H
#define BSA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bsa_stream_t;

typedef enum {
    BSA_OK = 0,
    BSA_ERR_INVALID_ARG = -1,   /* null pointer, bad size, N % block != 0, misaligned, overflow */
    BSA_ERR_UNSUPPORTED = -2,   /* head dim / block size / device outside what is built */
    BSA_ERR_CAPACITY = -3,      /* col_capacity smaller than the entries to write */
    BSA_ERR_CUDA = -4,          /* a CUDA runtime call or a launch failed */
    BSA_ERR_DEVICE_CHECK = -5   /* a kernel reported an error through the device error word */
} bsa_status;

/* Problem shape.  Query and key blocks have the same size `block`. */
typedef struct {
    int32_t B, H, N, D, block;
} bsa_shape;

#define BSA_MAX_GLOBAL_BLOCKS 64

/*
 * A fixed block-mask pattern (identical for every batch and head).
 * Query block i attends to key block j when
 *     (global_rows_attend_all and i is a global block)     -- global query row
 *  or (i - window_left <= j <= i + window_right)             -- sliding window, clipped
 *  or (j is a global block)                                  -- global key block
 * and, when causal, j <= i -- except in a global query row when
 * global_rows_noncausal is also set: such a row lists every key block and
 * attends to every key token even in a causal model (global tokens "attend
 * to everything": "Flash MSA Sparse Attention vs Full Attention", section
 * "Sparse Patterns Beyond Sliding Windows", "Global Tokens").  The forward
 * learns which rows those are from bsa_pattern_row_flags.
 * Window: "Mask[i][j] = 1 if |i - j| <= W" ("Flash MSA Sparse Attention vs
 * Full Attention", section "The Mechanics"), taken at block granularity with
 * independent left/right extents.  Global tokens "attend to everything and
 * are attended by everything" (same page, "Sparse Patterns Beyond Sliding
 * Windows", "Global Tokens"); attention sinks are global block 0.
 */
typedef struct {
    int32_t n_blocks;              /* must equal N / block of the forward call */
    int32_t window_left;           /* >= 0 */
    int32_t window_right;          /* >= 0 */
    int32_t causal;                /* 0 or 1 */
    int32_t n_global;              /* 0 .. BSA_MAX_GLOBAL_BLOCKS */
    const int32_t *global_blocks;  /* HOST array of n_global block ids in [0, n_blocks) */
    int32_t global_rows_attend_all;
    int32_t global_rows_noncausal; /* 0 or 1; 1 needs global_rows_attend_all */
} bsa_pattern;

/*
 * Number of CSR entries a pattern produces for B*H rows blocks (host only,
 * closed form, no device work).  *nnz_out = B * H * (entries per head).
 */
int bsa_pattern_nnz(const bsa_pattern *p, int32_t B, int32_t H, int64_t *nnz_out);

/*
 * Pattern -> block CSR, built on the device (no host round trip).
 *   row_ptr  device int32 [B*H*n_blocks + 1]
 *   col_idx  device int32 [col_capacity]; rows are written in ascending key
 *            order, identical for every (b, h)
 *   nnz_out  optional host int64: total entries (closed form, known before launch)
 * If col_idx is NULL nothing is launched and only *nnz_out is set.
 * BSA_ERR_CAPACITY when col_capacity < nnz.  Per-row lists of active key
 * blocks: "How Does Flash-MSA Sparse Attention Work?" (field guide, step 2).
 */
int bsa_build_mask_csr(const bsa_pattern *p, int32_t B, int32_t H,
                       int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                       int64_t *nnz_out, bsa_stream_t stream);

/*
 * Per-row flags of a pattern's CSR, built on the device:
 *   row_flags  device uint8 [B*H*n_blocks]; bit 0 set for the rows of global
 *              query blocks when global_rows_attend_all and
 *              global_rows_noncausal are both set (they take no causal cut),
 *              0 elsewhere.
 * Pass them to bsa_forward_ex with the same CSR.
 */
int bsa_pattern_row_flags(const bsa_pattern *p, int32_t B, int32_t H, uint8_t *row_flags,
                          bsa_stream_t stream);

#define BSA_MAX_WINDOWS 4
#define BSA_MAX_PATTERNS 8
#define BSA_MAX_PATTERN_GLOBALS 256
#define BSA_MAX_HEADS_EX 1024

/*
 * A fixed pattern built from dilated windows, a stride and global blocks.
 * Query block i attends to key block j when
 *     (global_rows_attend_all and i is a global block)             -- global query row
 *  or for some window w: j = i + window_dilation[w] * t with
 *         -window_left[w] <= t <= window_right[w]                    -- dilated window
 *  or (stride > 0 and (i - j) is a multiple of stride)              -- strided
 *  or (j is a global block)                                          -- global key block
 * and, when causal, j <= i.
 * Dilated windows: several windows of growing dilation (every block, every
 * 2nd, every 4th, ...) whose union gives a wide receptive field; strided:
 * keys sampled at a fixed interval ("Flash MSA Sparse Attention vs Full
 * Attention", section "Sparse Patterns Beyond Sliding Windows", "Strided
 * Patterns" and "Dilated Sliding Window"), taken at block granularity, the
 * stride in phase with the query block.  A window with dilation 1 is the
 * sliding window of bsa_pattern.
 */
typedef struct {
    int32_t n_blocks;                          /* N / block of the forward call */
    int32_t causal;                            /* 0 or 1 */
    int32_t n_windows;                         /* 0 .. BSA_MAX_WINDOWS */
    int32_t window_left[BSA_MAX_WINDOWS];      /* >= 0, in steps of the window's dilation */
    int32_t window_right[BSA_MAX_WINDOWS];     /* >= 0 */
    int32_t window_dilation[BSA_MAX_WINDOWS];  /* >= 1 */
    int32_t stride;                            /* 0 = none, else >= 1 */
    int32_t n_global;                          /* 0 .. BSA_MAX_GLOBAL_BLOCKS */
    const int32_t *global_blocks;              /* HOST array of n_global block ids in [0, n_blocks) */
    int32_t global_rows_attend_all;
} bsa_pattern_ex;

/*
 * Per-head patterns -> block CSR on the device: "different heads specialize
 * in different patterns" ("The Only Guide You Need for Sparse Attention
 * Kernels in Long-Context LLMs", section "Flash-MSA"), with fixed patterns.
 *   patterns       HOST array of n_patterns (1 .. BSA_MAX_PATTERNS) patterns,
 *                  all with the same n_blocks; their global blocks together
 *                  at most BSA_MAX_PATTERN_GLOBALS
 *   head_pattern   HOST int32 [H], head h follows patterns[head_pattern[h]];
 *                  NULL: head h follows patterns[h % n_patterns].  The same
 *                  for every batch element.  H <= BSA_MAX_HEADS_EX.
 *   row_ptr        device int32 [B*H*n_blocks + 1]
 *   col_idx        device int32 [col_capacity]; rows ascending
 *   nnz_out        optional host int64: total entries
 * If col_idx is NULL nothing is launched and only *nnz_out is set.  The
 * entry count is found on the host by walking each distinct pattern's rows
 * once (time proportional to its entries per head).  Three launches: row
 * lengths, an in-place scan into row_ptr, the row fill.  BSA_ERR_CAPACITY
 * when col_capacity < nnz.
 */
int bsa_build_mask_csr_heads(const bsa_pattern_ex *patterns, int32_t n_patterns,
                             const int32_t *head_pattern, int32_t B, int32_t H,
                             int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                             int64_t *nnz_out, bsa_stream_t stream);

/*
 * Content-based block mask: per (b, h) mean-pool Q and K over each block
 * (fp32), score every (query block i, key block j) by the dot product of
 * the pooled vectors, keep the `topk` best key blocks (score descending,
 * ties to the smaller index) plus the diagonal block i when include_diag is
 * set, and write them in ascending order.
 * Sources: "the model predicts importance scores and picks top-k" (field
 * guide, "What Exactly Is a Sparse Attention Kernel?"); pooled Q/K routing
 * features ("The Only Guide You Need ...", section "Flash-MSA").
 * Arithmetic (fixed so the selection is reproducible bit for bit):
 *   pooled[d] = pairwise-tree fp32 sum over the block's tokens * (1/block);
 *   score     = a0 + a1, a_c the fp32 chain of fused multiply-adds
 *               a_c <- fma(q[d], k[d], a_c) over d == c (mod 2), increasing d.
 *   q, k      device bf16 [B, H, N, D]
 *   row_ptr   device int32 [B*H*nb + 1]  (row_ptr[B*H*nb] = total entries)
 *   col_idx   device int32 [col_capacity], col_capacity >= B*H*nb*(topk + include_diag)
 * Limits: 1 <= topk <= min(32, nb); nb <= 4096; D in {64, 128}; block a
 * power of two in [16, 256].
 */
int bsa_topk_blocks(const bsa_shape *sh, const void *q, const void *k, int32_t topk,
                    int32_t include_diag, int32_t *row_ptr, int32_t *col_idx,
                    int64_t col_capacity, bsa_stream_t stream);

/*
 * Block-sparse attention forward.
 *   q, k, v   device bf16 [B, H, N, D], 16-byte aligned
 *   row_ptr, col_idx   device block CSR (see conventions)
 *   out       device bf16 [B, H, N, D]:  O = softmax(S) V over the allowed keys
 *   lse       device fp32 [B, H, N]:     natural-log log-sum-exp of the scaled
 *             logits of each row (-inf and O = 0 for a row with no allowed key)
 *   scale     logit scale, normally 1/sqrt(D)
 *   causal    1: key token k is allowed for query token q only if k <= q (key
 *             blocks j > i contribute nothing and are skipped; inside the
 *             diagonal block the mask is token-level)
 * Supported: D in {64, 128}; block in {64, 128}.
 * Out-of-range col_idx entries are skipped and flagged in the device error
 * word (read it with bsa_device_error).
 * Online softmax and tiling: "Flash MSA Sparse Attention vs Full Attention",
 * section "The Mechanics" (the flash_sparse_attention recurrence: running
 * max, rescale, running sum, final division).
 */
int bsa_forward(const bsa_shape *sh, const void *q, const void *k, const void *v,
                const int32_t *row_ptr, const int32_t *col_idx,
                void *out, float *lse, float scale, int32_t causal, bsa_stream_t stream);

/*
 * The forward with its geometry spelled out: key blocks held apart from the
 * query blocks (a query shard against its local plus received key blocks,
 * as in a sequence-sharded forward: "How Do Sparse Attention Kernels Work in
 * GPU Clusters?", section "Distributed Sparse Attention"), and rows that
 * take no causal cut (global query rows of a causal model, see bsa_pattern).
 * bsa_forward(sh, ...) is bsa_forward_ex with n_q_blocks = n_k_blocks =
 * N / block, q_block_offset = 0 and no row flags.
 */
typedef struct {
    int32_t B, H, D, block;
    int32_t n_q_blocks;       /* query blocks per (b, h): q, out, lse hold
                                 n_q_blocks * block rows per head, the CSR has
                                 B*H*n_q_blocks rows r = (b*H + h)*n_q_blocks + i */
    int32_t n_k_blocks;       /* key blocks per (b, h): k, v hold n_k_blocks *
                                 block rows per head; col_idx entries are in
                                 [0, n_k_blocks) (others are skipped and flagged) */
    int32_t q_block_offset;   /* key-block position of query block 0: with causal,
                                 query token t of block i sees key token u of block
                                 j only if (j*block + u) <= (i + q_block_offset)*block + t,
                                 so key blocks j > i + q_block_offset are skipped */
    const void *q, *k, *v;    /* device bf16, [B, H, rows, D] as above */
    const int32_t *row_ptr, *col_idx;
    const uint8_t *row_flags; /* optional device uint8 [B*H*n_q_blocks]: bit 0 lifts
                                 the causal cut for that row; NULL = none */
    void *out;                /* device bf16 [B, H, n_q_blocks*block, D] (fp32 with out_fp32) */
    float *lse;               /* device fp32 [B, H, n_q_blocks*block] */
    float scale;
    int32_t causal;
    int32_t out_fp32;         /* 0: O in bf16; 1: O in fp32 -- partial results that are
                                 merged later (bsa_merge_partial_blocks) keep their precision */
} bsa_forward_args;

int bsa_forward_ex(const bsa_forward_args *a, bsa_stream_t stream);

/*
 * FP8 scores: the same forward with Q and K given as OCP e4m3 (FN variant:
 * no infinities, largest finite value 448), one descale factor each, so the
 * logits are (q8 . k8) * q_descale * k_descale * scale; S = Q K^T runs on
 * the e4m3 tensor-core path (fp32 accumulation), softmax, P and V as in
 * bsa_forward.  Scores "in FP8" on Hopper/Blackwell tensor cores: "Flash MSA
 * Sparse Attention Kernels Explained", section "The Future of Attention
 * Kernels".
 *   q8, k8    device e4m3 bytes [B, H, N, D], 16-byte aligned (bsa_quantize_e4m3)
 *   v         device bf16 [B, H, N, D]
 *   q_descale, k_descale   > 0, finite (x = code value * descale)
 *   others    as bsa_forward
 * Supported: D = 128; block 128, or 64 (paired form).  Other shapes return
 * BSA_ERR_UNSUPPORTED before any launch.
 */
int bsa_forward_fp8(const bsa_shape *sh, const void *q8, const void *k8, const void *v,
                    const int32_t *row_ptr, const int32_t *col_idx, void *out, float *lse,
                    float q_descale, float k_descale, float scale, int32_t causal,
                    bsa_stream_t stream);

/*
 * FP8 scores with one scale per block: the same forward as bsa_forward_fp8,
 * but each (head, query block) and each (head, key block) has its own
 * descale factor, so the logits of a pair are
 * (q8 . k8) * q_descale[bh*nb + i] * k_descale[bh*nb + j] * scale.  One factor
 * per block instead of per tensor keeps a block of large values from
 * crushing the resolution of every other block (scores "in FP8": "Flash MSA
 * Sparse Attention Kernels Explained", "The Future of Attention Kernels").
 *   q8, k8      device e4m3 [B, H, N, D] (bsa_quantize_e4m3_blocks)
 *   q_descale, k_descale   device fp32 [B*H*nb], positive and finite
 *   others      as bsa_forward_fp8
 * Supported: D = 128; block 128, or 64 (paired form).
 */
int bsa_forward_fp8_blocks(const bsa_shape *sh, const void *q8, const void *k8, const void *v,
                           const float *q_descale, const float *k_descale, const int32_t *row_ptr,
                           const int32_t *col_idx, void *out, float *lse, float scale, int32_t causal,
                           bsa_stream_t stream);

/*
 * Per-block e4m3 quantisation for bsa_forward_fp8_blocks: for each (head,
 * block of sh->block tokens), amax = max |x| over its block x D values,
 * inv = fp32(448 / amax), y = e4m3(fp32(x * inv)) (nearest, ties to even,
 * saturating), descale = fp32(amax / 448); an all-zero block gets inv = 1 and
 * descale = 1.
 *   x        device bf16 [B, H, N, D];  y  device bytes, same shape
 *   descale  device fp32 [B*H*(N/block)]
 * Supported: block in {64, 128}, D in {64, 128}.
 */
int bsa_quantize_e4m3_blocks(const bsa_shape *sh, const void *x, void *y, float *descale, bsa_stream_t stream);

/*
 * e4m3 quantisation for bsa_forward_fp8: y[i] = e4m3(x[i] * inv_scale), the
 * product rounded once in fp32, then to the nearest e4m3 value (ties to
 * even), saturated to +-448; the sign of a zero result is kept.
 *   x   device bf16 [n];  y  device bytes [n]; both 16-byte aligned
 *   n   > 0 and a multiple of 16;  inv_scale > 0, finite
 * The caller keeps 1 / inv_scale as the descale factor.
 */
int bsa_quantize_e4m3(const void *x, void *y, int64_t n, float inv_scale, bsa_stream_t stream);

/*
 * Block-sparse attention backward: dQ, dK, dV of L = sum(dO * O) for the
 * attention bsa_forward computed with the same CSR, scale and causal flag.
 * Training differentiates through the sparse mask, which the backward reuses
 * ("How Do Sparse Attention Kernels Work in GPU Clusters?", FAQ on training
 * versus inference).  With P the forward's softmax weights, rebuilt from LSE:
 *   dP = dO V^T, dS = P o (dP - rowsum(dO o O)), dQ = scale dS K,
 *   dK = scale dS^T Q, dV = P^T dO.
 *   q, k, v, out, dout  device bf16 [B, H, N, D]; out and lse are bsa_forward's
 *   lse                 device fp32 [B, H, N]
 *   row_ptr, col_idx    the forward's block CSR; col_capacity >= its number of
 *                       entries (the col_idx allocation size will do): the
 *                       library transposes it into a workspace of that size
 *   dq, dk, dv          device bf16 [B, H, N, D], written (rows no query
 *                       attends get dK = dV = 0; rows with no key, dQ = 0)
 * Supported: block in {64, 128}, D in {64, 128}; other shapes
 * BSA_ERR_UNSUPPORTED.  Block 64 runs in a paired form: two 64-token key
 * blocks with overlapping transposed lists share a 128-row tile, and each
 * step takes two query blocks from the union of their lists.
 * Workspace: the transposed CSR (about 3 * B*H*nb + col_capacity int32, with
 * the work items' processing order), a float per query row, an fp32 dQ
 * accumulator (B*H*N*D floats) and, for block 64, the pairing buffers
 * (about 68 int32 per key block).
 * dQ is accumulated by fp32 additions (bulk tensor reductions) and the
 * transposed lists are filled in an order that depends on scheduling, so the
 * last bits of dQ, dK and dV may differ between runs.
 * Q, K, V and dO must be finite.
 */
int bsa_backward(const bsa_shape *sh, const void *q, const void *k, const void *v,
                 const void *out, const void *dout, const float *lse,
                 const int32_t *row_ptr, const int32_t *col_idx, int64_t col_capacity,
                 void *dq, void *dk, void *dv, float scale, int32_t causal, bsa_stream_t stream);

/*
 * bsa_backward with per-row causal flags, for the CSR of a causal model whose
 * global query rows attend every block (bsa_pattern.global_rows_noncausal;
 * "The Only Guide You Need for Sparse Attention Kernels", section "Sparse
 * Patterns Beyond Sliding Windows", Global Tokens): row_flags (device uint8,
 * one per CSR row, as bsa_pattern_row_flags writes and bsa_forward_ex reads)
 * with bit 0 set lifts the causal cut for that row, so its later key blocks
 * and every key of its diagonal block take part, exactly as in the forward
 * that produced out and lse.  row_flags == NULL, or causal == 0, is
 * bsa_backward.  Other arguments, errors and workspace as bsa_backward.
 */
int bsa_backward_ex(const bsa_shape *sh, const void *q, const void *k, const void *v,
                    const void *out, const void *dout, const float *lse,
                    const int32_t *row_ptr, const int32_t *col_idx, int64_t col_capacity,
                    const uint8_t *row_flags, void *dq, void *dk, void *dv, float scale,
                    int32_t causal, bsa_stream_t stream);

/*
 * Debug check of a block CSR on the device.  ORs into *d_err (device int32):
 *   1 = row_ptr[0] != 0 or row_ptr decreasing,  2 = col_idx entry outside
 *   [0, nb),  4 = duplicate entry in a row.  Does not clear *d_err.
 */
int bsa_validate_csr(const bsa_shape *sh, const int32_t *row_ptr, const int32_t *col_idx,
                     int32_t *d_err, bsa_stream_t stream);

/*
 * Read and clear the current device's error words (the workspace's, and the
 * fixed array's of bsa_forward_noalloc; their bits are ORed).  Synchronises
 * the device.  Allocates nothing: on a device where no workspace-using call
 * ran there is no workspace word to read.
 * *code_out: 0 = none; bit 1 = a kernel wait timed out (the kernel returned
 * early and its outputs are invalid); bit 2 = out-of-range col_idx entry
 * skipped; bit 4 = malformed row_ptr row treated as empty; bit 8 = a kernel
 * found its launch unusable (misaligned shared memory) and did nothing.  bit 16 =
 * the CSR held more entries than the col_capacity given to bsa_backward (the
 * extra ones were dropped).
 * Returns BSA_ERR_DEVICE_CHECK when the word was non-zero.
 */
int bsa_device_error(int32_t *code_out);

/*
 * Hang detection.  Every wait inside the pipelined kernels (bsa_forward,
 * bsa_forward_fp8, bsa_forward_noalloc, bsa_backward) is bounded: a wait
 * that lasts longer than this limit makes the launch drain its in-flight
 * copies and MMAs, free its tensor memory, return early and set bit 1 in the
 * device error word, so a hung pipeline surfaces as an error instead of a
 * stuck GPU.  (No page states this; it is a property of this library.)
 *   ns  new limit in nanoseconds for launches enqueued after this call,
 *       1000 .. 600e9; 0 restores the default of 2 s.
 * Process-wide; BSA_ERR_INVALID_ARG outside the range.
 */
int bsa_set_wait_limit(int64_t ns);
int64_t bsa_get_wait_limit(void);

/*
 * Test hook for the hang detection.  The next call of the forward family
 * (bsa_forward, bsa_forward_fp8 or bsa_forward_noalloc) runs with each
 * persistent CTA's work distributor handing out at most n_items work items
 * and then stopping without publishing the end of the work, so every other
 * role of the CTA waits until the wait limit runs out.  That call then
 * returns BSA_OK, its outputs are incomplete, and bsa_device_error reports
 * bit 1.  One-shot: later calls run normally.  n_items = -1 cancels a
 * pending stall.  Nothing faults: the waits are bounded, the kernels leave
 * through their normal exit.
 */
int bsa_debug_stall_next_forward(int32_t n_items);

/*
 * bsa_forward without any device allocation by the library.  (The pages
 * have no counterpart: this is a deployment variant of bsa_forward.)
 *
 * For callers that cannot let a library call cudaMalloc: serving loops that
 * must never hit the device-wide synchronisation cudaMalloc / cudaFree
 * imply, and applications that hand out every byte of device memory from
 * their own pre-reserved pools.  Arguments, layouts and results are those of
 * bsa_forward; the caller still owns Q, K, V, the CSR, O and LSE.
 * The schedule scratch (work counter, error word, one int32 per CSR row)
 * comes from a fixed array compiled into libbsa.so instead of the
 * workspace; every GPU that loads the library keeps that array (about
 * 1 MiB) until the process exits.
 *   - B*H*(N/block) must be <= BSA_NOALLOC_MAX_ROWS, else BSA_ERR_CAPACITY.
 *   - The first call on a device looks up the array's device address and the
 *     device's properties (no allocation); make that first call before any
 *     stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (on
 *     different streams, or from different threads) race and corrupt each
 *     other's schedule.  Order them on one stream.
 *   - Device-side error bits (timeouts, skipped out-of-range col_idx
 *     entries, malformed rows) land in a word of the fixed array and
 *     accumulate until bsa_device_error reads and clears them, as for
 *     bsa_forward's word; reading them allocates nothing.
 *   - The array's device address is looked up once per device and kept:
 *     calls after a device reset (cudaDeviceReset, which unloads the array)
 *     are not supported.
 */
#define BSA_NOALLOC_MAX_ROWS 262144
int bsa_forward_noalloc(const bsa_shape *sh, const void *q, const void *k, const void *v,
                        const int32_t *row_ptr, const int32_t *col_idx,
                        void *out, float *lse, float scale, int32_t causal, bsa_stream_t stream);

/*
 * Sequence-sharded forward ("How Do Sparse Attention Kernels Work in GPU
 * Clusters?", section "Distributed Sparse Attention": a sparse all-to-all of
 * the needed key/value blocks, indices first and blocks second; or local
 * attention with a global merge of partial outputs).  Shards are contiguous:
 * rank g of `world` owns query and key blocks [g*n_blocks/world,
 * (g+1)*n_blocks/world) of every (batch, head).  A rank's CSR holds its own
 * query blocks only: rows r = bh * count + i_local (count = its blocks),
 * entries are GLOBAL key-block ids.  The planners are host functions over
 * host copies of that CSR; the collectives themselves belong to the caller
 * (the Python layer uses torch.distributed all_to_all), the data movement to
 * bsa_copy_blocks and bsa_merge_partial_blocks.
 */
typedef struct {
    int32_t world, rank;   /* 1 <= world <= n_blocks, 0 <= rank < world */
    int32_t n_blocks;      /* blocks of the whole sequence */
    int32_t BH;            /* B * H */
} bsa_shard_geometry;

/* This rank's blocks: [*first, *first + *count).  Host only. */
int bsa_shard_range(const bsa_shard_geometry *g, int32_t *first, int32_t *count);

/*
 * Key/value exchange plan (host).  The extended key range of every head is:
 * n_before slots for remote blocks before the shard (a head's own remote
 * blocks end at slot n_before, ascending), the count own blocks, then
 * n_after slots for remote blocks after the shard (ascending); n_before and
 * n_after are maxima over the heads, and slots a head does not use are
 * never referenced.  The forward then runs as bsa_forward_ex with
 * n_q_blocks = count, n_k_blocks = n_before + count + n_after and
 * q_block_offset = n_before: every causal comparison keeps its meaning
 * because the extended order is the global order.
 *   row_ptr, col_idx  HOST, the rank's CSR (see above); row_ptr[0] == 0, monotone
 *   col_idx_ext       HOST out [nnz]: entries renumbered to extended key
 *                     blocks (-1 for entries outside [0, n_blocks): the
 *                     forward skips and flags them).  NULL: only the sizes
 *                     below are computed.
 *   need_bh, need_j, need_pos   HOST out [need_cap]: remote blocks to fetch
 *                     (head, global key block, extended slot), grouped by
 *                     owner rank (ascending), then head, then block
 *   need_count_by_rank          HOST out [world]: entries per owner (own rank 0)
 *   n_before_out, n_after_out   HOST out
 * BSA_ERR_CAPACITY when the fetch list exceeds need_cap (the local nnz is
 * always enough).
 */
int bsa_shard_plan_kv(const bsa_shard_geometry *g, const int32_t *row_ptr, const int32_t *col_idx,
                      int32_t *col_idx_ext, int32_t *need_bh, int32_t *need_j, int32_t *need_pos,
                      int64_t need_cap, int32_t *need_count_by_rank, int32_t *n_before_out,
                      int32_t *n_after_out);

/*
 * Partial-output plan (host).  The local part is the rank's rows restricted
 * to its own key blocks, renumbered to the shard (local_row_ptr [BH*count+1],
 * local_col_idx [<= nnz]); it runs as bsa_forward_ex with n_q_blocks =
 * n_k_blocks = count and the caller's causal flag and row flags.  The guest
 * part lists, for every other rank p (ascending), each local row that uses
 * key blocks of p: guest_q = its local CSR row, its entries in p's
 * numbering in guest_col[guest_ptr[x] .. guest_ptr[x+1]) (sorted, distinct).
 * With causal set, a row that is not flagged sends only blocks wholly before
 * its own block (blocks after it add nothing; its own block is local), so
 * the owner computes every guest row without a causal cut.
 *   cap  capacity of local_col_idx, guest_q, guest_ptr - 1 and guest_col (>= nnz)
 *   guest_rows_by_rank, guest_entries_by_rank  HOST out [world]
 */
int bsa_shard_plan_partial(const bsa_shard_geometry *g, const int32_t *row_ptr, const int32_t *col_idx,
                           const uint8_t *row_flags, int32_t causal, int32_t *local_row_ptr,
                           int32_t *local_col_idx, int32_t *guest_q, int32_t *guest_ptr, int32_t *guest_col,
                           int64_t cap, int32_t *guest_rows_by_rank, int32_t *guest_entries_by_rank);

/*
 * Block copy on the device: block n of rows_per_block rows of row_bytes
 * bytes each goes from src rows src_row[n] .. to dst rows dst_row[n] ..
 * (src_row, dst_row: device int64 [n_blocks]).  Gathers blocks into a send
 * buffer, places received ones, and copies a shard into the extended range.
 * row_bytes % 16 == 0; src, dst 16-byte aligned; blocks must not overlap.
 */
int bsa_copy_blocks(const void *src, void *dst, const int64_t *src_row, const int64_t *dst_row,
                    int64_t n_blocks, int32_t rows_per_block, int32_t row_bytes, bsa_stream_t stream);

/*
 * Merge partial attention results into an accumulated one, row by row:
 * LSE = log(exp(LSE_acc) + exp(LSE_part)), O = exp(LSE_acc - LSE) O_acc +
 * exp(LSE_part - LSE) O_part -- the online-softmax rescale ("Flash MSA
 * Sparse Attention vs Full Attention", "The Mechanics") applied to whole
 * partial results, i.e. the global merge of partial outputs.  A part row with
 * LSE = -inf changes nothing.  O stays fp32 until the last merge (a bf16
 * partial would add its rounding to the result's).
 *   o_acc, lse_acc    device fp32 [rows, D] / fp32 [rows], updated in place
 *   o_part, lse_part  device fp32 [n_blocks*rows_per_block, D] / fp32, compact
 *   dst_row           device int64 [n_blocks]: first accumulator row of part block n
 * Parts merged by one call must cover distinct rows.
 */
int bsa_merge_partial_blocks(float *o_acc, float *lse_acc, const float *o_part, const float *lse_part,
                             const int64_t *dst_row, int64_t n_blocks, int32_t rows_per_block, int32_t D,
                             bsa_stream_t stream);

/* y = bf16(x), round to nearest even; n % 8 == 0, x and y 16-byte aligned. */
int bsa_convert_f32_bf16(const float *x, void *y, int64_t n, bsa_stream_t stream);

/* Human-readable text of a bsa_status (static storage). */
const char *bsa_status_string(int status);

/* Free the workspace of every device (synchronises them first). */
void bsa_release_workspace(void);

/* ABI version: 100 * major + minor. */
int bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H */
