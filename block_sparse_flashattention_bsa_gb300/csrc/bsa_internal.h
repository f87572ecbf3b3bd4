// bsa_internal.h -- declarations shared by the host layer and the kernel
// translation units of libbsa.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bsa {

struct FwdParams {
    const int32_t* row_ptr;
    const int32_t* col_idx;
    // Paired block-64 forward: work items from the pairing pass.  Item w is
    // CSR row item_a[w] = (b*H + h)*nb + i plus, when item_b[w] >= 0, query
    // block item_b[w] of the same head (a pair), whose key blocks are the
    // item_cnt[w] entries of slots[w * kPairSlot ...]: j | in_a << 30 | in_b << 31,
    // ascending.  A single (item_b < 0) reads its row from the CSR.
    const int32_t* item_a;
    const int32_t* item_b;
    const int32_t* item_cnt;
    const uint32_t* slots;
    const int32_t* n_items_dev;  // item count (device), used instead of n_items when set
    const int32_t* perm;   // work items, longest row first
    int32_t* counter;      // next position in perm to claim (zeroed by the schedule kernel)
    void* out;             // bf16 [BH, N, D]
    float* out_f32;        // when set: O goes here as fp32 [BH, N, D] instead (partial results)
    float* lse;            // fp32 [BH, N]
    int32_t* err;          // device error word
    int32_t BH, N, nb, n_items, causal;  // N, nb: query rows / blocks per head (Q, O, LSE, CSR rows)
    int32_t Nk, nbk;       // key rows / blocks per head (K, V); col_idx entries are in [0, nbk)
    int32_t q_off;         // key-block position of query block 0 (causal cut: j <= i + q_off)
    const uint8_t* row_flags;  // optional, per CSR row: bit 0 lifts the causal cut for that row
    // FP8 scores with per-block scales (else null): descale of every query
    // block [BH * nb] and key block [BH * nbk]; the logit scale of a pair is
    // scale_log2 * q_descale * k_descale.
    const float* q_descale;
    const float* k_descale;
    float scale_log2;      // scale * log2(e)
    unsigned long long wait_limit_ns;  // a pipeline wait longer than this aborts the launch (ERR_TIMEOUT)
    int32_t stall_after;   // test hook: the work distributor stops after this many items (-1: off)
};

// Process-wide limit of the kernels' pipeline waits (bsa_set_wait_limit) and
// the one-shot stall of the next forward (bsa_debug_stall_next_forward).
unsigned long long wait_limit_ns();
int32_t take_forward_stall();
// Read and clear the allocation-free forward's device error word on device
// `dev` (0 when that entry point never ran there).  Allocates nothing.
cudaError_t noalloc_take_error(int dev, int32_t* code);

// Forward kernel shared-memory bytes for a (block, head_dim) instance, or 0
// when the pair is not built.  paired: the paired form of 64-token blocks.
int fwd_smem_bytes(int block, int D, bool paired);

// Persistent forward kernel.  grid = number of CTAs (<= SM count).
// tq, tk, tv: loads of Q, K, V tiles; to: stores of O tiles (box 64 x block).
cudaError_t launch_forward(int block, int D, bool paired, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int grid,
                           cudaStream_t stream);
// FP8 scores: Q and K e4m3 (D = 128; block 128, or 64 in the paired form).
cudaError_t launch_forward_f8(int block, int D, bool paired, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int grid,
                              cudaStream_t stream);
// Per (head, block of `block` tokens): amax, inv = 448 / amax, codes
// e4m3(x * inv), descale = amax / 448 (1 and inv 1 for an all-zero block).
cudaError_t launch_quantize_e4m3_blocks(const void* x, void* y, float* descale, int64_t n_blocks, int32_t block,
                                        int32_t D, cudaStream_t stream);
// y = e4m3(x * inv_scale), round to nearest even, saturating; n % 16 == 0.
cudaError_t launch_quantize_e4m3(const void* x, void* y, int64_t n, float inv_scale, int sm_count,
                                 cudaStream_t stream);

// Longest-first, stable schedule of the R = BH * nb rows; zeroes *counter.
cudaError_t launch_schedule(const int32_t* row_ptr, int32_t R, int32_t* perm, int32_t* counter,
                            cudaStream_t stream);
// The same over items with given lengths: lens[0 .. *n_dev), *n_dev <= R_max,
// sorted in classes of 2^lens_shift steps (stable: each class keeps the
// items' order, which the pairing pass groups by head).
cudaError_t launch_schedule_lens(const int32_t* lens, const int32_t* n_dev, int32_t R_max, int32_t* perm,
                                 int32_t* counter, int lens_shift, cudaStream_t stream);

// Pairing of 64-token query blocks (csrc/bsa_pair.cu).
constexpr int kPairRowMax = 32;  // rows with more raw entries stay single
constexpr int kPairSlot = 64;    // union entries of a pair (2 x kPairRowMax)
struct PairingBuffers {
    int32_t* item_a;
    int32_t* item_b;
    int32_t* item_cnt;
    int32_t* item_len;  // steps (two key blocks each): the schedule's length
    int32_t* n_items;
    uint32_t* slots;
};
size_t pairing_workspace_bytes(int32_t BH, int32_t nb);
PairingBuffers pairing_buffers(void* ws, int32_t BH, int32_t nb);
// Geometry of the CSR rows the pairing pass reads: nb query blocks per head
// (rows), nbk key blocks, causal cut j <= i + q_off unless the row's flag bit 0
// lifts it (flagged rows are never paired).
struct PairGeom {
    int32_t nb, nbk, q_off, causal;
    const uint8_t* row_flags;
    int64_t col_cap;  // entries col_idx holds: rows are read only below it
};
cudaError_t launch_pairing(const int32_t* row_ptr, const int32_t* col_idx, int32_t BH, const PairGeom& g,
                           const PairingBuffers& b, int32_t* err, int sm_count, cudaStream_t stream);

// Pattern mask builder.
struct PatternDev {
    int32_t nb, wl, wr, causal, n_global, gra;
    int32_t grnc;         // global query rows take no causal cut (and list every block)
    int32_t globals[64];  // sorted, distinct
};
cudaError_t launch_mask(const PatternDev& p, int32_t BH, int64_t nnz_head, int32_t* row_ptr, int32_t* col_idx,
                        cudaStream_t stream);
// flags[r] = 1 for the rows of non-causal global query rows, else 0.
cudaError_t launch_row_flags(const PatternDev& p, int32_t BH, uint8_t* flags, cudaStream_t stream);
// Host mirror of the mask builder's row length (closed form).
int32_t pattern_row_len(const PatternDev& p, int32_t i);

// Per-head patterns of dilated windows, a stride and global blocks.
constexpr int kMaxWindows = 4;
constexpr int kMaxPatterns = 8;
constexpr int kMaxPatternGlobals = 256;
constexpr int kMaxHeadsEx = 1024;
struct PatternExDev {
    int32_t causal, gra, n_win, stride;  // stride 0 = none
    int32_t g_off, g_cnt;                // this pattern's globals: PatternSetDev::globals[g_off .. g_off + g_cnt)
    int32_t wl[kMaxWindows], wr[kMaxWindows], wd[kMaxWindows];
};
struct PatternSetDev {
    int32_t nb, H, n_pat;
    PatternExDev pat[kMaxPatterns];
    int32_t globals[kMaxPatternGlobals];  // per pattern: sorted, distinct
    uint8_t head_pat[kMaxHeadsEx];        // pattern of head h
};
// Entries of row i of pattern p (host mirror of the device walk).
int32_t pattern_ex_row_len(const PatternSetDev& s, const PatternExDev& p, int32_t i);
// Row lengths into row_ptr[1..R], in-place scan, row fill.
cudaError_t launch_mask_ex(const PatternSetDev& s, int32_t B, int32_t* row_ptr, int32_t* col_idx,
                           cudaStream_t stream);

// row_ptr[0] = 0, row_ptr[r + 1] = lens[0] + ... + lens[r] (one CTA).  lens
// may alias row_ptr + 1.
cudaError_t launch_row_ptr_scan(const int32_t* lens, int64_t R, int32_t* row_ptr, cudaStream_t stream);

// Backward (csrc/bsa_bwd.cu): transposed CSR, Dv, the key-stationary kernel, dQ.
struct BwdLaunch {
    CUtensorMap tq, tk, tv, tdo;  // 64-column x 128-row boxes
    CUtensorMap tdq;               // fp32 dQ buffer in the workspace, 32 x 32 boxes (bulk reductions)
    CUtensorMap tdk, tdv;          // bf16 outputs, 64-column x block-row boxes (stores)
    const int32_t* row_ptr;
    const int32_t* col_idx;
    int64_t col_capacity;
    const uint8_t* row_flags;  // per CSR row, bit 0 lifts the causal cut; may be null
    const void* out;    // bf16 [BH, N, D]
    const void* dout;   // bf16 [BH, N, D]
    const float* lse;   // [BH, N]
    void* dq;           // bf16 outputs [BH, N, D]
    void* dk;
    void* dv;
    void* workspace;    // bwd_workspace_bytes
    int32_t* err;
    int32_t BH, N, D, block, nb, causal, sm_count;
    float scale;
};
size_t bwd_workspace_bytes(int32_t BH, int32_t N, int32_t D, int32_t block, int32_t nb, int64_t col_capacity);
size_t bwd_dq_acc_offset(int32_t BH, int32_t N, int32_t nb, int64_t col_capacity);
cudaError_t launch_backward(const BwdLaunch& L, cudaStream_t stream);

// Content top-k: workspace bytes it needs and the launch sequence.
size_t topk_workspace_bytes(int32_t BH, int32_t nb, int32_t D, int32_t topk);
cudaError_t launch_topk(int32_t BH, int32_t N, int32_t D, int32_t block, const void* q, const void* k,
                        int32_t topk, int32_t include_diag, int32_t* row_ptr, int32_t* col_idx, void* workspace,
                        cudaStream_t stream);

cudaError_t launch_validate(int32_t R, int32_t nb, const int32_t* row_ptr, const int32_t* col_idx, int32_t* d_err,
                            cudaStream_t stream);

}  // namespace bsa
