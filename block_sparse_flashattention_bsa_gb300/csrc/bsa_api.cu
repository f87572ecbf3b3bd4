// bsa_api.cu -- host side of libbsa.so: argument checks, per-device state
// and workspace, TMA descriptors, launches.  Declarations and contracts are
// in include/bsa.h.

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

using bsa::FwdParams;
using bsa::PatternDev;

constexpr int kMaxDevices = 64;

struct DevState {
    bool init = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int32_t* err = nullptr;  // device error word
    void* ws = nullptr;      // workspace
    size_t ws_bytes = 0;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];

// Limit of the kernels' pipeline waits, and the one-shot test stall of the
// next forward (-1: none).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int32_t> g_stall_next{-1};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int cuda_fail(cudaError_t) { return BSA_ERR_CUDA; }

// Current device's state (initialised on first use).  Caller holds g_mu.
int dev_state(DevState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
    DevState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (cudaMalloc(&d.err, 256) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaMemset(d.err, 0, 256) != cudaSuccess) return BSA_ERR_CUDA;
        d.init = true;
    }
    *out = &d;
    return BSA_OK;
}

// The kernels are built for sm_103a only.
int check_arch(const DevState* d) { return (d->cc_major == 10 && d->cc_minor == 3) ? BSA_OK : BSA_ERR_UNSUPPORTED; }

int ensure_workspace(DevState* d, size_t bytes) {
    if (d->ws_bytes >= bytes) return BSA_OK;
    // Growing: wait for every user of the old buffer first.
    if (d->ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return BSA_ERR_CUDA;
        cudaFree(d->ws);
        d->ws = nullptr;
        d->ws_bytes = 0;
    }
    const size_t want = align256(std::max(bytes, (size_t)1 << 20));
    if (cudaMalloc(&d->ws, want) != cudaSuccess) return BSA_ERR_CUDA;
    d->ws_bytes = want;
    return BSA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view [rows, D] of a bf16 [B, H, N, D] tensor; box = 64 columns (one
// 128-byte swizzled row) x box_rows rows.
int make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t D, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return BSA_ERR_CUDA;
    cuuint64_t dims[2] = {D, rows};
    cuuint64_t strides[1] = {D * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSA_OK : BSA_ERR_CUDA;
}

// 2-D view [rows, D] of an e4m3 tensor (one byte per element, D = 128: one
// 128-byte swizzled box per row); box = D x box_rows.
int make_map_e4m3(CUtensorMap* m, const void* base, uint64_t rows, uint64_t D, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return BSA_ERR_CUDA;
    cuuint64_t dims[2] = {D, rows};
    cuuint64_t strides[1] = {D};
    cuuint32_t box[2] = {(cuuint32_t)D, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSA_OK : BSA_ERR_CUDA;
}

// 2-D view [rows, D] of an fp32 buffer; box = 32 columns (one 128-byte
// swizzled row) x 32 rows: the backward's dQ reductions.
int make_map_f32_32x32(CUtensorMap* m, void* base, uint64_t rows, uint64_t D) {
    auto fn = encode_fn();
    if (!fn) return BSA_ERR_CUDA;
    cuuint64_t dims[2] = {D, rows};
    cuuint64_t strides[1] = {D * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSA_OK : BSA_ERR_CUDA;
}

int check_shape(const bsa_shape* sh) {
    if (!sh) return BSA_ERR_INVALID_ARG;
    if (sh->B <= 0 || sh->H <= 0 || sh->N <= 0 || sh->D <= 0 || sh->block <= 0) return BSA_ERR_INVALID_ARG;
    if (sh->N % sh->block != 0) return BSA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)sh->B * sh->H * sh->N;
    if (rows > INT32_MAX) return BSA_ERR_INVALID_ARG;
    return BSA_OK;
}

int to_pattern(const bsa_pattern* p, PatternDev* out) {
    if (!p) return BSA_ERR_INVALID_ARG;
    if (p->n_blocks <= 0 || p->window_left < 0 || p->window_right < 0) return BSA_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return BSA_ERR_INVALID_ARG;
    if (p->n_global < 0 || p->n_global > BSA_MAX_GLOBAL_BLOCKS) return BSA_ERR_INVALID_ARG;
    if (p->n_global > 0 && !p->global_blocks) return BSA_ERR_INVALID_ARG;
    if (p->global_rows_noncausal != 0 && p->global_rows_noncausal != 1) return BSA_ERR_INVALID_ARG;
    if (p->global_rows_noncausal && !p->global_rows_attend_all) return BSA_ERR_INVALID_ARG;
    std::vector<int32_t> g(p->global_blocks, p->global_blocks + p->n_global);
    for (int32_t x : g)
        if (x < 0 || x >= p->n_blocks) return BSA_ERR_INVALID_ARG;
    std::sort(g.begin(), g.end());
    g.erase(std::unique(g.begin(), g.end()), g.end());
    std::memset(out, 0, sizeof(*out));
    out->nb = p->n_blocks;
    // clip the window to the sequence (keeps i +- w inside int32)
    out->wl = std::min(p->window_left, p->n_blocks);
    out->wr = std::min(p->window_right, p->n_blocks);
    out->causal = p->causal;
    out->gra = p->global_rows_attend_all ? 1 : 0;
    out->grnc = p->global_rows_noncausal ? 1 : 0;
    out->n_global = (int32_t)g.size();
    for (size_t x = 0; x < g.size(); ++x) out->globals[x] = g[x];
    return BSA_OK;
}

int64_t pattern_nnz_head(const PatternDev& p) {
    int64_t n = 0;
    for (int32_t i = 0; i < p.nb; ++i) n += bsa::pattern_row_len(p, i);
    return n;
}

// Validates n_patterns patterns and the head map, fills the device pattern
// set.  Windows, dilations and the stride are clipped to the sequence: a
// dilation or stride >= n_blocks reaches no block but i, so clipping keeps
// every progression inside int32 without changing the pattern.
int to_pattern_set(const bsa_pattern_ex* pats, int32_t n_patterns, const int32_t* head_pattern, int32_t H,
                   bsa::PatternSetDev* out) {
    if (!pats || n_patterns < 1 || n_patterns > BSA_MAX_PATTERNS) return BSA_ERR_INVALID_ARG;
    if (H <= 0 || H > BSA_MAX_HEADS_EX) return BSA_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    const int32_t nb = pats[0].n_blocks;
    if (nb <= 0) return BSA_ERR_INVALID_ARG;
    out->nb = nb;
    out->H = H;
    out->n_pat = n_patterns;
    int32_t g_used = 0;
    for (int32_t q = 0; q < n_patterns; ++q) {
        const bsa_pattern_ex& p = pats[q];
        bsa::PatternExDev& d = out->pat[q];
        if (p.n_blocks != nb) return BSA_ERR_INVALID_ARG;
        if (p.causal != 0 && p.causal != 1) return BSA_ERR_INVALID_ARG;
        if (p.n_windows < 0 || p.n_windows > BSA_MAX_WINDOWS) return BSA_ERR_INVALID_ARG;
        if (p.stride < 0) return BSA_ERR_INVALID_ARG;
        if (p.n_global < 0 || p.n_global > BSA_MAX_GLOBAL_BLOCKS) return BSA_ERR_INVALID_ARG;
        if (p.n_global > 0 && !p.global_blocks) return BSA_ERR_INVALID_ARG;
        d.causal = p.causal;
        d.gra = p.global_rows_attend_all ? 1 : 0;
        d.n_win = p.n_windows;
        for (int w = 0; w < p.n_windows; ++w) {
            if (p.window_left[w] < 0 || p.window_right[w] < 0 || p.window_dilation[w] < 1)
                return BSA_ERR_INVALID_ARG;
            d.wl[w] = std::min(p.window_left[w], nb);
            d.wr[w] = std::min(p.window_right[w], nb);
            d.wd[w] = std::min(p.window_dilation[w], nb);
        }
        d.stride = std::min(p.stride, nb);
        std::vector<int32_t> g(p.global_blocks, p.global_blocks + p.n_global);
        for (int32_t x : g)
            if (x < 0 || x >= nb) return BSA_ERR_INVALID_ARG;
        std::sort(g.begin(), g.end());
        g.erase(std::unique(g.begin(), g.end()), g.end());
        if (g_used + (int32_t)g.size() > BSA_MAX_PATTERN_GLOBALS) return BSA_ERR_INVALID_ARG;
        d.g_off = g_used;
        d.g_cnt = (int32_t)g.size();
        for (int32_t x : g) out->globals[g_used++] = x;
    }
    for (int32_t h = 0; h < H; ++h) {
        const int32_t q = head_pattern ? head_pattern[h] : h % n_patterns;
        if (q < 0 || q >= n_patterns) return BSA_ERR_INVALID_ARG;
        out->head_pat[h] = (uint8_t)q;
    }
    return BSA_OK;
}

}  // namespace

namespace bsa {
unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int32_t take_forward_stall() { return g_stall_next.exchange(-1); }
}  // namespace bsa

extern "C" {

int bsa_version(void) { return 102; }

int bsa_set_wait_limit(int64_t ns) {
    if (ns == 0) ns = (int64_t)kDefaultWaitLimitNs;
    if (ns < 1000 || ns > 600ll * 1000000000ll) return BSA_ERR_INVALID_ARG;
    g_wait_limit_ns.store((unsigned long long)ns);
    return BSA_OK;
}

int64_t bsa_get_wait_limit(void) { return (int64_t)g_wait_limit_ns.load(); }

int bsa_debug_stall_next_forward(int32_t n_items) {
    if (n_items < -1) return BSA_ERR_INVALID_ARG;
    g_stall_next.store(n_items);
    return BSA_OK;
}

const char* bsa_status_string(int status) {
    switch (status) {
        case BSA_OK: return "ok";
        case BSA_ERR_INVALID_ARG: return "invalid argument";
        case BSA_ERR_UNSUPPORTED: return "unsupported shape, option or device";
        case BSA_ERR_CAPACITY: return "output capacity too small";
        case BSA_ERR_CUDA: return "CUDA error";
        case BSA_ERR_DEVICE_CHECK: return "device-side check failed";
        default: return "unknown status";
    }
}

int bsa_pattern_nnz(const bsa_pattern* p, int32_t B, int32_t H, int64_t* nnz_out) {
    if (B <= 0 || H <= 0 || !nnz_out) return BSA_ERR_INVALID_ARG;
    PatternDev pd;
    int st = to_pattern(p, &pd);
    if (st != BSA_OK) return st;
    *nnz_out = pattern_nnz_head(pd) * B * H;
    return BSA_OK;
}

int bsa_build_mask_csr(const bsa_pattern* p, int32_t B, int32_t H, int32_t* row_ptr, int32_t* col_idx,
                       int64_t col_capacity, int64_t* nnz_out, bsa_stream_t stream) {
    if (B <= 0 || H <= 0) return BSA_ERR_INVALID_ARG;
    PatternDev pd;
    int st = to_pattern(p, &pd);
    if (st != BSA_OK) return st;
    const int64_t R = (int64_t)B * H * pd.nb;
    if (R >= INT32_MAX) return BSA_ERR_INVALID_ARG;
    const int64_t nnz_head = pattern_nnz_head(pd);
    const int64_t nnz = nnz_head * B * H;
    if (nnz > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if (nnz_out) *nnz_out = nnz;
    if (!col_idx) return BSA_OK;
    if (!row_ptr) return BSA_ERR_INVALID_ARG;
    if (col_capacity < nnz) return BSA_ERR_CAPACITY;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    cudaError_t e = bsa::launch_mask(pd, B * H, nnz_head, row_ptr, col_idx, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_pattern_row_flags(const bsa_pattern* p, int32_t B, int32_t H, uint8_t* row_flags, bsa_stream_t stream) {
    if (B <= 0 || H <= 0 || !row_flags) return BSA_ERR_INVALID_ARG;
    PatternDev pd;
    int st = to_pattern(p, &pd);
    if (st != BSA_OK) return st;
    if ((int64_t)B * H * pd.nb >= INT32_MAX) return BSA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    cudaError_t e = bsa::launch_row_flags(pd, B * H, row_flags, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_build_mask_csr_heads(const bsa_pattern_ex* patterns, int32_t n_patterns, const int32_t* head_pattern,
                             int32_t B, int32_t H, int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                             int64_t* nnz_out, bsa_stream_t stream) {
    if (B <= 0 || H <= 0) return BSA_ERR_INVALID_ARG;
    bsa::PatternSetDev ps;
    int st = to_pattern_set(patterns, n_patterns, head_pattern, H, &ps);
    if (st != BSA_OK) return st;
    const int64_t R = (int64_t)B * H * ps.nb;
    if (R >= INT32_MAX) return BSA_ERR_INVALID_ARG;
    // entries of one head of each pattern, then of every head of one batch element
    int64_t per_pat[BSA_MAX_PATTERNS] = {0};
    for (int32_t q = 0; q < n_patterns; ++q)
        for (int32_t i = 0; i < ps.nb; ++i) per_pat[q] += bsa::pattern_ex_row_len(ps, ps.pat[q], i);
    int64_t per_b = 0;
    for (int32_t h = 0; h < H; ++h) per_b += per_pat[ps.head_pat[h]];
    const int64_t nnz = per_b * B;
    if (nnz > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if (nnz_out) *nnz_out = nnz;
    if (!col_idx) return BSA_OK;
    if (!row_ptr) return BSA_ERR_INVALID_ARG;
    if (col_capacity < nnz) return BSA_ERR_CAPACITY;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    cudaError_t e = bsa::launch_mask_ex(ps, B, row_ptr, col_idx, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_topk_blocks(const bsa_shape* sh, const void* q, const void* k, int32_t topk, int32_t include_diag,
                    int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, bsa_stream_t stream) {
    int st = check_shape(sh);
    if (st != BSA_OK) return st;
    if (!q || !k || !row_ptr || !col_idx) return BSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16)) return BSA_ERR_INVALID_ARG;
    if (include_diag != 0 && include_diag != 1) return BSA_ERR_INVALID_ARG;
    if (sh->D != 64 && sh->D != 128) return BSA_ERR_UNSUPPORTED;
    const int b = sh->block;
    if (b != 16 && b != 32 && b != 64 && b != 128 && b != 256) return BSA_ERR_UNSUPPORTED;
    const int32_t nb = sh->N / b;
    if (nb > 4096) return BSA_ERR_UNSUPPORTED;
    if (topk < 1 || topk > nb) return BSA_ERR_INVALID_ARG;
    if (topk > 32) return BSA_ERR_UNSUPPORTED;
    const int32_t BH = sh->B * sh->H;
    const int64_t R = (int64_t)BH * nb;
    const int64_t need = R * (topk + include_diag);
    if (need > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if (col_capacity < need) return BSA_ERR_CAPACITY;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    if ((st = ensure_workspace(d, bsa::topk_workspace_bytes(BH, nb, sh->D, topk))) != BSA_OK) return st;
    cudaError_t e = bsa::launch_topk(BH, sh->N, sh->D, b, q, k, topk, include_diag, row_ptr, col_idx, d->ws,
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

namespace {

// The forward of bsa_forward / bsa_forward_ex (fp8 = false: bf16 Q, K) and
// bsa_forward_fp8 (e4m3 Q, K; `scale` already includes their descale factors).
struct FwdCall {
    int32_t B, H, D, block;
    int32_t nbq, nbk, q_off;  // query blocks, key blocks per head; key position of query block 0
    const void *q, *k, *v;
    const int32_t *row_ptr, *col_idx;
    const uint8_t* row_flags;
    void* out;
    float* lse;
    float scale;
    int32_t causal;
    const float* q_descale = nullptr;  // FP8 with per-block scales
    const float* k_descale = nullptr;
    bool out_f32 = false;              // O written as fp32
};

int forward_impl(const FwdCall& a, bsa_stream_t stream, bool fp8) {
    if (a.B <= 0 || a.H <= 0 || a.D <= 0 || a.block <= 0 || a.nbq <= 0 || a.nbk <= 0) return BSA_ERR_INVALID_ARG;
    if (a.q_off < 0 || a.q_off > a.nbk) return BSA_ERR_INVALID_ARG;
    const int64_t BH64 = (int64_t)a.B * a.H;
    if (BH64 * a.nbq * a.block > INT32_MAX || BH64 * a.nbk * a.block > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if (!a.q || !a.k || !a.v || !a.row_ptr || !a.col_idx || !a.out || !a.lse) return BSA_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.out, 16) || !aligned(a.lse, 4))
        return BSA_ERR_INVALID_ARG;
    if (a.causal != 0 && a.causal != 1) return BSA_ERR_INVALID_ARG;
    if (!(a.scale > 0.f) || !std::isfinite(a.scale)) return BSA_ERR_INVALID_ARG;
    // 64-token blocks run in the paired form: two query blocks per 128-row tile
    const bool paired = a.block == 64;
    if (bsa::fwd_smem_bytes(a.block, a.D, paired) == 0) return BSA_ERR_UNSUPPORTED;
    if (fp8 && (a.D != 128 || (a.block != 128 && a.block != 64))) return BSA_ERR_UNSUPPORTED;
    const int32_t BH = (int32_t)BH64;
    const int64_t R = BH64 * a.nbq;
    const int32_t Nq = a.nbq * a.block, Nk = a.nbk * a.block;
    int st;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    // workspace: [counter | perm | pairing buffers (paired form)]
    const size_t perm_bytes = 256 + align256((size_t)R * sizeof(int32_t));
    const size_t pair_bytes = paired ? bsa::pairing_workspace_bytes(BH, a.nbq) : 0;
    if ((st = ensure_workspace(d, perm_bytes + pair_bytes)) != BSA_OK) return st;
    int32_t* counter = static_cast<int32_t*>(d->ws);
    int32_t* perm = reinterpret_cast<int32_t*>(static_cast<char*>(d->ws) + 256);
    const uint64_t qrows = (uint64_t)BH * Nq, krows = (uint64_t)BH * Nk;
    CUtensorMap tq, tk, tv, to;
    if (fp8) {
        if ((st = make_map_e4m3(&tq, a.q, qrows, a.D, a.block)) != BSA_OK) return st;
        if ((st = make_map_e4m3(&tk, a.k, krows, a.D, a.block)) != BSA_OK) return st;
    } else {
        if ((st = make_map(&tq, a.q, qrows, a.D, a.block)) != BSA_OK) return st;
        if ((st = make_map(&tk, a.k, krows, a.D, a.block)) != BSA_OK) return st;
    }
    if ((st = make_map(&tv, a.v, krows, a.D, a.block)) != BSA_OK) return st;
    if ((st = make_map(&to, a.out, qrows, a.D, a.block)) != BSA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    FwdParams p{};
    cudaError_t e;
    if (paired) {
        const bsa::PairingBuffers pb = bsa::pairing_buffers(static_cast<char*>(d->ws) + perm_bytes, BH, a.nbq);
        bsa::PairGeom pg{a.nbq, a.nbk, a.q_off, a.causal, a.row_flags, INT64_MAX};
        e = bsa::launch_pairing(a.row_ptr, a.col_idx, BH, pg, pb, d->err, d->sm_count, s);
        if (e != cudaSuccess) return cuda_fail(e);
        // classes of 32 steps: pairs (at most 32 steps) run head by head, so a
        // head's K/V is read from HBM about once (content top-k: 1.80 -> 1.06 GB
        // per launch; classes of 8 steps: 1.46 GB)
        e = bsa::launch_schedule_lens(pb.item_len, pb.n_items, (int32_t)R, perm, counter, 5, s);
        p.item_a = pb.item_a;
        p.item_b = pb.item_b;
        p.item_cnt = pb.item_cnt;
        p.slots = pb.slots;
        p.n_items_dev = pb.n_items;
    } else {
        e = bsa::launch_schedule(a.row_ptr, (int32_t)R, perm, counter, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    p.row_ptr = a.row_ptr;
    p.col_idx = a.col_idx;
    p.perm = perm;
    p.counter = counter;
    p.out = a.out;
    p.out_f32 = a.out_f32 ? static_cast<float*>(a.out) : nullptr;
    p.lse = a.lse;
    p.err = d->err;
    p.BH = BH;
    p.N = Nq;
    p.nb = a.nbq;
    p.Nk = Nk;
    p.nbk = a.nbk;
    p.q_off = a.q_off;
    p.row_flags = a.row_flags;
    p.q_descale = a.q_descale;
    p.k_descale = a.k_descale;
    p.n_items = (int32_t)R;
    p.causal = a.causal;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_limit_ns = bsa::wait_limit_ns();
    p.stall_after = bsa::take_forward_stall();
    const int grid = (int)std::min<int64_t>(R, d->sm_count);
    e = fp8 ? bsa::launch_forward_f8(a.block, a.D, paired, tq, tk, tv, to, p, grid, s)
            : bsa::launch_forward(a.block, a.D, paired, tq, tk, tv, to, p, grid, s);
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int shape_call(const bsa_shape* sh, const void* q, const void* k, const void* v, const int32_t* row_ptr,
               const int32_t* col_idx, void* out, float* lse, float scale, int32_t causal, FwdCall* c) {
    int st = check_shape(sh);
    if (st != BSA_OK) return st;
    const int32_t nb = sh->N / sh->block;
    *c = FwdCall{sh->B, sh->H, sh->D, sh->block, nb, nb, 0, q, k, v, row_ptr, col_idx, nullptr, out, lse,
                 scale, causal};
    return BSA_OK;
}

}  // namespace

int bsa_forward(const bsa_shape* sh, const void* q, const void* k, const void* v, const int32_t* row_ptr,
                const int32_t* col_idx, void* out, float* lse, float scale, int32_t causal, bsa_stream_t stream) {
    FwdCall c;
    int st = shape_call(sh, q, k, v, row_ptr, col_idx, out, lse, scale, causal, &c);
    if (st != BSA_OK) return st;
    return forward_impl(c, stream, false);
}

int bsa_forward_ex(const bsa_forward_args* a, bsa_stream_t stream) {
    if (!a) return BSA_ERR_INVALID_ARG;
    if (a->out_fp32 != 0 && a->out_fp32 != 1) return BSA_ERR_INVALID_ARG;
    FwdCall c{a->B, a->H, a->D, a->block, a->n_q_blocks, a->n_k_blocks, a->q_block_offset, a->q, a->k, a->v,
              a->row_ptr, a->col_idx, a->row_flags, a->out, a->lse, a->scale, a->causal};
    c.out_f32 = a->out_fp32 == 1;
    return forward_impl(c, stream, false);
}

int bsa_forward_fp8(const bsa_shape* sh, const void* q8, const void* k8, const void* v, const int32_t* row_ptr,
                    const int32_t* col_idx, void* out, float* lse, float q_descale, float k_descale, float scale,
                    int32_t causal, bsa_stream_t stream) {
    if (!(q_descale > 0.f) || !std::isfinite(q_descale) || !(k_descale > 0.f) || !std::isfinite(k_descale))
        return BSA_ERR_INVALID_ARG;
    const float eff = scale * q_descale * k_descale;
    if (!(scale > 0.f) || !std::isfinite(scale) || !(eff > 0.f) || !std::isfinite(eff)) return BSA_ERR_INVALID_ARG;
    FwdCall c;
    int st = shape_call(sh, q8, k8, v, row_ptr, col_idx, out, lse, eff, causal, &c);
    if (st != BSA_OK) return st;
    return forward_impl(c, stream, true);
}

int bsa_forward_fp8_blocks(const bsa_shape* sh, const void* q8, const void* k8, const void* v,
                           const float* q_descale, const float* k_descale, const int32_t* row_ptr,
                           const int32_t* col_idx, void* out, float* lse, float scale, int32_t causal,
                           bsa_stream_t stream) {
    if (!q_descale || !k_descale || !aligned(q_descale, 4) || !aligned(k_descale, 4)) return BSA_ERR_INVALID_ARG;
    FwdCall c;
    int st = shape_call(sh, q8, k8, v, row_ptr, col_idx, out, lse, scale, causal, &c);
    if (st != BSA_OK) return st;
    c.q_descale = q_descale;
    c.k_descale = k_descale;
    return forward_impl(c, stream, true);
}

int bsa_quantize_e4m3_blocks(const bsa_shape* sh, const void* x, void* y, float* descale, bsa_stream_t stream) {
    int st = check_shape(sh);
    if (st != BSA_OK) return st;
    if (!x || !y || !descale || !aligned(x, 16) || !aligned(y, 16) || !aligned(descale, 4)) return BSA_ERR_INVALID_ARG;
    if ((sh->block != 64 && sh->block != 128) || (sh->D != 64 && sh->D != 128)) return BSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    const int64_t nblk = (int64_t)sh->B * sh->H * (sh->N / sh->block);
    const cudaError_t e = bsa::launch_quantize_e4m3_blocks(x, y, descale, nblk, sh->block, sh->D,
                                                           reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_quantize_e4m3(const void* x, void* y, int64_t n, float inv_scale, bsa_stream_t stream) {
    if (!x || !y || n <= 0 || n % 16 != 0) return BSA_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return BSA_ERR_INVALID_ARG;
    if (!(inv_scale > 0.f) || !std::isfinite(inv_scale)) return BSA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    int st;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    const cudaError_t e =
        bsa::launch_quantize_e4m3(x, y, n, inv_scale, d->sm_count, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_backward(const bsa_shape* sh, const void* q, const void* k, const void* v, const void* out,
                 const void* dout, const float* lse, const int32_t* row_ptr, const int32_t* col_idx,
                 int64_t col_capacity, void* dq, void* dk, void* dv, float scale, int32_t causal,
                 bsa_stream_t stream) {
    return bsa_backward_ex(sh, q, k, v, out, dout, lse, row_ptr, col_idx, col_capacity, nullptr, dq, dk, dv, scale,
                           causal, stream);
}

int bsa_backward_ex(const bsa_shape* sh, const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, const int32_t* row_ptr, const int32_t* col_idx,
                    int64_t col_capacity, const uint8_t* row_flags, void* dq, void* dk, void* dv, float scale,
                    int32_t causal, bsa_stream_t stream) {
    int st = check_shape(sh);
    if (st != BSA_OK) return st;
    if (!q || !k || !v || !out || !dout || !lse || !row_ptr || !col_idx || !dq || !dk || !dv)
        return BSA_ERR_INVALID_ARG;
    for (const void* x : {q, k, v, out, dout, (const void*)dq, (const void*)dk, (const void*)dv})
        if (!aligned(x, 16)) return BSA_ERR_INVALID_ARG;
    if (!aligned(lse, 4)) return BSA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BSA_ERR_INVALID_ARG;
    if (col_capacity < 0 || col_capacity > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if ((sh->block != 128 && sh->block != 64) || (sh->D != 64 && sh->D != 128)) return BSA_ERR_UNSUPPORTED;
    const int32_t nb = sh->N / sh->block;
    const int32_t BH = sh->B * sh->H;
    const int64_t R = (int64_t)BH * nb;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    if ((st = ensure_workspace(d, bsa::bwd_workspace_bytes(BH, sh->N, sh->D, sh->block, nb, col_capacity))) != BSA_OK)
        return st;
    bsa::BwdLaunch L{};
    const uint64_t rows = (uint64_t)BH * sh->N;
    if ((st = make_map(&L.tq, q, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&L.tk, k, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&L.tv, v, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&L.tdo, dout, rows, sh->D, sh->block)) != BSA_OK) return st;
    void* dq_acc = static_cast<char*>(d->ws) + bsa::bwd_dq_acc_offset(BH, sh->N, nb, col_capacity);
    if ((st = make_map_f32_32x32(&L.tdq, dq_acc, rows, sh->D)) != BSA_OK) return st;
    if ((st = make_map(&L.tdk, dk, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&L.tdv, dv, rows, sh->D, sh->block)) != BSA_OK) return st;
    L.row_ptr = row_ptr;
    L.col_idx = col_idx;
    L.col_capacity = col_capacity;
    L.row_flags = causal ? row_flags : nullptr;  // flags only lift the causal cut
    L.out = out;
    L.dout = dout;
    L.lse = lse;
    L.dq = dq;
    L.dk = dk;
    L.dv = dv;
    L.workspace = d->ws;
    L.err = d->err;
    L.BH = BH;
    L.N = sh->N;
    L.D = sh->D;
    L.block = sh->block;
    L.nb = nb;
    L.causal = causal;
    L.sm_count = d->sm_count;
    L.scale = scale;
    (void)R;
    const cudaError_t e = bsa::launch_backward(L, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_validate_csr(const bsa_shape* sh, const int32_t* row_ptr, const int32_t* col_idx, int32_t* d_err,
                     bsa_stream_t stream) {
    int st = check_shape(sh);
    if (st != BSA_OK) return st;
    if (!row_ptr || !col_idx || !d_err) return BSA_ERR_INVALID_ARG;
    const int32_t nb = sh->N / sh->block;
    const int64_t R = (int64_t)sh->B * sh->H * nb;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState* d;
    if ((st = dev_state(&d)) != BSA_OK) return st;
    if ((st = check_arch(d)) != BSA_OK) return st;
    cudaError_t e = bsa::launch_validate((int32_t)R, nb, row_ptr, col_idx, d_err, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : cuda_fail(e);
}

int bsa_device_error(int32_t* code_out) {
    if (!code_out) return BSA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
    if (cudaDeviceSynchronize() != cudaSuccess) return BSA_ERR_CUDA;
    int32_t v = 0;
    // The workspace's word exists once a workspace-using call ran on this
    // device; nothing is allocated here for a caller that never made one.
    const DevState& d = g_dev[dev];
    if (d.init) {
        if (cudaMemcpy(&v, d.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaMemset(d.err, 0, sizeof v) != cudaSuccess) return BSA_ERR_CUDA;
    }
    // The allocation-free forward keeps its word in its fixed array.
    int32_t w = 0;
    if (bsa::noalloc_take_error(dev, &w) != cudaSuccess) return BSA_ERR_CUDA;
    v |= w;
    *code_out = v;
    return v ? BSA_ERR_DEVICE_CHECK : BSA_OK;
}

void bsa_release_workspace(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        DevState& d = g_dev[dev];
        if (!d.init) continue;
        cudaSetDevice(dev);
        cudaDeviceSynchronize();
        if (d.ws) cudaFree(d.ws);
        if (d.err) cudaFree(d.err);
        d = DevState();
    }
    cudaSetDevice(cur);
}

}  // extern "C"
