// bsa_noalloc.cu -- bsa_forward_noalloc: the forward pass without any device
// allocation by the library.
//
// bsa_forward keeps its schedule (the longest-first order of the rows and the
// work counter the persistent CTAs claim rows from) in a workspace that the
// library cudaMallocs on first use and grows on demand.  Some callers cannot
// allow that: serving loops that must never hit the device-wide
// synchronisation that cudaMalloc / cudaFree imply, and applications that
// hand out every byte of device memory from their own pre-reserved pools.
// For them this entry point takes its scratch from a fixed array compiled
// into the library instead.  Apart from where the scratch lives it launches
// exactly the kernels bsa_forward launches.

#include <algorithm>
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

// Scratch layout (int32 words): [0] work counter, [1] device error word,
// [64 ..) schedule permutation, one word per CSR row.
constexpr int kHeader = 64;
static __device__ __align__(256) int32_t g_noalloc_scratch[kHeader + BSA_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
int g_sms[kMaxDevices];
int g_ok[kMaxDevices];        // 1 = sm_103 device

// Once per device, with that device current: the device address of the
// array (in host code its name is only a host-side stand-in) and the facts
// the launch needs.  None of these calls allocates.  The address is kept for
// the life of the process, so a device reset (which unloads the module and
// the array with it) is not supported between calls.
int setup_device(int dev) {
    if (g_ptr[dev]) return BSA_OK;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return BSA_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BSA_ERR_CUDA;
    g_sms[dev] = sms;
    g_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
    g_ptr[dev] = static_cast<int32_t*>(ptr);
    return BSA_OK;
}

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

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace bsa {
// The error word of this entry point (word 1 of the array), read and cleared
// through the symbol: cudaMemcpyFromSymbol / ToSymbol allocate nothing.  A
// device where the entry point never ran has nothing to report, and its
// module is not loaded just to look.
cudaError_t noalloc_take_error(int dev, int32_t* code) {
    *code = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= kMaxDevices || !g_ptr[dev]) return cudaSuccess;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_noalloc_scratch, sizeof v, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    if (v) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof zero, sizeof(int32_t), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    *code = v;
    return cudaSuccess;
}
}  // namespace bsa

extern "C" int bsa_forward_noalloc(const bsa_shape* sh, const void* q, const void* k, const void* v,
                                   const int32_t* row_ptr, const int32_t* col_idx, void* out, float* lse,
                                   float scale, int32_t causal, bsa_stream_t stream) {
    if (!sh || sh->B <= 0 || sh->H <= 0 || sh->N <= 0 || sh->D <= 0 || sh->block <= 0) return BSA_ERR_INVALID_ARG;
    if (sh->N % sh->block != 0) return BSA_ERR_INVALID_ARG;
    if ((int64_t)sh->B * sh->H * sh->N > INT32_MAX) return BSA_ERR_INVALID_ARG;
    if (!q || !k || !v || !row_ptr || !col_idx || !out || !lse) return BSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
        return BSA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BSA_ERR_INVALID_ARG;
    if (bsa::fwd_smem_bytes(sh->block, sh->D, false) == 0) return BSA_ERR_UNSUPPORTED;
    const int32_t nb = sh->N / sh->block;
    const int32_t BH = sh->B * sh->H;
    const int64_t R = (int64_t)BH * nb;
    if (R > BSA_NOALLOC_MAX_ROWS) return BSA_ERR_CAPACITY;  // the fixed scratch holds one word per row

    std::lock_guard<std::mutex> lk(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
    int st = setup_device(dev);
    if (st != BSA_OK) return st;
    if (!g_ok[dev]) return BSA_ERR_UNSUPPORTED;
    int32_t* counter = g_ptr[dev];
    int32_t* err = g_ptr[dev] + 1;
    int32_t* perm = g_ptr[dev] + kHeader;

    const uint64_t rows = (uint64_t)BH * sh->N;
    CUtensorMap tq, tk, tv, to;
    if ((st = make_map(&tq, q, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&tk, k, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&tv, v, rows, sh->D, sh->block)) != BSA_OK) return st;
    if ((st = make_map(&to, out, rows, sh->D, sh->block)) != BSA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents.  The schedule kernel
    // zeroes the work counter and rewrites every permutation word it uses;
    // the error word accumulates like bsa_forward's until bsa_device_error
    // reads and clears it (the array starts zeroed when the module loads).
    if (bsa::launch_schedule(row_ptr, (int32_t)R, perm, counter, s) != cudaSuccess) return BSA_ERR_CUDA;
    bsa::FwdParams p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.perm = perm;
    p.counter = counter;
    p.out = out;
    p.lse = lse;
    p.err = err;
    p.BH = BH;
    p.N = sh->N;
    p.nb = nb;
    p.Nk = sh->N;   // keys: the same blocks as the queries
    p.nbk = nb;
    p.q_off = 0;
    p.row_flags = nullptr;
    p.n_items = (int32_t)R;
    p.causal = causal;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = bsa::wait_limit_ns();
    p.stall_after = bsa::take_forward_stall();
    const int grid = (int)std::min<int64_t>(R, g_sms[dev]);
    return bsa::launch_forward(sh->block, sh->D, false, tq, tk, tv, to, p, grid, s) == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}
