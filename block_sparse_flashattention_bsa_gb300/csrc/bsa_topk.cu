// bsa_topk.cu -- content-based block selection on the device.
//
// "the model predicts importance scores and picks top-k" ("How Do Sparse
// Attention Kernels Work in GPU Clusters?", section "What Exactly Is a Sparse
// Attention Kernel?"), with mean-pooled Q and K as the routing features ("The
// Only Guide You Need for Sparse Attention Kernels in Long-Context LLMs",
// section "Flash-MSA", pooled per block here), plus the diagonal block.
//
// The selection is an integer decision taken on fp32 scores, so the
// arithmetic order is fixed and identical to the stated contract:
//   pooled[d]  = pairwise-tree fp32 sum over the block's tokens, times 1/block
//   score(i,j) = (a0 + a1) + (a2 + a3), a_c = fp32 running sum over d == c
//                (mod 4), increasing d, of fp32-rounded products
//   order      = score descending, ties to the smaller key block.
// Every multiply and add uses the _rn intrinsics so nothing is contracted.
//
// Kernels: pool (HBM-bound: reads Q and K once), score+select (one warp per
// query block), row_ptr scan, compaction into the caller's CSR.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

namespace {

// ---------------------------------------------------------------- pooling
// grid (BH * nb, 2): blockIdx.y 0 = Q, 1 = K.  D/2 threads, two columns each.
template <int BS, int D>
__global__ void __launch_bounds__(D / 2) pool_kernel(const __nv_bfloat162* __restrict__ q,
                                                     const __nv_bfloat162* __restrict__ k,
                                                     float2* __restrict__ qbar, float2* __restrict__ kbar) {
    const int64_t blk = blockIdx.x;  // bh * nb + i
    const __nv_bfloat162* src = (blockIdx.y == 0 ? q : k) + blk * BS * (D / 2) + threadIdx.x;
    float2* dst = (blockIdx.y == 0 ? qbar : kbar) + blk * (D / 2) + threadIdx.x;
    // Streaming pairwise tree: a stack of partial sums whose sizes are powers
    // of two; equal-sized neighbours are merged (left + right) as soon as they
    // exist, which reproduces the level-by-level pairwise tree exactly.
    constexpr int DEPTH = 10;
    float sx[DEPTH], sy[DEPTH];
    int top = 0;
#pragma unroll
    for (int t0 = 0; t0 < BS; t0 += 16) {
        float2 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = __bfloat1622float2(src[(t0 + u) * (D / 2)]);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            sx[top] = v[u].x;
            sy[top] = v[u].y;
            ++top;
            // merge while the two top entries cover equal token counts
            const int t = t0 + u + 1;  // tokens consumed so far
#pragma unroll
            for (int lvl = 1; lvl < DEPTH; ++lvl) {
                if ((t & ((1 << lvl) - 1)) == 0) {
                    sx[top - 2] = __fadd_rn(sx[top - 2], sx[top - 1]);
                    sy[top - 2] = __fadd_rn(sy[top - 2], sy[top - 1]);
                    --top;
                }
            }
        }
    }
    const float inv = 1.0f / (float)BS;  // exact: BS is a power of two
    *dst = make_float2(__fmul_rn(sx[0], inv), __fmul_rn(sy[0], inv));
}

// ---------------------------------------------------------------- scores + select
constexpr int kRows = 8;     // query blocks per CTA, one warp each
constexpr int kKeyChunk = 64;

__device__ __forceinline__ bool ahead(float s1, int j1, float s2, int j2) {
    return (s1 > s2) || (s1 == s2 && j1 < j2);
}

template <int D>
__global__ void __launch_bounds__(kRows * 32) score_select_kernel(const float* __restrict__ qbar,
                                                                  const float* __restrict__ kbar, int nb, int topk,
                                                                  int include_diag, int32_t* __restrict__ sel,
                                                                  int32_t* __restrict__ lens) {
    extern __shared__ __align__(16) float sm[];
    float* sq = sm;                            // [kRows][D]
    float* sk = sq + kRows * D;                // [kKeyChunk][D + 4]  (padding: conflict-free float4 rows)
    float* ss = sk + kKeyChunk * (D + 4);      // [kRows][nb]
    const int bh = blockIdx.y;
    const int i0 = blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* qb = qbar + (int64_t)bh * nb * D;
    const float* kb = kbar + (int64_t)bh * nb * D;
    for (int x = threadIdx.x; x < kRows * D; x += kRows * 32) {
        const int r = x / D;
        sq[x] = (i0 + r < nb) ? qb[(int64_t)(i0 + r) * D + (x - r * D)] : 0.f;
    }
    for (int kc = 0; kc < nb; kc += kKeyChunk) {
        __syncthreads();
        for (int x = threadIdx.x; x < kKeyChunk * (D / 4); x += kRows * 32) {
            const int kr = x / (D / 4), d4 = x - kr * (D / 4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kc + kr < nb) v = reinterpret_cast<const float4*>(kb + (int64_t)(kc + kr) * D)[d4];
            *reinterpret_cast<float4*>(sk + kr * (D + 4) + d4 * 4) = v;
        }
        __syncthreads();
        const float* qrow = sq + warp * D;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int kr = lane + half * 32;
            const float* krow = sk + kr * (D + 4);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; d += 4) {
                const float4 qv = *reinterpret_cast<const float4*>(qrow + d);
                const float4 kv = *reinterpret_cast<const float4*>(krow + d);
                a0 = __fadd_rn(a0, __fmul_rn(qv.x, kv.x));
                a1 = __fadd_rn(a1, __fmul_rn(qv.y, kv.y));
                a2 = __fadd_rn(a2, __fmul_rn(qv.z, kv.z));
                a3 = __fadd_rn(a3, __fmul_rn(qv.w, kv.w));
            }
            if (kc + kr < nb) ss[warp * nb + kc + kr] = __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
        }
    }
    __syncthreads();
    const int i = i0 + warp;
    if (i >= nb) return;
    const float* srow = ss + warp * nb;
    // lane owns key blocks lane + 32 m; taken[m / 32] bit (m % 32) marks selected ones
    uint32_t taken[4] = {0u, 0u, 0u, 0u};
    const int per_lane = (nb + 31) / 32;  // <= 128
    float bs;
    int bj;
    auto local_best = [&]() {
        bs = -INFINITY;
        bj = 0x7fffffff;
        for (int m = 0; m < per_lane; ++m) {
            const int j = lane + 32 * m;
            if (j < nb && !((taken[m >> 5] >> (m & 31)) & 1u)) {
                const float s = srow[j];
                if (ahead(s, j, bs, bj)) {
                    bs = s;
                    bj = j;
                }
            }
        }
    };
    local_best();
    int my_sel = 0x7fffffff;
    for (int a = 0; a < topk; ++a) {
        float ws = bs;
        int wj = bj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, ws, o);
            const int oj = __shfl_xor_sync(0xffffffffu, wj, o);
            if (ahead(os, oj, ws, wj)) {
                ws = os;
                wj = oj;
            }
        }
        if (lane == a) my_sel = wj;
        if ((wj & 31) == lane) {
            const int m = wj >> 5;
            taken[m >> 5] |= 1u << (m & 31);
            local_best();
        }
    }
    const bool mine = lane < topk;
    const bool has_diag = __any_sync(0xffffffffu, mine && my_sel == i);
    const bool add = include_diag && !has_diag;
    int rank = 0;
    for (int b = 0; b < topk; ++b) {
        const int xb = __shfl_sync(0xffffffffu, my_sel, b);
        rank += (xb < my_sel) ? 1 : 0;
    }
    if (add && i < my_sel) ++rank;
    const int64_t r = (int64_t)bh * nb + i;
    int32_t* out = sel + r * (topk + 1);
    if (mine) out[rank] = my_sel;
    const int below = __popc(__ballot_sync(0xffffffffu, mine && my_sel < i));
    if (lane == 0) {
        if (add) out[below] = i;
        lens[r] = topk + (add ? 1 : 0);
    }
}

// ---------------------------------------------------------------- CSR assembly
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) lens_scan_kernel(const int32_t* __restrict__ lens, int64_t R,
                                                                 int32_t* __restrict__ row_ptr) {
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t per = (R + kScanThreads - 1) / kScanThreads;
    const int64_t r0 = tid * per;
    int32_t local = 0;
    for (int64_t r = r0; r < r0 + per && r < R; ++r) local += lens[r];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        warp_tot[lane] = ti - t;
    }
    __syncthreads();
    int32_t run = incl - local + warp_tot[warp];
    if (tid == 0) row_ptr[0] = 0;
    for (int64_t r = r0; r < r0 + per && r < R; ++r) {
        run += lens[r];
        row_ptr[r + 1] = run;
    }
}

__global__ void compact_kernel(const int32_t* __restrict__ sel, const int32_t* __restrict__ lens,
                               const int32_t* __restrict__ row_ptr, int64_t R, int topk,
                               int32_t* __restrict__ col_idx) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const int32_t* s = sel + r * (topk + 1);
    int32_t* d = col_idx + row_ptr[r];
    const int n = lens[r];
    for (int a = 0; a < n; ++a) d[a] = s[a];
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int D>
cudaError_t launch_pool(int block, int64_t nblk, const void* q, const void* k, float* qbar, float* kbar,
                        cudaStream_t s) {
    dim3 grid((unsigned)nblk, 2);
    auto* q2 = static_cast<const __nv_bfloat162*>(q);
    auto* k2 = static_cast<const __nv_bfloat162*>(k);
    auto* qb = reinterpret_cast<float2*>(qbar);
    auto* kb = reinterpret_cast<float2*>(kbar);
    switch (block) {
        case 16: pool_kernel<16, D><<<grid, D / 2, 0, s>>>(q2, k2, qb, kb); break;
        case 32: pool_kernel<32, D><<<grid, D / 2, 0, s>>>(q2, k2, qb, kb); break;
        case 64: pool_kernel<64, D><<<grid, D / 2, 0, s>>>(q2, k2, qb, kb); break;
        case 128: pool_kernel<128, D><<<grid, D / 2, 0, s>>>(q2, k2, qb, kb); break;
        case 256: pool_kernel<256, D><<<grid, D / 2, 0, s>>>(q2, k2, qb, kb); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_select(int32_t BH, int32_t nb, int32_t topk, int32_t include_diag, const float* qbar,
                          const float* kbar, int32_t* sel, int32_t* lens, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)kRows * D + (size_t)kKeyChunk * (D + 4) + (size_t)kRows * nb);
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((nb + kRows - 1) / kRows), (unsigned)BH);
    score_select_kernel<D><<<grid, kRows * 32, smem, s>>>(qbar, kbar, nb, topk, include_diag, sel, lens);
    return cudaGetLastError();
}

}  // namespace

size_t topk_workspace_bytes(int32_t BH, int32_t nb, int32_t D, int32_t topk) {
    const size_t R = (size_t)BH * nb;
    return 2 * align256(R * D * sizeof(float)) + align256(R * (topk + 1) * sizeof(int32_t)) +
           align256(R * sizeof(int32_t));
}

cudaError_t launch_topk(int32_t BH, int32_t N, int32_t D, int32_t block, const void* q, const void* k,
                        int32_t topk, int32_t include_diag, int32_t* row_ptr, int32_t* col_idx, void* workspace,
                        cudaStream_t stream) {
    const int32_t nb = N / block;
    const int64_t R = (int64_t)BH * nb;
    char* w = static_cast<char*>(workspace);
    float* qbar = reinterpret_cast<float*>(w);
    w += align256((size_t)R * D * sizeof(float));
    float* kbar = reinterpret_cast<float*>(w);
    w += align256((size_t)R * D * sizeof(float));
    int32_t* sel = reinterpret_cast<int32_t*>(w);
    w += align256((size_t)R * (topk + 1) * sizeof(int32_t));
    int32_t* lens = reinterpret_cast<int32_t*>(w);
    cudaError_t e = (D == 128) ? launch_pool<128>(block, R, q, k, qbar, kbar, stream)
                               : launch_pool<64>(block, R, q, k, qbar, kbar, stream);
    if (e != cudaSuccess) return e;
    e = (D == 128) ? launch_select<128>(BH, nb, topk, include_diag, qbar, kbar, sel, lens, stream)
                   : launch_select<64>(BH, nb, topk, include_diag, qbar, kbar, sel, lens, stream);
    if (e != cudaSuccess) return e;
    lens_scan_kernel<<<1, kScanThreads, 0, stream>>>(lens, R, row_ptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    compact_kernel<<<(unsigned)((R + 255) / 256), 256, 0, stream>>>(sel, lens, row_ptr, R, topk, col_idx);
    return cudaGetLastError();
}

}  // namespace bsa
