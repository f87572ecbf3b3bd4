// bsa_fp8.cu -- e4m3 quantisation of bf16 Q and K for the FP8-score forward.
//
// The scores may be computed in FP8 on tensor cores that have such
// instructions ("Flash MSA Sparse Attention Kernels Explained", section "The
// Future of Attention Kernels").  Q and K are stored as OCP e4m3 (FN: no
// infinities, largest finite 448) with one scale per tensor:
// y = e4m3(x * inv_scale), the product rounded once in fp32, then rounded to
// the nearest e4m3 value (ties to even) and saturated to +-448.  A second
// form takes one scale per (head, block of tokens) instead.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

#include <cuda_bf16.h>

namespace bsa {
namespace {

// Two floats to two e4m3 codes: lo lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16 elements per thread: two 16-byte loads of bf16, one 16-byte store.
__global__ void quantize_e4m3_kernel(const uint4* __restrict__ x, uint4* __restrict__ y, int64_t n16,
                                     float inv_scale) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n16; t += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = x[2 * t], b = x[2 * t + 1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * u]));
            const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * u + 1]));
            const uint16_t lo = e4m3x2(__fmul_rn(f0.x, inv_scale), __fmul_rn(f0.y, inv_scale));
            const uint16_t hi = e4m3x2(__fmul_rn(f1.x, inv_scale), __fmul_rn(f1.y, inv_scale));
            o[u] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        y[t] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One CTA of 256 threads per (head, block): the block's block x D bf16
// values stay in registers (CH chunks of 16 per thread), the CTA reduces
// their largest magnitude, then scales, rounds and stores them.  Scales per
// block keep a peaked block from crushing the precision of the others.
template <int CH>
__global__ void __launch_bounds__(256) quantize_e4m3_blocks_kernel(const uint4* __restrict__ x, uint4* __restrict__ y,
                                                                   float* __restrict__ descale, int32_t chunks) {
    __shared__ float red[8];
    const int64_t b = blockIdx.x;
    const uint4* xb = x + b * (int64_t)chunks * 2;
    uint4* yb = y + b * (int64_t)chunks;
    uint32_t w[CH][8];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = threadIdx.x + u * 256;
        if (c < chunks) {
            const uint4 a = xb[2 * c], bq = xb[2 * c + 1];
            w[u][0] = a.x; w[u][1] = a.y; w[u][2] = a.z; w[u][3] = a.w;
            w[u][4] = bq.x; w[u][5] = bq.y; w[u][6] = bq.z; w[u][7] = bq.w;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u][q]));
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) amax = fmaxf(amax, red[q]);
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    if (threadIdx.x == 0) descale[b] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = threadIdx.x + u * 256;
        if (c < chunks) {
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u][2 * q]));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u][2 * q + 1]));
                const uint16_t lo = e4m3x2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv));
                const uint16_t hi = e4m3x2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv));
                o[q] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            yb[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_e4m3_blocks(const void* x, void* y, float* descale, int64_t n_blocks, int32_t block,
                                        int32_t D, cudaStream_t stream) {
    const int32_t chunks = block * D / 16;  // 16 elements per chunk
    const uint4* xs = static_cast<const uint4*>(x);
    uint4* ys = static_cast<uint4*>(y);
    if (chunks <= 256)
        quantize_e4m3_blocks_kernel<1><<<(unsigned)n_blocks, 256, 0, stream>>>(xs, ys, descale, chunks);
    else if (chunks <= 512)
        quantize_e4m3_blocks_kernel<2><<<(unsigned)n_blocks, 256, 0, stream>>>(xs, ys, descale, chunks);
    else if (chunks <= 1024)
        quantize_e4m3_blocks_kernel<4><<<(unsigned)n_blocks, 256, 0, stream>>>(xs, ys, descale, chunks);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* x, void* y, int64_t n, float inv_scale, int sm_count,
                                 cudaStream_t stream) {
    const int64_t n16 = n / 16;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 8 * (int64_t)sm_count) blocks = 8 * (int64_t)sm_count;
    if (blocks < 1) blocks = 1;
    quantize_e4m3_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4*>(x), static_cast<uint4*>(y),
                                                               n16, inv_scale);
    return cudaGetLastError();
}

}  // namespace bsa
