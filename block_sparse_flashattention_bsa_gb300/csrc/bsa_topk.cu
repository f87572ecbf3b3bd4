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
//   score(i,j) = a0 + a1, a_c = fp32 chain of fused multiply-adds over
//                d == c (mod 2), increasing d, from 0
//   order      = score descending, ties to the smaller key block.
// The pooling uses the _rn intrinsics so nothing is contracted; the score
// chains use the packed fma.rn.f32x2, which rounds each lane once.
//
// Kernels: pool (HBM-bound: reads Q and K once), scores (register-blocked,
// into the workspace) then selection (warp per row) -- or, above 1024 key
// blocks or 256 MB of scores, one fused score+select kernel -- row_ptr scan,
// compaction into the caller's CSR.

#include <algorithm>

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
// One CTA = RPC query blocks of one (b, h); 8 warps.
// Scores: warp w owns rows RT*w .. RT*w+RT-1 (RT = RPC / 8) and each lane two
// key blocks of the current 64-key chunk, so every pooled value loaded from
// shared memory is used RT (queries) or 2 (keys) times.  Each (row, key)
// keeps the two fused multiply-add chains (even and odd d) of the stated order.
// Selection: one warp per row, lane l holding the key blocks l + 32 t.  The
// topk-th largest of the 32 lane maxima is a lower bound on the topk-th best
// score (it and the topk - 1 lane maxima above it are topk distinct scores at
// least that large), so only scores at or above it can be chosen.  When at
// most 32 pass, each is ranked exactly among them (score descending, ties to
// the smaller index); otherwise (many equal scores) the best remaining entry
// is taken topk times.  A per-warp bitmap then emits the chosen blocks plus
// the diagonal in ascending order.
constexpr int kKeyChunk = 64;

__device__ __forceinline__ bool ahead(float s1, int j1, float s2, int j2) {
    return (s1 > s2) || (s1 == s2 && j1 < j2);
}

// Selection of query block i from its score row srow[0 .. nb) (shared or
// global memory), by one warp: the chosen blocks in ascending order into
// out[0 .. n) and n into *len.  cv, cj: 32 floats and ints of scratch; bits:
// (nb + 31) / 32 words of scratch; all of them the warp's own.
__device__ void select_row(const float* srow, int nb, int i, int topk, int include_diag, float* cv, int* cj,
                           uint32_t* bits, int32_t* out, int32_t* len) {
    const int lane = threadIdx.x & 31;
    const int nbits = (nb + 31) >> 5;
    const int wpl = (nbits + 31) >> 5;  // bitmap words per lane
    float mx = -INFINITY;
    for (int j = lane; j < nb; j += 32) mx = fmaxf(mx, srow[j]);
    // bitonic sort of the lane maxima, descending; the topk-th of them
    // bounds the topk-th best score from below
    float v = mx;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int h = k >> 1; h > 0; h >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, h);
            v = (((lane & h) == 0) == ((lane & k) == 0)) ? fmaxf(v, o) : fminf(v, o);
        }
    const float thr = __shfl_sync(0xffffffffu, v, topk - 1);
    int cnt = 0;
    for (int j = lane; j < nb; j += 32) cnt += (srow[j] >= thr) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    for (int x = lane; x < nbits; x += 32) bits[x] = 0u;
    __syncwarp();
    if (total <= 32) {
        // rank each candidate among the candidates
        int pos = incl - cnt;
        for (int j = lane; j < nb; j += 32) {
            const float x = srow[j];
            if (x >= thr) {
                cv[pos] = x;
                cj[pos] = j;
                ++pos;
            }
        }
        __syncwarp();
        const bool has = lane < total;
        const float x = has ? cv[lane] : -INFINITY;
        const int jx = has ? cj[lane] : 0x7fffffff;
        int rank = 0;
        for (int c = 0; c < total; ++c) rank += ahead(cv[c], cj[c], x, jx) ? 1 : 0;
        if (has && rank < topk) atomicOr(&bits[jx >> 5], 1u << (jx & 31));
    } else {
        // many equal scores: take the best remaining entry topk times,
        // each strictly behind the previous one in the total order
        float pv = INFINITY;
        int pj = -1;
        for (int a = 0; a < topk; ++a) {
            float bv = -INFINITY;
            int bj = 0x7fffffff;
            bool found = false;
            for (int j = lane; j < nb; j += 32) {
                const float x = srow[j];
                if (ahead(pv, pj, x, j) && (!found || ahead(x, j, bv, bj))) {
                    bv = x;
                    bj = j;
                    found = true;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
                const bool of = __shfl_xor_sync(0xffffffffu, found ? 1 : 0, o) != 0;
                if (of && (!found || ahead(ov, oj, bv, bj))) {
                    bv = ov;
                    bj = oj;
                    found = true;
                }
            }
            if (!found) break;
            pv = bv;
            pj = bj;
            if (lane == 0) bits[bj >> 5] |= 1u << (bj & 31);
        }
    }
    if (include_diag && lane == 0) atomicOr(&bits[i >> 5], 1u << (i & 31));
    __syncwarp();
    // emit in ascending order: lane l owns bitmap words [l * wpl, l * wpl + wpl)
    const int wb = min(nbits, lane * wpl), we = min(nbits, wb + wpl);
    int c = 0;
    for (int x = wb; x < we; ++x) c += __popc(bits[x]);
    int ci = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ci, o);
        if (lane >= o) ci += y;
    }
    int n = ci - c;
    for (int x = wb; x < we; ++x) {
        uint32_t bw = bits[x];
        while (bw) {
            out[n++] = x * 32 + __ffs(bw) - 1;
            bw &= bw - 1;
        }
    }
    if (lane == 31) *len = ci;
    __syncwarp();
}

template <int D, int RPC>
__global__ void __launch_bounds__(256, 2) score_select_kernel(const float* __restrict__ qbar,
                                                           const float* __restrict__ kbar, int nb, int topk,
                                                           int include_diag, int32_t* __restrict__ sel,
                                                           int32_t* __restrict__ lens) {
    constexpr int RT = RPC / 8;
    extern __shared__ __align__(16) float sm[];
    const int ldss = nb + 1;                   // padded score row: thread-per-row reads are conflict-free
    float* sq = sm;                            // [RPC][D]
    float* sk = sq + RPC * D;                  // [kKeyChunk][D + 4]; later the selection scratch
    float* ss = sk + kKeyChunk * (D + 4);      // [RPC][nb + 1]
    const int bh = blockIdx.y;
    const int i0 = blockIdx.x * RPC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* qb = qbar + (int64_t)bh * nb * D;
    const float* kb = kbar + (int64_t)bh * nb * D;
    for (int x = threadIdx.x; x < RPC * (D / 4); x += 256) {
        const int r = x / (D / 4), d4 = x - r * (D / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i0 + r < nb) v = reinterpret_cast<const float4*>(qb + (int64_t)(i0 + r) * D)[d4];
        reinterpret_cast<float4*>(sq)[x] = v;
    }
    // The next 64-key chunk is loaded into registers while this one is scored.
    constexpr int PER = kKeyChunk * (D / 4) / 256;  // float4 per thread per chunk
    float4 nxt[PER];
    auto load_chunk = [&](int kc0) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int x = threadIdx.x + u * 256;
            const int kr = x / (D / 4), d4 = x - kr * (D / 4);
            nxt[u] = kc0 + kr < nb ? reinterpret_cast<const float4*>(kb + (int64_t)(kc0 + kr) * D)[d4]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    load_chunk(0);
    for (int kc = 0; kc < nb; kc += kKeyChunk) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int x = threadIdx.x + u * 256;
            const int kr = x / (D / 4), d4 = x - kr * (D / 4);
            *reinterpret_cast<float4*>(sk + kr * (D + 4) + d4 * 4) = nxt[u];
        }
        if (kc + kKeyChunk < nb) load_chunk(kc + kKeyChunk);
        __syncthreads();
        // acc[r][k] = {a0, a1}: the fused multiply-add chains over even and odd
        // d, one packed f32x2 FMA per pair of consecutive d (each lane rounds
        // once, like fmaf)
        f2 acc[RT][2];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            acc[r][0] = {0.f, 0.f};
            acc[r][1] = {0.f, 0.f};
        }
        const float* k0 = sk + lane * (D + 4);
        const float* k1 = sk + (lane + 32) * (D + 4);
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
            const float4 kv0 = *reinterpret_cast<const float4*>(k0 + d);
            const float4 kv1 = *reinterpret_cast<const float4*>(k1 + d);
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                const float4 qv = *reinterpret_cast<const float4*>(sq + (warp * RT + r) * D + d);
                const f2 qlo = {qv.x, qv.y}, qhi = {qv.z, qv.w};
                acc[r][0] = fma2(qlo, {kv0.x, kv0.y}, acc[r][0]);
                acc[r][1] = fma2(qlo, {kv1.x, kv1.y}, acc[r][1]);
                acc[r][0] = fma2(qhi, {kv0.z, kv0.w}, acc[r][0]);
                acc[r][1] = fma2(qhi, {kv1.z, kv1.w}, acc[r][1]);
            }
        }
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int kr = lane + 32 * k;
                if (kc + kr < nb) ss[(warp * RT + r) * ldss + kc + kr] = __fadd_rn(acc[r][k].x, acc[r][k].y);
            }
    }
    __syncthreads();
    // ---- selection: warp w takes rows w, w + 8, ...; lane l sees key blocks l + 32 t
    float* cv = sk + warp * 32;                                         // [8][32] candidate scores
    int* cj = reinterpret_cast<int*>(sk + 8 * 32) + warp * 32;          // [8][32] candidate blocks
    const int nbits = (nb + 31) >> 5;
    uint32_t* bits = reinterpret_cast<uint32_t*>(sk + 16 * 32) + warp * nbits;  // [8][nbits]
    for (int rr = warp; rr < RPC; rr += 8) {
        const int i = i0 + rr;
        if (i >= nb) break;
        const int64_t r = (int64_t)bh * nb + i;
        select_row(ss + rr * ldss, nb, i, topk, include_diag, cv, cj, bits, sel + r * (topk + 1), lens + r);
    }
}

// ---------------------------------------------------------------- scores, then select
// Up to 1024 key blocks the score matrix of every head goes to the workspace
// (4 nb^2 bytes a head, read back from the L2) and the two steps run as
// separate kernels.  score_kernel: one CTA = 64 query blocks x 128 key blocks
// of one head, 256 threads in a 16 x 16 grid; thread (ty, tx) owns query
// blocks 4 ty .. 4 ty + 3 and key blocks tx + 16 c (c < 8), 32 scores of two
// fused multiply-add chains each, so one pooled value read from shared
// memory feeds 8 (queries) or 4 (keys) packed FMAs.  Same chains and order as
// above, so the scores are bit-identical.
constexpr int kScoreTQ = 64, kScoreTK = 128;

template <int D>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ qbar, const float* __restrict__ kbar,
                                                    int nb, float* __restrict__ scores) {
    constexpr int LD = D + 4;  // padded rows: a warp's 16 key rows cover the banks twice
    extern __shared__ __align__(16) float sm[];
    float* sq = sm;                 // [kScoreTQ][LD]
    float* sk = sq + kScoreTQ * LD;  // [kScoreTK][LD]
    const int bh = blockIdx.z;
    const int i0 = blockIdx.x * kScoreTQ, j0 = blockIdx.y * kScoreTK;
    const float* qb = qbar + (int64_t)bh * nb * D;
    const float* kb = kbar + (int64_t)bh * nb * D;
    // every load of the tile issued before the first store, so the copies overlap
    constexpr int NQL = kScoreTQ * (D / 4) / 256, NKL = kScoreTK * (D / 4) / 256;
    static_assert(NQL * 256 == kScoreTQ * (D / 4) && NKL * 256 == kScoreTK * (D / 4), "whole tiles per thread");
    float4 vq[NQL], vk[NKL];
#pragma unroll
    for (int u = 0; u < NQL; ++u) {
        const int x = threadIdx.x + 256 * u, r = x / (D / 4), d4 = x - r * (D / 4);
        vq[u] = i0 + r < nb ? reinterpret_cast<const float4*>(qb + (int64_t)(i0 + r) * D)[d4]
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NKL; ++u) {
        const int x = threadIdx.x + 256 * u, r = x / (D / 4), d4 = x - r * (D / 4);
        vk[u] = j0 + r < nb ? reinterpret_cast<const float4*>(kb + (int64_t)(j0 + r) * D)[d4]
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NQL; ++u) {
        const int x = threadIdx.x + 256 * u, r = x / (D / 4), d4 = x - r * (D / 4);
        *reinterpret_cast<float4*>(sq + r * LD + d4 * 4) = vq[u];
    }
#pragma unroll
    for (int u = 0; u < NKL; ++u) {
        const int x = threadIdx.x + 256 * u, r = x / (D / 4), d4 = x - r * (D / 4);
        *reinterpret_cast<float4*>(sk + r * LD + d4 * 4) = vk[u];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tx = lane & 15, ty = warp * 2 + (lane >> 4);
    f2 acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = {0.f, 0.f};
#pragma unroll 2
    for (int d = 0; d < D; d += 4) {
        float4 qv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) qv[r] = *reinterpret_cast<const float4*>(sq + (ty * 4 + r) * LD + d);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float4 kv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                kv[c] = *reinterpret_cast<const float4*>(sk + (tx + 16 * (4 * half + c)) * LD + d);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    f2& a = acc[r][4 * half + c];
                    a = fma2({qv[r].x, qv[r].y}, {kv[c].x, kv[c].y}, a);
                    a = fma2({qv[r].z, qv[r].w}, {kv[c].z, kv[c].w}, a);
                }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = i0 + ty * 4 + r;
        if (i >= nb) continue;
        float* dst = scores + ((int64_t)bh * nb + i) * nb;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j = j0 + tx + 16 * c;
            if (j < nb) dst[j] = __fadd_rn(acc[r][c].x, acc[r][c].y);
        }
    }
}

// One warp per query block: select_row on its score row.
__global__ void __launch_bounds__(256) select_kernel(const float* __restrict__ scores, int64_t R, int nb, int topk,
                                                     int include_diag, int32_t* __restrict__ sel,
                                                     int32_t* __restrict__ lens) {
    extern __shared__ uint32_t ws[];  // per warp: 32 scores, 32 blocks, the bitmap
    const int warp = threadIdx.x >> 5;
    const int nbits = (nb + 31) >> 5;
    uint32_t* mine = ws + warp * (64 + nbits);
    const int64_t r = (int64_t)blockIdx.x * 8 + warp;
    if (r >= R) return;
    const int i = (int)(r % nb);
    select_row(scores + r * nb, nb, i, topk, include_diag, reinterpret_cast<float*>(mine),
               reinterpret_cast<int*>(mine + 32), mine + 64, sel + r * (topk + 1), lens + r);
}

// ---------------------------------------------------------------- CSR assembly
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

template <int D, int RPC>
cudaError_t launch_select_rpc(int32_t BH, int32_t nb, int32_t topk, int32_t include_diag, const float* qbar,
                              const float* kbar, int32_t* sel, int32_t* lens, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)RPC * D + (size_t)kKeyChunk * (D + 4) + (size_t)RPC * (nb + 1));
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel<D, RPC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((nb + RPC - 1) / RPC), (unsigned)BH);
    score_select_kernel<D, RPC><<<grid, 256, smem, s>>>(qbar, kbar, nb, topk, include_diag, sel, lens);
    return cudaGetLastError();
}

// Up to kSplitMaxNb key blocks (and kSplitMaxScoreBytes of scores in all):
// score_kernel into the workspace, then select_kernel; otherwise (scores ==
// nullptr) the fused kernel with 8 query blocks per CTA (their score rows in
// shared memory).
constexpr int kSplitMaxNb = 1024;
constexpr size_t kSplitMaxScoreBytes = (size_t)256 << 20;  // the score matrices of all heads

// The split path: few enough key blocks, and every head's score matrix fits
// the budget (beyond it, the fused kernel needs no score workspace).
inline bool use_split(int64_t BH, int32_t nb) {
    return nb <= kSplitMaxNb && (size_t)BH * nb * nb * sizeof(float) <= kSplitMaxScoreBytes;
}

template <int D>
cudaError_t launch_select(int32_t BH, int32_t nb, int32_t topk, int32_t include_diag, const float* qbar,
                          const float* kbar, float* scores, int32_t* sel, int32_t* lens, cudaStream_t s) {
    if (scores == nullptr) return launch_select_rpc<D, 8>(BH, nb, topk, include_diag, qbar, kbar, sel, lens, s);
    const size_t smem = sizeof(float) * (size_t)(kScoreTQ + kScoreTK) * (D + 4);
    cudaError_t e = cudaFuncSetAttribute(score_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((nb + kScoreTQ - 1) / kScoreTQ), (unsigned)((nb + kScoreTK - 1) / kScoreTK), (unsigned)BH);
    score_kernel<D><<<grid, 256, smem, s>>>(qbar, kbar, nb, scores);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t R = (int64_t)BH * nb;
    const size_t smem_sel = sizeof(uint32_t) * 8 * (64 + (size_t)((nb + 31) >> 5));
    select_kernel<<<(unsigned)((R + 7) / 8), 256, smem_sel, s>>>(scores, R, nb, topk, include_diag, sel, lens);
    return cudaGetLastError();
}

}  // namespace

size_t topk_workspace_bytes(int32_t BH, int32_t nb, int32_t D, int32_t topk) {
    const size_t R = (size_t)BH * nb;
    return 2 * align256(R * D * sizeof(float)) + align256(R * (topk + 1) * sizeof(int32_t)) +
           align256(R * sizeof(int32_t)) + (use_split(BH, nb) ? align256(R * nb * sizeof(float)) : 0);
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
    w += align256((size_t)R * sizeof(int32_t));
    float* scores = use_split(BH, nb) ? reinterpret_cast<float*>(w) : nullptr;
    cudaError_t e = (D == 128) ? launch_pool<128>(block, R, q, k, qbar, kbar, stream)
                               : launch_pool<64>(block, R, q, k, qbar, kbar, stream);
    if (e != cudaSuccess) return e;
    e = (D == 128) ? launch_select<128>(BH, nb, topk, include_diag, qbar, kbar, scores, sel, lens, stream)
                   : launch_select<64>(BH, nb, topk, include_diag, qbar, kbar, scores, sel, lens, stream);
    if (e != cudaSuccess) return e;
    if ((e = launch_row_ptr_scan(lens, R, row_ptr, stream)) != cudaSuccess) return e;
    compact_kernel<<<(unsigned)((R + 255) / 256), 256, 0, stream>>>(sel, lens, row_ptr, R, topk, col_idx);
    return cudaGetLastError();
}

}  // namespace bsa
