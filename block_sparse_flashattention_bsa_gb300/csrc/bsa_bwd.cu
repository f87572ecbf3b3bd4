// bsa_bwd.cu -- block-sparse attention backward on the device.
//
// Training differentiates through the sparse mask, which the backward pass
// reuses ("How Do Sparse Attention Kernels Work in GPU Clusters?", FAQ on
// training versus inference).  For L = sum(dO * O), with P the softmax
// weights the forward used (rebuilt from its LSE):
//   dP = dO V^T,  dS = P o (dP - Dv),  Dv = rowsum(dO o O),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
//
// Kernels (one pass each, stream-ordered):
//   tcsr_count / row_ptr scan / tcsr_fill  the block CSR transposed: for every
//        key block, the query blocks whose rows list it (causal: j <= i);
//   bwd_prep_kernel                       Dv per query row;
//   bsa_bwd_kernel<D>                     one CTA per key block j: K_j and V_j
//        stay in shared memory; for each listed query block i, S = Q K^T and
//        dP = dO V^T go to TMEM, the row warps form P and dS in shared memory,
//        then dV += P^T dO and dK += dS^T Q accumulate in TMEM and dQ_i = dS K
//        (in dP's columns) is added to an fp32 buffer by bulk tensor
//        reductions of 32 x 32 blocks staged in the P tile.  Q is double
//        buffered and dQ does not share TMEM with S, so the next query block's
//        Q is resident and its S product runs while dQ_i is read out, and its
//        dO is copied in while dK_i and dQ_i are computed;
//   bwd_dq_kernel                         dQ = scale * buffer, to bf16.
// Block 128, and block 64 in a padded form: a 64-token block fills half of a
// 128-row tile (the other half is read from outside the tensor, as zeros),
// and the padded rows and key columns are masked out of P.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

#include <cuda_bf16.h>

namespace bsa {

namespace {

constexpr int kBwdThreads = 192;  // warps 0-3: row math, 4: producer, 5: MMA
constexpr int kBwdProducer = 4;
constexpr int kBwdMma = 5;

template <int D>
struct BCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int BOX = 128 * 128;     // one 64-column (128-byte) box of a 128-row tile
    static constexpr int TILE = NBOX * BOX;   // a [128][D] bf16 tile: K, V, Q, dO
    static constexpr int PTILE = 2 * BOX;     // a [128][128] bf16 tile: P, dS (boxes of 64 keys)
    // K, V, two Q buffers, dO, P, dS
    static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE, OFF_DO = 4 * TILE;
    static constexpr int OFF_P = 5 * TILE, OFF_DS = 5 * TILE + PTILE;
    // While dQ_i is read out the P and dS tiles are idle: row warp w stages
    // 32-row x 32-column fp32 blocks of dQ in its own rows of them, 4 KB in
    // each 64-key box: P box 0, P box 1, dS box 0, dS box 1.
    static constexpr int SLAB = 32 * 32 * 4;
    static_assert(D / 32 <= 4, "one staging slab per dQ chunk: two in P, two in dS");
    static constexpr int OFF_CTRL = 5 * TILE + 2 * PTILE;
    static constexpr int SMEM = OFF_CTRL + 256;
    // TMEM columns: S, dP, dV, dK; dQ reuses dP's columns
    static constexpr int C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D, C_DQ = 128;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t ID_S = idesc_bf16_f32_ab(128, 128, false, false);  // S, dP
    static constexpr uint32_t ID_KV = idesc_bf16_f32_ab(128, D, true, true);     // dV, dK: A = P^T / dS^T
    static constexpr uint32_t ID_Q = idesc_bf16_f32_ab(128, D, false, true);     // dQ: B = K, MN-major
    static constexpr uint32_t TX_TILE = 128 * D * 2;
    static_assert(SMEM <= 232448, "shared memory overflow");
};

struct BCtrl {
    uint64_t kv_full, q_full[2], q_empty[2], do_full, do_empty, s_full, dp_full, ps_full, dq_full, dq_free, kv_done,
        staged, drain;
    uint32_t tmem_base;
    int32_t abort;
};

struct BwdParams {
    const int32_t* trp;  // transposed CSR: query blocks of key block r in tci[trp[r] .. trp[r+1])
    const int32_t* tci;
    int64_t tci_cap;     // entries tci holds
    const float* lse;    // [BH, N]
    const float* dvec;   // [BH, N]
    float* dq_acc;       // [BH, N, D] fp32
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int32_t* err;
    int32_t N, nb, causal;
    float scale, scale_log2;
};

__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// ---------------------------------------------------------------- transposed CSR
__global__ void tcsr_count_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
                                  int64_t R, int32_t nb, int32_t causal, int32_t* __restrict__ cnt, int32_t* err) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bh = r / nb;
        const int32_t i = (int32_t)(r - bh * nb);
        int32_t beg = row_ptr[r], end = row_ptr[r + 1];
        if (end < beg) {
            atomicOr(err, ERR_BAD_ROW);
            end = beg;
        }
        for (int32_t e = beg; e < end; ++e) {
            const int32_t j = col_idx[e];
            if ((unsigned)j >= (unsigned)nb) {
                atomicOr(err, ERR_BAD_COL);
            } else if (!(causal && j > i)) {
                atomicAdd(&cnt[bh * nb + j], 1);
            }
        }
    }
}

__global__ void tcsr_fill_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx, int64_t R,
                                 int32_t nb, int32_t causal, const int32_t* __restrict__ trp,
                                 int32_t* __restrict__ cursor, int32_t* __restrict__ tci, int64_t cap,
                                 int32_t* err) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bh = r / nb;
        const int32_t i = (int32_t)(r - bh * nb);
        const int32_t beg = row_ptr[r];
        int32_t end = row_ptr[r + 1];
        if (end < beg) end = beg;
        for (int32_t e = beg; e < end; ++e) {
            const int32_t j = col_idx[e];
            if ((unsigned)j < (unsigned)nb && !(causal && j > i)) {
                const int64_t c = bh * nb + j;
                const int64_t pos = (int64_t)trp[c] + atomicAdd(&cursor[c], 1);
                if (pos < cap) tci[pos] = i;  // more entries than col_capacity: dropped and flagged
                else atomicOr(err, ERR_CAPACITY);
            }
        }
    }
}

// ---------------------------------------------------------------- Dv = rowsum(dO o O)
__global__ void bwd_prep_kernel(const __nv_bfloat162* __restrict__ o, const __nv_bfloat162* __restrict__ dout,
                                float* __restrict__ dvec, int64_t rows, int32_t D) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int half = D >> 1;
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        float acc = 0.f;
        for (int x = lane; x < half; x += 32) {
            const float2 a = __bfloat1622float2(o[r * half + x]);
            const float2 b = __bfloat1622float2(dout[r * half + x]);
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (lane == 0) dvec[r] = acc;
    }
}

// ---------------------------------------------------------------- dQ to bf16
__global__ void bwd_dq_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, int64_t n4, float scale) {
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = acc[x];
        dq[x] = make_uint2(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale));
    }
}

// ---------------------------------------------------------------- main kernel
// KB: tokens per block (128, or 64 padded to the 128-row tile).
template <int D, int KB>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bsa_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                   const __grid_constant__ CUtensorMap tdv, const BwdParams p) {
    using C = BCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_LAUNCH);
        return;
    }
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint8_t* sQ = smem + C::OFF_Q;  // buffer b at sQ + b * TILE
    uint8_t* sDO = smem + C::OFF_DO;
    uint8_t* sP = smem + C::OFF_P;
    uint8_t* sDS = smem + C::OFF_DS;
    BCtrl* c = reinterpret_cast<BCtrl*>(smem + C::OFF_CTRL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x;  // key block (b * H + h) * nb + j
    const int bh = item / p.nb;
    const int j = item - bh * p.nb;
    const int row0 = bh * p.N;
    const int beg = p.trp[item];
    int n = p.trp[item + 1] - beg;
    if ((int64_t)beg + n > p.tci_cap) n = (int64_t)beg < p.tci_cap ? (int)(p.tci_cap - beg) : 0;  // flagged by the fill

    if (threadIdx.x == 0) {
        mbar_init(&c->kv_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c->q_full[b], 1);
            mbar_init(&c->q_empty[b], 1);
        }
        mbar_init(&c->do_full, 1);
        mbar_init(&c->do_empty, 1);
        mbar_init(&c->s_full, 1);
        mbar_init(&c->dp_full, 1);
        mbar_init(&c->ps_full, 4);
        mbar_init(&c->dq_full, 1);
        mbar_init(&c->dq_free, 4);
        mbar_init(&c->kv_done, 1);
        mbar_init(&c->staged, 4);
        mbar_init(&c->drain, 1);
        c->abort = 0;
        fence_mbar_init();
    }
    if (warp == kBwdMma) {
        tmem_alloc(&c->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c->tmem_base;
    volatile int* abort = &c->abort;

    if (warp == kBwdProducer && n > 0) {
        const bool leader = elect_one();
        if (leader) {
            mbar_arrive_expect_tx(&c->kv_full, 2 * C::TX_TILE);
#pragma unroll
            for (int b = 0; b < C::NBOX; ++b) {
                tma_load_2d(sK + b * C::BOX, &tk, &c->kv_full, b * 64, row0 + j * KB);
                tma_load_2d(sV + b * C::BOX, &tv, &c->kv_full, b * 64, row0 + j * KB);
                if (KB == 64) {  // rows 64-127: zeros, read from outside the tensor
                    tma_load_2d(sK + b * C::BOX + 64 * 128, &tk, &c->kv_full, b * 64, -64);
                    tma_load_2d(sV + b * C::BOX + 64 * 128, &tv, &c->kv_full, b * 64, -64);
                }
            }
        }
        // Q_t goes to buffer t & 1 once dK of step t - 2 has read it; dO_t to
        // its one buffer once dV of step t - 1 has read it.
        int nq0 = 0, nq1 = 0, nd = 0;  // copies issued per buffer
        auto load_q = [&](int t) {
            const int b = t & 1, i = p.tci[beg + t];
            uint8_t* dst = sQ + b * C::TILE;
            if (leader) {
                mbar_arrive_expect_tx(&c->q_full[b], C::TX_TILE);
#pragma unroll
                for (int x = 0; x < C::NBOX; ++x) {
                    tma_load_2d(dst + x * C::BOX, &tq, &c->q_full[b], x * 64, row0 + i * KB);
                    if (KB == 64) tma_load_2d(dst + x * C::BOX + 64 * 128, &tq, &c->q_full[b], x * 64, -64);
                }
            }
            if (b) ++nq1; else ++nq0;
        };
        auto load_do = [&](int t) {
            const int i = p.tci[beg + t];
            if (leader) {
                mbar_arrive_expect_tx(&c->do_full, C::TX_TILE);
#pragma unroll
                for (int x = 0; x < C::NBOX; ++x) {
                    tma_load_2d(sDO + x * C::BOX, &tdo, &c->do_full, x * 64, row0 + i * KB);
                    if (KB == 64) tma_load_2d(sDO + x * C::BOX + 64 * 128, &tdo, &c->do_full, x * 64, -64);
                }
            }
            ++nd;
        };
        load_q(0);
        load_do(0);
        if (n > 1) load_q(1);
        for (int t = 1; t < n; ++t) {
            if (!wwait(&c->do_empty, (t - 1) & 1, abort)) break;
            load_do(t);
            if (t + 1 < n) {
                if (!wwait(&c->q_empty[(t + 1) & 1], (((t + 1) >> 1) - 1) & 1, abort)) break;
                load_q(t + 1);
            }
        }
        if (*abort && leader) {
            // the copies in flight must land before the CTA exits
            mbar_wait_drain(&c->kv_full, 0);
            if (nq0 > 0) mbar_wait_drain(&c->q_full[0], (nq0 - 1) & 1);
            if (nq1 > 0) mbar_wait_drain(&c->q_full[1], (nq1 - 1) & 1);
            if (nd > 0) mbar_wait_drain(&c->do_full, (nd - 1) & 1);
        }
    } else if (warp == kBwdMma && n > 0) {
        const bool leader = elect_one();
        constexpr uint64_t KDESC = sdesc_sw128_base(16, 1024);       // K-major, 128-byte swizzle
        constexpr uint64_t MDESC = sdesc_sw128_base(C::BOX, 1024);   // MN-major: 64-element groups a box apart
        const uint64_t k_k = KDESC + (smem_u32(sK) >> 4);
        const uint64_t do_k = KDESC + (smem_u32(sDO) >> 4), v_k = KDESC + (smem_u32(sV) >> 4);
        const uint64_t ds_k = KDESC + (smem_u32(sDS) >> 4);
        const uint64_t p_m = MDESC + (smem_u32(sP) >> 4), ds_m = MDESC + (smem_u32(sDS) >> 4);
        const uint64_t do_m = MDESC + (smem_u32(sDO) >> 4);
        const uint64_t k_m = MDESC + (smem_u32(sK) >> 4);
        bool ok = wwait(&c->kv_full, 0, abort);
        for (int t = 0; t < n && ok; ++t) {
            const int b = t & 1;
            const uint64_t q_k = KDESC + (smem_u32(sQ + b * C::TILE) >> 4);
            const uint64_t q_m = MDESC + (smem_u32(sQ + b * C::TILE) >> 4);
            // S = Q K^T: S's columns were read before step t - 1's P was published
            if (!wwait(&c->q_full[b], (t >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                // K-major operands: 16 columns (32 bytes) per MMA inside a box, the next box every 4
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                    mma_ss(tmem + C::C_S, q_k + off, k_k + off, C::ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit(&c->s_full);
            }
            __syncwarp();
            // dP = dO V^T, into the columns dQ of step t - 1 occupied until read out
            if (!wwait(&c->do_full, t & 1, abort) || (t > 0 && !wwait(&c->dq_free, (t - 1) & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                    mma_ss(tmem + C::C_DP, do_k + off, v_k + off, C::ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit(&c->dp_full);
            }
            __syncwarp();
            if (!wwait(&c->ps_full, t & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                // dV += P^T dO, dK += dS^T Q: the reduction runs over the 128 query
                // rows, 16 (2048 bytes of every box) per MMA
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const uint64_t off = (uint64_t)((kq * 2048) >> 4);
                    mma_ss(tmem + C::C_DV, p_m + off, do_m + off, C::ID_KV, (t > 0 || kq > 0) ? 1u : 0u);
                }
                mma_commit(&c->do_empty);
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const uint64_t off = (uint64_t)((kq * 2048) >> 4);
                    mma_ss(tmem + C::C_DK, ds_m + off, q_m + off, C::ID_KV, (t > 0 || kq > 0) ? 1u : 0u);
                }
                mma_commit(&c->q_empty[b]);
                // dQ_i = dS K: the reduction runs over the 128 keys
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t aoff = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                    const uint64_t boff = (uint64_t)((kk * 2048) >> 4);
                    mma_ss(tmem + C::C_DQ, ds_k + aoff, k_m + boff, C::ID_Q, kk > 0 ? 1u : 0u);
                }
                mma_commit(&c->dq_full);
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(&c->kv_done);
            mma_commit(&c->drain);
            mbar_wait_drain(&c->drain, 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        const int tid = threadIdx.x;  // query row (steps) or key row (end) = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t xr = (uint32_t)(tid & 7);
        const bool row_real = KB == 128 || tid < KB;  // padded rows of a 64-token block: no data
        bool ok = true;
        for (int t = 0; t < n && ok; ++t) {
            const int i = p.tci[beg + t];
            const int64_t row = (int64_t)row0 + (int64_t)i * KB + tid;
            const float lse2 = row_real ? p.lse[row] * 1.4426950408889634f : 0.f;
            const float dv_row = row_real ? p.dvec[row] : 0.f;
            const f2 sl2 = {p.scale_log2, p.scale_log2}, nl2 = {-lse2, -lse2}, ndv = {-dv_row, -dv_row};
            const bool diag = p.causal && i == j;
            if (!wwait(&c->s_full, t & 1, abort) || !wwait(&c->dp_full, t & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // this warp's rows of P and dS held its dQ blocks of step t - 1:
            // the reductions must have read them
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t s[32], dp[32];
                tmem_ld32(tmem + lane_base + C::C_S + ch * 32, s);
                tmem_ld32(tmem + lane_base + C::C_DP + ch * 32, dp);
                tmem_wait_ld();
                reg_fence(s);
                reg_fence(dp);
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int col = ch * 32 + 2 * x;
                    const f2 tt = fma2({__uint_as_float(s[2 * x]), __uint_as_float(s[2 * x + 1])}, sl2, nl2);
                    float p0 = ex2_approx(tt.x), p1 = ex2_approx(tt.y);
                    if (diag && col > tid) p0 = 0.f;          // key token after the query token
                    if (diag && col + 1 > tid) p1 = 0.f;
                    if (!row_real || col >= KB) p0 = 0.f;     // padding of a 64-token block
                    if (!row_real || col + 1 >= KB) p1 = 0.f;
                    pk[x] = pack_bf16x2(p0, p1);
                    const f2 ds = mul2({p0, p1}, add2({__uint_as_float(dp[2 * x]), __uint_as_float(dp[2 * x + 1])}, ndv));
                    dk[x] = pack_bf16x2(ds.x, ds.y);
                }
                // [query][key] bf16, 128-byte swizzle, boxes of 64 keys
                uint8_t* bp = sP + (ch >> 1) * C::BOX + tid * 128;
                uint8_t* bd = sDS + (ch >> 1) * C::BOX + tid * 128;
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    const uint32_t sw = ((uint32_t)((ch & 1) * 4 + v4) ^ xr) << 4;
                    *reinterpret_cast<uint4*>(bp + sw) = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    *reinterpret_cast<uint4*>(bd + sw) = make_uint4(dk[4 * v4], dk[4 * v4 + 1], dk[4 * v4 + 2], dk[4 * v4 + 3]);
                }
            }
            fence_proxy_async_smem();  // P and dS are read by the tensor cores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->ps_full);
            if (!wwait(&c->dq_full, t & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // dQ_i: each 32-column chunk of this warp's 32 rows goes through a
            // swizzled slab (16-byte chunk c of slab row r at r * 128 + ((c ^ (r & 7)) << 4))
            // and is added to the fp32 buffer by one bulk tensor reduction, so
            // the L2 sees whole lines.  The slabs are this warp's rows of the P
            // and dS tiles (both idle until the next step's row math, which
            // first waits for these reductions to have read them): one per
            // chunk, so no chunk waits for an earlier reduction.
            if (warp * 32 < KB) {  // padded rows add nothing
                uint32_t o[2][32];
                tmem_ld32(tmem + lane_base + C::C_DQ, o[0]);
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    const int cb = ch & 1;
                    tmem_wait_ld();
                    if (ch + 1 < D / 32) tmem_ld32(tmem + lane_base + C::C_DQ + (ch + 1) * 32, o[cb ^ 1]);
                    reg_fence(o[cb]);
                    uint8_t* slab = (ch < 2 ? sP : sDS) + (ch & 1) * C::BOX + warp * C::SLAB;
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4)
                        *reinterpret_cast<uint4*>(slab + lane * 128 + ((c4 ^ (lane & 7)) << 4)) =
                            make_uint4(o[cb][4 * c4], o[cb][4 * c4 + 1], o[cb][4 * c4 + 2], o[cb][4 * c4 + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_2d(&tdq, slab, ch * 32, row0 + i * KB + warp * 32);
                        bulk_commit_group();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->dq_free);
        }
        if (lane == 0) bulk_wait_read_all();  // the dQ reductions have read their slabs
        __syncwarp();
        // dK and dV of this key block (zero when no query block lists it).
        // Thread tid owns key row tid: its rows of dK (x scale) and dV are
        // staged as bf16 in the two Q buffers (idle once every MMA has
        // completed) in the 128-byte swizzled box layout of the dK / dV
        // tensor maps, and written by one TMA store per 64-column box.
        if (n == 0) {
            if (row_real) {
                const int64_t krow = (int64_t)row0 + (int64_t)j * KB + tid;
                uint4* gk = reinterpret_cast<uint4*>(p.dk + krow * D);
                uint4* gv = reinterpret_cast<uint4*>(p.dv + krow * D);
#pragma unroll 1
                for (int x = 0; x < D / 8; ++x) {
                    gk[x] = make_uint4(0u, 0u, 0u, 0u);
                    gv[x] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        } else {
            uint8_t* stk = sQ;
            uint8_t* stv = sQ + C::TILE;
            if (ok && wwait(&c->kv_done, 0, abort) && row_real) {
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t a[32], b[32];
                    tmem_ld32(tmem + lane_base + C::C_DK + ch * 32, a);
                    tmem_ld32(tmem + lane_base + C::C_DV + ch * 32, b);
                    tmem_wait_ld();
                    reg_fence(a);
                    reg_fence(b);
                    const int off = (ch >> 1) * C::BOX + tid * 128;
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint32_t ka[4], va[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int x = v4 * 8 + 2 * u;
                            ka[u] = pack_bf16x2(__uint_as_float(a[x]) * p.scale, __uint_as_float(a[x + 1]) * p.scale);
                            va[u] = pack_bf16x2(__uint_as_float(b[x]), __uint_as_float(b[x + 1]));
                        }
                        const int sw = (((ch & 1) * 4 + v4) ^ (int)xr) << 4;
                        *reinterpret_cast<uint4*>(stk + off + sw) = make_uint4(ka[0], ka[1], ka[2], ka[3]);
                        *reinterpret_cast<uint4*>(stv + off + sw) = make_uint4(va[0], va[1], va[2], va[3]);
                    }
                }
            }
            fence_proxy_async_smem();  // read next by the TMA unit
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->staged);
            if (warp == 0 && wwait(&c->staged, 0, abort) && lane == 0 && !*abort) {
#pragma unroll
                for (int x = 0; x < C::NBOX; ++x) {
                    tma_store_2d(&tdk, stk + x * C::BOX, x * 64, row0 + j * KB);
                    tma_store_2d(&tdv, stv + x * C::BOX, x * 64, row0 + j * KB);
                }
                bulk_commit_group();
                bulk_wait_read_all();  // the staging must be read before the CTA exits
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && c->abort) atomicOr(p.err, ERR_TIMEOUT);
}

}  // namespace

size_t bwd_workspace_bytes(int32_t BH, int32_t N, int32_t D, int32_t nb, int64_t col_capacity) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t R = (size_t)BH * nb;
    return a((R + 1) * 4) + a(R * 4) + a((size_t)col_capacity * 4 + 4) + a((size_t)BH * N * 4) +
           a((size_t)BH * N * D * 4);
}

size_t bwd_dq_acc_offset(int32_t BH, int32_t N, int32_t nb, int64_t col_capacity) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t R = (size_t)BH * nb;
    return a((R + 1) * 4) + a(R * 4) + a((size_t)col_capacity * 4 + 4) + a((size_t)BH * N * 4);
}

cudaError_t launch_backward(const BwdLaunch& L, cudaStream_t s) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const int64_t R = (int64_t)L.BH * L.nb;
    const int64_t rows = (int64_t)L.BH * L.N;
    char* w = static_cast<char*>(L.workspace);
    int32_t* trp = reinterpret_cast<int32_t*>(w);
    w += a((size_t)(R + 1) * 4);
    int32_t* cursor = reinterpret_cast<int32_t*>(w);
    w += a((size_t)R * 4);
    int32_t* tci = reinterpret_cast<int32_t*>(w);
    w += a((size_t)L.col_capacity * 4 + 4);
    float* dvec = reinterpret_cast<float*>(w);
    w += a((size_t)rows * 4);
    float* dq_acc = reinterpret_cast<float*>(w);
    cudaError_t e;
    if ((e = cudaMemsetAsync(trp, 0, (size_t)(R + 1) * 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(cursor, 0, (size_t)R * 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dq_acc, 0, (size_t)rows * L.D * 4, s)) != cudaSuccess) return e;
    int64_t blocks = (R + 255) / 256;
    if (blocks > 8 * (int64_t)L.sm_count) blocks = 8 * (int64_t)L.sm_count;
    tcsr_count_kernel<<<(unsigned)blocks, 256, 0, s>>>(L.row_ptr, L.col_idx, R, L.nb, L.causal, trp + 1, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_row_ptr_scan(trp + 1, R, trp, s)) != cudaSuccess) return e;
    tcsr_fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(L.row_ptr, L.col_idx, R, L.nb, L.causal, trp, cursor, tci,
                                                      L.col_capacity, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int64_t pblocks = (rows + 7) / 8;
    if (pblocks > 16 * (int64_t)L.sm_count) pblocks = 16 * (int64_t)L.sm_count;
    bwd_prep_kernel<<<(unsigned)pblocks, 256, 0, s>>>(static_cast<const __nv_bfloat162*>(L.out),
                                                      static_cast<const __nv_bfloat162*>(L.dout), dvec, rows, L.D);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    BwdParams p;
    p.trp = trp;
    p.tci = tci;
    p.tci_cap = L.col_capacity;
    p.lse = L.lse;
    p.dvec = dvec;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(L.dk);
    p.dv = static_cast<__nv_bfloat16*>(L.dv);
    p.err = L.err;
    p.N = L.N;
    p.nb = L.nb;
    p.causal = L.causal;
    p.scale = L.scale;
    p.scale_log2 = L.scale * 1.4426950408889634f;
    auto run = [&](auto kernel, int smem) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        kernel<<<(unsigned)R, kBwdThreads, smem, s>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, L.tdk, L.tdv, p);
        return cudaGetLastError();
    };
    if (L.block == 128)
        e = L.D == 128 ? run(bsa_bwd_kernel<128, 128>, BCfg<128>::SMEM) : run(bsa_bwd_kernel<64, 128>, BCfg<64>::SMEM);
    else
        e = L.D == 128 ? run(bsa_bwd_kernel<128, 64>, BCfg<128>::SMEM) : run(bsa_bwd_kernel<64, 64>, BCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n4 = rows * L.D / 4;
    int64_t cblocks = (n4 + 255) / 256;
    if (cblocks > 16 * (int64_t)L.sm_count) cblocks = 16 * (int64_t)L.sm_count;
    bwd_dq_kernel<<<(unsigned)cblocks, 256, 0, s>>>(reinterpret_cast<const float4*>(dq_acc),
                                                    static_cast<uint2*>(L.dq), n4, L.scale);
    return cudaGetLastError();
}

}  // namespace bsa
