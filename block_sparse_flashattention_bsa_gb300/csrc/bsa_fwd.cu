// bsa_fwd.cu -- persistent block-sparse FlashAttention forward for sm_103a.
//
// Method: "How Do Sparse Attention Kernels Work in GPU Clusters? A 2026 Field
// Guide", section "How Does Flash-MSA Sparse Attention Work?" (for each query
// block load only the active key/value blocks, FlashAttention tiling over
// them, online softmax, write the output), with the recurrence of "Flash MSA
// Sparse Attention vs Full Attention", section "The Mechanics" (running max,
// rescale of the accumulator and of the running sum, division at the end).
// Load balance: "bucket queries by sparsity level" (field guide, "When Sparse
// Kernels Break", item 1) -- work items are claimed longest row first.
//
// GB300 design (one CTA per SM, 6 warps, warp-specialised):
//   warp 4     producer: claims work items from a global counter, TMA-loads
//              the Q tile (2 buffers) and the K_j / V_j tiles of the row's
//              col_idx list into a ring of NT shared-memory tiles;
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T (tcgen05.mma, both
//              operands in shared memory, fp32 accumulator in TMEM, two S
//              buffers), then O += P_j V_j (P from TMEM, V in shared memory,
//              MN-major); completions are signalled with tcgen05.commit;
//   warps 0-3  softmax + epilogue: thread t owns query row t of the tile, so
//              row max and row sum stay inside one thread.  Reads S_j from
//              TMEM, applies the token-level causal mask on the diagonal
//              block, updates the running max (rescaling O only when the max
//              grows by more than 2^8, which keeps every exponent <= 2^8 and is
//              exact after the final division), writes P_j (bf16) to TMEM,
//              and at the end writes O / l (bf16) and LSE (fp32).
// The issue order QK_0, QK_1, PV_0, QK_2, PV_1, ... lets the softmax of block
// j overlap the tensor-core work of blocks j-1 and j+1.
//
// Every wait is bounded: on a timeout the kernel raises an abort flag, every
// role leaves its loop, in-flight copies and MMAs are drained (bounded), TMEM
// is freed and ERR_TIMEOUT is written to the device error word.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {
namespace {

constexpr int kSmemLimit = 232448;  // maximum dynamic shared memory per CTA
constexpr int kCtrlBytes = 1024;
constexpr int kAlign = 1024;        // 128-byte swizzle atoms need 1024-byte alignment
constexpr int kThreads = 192;

template <int BS, int D>
struct Cfg {
    static constexpr int M = 128;                 // MMA rows (query rows; BS = 64 pads to 128)
    static constexpr int NBOX = D / 64;           // 64 bf16 = one 128-byte swizzled row per box
    static constexpr int Q_BOX = M * 128;         // bytes of one box of the Q tile
    static constexpr int Q_BYTES = NBOX * Q_BOX;
    static constexpr int T_BOX = BS * 128;        // bytes of one box of a K or V tile
    static constexpr int T_BYTES = NBOX * T_BOX;
    static constexpr int NQ = 2;
    static constexpr int NT_FIT = (kSmemLimit - kCtrlBytes - kAlign - NQ * Q_BYTES) / T_BYTES;
    static constexpr int NT = NT_FIT > 8 ? 8 : NT_FIT;
    static constexpr int SMEM = kAlign + NQ * Q_BYTES + NT * T_BYTES + kCtrlBytes;
    // TMEM columns: S buffers, O accumulator, P buffers (bf16 pairs).
    static constexpr int S_COL = 0;
    static constexpr int O_COL = 2 * BS;
    static constexpr int P_COL = 2 * BS + D;
    static constexpr int USED_COLS = 3 * BS + D;
    static constexpr int TMEM_COLS = USED_COLS <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(M, BS, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(M, D, true);
    static constexpr uint32_t TX_BYTES = BS * D * 2;
    static_assert(NT >= 2, "shared memory ring too small");
    static_assert(USED_COLS <= 512, "TMEM overflow");
    static_assert(SMEM <= kSmemLimit, "shared memory overflow");
};

struct Ctrl {
    uint64_t item_full[4];
    uint64_t item_empty[4];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t t_full[8];
    uint64_t t_empty[8];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t pv_done[2];
    uint64_t o_free;
    uint64_t drain;
    int32_t ring[4];
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

__device__ __forceinline__ void row_range(const FwdParams& p, int item, int& beg, int& end) {
    beg = p.row_ptr[item];
    end = p.row_ptr[item + 1];
    if (end < beg) end = beg;
}

__device__ __forceinline__ bool block_ok(const FwdParams& p, int j, int i) {
    return (unsigned)j < (unsigned)p.nb && !(p.causal && j > i);
}

// ---------------------------------------------------------------- producer
template <int BS, int D>
__device__ void producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const FwdParams& p,
                         uint8_t* sQ, uint8_t* sT, Ctrl* c, volatile int* abort) {
    using C = Cfg<BS, D>;
    uint32_t tt = 0, nq = 0;
    for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it & 3;
        if (!mbar_wait(&c->item_empty[slot], ((it >> 2) & 1) ^ 1, abort)) break;
        const int w = atomicAdd(p.counter, 1);
        const int item = w < p.n_items ? p.perm[w] : -1;
        c->ring[slot] = item;
        mbar_arrive(&c->item_full[slot]);
        if (item < 0) break;
        const int bh = item / p.nb;
        const int i = item - bh * p.nb;
        const int row0 = bh * p.N;
        const uint32_t qb = it & 1;
        if (!mbar_wait(&c->q_empty[qb], ((it >> 1) & 1) ^ 1, abort)) break;
        mbar_arrive_expect_tx(&c->q_full[qb], C::TX_BYTES);
#pragma unroll
        for (int b = 0; b < C::NBOX; ++b)
            tma_load_2d(sQ + qb * C::Q_BYTES + b * C::Q_BOX, tq, &c->q_full[qb], b * 64, row0 + i * BS);
        ++nq;
        int beg = p.row_ptr[item], end = p.row_ptr[item + 1];
        if (end < beg) {
            atomicOr(p.err, ERR_BAD_ROW);
            end = beg;
        }
        bool ok = true;
        for (int e = beg; e < end && ok; ++e) {
            const int j = p.col_idx[e];
            if ((unsigned)j >= (unsigned)p.nb) {
                atomicOr(p.err, ERR_BAD_COL);
                continue;
            }
            if (p.causal && j > i) continue;
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t t = tt % C::NT;
                if (!mbar_wait(&c->t_empty[t], ((tt / C::NT) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&c->t_full[t], C::TX_BYTES);
#pragma unroll
                for (int b = 0; b < C::NBOX; ++b)
                    tma_load_2d(sT + t * C::T_BYTES + b * C::T_BOX, kv ? tv : tk, &c->t_full[t], b * 64,
                                row0 + j * BS);
                ++tt;
            }
        }
        if (!ok) break;
    }
    if (*abort) {
        // Drain the copies still in flight before the CTA exits.
        for (uint32_t n = (tt > (uint32_t)C::NT ? tt - C::NT : 0); n < tt; ++n)
            mbar_wait_drain(&c->t_full[n % C::NT], (n / C::NT) & 1);
        for (uint32_t n = (nq > 2 ? nq - 2 : 0); n < nq; ++n) mbar_wait_drain(&c->q_full[n & 1], (n >> 1) & 1);
    }
}

// ---------------------------------------------------------------- MMA issuer
template <int BS, int D>
__device__ bool issue_pv(const FwdParams& p, uint8_t* sT, Ctrl* c, uint32_t tmem, volatile int* abort, uint32_t gp,
                         uint32_t vseq, bool first, uint32_t it) {
    using C = Cfg<BS, D>;
    const uint32_t pb = gp & 1;
    if (!mbar_wait(&c->p_full[pb], (gp >> 1) & 1, abort)) return false;
    const uint32_t vt = vseq % C::NT;
    if (!mbar_wait(&c->t_full[vt], (vseq / C::NT) & 1, abort)) return false;
    if (first && it > 0 && !mbar_wait(&c->o_free, (it - 1) & 1, abort)) return false;
    tc_fence_after();
    const uint32_t v_addr = smem_u32(sT + vt * C::T_BYTES);
#pragma unroll
    for (int kk = 0; kk < BS / 16; ++kk) {
        // V tile is [keys][D]: MN-major B operand.  16 keys per MMA = 2 groups
        // of 8 swizzled 128-byte rows (SBO = 1024); the next 64 columns of D
        // live in the next box (LBO = box size).
        const uint64_t bdesc = smem_desc_sw128(v_addr + kk * 16 * 128, C::T_BOX, 1024);
        mma_ts(tmem + C::O_COL, tmem + C::P_COL + pb * (BS / 2) + kk * 8, bdesc, C::IDESC_PV,
               (first && kk == 0) ? 0u : 1u);
    }
    mma_commit(&c->pv_done[pb]);
    mma_commit(&c->t_empty[vt]);
    return true;
}

template <int BS, int D>
__device__ void mma_issuer(const FwdParams& p, uint8_t* sQ, uint8_t* sT, Ctrl* c, uint32_t tmem,
                           volatile int* abort) {
    using C = Cfg<BS, D>;
    uint32_t g = 0, tt = 0;
    bool ok = true;
    for (uint32_t it = 0; ok; ++it) {
        const uint32_t slot = it & 3;
        if (!mbar_wait(&c->item_full[slot], (it >> 2) & 1, abort)) break;
        const int item = c->ring[slot];
        mbar_arrive(&c->item_empty[slot]);
        if (item < 0) break;
        const int i = item % p.nb;
        const uint32_t qb = it & 1;
        if (!mbar_wait(&c->q_full[qb], (it >> 1) & 1, abort)) break;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(sQ + qb * C::Q_BYTES);
        int beg, end;
        row_range(p, item, beg, end);
        uint32_t s = 0, pend_g = 0, pend_v = 0;
        for (int e = beg; e < end; ++e) {
            const int j = p.col_idx[e];
            if (!block_ok(p, j, i)) continue;
            const uint32_t kseq = tt, vseq = tt + 1;
            tt += 2;
            const uint32_t kt = kseq % C::NT;
            if (!mbar_wait(&c->t_full[kt], (kseq / C::NT) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sb = g & 1;
            const uint32_t k_addr = smem_u32(sT + kt * C::T_BYTES);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                // Q and K tiles are K-major with 128-byte swizzle: 16 columns
                // (32 bytes) per MMA inside a box, next box every 4 steps.
                const uint64_t adesc = smem_desc_sw128(q_addr + (kk >> 2) * C::Q_BOX + (kk & 3) * 32, 16, 1024);
                const uint64_t bdesc = smem_desc_sw128(k_addr + (kk >> 2) * C::T_BOX + (kk & 3) * 32, 16, 1024);
                mma_ss(tmem + C::S_COL + sb * BS, adesc, bdesc, C::IDESC_QK, kk > 0 ? 1u : 0u);
            }
            mma_commit(&c->s_full[sb]);
            mma_commit(&c->t_empty[kt]);
            if (s > 0 && !issue_pv<BS, D>(p, sT, c, tmem, abort, pend_g, pend_v, s == 1, it)) {
                ok = false;
                break;
            }
            pend_g = g;
            pend_v = vseq;
            ++g;
            ++s;
        }
        if (!ok) break;
        if (s > 0 && !issue_pv<BS, D>(p, sT, c, tmem, abort, pend_g, pend_v, s == 1, it)) break;
        mma_commit(&c->q_empty[qb]);
    }
    // Every MMA this thread issued must finish before TMEM is freed.
    mma_commit(&c->drain);
    mbar_wait_drain(&c->drain, 0);
}

// ---------------------------------------------------------------- softmax
template <int BS, int D>
__device__ void softmax_role(const FwdParams& p, Ctrl* c, uint32_t tmem, volatile int* abort) {
    using C = Cfg<BS, D>;
    const int tid = threadIdx.x;  // 0..127 = TMEM lane = query row in the tile
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::S_COL;
    const uint32_t t_o = tmem + lane_base + C::O_COL;
    const uint32_t t_p = tmem + lane_base + C::P_COL;
    const bool row_valid = tid < BS;
    const float sl = p.scale_log2;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t it = 0; ok; ++it) {
        const uint32_t slot = it & 3;
        if (!warp_wait(&c->item_full[slot], (it >> 2) & 1, abort)) break;
        const int item = c->ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->item_empty[slot]);
        if (item < 0) break;
        const int bh = item / p.nb;
        const int i = item - bh * p.nb;
        int beg, end;
        row_range(p, item, beg, end);
        // l: fp32 sum of the exponentials (for LSE); lr: sum of the same
        // values after rounding to bf16, i.e. of the weights the PV MMA
        // actually uses, so O / lr is an exact convex combination of them.
        float m_used = -INFINITY, l = 0.f, lr = 0.f;
        uint32_t s = 0;
        for (int e = beg; e < end; ++e) {
            const int j = p.col_idx[e];
            if (!block_ok(p, j, i)) continue;
            const uint32_t sb = g & 1;
            if (!warp_wait(&c->s_full[sb], (g >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[BS / 32][32];
#pragma unroll
            for (int ch = 0; ch < BS / 32; ++ch) tmem_ld32(t_s + sb * BS + ch * 32, sr[ch]);
            tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < BS / 32; ++ch) reg_fence(sr[ch]);
            if (p.causal && j == i) {
                // token-level causal mask inside the diagonal block
#pragma unroll
                for (int ch = 0; ch < BS / 32; ++ch)
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (ch * 32 + x > tid) sr[ch][x] = __float_as_uint(-INFINITY);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < BS / 32; ++ch)
#pragma unroll
                for (int x = 0; x < 32; x += 4) {
                    mx0 = fmaxf(mx0, __uint_as_float(sr[ch][x]));
                    mx1 = fmaxf(mx1, __uint_as_float(sr[ch][x + 1]));
                    mx2 = fmaxf(mx2, __uint_as_float(sr[ch][x + 2]));
                    mx3 = fmaxf(mx3, __uint_as_float(sr[ch][x + 3]));
                }
            const float mnew = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl;
            float alpha = 1.f;
            bool need = false;
            if (s == 0) {
                m_used = mnew;
            } else if (mnew > m_used + 8.f) {
                alpha = ex2_approx(m_used - mnew);
                m_used = mnew;
                l *= alpha;
                lr *= alpha;
                need = true;
            }
            if (__any_sync(0xffffffffu, need)) {
                // The running max grew by more than 2^8 for some row of this
                // warp: rescale its rows of O once PV_{g-1} has landed.
                const uint32_t gp = g - 1;
                if (!warp_wait(&c->pv_done[gp & 1], (gp >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(t_o + ch * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
#pragma unroll
                    for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                    tmem_st32(t_o + ch * 32, o);
                }
                tmem_wait_st();
            }
            const float mo = (m_used == -INFINITY) ? 0.f : m_used;
            // P buffer sb is free once PV_{g-2} has completed.
            if (g >= 2 && !warp_wait(&c->pv_done[sb], ((g - 2) >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            float sum0 = 0.f, sum1 = 0.f, rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int ch = 0; ch < BS / 32; ++ch) {
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sr[ch][2 * x]), sl, -mo));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sr[ch][2 * x + 1]), sl, -mo));
                    sum0 += p0;
                    sum1 += p1;
                    pk[x] = pack_bf16x2(p0, p1);
                    rs0 += __uint_as_float(pk[x] << 16);
                    rs1 += __uint_as_float(pk[x] & 0xffff0000u);
                }
                tmem_st16(t_p + sb * (BS / 2) + ch * 16, pk);
            }
            l += sum0 + sum1;
            lr += rs0 + rs1;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->p_full[sb]);
            ++g;
            ++s;
        }
        if (!ok) break;
        // ---- epilogue: O / l -> bf16, LSE
        float lse_v = -INFINITY;
        const size_t row = (size_t)bh * p.N + (size_t)i * BS + tid;
        uint4* dst = reinterpret_cast<uint4*>(out + row * D);
        if (s > 0) {
            const uint32_t gp = g - 1;
            if (!warp_wait(&c->pv_done[gp & 1], (gp >> 1) & 1, abort)) break;
            tc_fence_after();
            const float inv_l = 1.f / lr;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(t_o + ch * 32, o);
                tmem_wait_ld();
                reg_fence(o);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                    pk[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * inv_l, __uint_as_float(o[2 * x + 1]) * inv_l);
                if (row_valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[ch * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            lse_v = (m_used + __log2f(l)) * 0.69314718055994531f;
        } else if (row_valid) {
#pragma unroll 1
            for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (row_valid) p.lse[row] = lse_v;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->o_free);
    }
}

// ---------------------------------------------------------------- kernel
template <int BS, int D>
__global__ void __launch_bounds__(kThreads, 1)
    bsa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const FwdParams p) {
    using C = Cfg<BS, D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + ((kAlign - (raw & (kAlign - 1))) & (kAlign - 1));
    uint8_t* sQ = base;
    uint8_t* sT = base + C::NQ * C::Q_BYTES;
    Ctrl* c = reinterpret_cast<Ctrl*>(sT + C::NT * C::T_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 4; ++x) {
            mbar_init(&c->item_full[x], 1);
            mbar_init(&c->item_empty[x], 1 + 4);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&c->q_full[x], 1);
            mbar_init(&c->q_empty[x], 1);
            mbar_init(&c->s_full[x], 1);
            mbar_init(&c->p_full[x], 4);
            mbar_init(&c->pv_done[x], 1);
        }
        for (int x = 0; x < C::NT; ++x) {
            mbar_init(&c->t_full[x], 1);
            mbar_init(&c->t_empty[x], 1);
        }
        mbar_init(&c->o_free, 4);
        mbar_init(&c->drain, 1);
        c->abort = 0;
        fence_mbar_init();
    }
    if (BS < C::M) {
        // Rows BS..127 of the Q tiles are never loaded; keep them zero so the
        // padded rows of S stay finite.
        for (int b = 0; b < C::NQ * C::NBOX; ++b) {
            uint4* z = reinterpret_cast<uint4*>(sQ + b * C::Q_BOX + BS * 128);
            for (int x = threadIdx.x; x < (C::M - BS) * 128 / 16; x += kThreads) z[x] = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    if (warp == 5) {
        tmem_alloc(&c->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c->tmem_base;
    volatile int* abort = &c->abort;

    if (warp == 4) {
        if (lane == 0) producer<BS, D>(&tq, &tk, &tv, p, sQ, sT, c, abort);
    } else if (warp == 5) {
        if (lane == 0) mma_issuer<BS, D>(p, sQ, sT, c, tmem, abort);
    } else {
        softmax_role<BS, D>(p, c, tmem, abort);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && c->abort) atomicOr(p.err, ERR_TIMEOUT);
}

template <int BS, int D>
cudaError_t launch_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                        int grid, cudaStream_t stream) {
    using C = Cfg<BS, D>;
    cudaError_t e = cudaFuncSetAttribute(bsa_fwd_kernel<BS, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    bsa_fwd_kernel<BS, D><<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- schedule
constexpr int kSchedThreads = 1024;
constexpr int kSchedBins = 1024;

__device__ __forceinline__ int sched_key(int len) {
    len = len < 0 ? 0 : (len > kSchedBins - 1 ? kSchedBins - 1 : len);
    return kSchedBins - 1 - len;  // ascending key = descending row length
}

// Stable longest-first order of the rows (a counting sort on the row length,
// ties kept in row order so concurrently running CTAs share a head's K/V in
// L2).  One CTA; also zeroes the work counter of the forward kernel.
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const int32_t* __restrict__ row_ptr, int32_t R,
                                                                 int32_t* __restrict__ perm, int32_t* counter) {
    __shared__ int32_t hist[kSchedBins];
    __shared__ int32_t start[kSchedBins];
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) *counter = 0;
    hist[tid] = 0;
    __syncthreads();
    for (int r = tid; r < R; r += kSchedThreads) atomicAdd(&hist[sched_key(row_ptr[r + 1] - row_ptr[r])], 1);
    __syncthreads();
    // exclusive scan of hist (one bin per thread)
    const int v = hist[tid];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        warp_tot[lane] = ti - t;
    }
    __syncthreads();
    start[tid] = incl - v + warp_tot[warp];
    __syncthreads();
    for (int base = 0; base < R; base += kSchedThreads) {
        const int r = base + tid;
        const bool valid = r < R;
        const int key = valid ? sched_key(row_ptr[r + 1] - row_ptr[r]) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int leader = __ffs(peers) - 1;
        for (int w = 0; w < kSchedThreads / 32; ++w) {
            if (warp == w) {
                const int pos = valid ? start[key] + rank : 0;
                __syncwarp();
                if (valid) {
                    perm[pos] = r;
                    if (lane == leader) start[key] += __popc(peers);
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace

int fwd_smem_bytes(int block, int D) {
    if (block == 128 && D == 128) return Cfg<128, 128>::SMEM;
    if (block == 128 && D == 64) return Cfg<128, 64>::SMEM;
    if (block == 64 && D == 128) return Cfg<64, 128>::SMEM;
    if (block == 64 && D == 64) return Cfg<64, 64>::SMEM;
    return 0;
}

cudaError_t launch_forward(int block, int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, int grid, cudaStream_t stream) {
    if (block == 128 && D == 128) return launch_impl<128, 128>(tq, tk, tv, p, grid, stream);
    if (block == 128 && D == 64) return launch_impl<128, 64>(tq, tk, tv, p, grid, stream);
    if (block == 64 && D == 128) return launch_impl<64, 128>(tq, tk, tv, p, grid, stream);
    if (block == 64 && D == 64) return launch_impl<64, 64>(tq, tk, tv, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_schedule(const int32_t* row_ptr, int32_t R, int32_t* perm, int32_t* counter,
                            cudaStream_t stream) {
    schedule_kernel<<<1, kSchedThreads, 0, stream>>>(row_ptr, R, perm, counter);
    return cudaGetLastError();
}

}  // namespace bsa
