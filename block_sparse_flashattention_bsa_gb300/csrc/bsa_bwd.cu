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
//   schedule (the forward's)              key blocks ordered by the length
//        of their transposed lists, longest first;
//   bwd_prep_kernel                       Dv per query row;
//   bwd_zero_kernel                       dK = dV = 0 for unlisted key blocks;
//   bsa_bwd_kernel<D>                     persistent, one CTA per SM claiming
//        key blocks j in that order: K_j and V_j stay in shared memory; for
//        each listed query block i, S = Q K^T and dP = dO V^T go to TMEM, the
//        row warps form P and dS in shared memory, then dV += P^T dO,
//        dQ_i = dS K (in dP's columns) and dK += dS^T Q run in that order; dQ_i
//        is added to an fp32 buffer by bulk tensor reductions of 32 x 32 blocks
//        staged in the P tile while dK runs.  Q is double buffered and dQ does
//        not share TMEM with S, so the next query block's Q is resident and its
//        S product runs while dQ_i is read out, and its dO is copied in while
//        dQ_i and dK are computed; a key block's dK and dV are written by TMA
//        stores while the next block's copies and first products run.  In
//        the unpaired form the next query block's S is issued while the row
//        warps still compute P and dS (they load S first), P is posted before
//        dP is awaited so that dV runs on it, and K and V alternate between
//        two tile slots from one key block to the next;
//   bwd_dq_kernel                         dQ = scale * buffer, to bf16.
// Block 128, and block 64 in a paired form: a tile holds two 64-token key
// blocks whose transposed lists overlap (the forward's pairing pass on the
// transposed CSR), and each step two query blocks from the union of their
// lists; a (query block, key block) quarter of the step that no list names
// is zeroed in P and dS.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

#include <cuda_bf16.h>

namespace bsa {

namespace {

// warps 0 .. kBwdRowWarps - 1: row math (warp w: rows 32 (w & 3) .. + 31;
// with eight, column half w >> 2), then the producer and the MMA warp.
// Eight row warps (two per SM sub-partition, 168 registers a thread at most)
// measured 2-5 % faster than four.
constexpr int kBwdRowWarps = 8;
constexpr int kBwdThreads = (kBwdRowWarps + 2) * 32;
static_assert(kBwdRowWarps == 8, "warpgroup h owns dP / dQ half h");
constexpr int kBwdProducer = kBwdRowWarps;
constexpr int kBwdMma = kBwdRowWarps + 1;

template <int D>
struct BCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int BOX = 128 * 128;     // one 64-column (128-byte) box of a 128-row tile
    static constexpr int TILE = NBOX * BOX;   // a [128][D] bf16 tile: K, V, Q, dO
    static constexpr int PTILE = 2 * BOX;     // a [128][128] bf16 tile: P, dS (boxes of 64 keys)
    // K, V, two Q buffers, dO, P, dS
    static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE, OFF_DO = 4 * TILE;
    static constexpr int OFF_P = 5 * TILE, OFF_DS = 5 * TILE + PTILE;
    // While dQ_i is read out the P tile is idle (dV has read it): a row warp
    // stages 32-row x 32-column fp32 blocks of dQ in its own 32 rows of box h
    // of it (4 KB), one chunk after the other.
    static constexpr int SLAB = 32 * 32 * 4;
    static_assert(D / 32 <= 4, "at most two dQ chunks per row warp");
    static constexpr int OFF_CTRL = 5 * TILE + 2 * PTILE;
    static constexpr int CTRL_BYTES = 512;  // the control block (BCtrl), checked below
    static constexpr int SMEM = OFF_CTRL + CTRL_BYTES;
    // TMEM columns: S, dP, dV, dK; dQ reuses dP's columns
    static constexpr int C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D, C_DQ = 128;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t ID_S = idesc_bf16_f32_ab(128, 128, false, false);  // S, dP
    static constexpr uint32_t ID_KV = idesc_bf16_f32_ab(128, D, true, true);     // dV, dK: A = P^T / dS^T
    // dP and dQ in halves of 64 columns: dP half h (keys 64h ..) and dQ half h
    // (D columns 64h ..) share TMEM columns C_DP + 64h .. + 63
    static constexpr int NQH = D / 64;                                           // dQ halves
    static constexpr uint32_t ID_S64 = idesc_bf16_f32_ab(128, 64, false, false);  // dP half
    static constexpr uint32_t ID_Q64 = idesc_bf16_f32_ab(128, 64, false, true);   // dQ half
    static constexpr uint32_t TX_TILE = 128 * D * 2;
    static_assert(SMEM <= 232448, "shared memory overflow");
};

// mbarriers (completed by -> waited on by; "step" = one query block of a
// key block, "block" = one claimed key block):
//   slot_full[x] the copy into tile slot x     -> MMA (K or V of a block)
//   slot_free[x] the MMAs of a block done with slot x -> producer (next copy into x)
//   q_full[b] Q copy of a step (buffer b)    -> MMA
//   q_empty[b] dK of a step read Q           -> producer (next copy into b)
//   do_full   dO copy of a step              -> MMA
//   do_empty  dV of a step read dO           -> producer
//   s_full    S of a step                    -> row warps
//   s_read    S of a step loaded (row warps)  -> MMA (S of the next step of the block)
//   dp_full[h] half h of dP (keys 64h ..)   -> warpgroup h
//   ps_full   P, dS written (row warps)      -> MMA (paired form)
//   p_full    P written (row warps)          -> MMA (dV; unpaired form)
//   ds_full   dS written (row warps)         -> MMA (dQ, dK; unpaired form)
//   dq_full[h] dV and half h of dQ done      -> warpgroup h (dK may still run)
//   dq_free[h] half h of dQ read out          -> MMA (half h of the next dP overwrites it)
//   kv_done   every MMA of a block done      -> row warps (dK, dV)
//   acc_free  dK, dV read out (row warps)    -> MMA (next block's first dV, dK)
//   staged    dK, dV staged (row warps)      -> warp 0 (TMA stores)
//   st_read   the stores read the staging    -> row warps (next block's P, dS)
struct BCtrl {
    uint64_t slot_full[2], slot_free[2], q_full[2], q_empty[2], do_full, do_empty, s_full, s_read, dp_full[2], ps_full, p_full, ds_full, dq_full[2], dq_free[2], kv_done,
        staged, acc_free, st_read, drain;
    uint64_t item_full[4], item_empty[4];  // ring of claimed key blocks (producer -> MMA, row warps)
    int32_t ring[4];
    uint32_t tmem_base;
    WaitFlag wf;
};

static_assert(sizeof(BCtrl) <= BCfg<128>::CTRL_BYTES && sizeof(BCtrl) <= BCfg<64>::CTRL_BYTES,
              "control block larger than its shared-memory slot");

struct BwdParams {
    const int32_t* trp;  // transposed CSR: query blocks of key block r in tci[trp[r] .. trp[r+1])
    const int32_t* tci;
    int64_t tci_cap;     // entries tci holds
    const float* lse;    // [BH, N]
    const float* dvec;   // [BH, N]
    const uint8_t* row_flags;  // per CSR row (query block), bit 0 lifts the causal cut; may be null
    float* dq_acc;       // [BH, N, D] fp32
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int32_t* err;
    int32_t N, nb, causal;
    int32_t n_items;     // key blocks, BH * nb (the paired form: items, from n_items_dev)
    const int32_t* perm; // key blocks (paired form: items) by steps, longest first
    // paired form (64-token blocks), from the pairing pass on the transposed
    // lists: item w is key block item_a[w] (global row of the transposed CSR)
    // with key block item_b[w] of the same head, or alone (item_b[w] < 0);
    // item_cnt[w] union entries, in slots[w * kPairSlot ...] for a pair
    // (query block | in_a << 30 | in_b << 31) and in the transposed row of
    // item_a[w] for a single.
    const int32_t* item_a;
    const int32_t* item_b;
    const int32_t* item_cnt;
    const uint32_t* slots;
    const int32_t* n_items_dev;
    int32_t* counter;    // next entry of perm to claim
    float scale, scale_log2;
    unsigned long long wait_limit_ns;  // a pipeline wait longer than this aborts the launch
};

// Key block r (global row of the transposed CSR): its entries, without
// those beyond the capacity (dropped and flagged by the fill).
__device__ __forceinline__ int tcsr_len(const BwdParams& p, int r, int* beg) {
    *beg = p.trp[r];
    int n = p.trp[r + 1] - *beg;
    if ((int64_t)*beg + n > p.tci_cap) n = (int64_t)*beg < p.tci_cap ? (int)(p.tci_cap - *beg) : 0;
    return n;
}

// A claimed work item.  Block 128: key block j of head bh, one query block
// per step.  Paired form (64-token blocks): key blocks j (rows 0-63 of the
// tile) and jb (rows 64-127, or none when jb < 0), two union entries per step
// (query blocks in rows 0-63 and 64-127 of the step's Q tile).
struct BItem {
    int item, bh, j, jb, row0, beg, n, cnt;
    bool pair;
};
__device__ __forceinline__ BItem bitem(const BwdParams& p, int item) {
    BItem it;
    it.item = item;
    if (p.item_a) {
        const int ra = p.item_a[item];
        it.bh = ra / p.nb;
        it.j = ra - it.bh * p.nb;
        it.jb = p.item_b[item];
        it.pair = it.jb >= 0;
        it.cnt = p.item_cnt[item];
        if (it.pair) {
            it.beg = item * kPairSlot;
        } else {
            const int n = tcsr_len(p, ra, &it.beg);
            if (it.cnt > n) it.cnt = n;
        }
        it.n = (it.cnt + 1) >> 1;
    } else {
        it.bh = item / p.nb;
        it.j = item - it.bh * p.nb;
        it.jb = -1;
        it.pair = false;
        it.n = it.cnt = tcsr_len(p, item, &it.beg);
    }
    it.row0 = it.bh * p.N;
    return it;
}
// Union entry e of an item: query block | in_a << 30 | in_b << 31.
__device__ __forceinline__ uint32_t bentry(const BwdParams& p, const BItem& it, int e) {
    return it.pair ? p.slots[it.beg + e] : ((uint32_t)p.tci[it.beg + e] | (1u << 30));
}

// dK = dV = 0 for the key blocks no query block lists (the main kernel
// never claims them); one thread per key row.
template <int D, int KB>
__global__ void bwd_zero_kernel(const BwdParams p) {
    const int64_t rows = (int64_t)p.n_items * KB;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < rows; x += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(x / KB), t = (int)(x - (int64_t)r * KB);
        int beg;
        if (tcsr_len(p, r, &beg) > 0) continue;
        const int bh = r / p.nb, j = r - bh * p.nb;
        const int64_t krow = (int64_t)bh * p.N + (int64_t)j * KB + t;
        uint4* gk = reinterpret_cast<uint4*>(p.dk + krow * D);
        uint4* gv = reinterpret_cast<uint4*>(p.dv + krow * D);
#pragma unroll 1
        for (int y = 0; y < D / 8; ++y) {
            gk[y] = make_uint4(0u, 0u, 0u, 0u);
            gv[y] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, volatile WaitFlag* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// ---------------------------------------------------------------- transposed CSR
// The causal cut applies to CSR row r unless its flag lifts it.
__device__ __forceinline__ bool row_causal_b(int32_t causal, const uint8_t* flags, int64_t r) {
    return causal && !(flags && (flags[r] & 1));
}

__global__ void tcsr_count_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
                                  int64_t R, int32_t nb, int32_t causal_all, const uint8_t* __restrict__ flags,
                                  int32_t* __restrict__ cnt, int32_t* err) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bh = r / nb;
        const int32_t i = (int32_t)(r - bh * nb);
        const bool causal = row_causal_b(causal_all, flags, r);
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
                                 int32_t nb, int32_t causal_all, const uint8_t* __restrict__ flags,
                                 const int32_t* __restrict__ trp, int32_t* __restrict__ cursor,
                                 int32_t* __restrict__ tci, int64_t cap, int32_t* err) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bh = r / nb;
        const int32_t i = (int32_t)(r - bh * nb);
        const bool causal = row_causal_b(causal_all, flags, r);
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
// KB: tokens per block (128, or 64 in the paired form).
template <int D, int KB>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bsa_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                   const __grid_constant__ CUtensorMap tdv, const BwdParams p) {
    using C = BCfg<D>;
    constexpr bool PAIR = KB == 64;
    // Unpaired form: S of the next step of a block is issued while the row
    // warps compute this step's P and dS (they load S first), and dQ's TMEM
    // columns are released once read into registers.  The paired form keeps
    // S at the start of its step: holding S in registers there spills.
    constexpr bool SAHEAD = !PAIR;
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

    if (threadIdx.x == 0) {
        mbar_init(&c->slot_full[0], 1);
        mbar_init(&c->slot_full[1], 1);
        mbar_init(&c->slot_free[0], 1);
        mbar_init(&c->slot_free[1], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c->q_full[b], 1);
            mbar_init(&c->q_empty[b], 1);
        }
        mbar_init(&c->do_full, 1);
        mbar_init(&c->do_empty, 1);
        mbar_init(&c->s_full, 1);
        mbar_init(&c->s_read, kBwdRowWarps);
        mbar_init(&c->dp_full[0], 1);
        mbar_init(&c->dp_full[1], 1);
        mbar_init(&c->ps_full, kBwdRowWarps);
        mbar_init(&c->p_full, kBwdRowWarps);
        mbar_init(&c->ds_full, kBwdRowWarps);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&c->dq_full[x], 1);
            mbar_init(&c->dq_free[x], 4);  // the warpgroup of half x
        }
        mbar_init(&c->kv_done, 1);
        mbar_init(&c->staged, kBwdRowWarps);
        mbar_init(&c->acc_free, kBwdRowWarps);
        mbar_init(&c->st_read, 1);
        for (int x = 0; x < 4; ++x) {
            mbar_init(&c->item_full[x], 1);
            mbar_init(&c->item_empty[x], kBwdRowWarps + 1);  // the MMA warp and the row warps
        }
        mbar_init(&c->drain, 1);
        c->wf.abort = 0;
        c->wf.limit_ns = p.wait_limit_ns;
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
    volatile WaitFlag* abort = &c->wf;
    // The producer claims key blocks longest list first from a global counter
    // (the claim order stops at the first block no query block lists: those
    // get zeros from bwd_zero_kernel) and hands them to the MMA warp and the
    // row warps through a ring of 4.  Barrier phases count global steps g (all
    // steps of this CTA's blocks in order) and blocks u.

    if (warp == kBwdProducer) {
        const bool leader = elect_one();
        // Copies in global step order: dO_g once dV of step g - 1 has read the
        // buffer; K and V of a block into the tile slots the previous block's
        // V and K held, each once that block's last dP / last dQ has run;
        // Q_{g+1} (one step ahead, possibly of the next block) into buffer
        // (g + 1) & 1 once dK of step g - 1 has read it.
        int nkv = 0, nq0 = 0, nq1 = 0, nd = 0;
        int nsl0 = 0, nsl1 = 0;  // copies into tile slots 0 and 1
        // Paired form: every tile is two 64-row boxes (key blocks j, jb; the
        // step's two query blocks); a missing second block is read from
        // outside the tensor, which the copy fills with zeros.
        // K or V of a block into tile slot x.  Block u (the u-th this CTA
        // takes) holds K in slot u & 1 and V in the other, so the next
        // block's K goes where this block's V was, which frees once the
        // block's last dP has run, well before its last dQ and dK.
        auto load_slot = [&](int x, const CUtensorMap* tm, const BItem& it) {
            uint8_t* dst = x ? sV : sK;
            if (leader) {
                mbar_arrive_expect_tx(&c->slot_full[x], C::TX_TILE);
#pragma unroll
                for (int b = 0; b < C::NBOX; ++b) {
                    tma_load_2d(dst + b * C::BOX, tm, &c->slot_full[x], b * 64, it.row0 + it.j * KB);
                    if (PAIR) {
                        const int y = it.jb >= 0 ? it.row0 + it.jb * KB : -KB;
                        tma_load_2d(dst + b * C::BOX + 64 * 128, tm, &c->slot_full[x], b * 64, y);
                    }
                }
            }
            if (x) ++nsl1; else ++nsl0;
        };
        // query rows of step t: [first, second] (second < 0: none)
        auto step_rows = [&](const BItem& it, int t, int& y0, int& y1) {
            if (PAIR) {
                y0 = it.row0 + (int)(bentry(p, it, 2 * t) & 0x3fffffffu) * KB;
                y1 = 2 * t + 1 < it.cnt ? it.row0 + (int)(bentry(p, it, 2 * t + 1) & 0x3fffffffu) * KB : -KB;
            } else {
                y0 = it.row0 + p.tci[it.beg + t] * KB;
                y1 = -1;
            }
        };
        auto load_q = [&](const BItem& it, int t, int g) {
            const int b = g & 1;
            int y0, y1;
            step_rows(it, t, y0, y1);
            uint8_t* dst = sQ + b * C::TILE;
            if (leader) {
                mbar_arrive_expect_tx(&c->q_full[b], C::TX_TILE);
#pragma unroll
                for (int x = 0; x < C::NBOX; ++x) {
                    tma_load_2d(dst + x * C::BOX, &tq, &c->q_full[b], x * 64, y0);
                    if (PAIR) tma_load_2d(dst + x * C::BOX + 64 * 128, &tq, &c->q_full[b], x * 64, y1);
                }
            }
            if (b) ++nq1; else ++nq0;
        };
        auto load_do = [&](const BItem& it, int t) {
            int y0, y1;
            step_rows(it, t, y0, y1);
            if (leader) {
                mbar_arrive_expect_tx(&c->do_full, C::TX_TILE);
#pragma unroll
                for (int x = 0; x < C::NBOX; ++x) {
                    tma_load_2d(sDO + x * C::BOX, &tdo, &c->do_full, x * 64, y0);
                    if (PAIR) tma_load_2d(sDO + x * C::BOX + 64 * 128, &tdo, &c->do_full, x * 64, y1);
                }
            }
            ++nd;
        };
        // Claims: each claimed block is published in the ring (slot k & 3);
        // -1 ends the sequence.  The producer runs at most two steps ahead of
        // the step whose dO it copies, so it holds at most three claimed
        // blocks: qa (the dO / K / V cursor's), qb, qc.
        int nclaim = 0;
        bool ended = false, ok = true;
        const int n_items = PAIR ? *p.n_items_dev : p.n_items;
        auto claim = [&]() -> BItem {
            BItem it;
            it.item = -1;
            it.n = 0;
            if (ended) return it;
            int w = 0;
            if (lane == 0) w = atomicAdd(p.counter, 1);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (w < n_items) {
                it = bitem(p, p.perm[w]);
                if (it.n == 0) it.item = -1;  // sorted: no later block is listed either
            }
            const int slot = nclaim & 3;
            if (!wwait(&c->item_empty[slot], ((nclaim >> 2) & 1) ^ 1, abort)) {
                ok = false;
                it.item = -1;
                return it;
            }
            if (lane == 0) {
                c->ring[slot] = it.item;
                mbar_arrive(&c->item_full[slot]);
            }
            __syncwarp();
            ++nclaim;
            if (it.item < 0) ended = true;
            return it;
        };
        // a: the step whose dO (and, at a block start, K and V) is copied;
        // b: the next step, whose Q is copied ahead
        BItem qa = claim(), qb, qc;
        qb.item = qc.item = -1;
        qb.n = qc.n = 0;
        int nq_blocks = qa.item >= 0 ? 1 : 0;  // claimed blocks held: qa [, qb [, qc]]
        int ib = 0, ta = 0, tb = 0;            // b's block: 0 = qa, 1 = qb, 2 = qc
        ok = ok && qa.item >= 0;
        auto bblock = [&]() -> BItem { return ib == 0 ? qa : (ib == 1 ? qb : qc); };
        bool b_valid = ok;
        auto advance_b = [&]() {
            if (++tb == bblock().n) {
                tb = 0;
                BItem nx = claim();
                if (nx.item < 0) {
                    b_valid = false;
                    return;
                }
                if (nq_blocks >= 3) {  // never: b is at most two steps ahead of a
                    if (lane == 0) atomicOr(p.err, ERR_LAUNCH);
                    ok = b_valid = false;
                    return;
                }
                if (nq_blocks == 1) qb = nx; else qc = nx;
                ib = nq_blocks;
                ++nq_blocks;
            }
        };
        if (ok) {
            load_slot(0, &tk, qa);
            load_slot(1, &tv, qa);
            ++nkv;
            load_q(qa, 0, 0);
            advance_b();
            load_do(qa, ta);
            if (b_valid) {
                load_q(bblock(), tb, 1);
                advance_b();
            }
        }
        for (int g = 1; ok; ++g) {
            if (++ta == qa.n) {
                if (nq_blocks < 2) break;  // no further block
                qa = qb;
                qb = qc;
                --nq_blocks;
                --ib;
                ta = 0;
            }
            // a new block u: its K into the slot of block u - 1's V (free after
            // that block's last dP), then dO, then its V into the slot of
            // block u - 1's K (free after its last dQ)
            const int kx = nkv & 1;
            if (ta == 0) {
                if (!wwait(&c->slot_free[kx], (nkv - 1) & 1, abort)) break;
                load_slot(kx, &tk, qa);
            }
            if (!wwait(&c->do_empty, (g - 1) & 1, abort)) break;
            load_do(qa, ta);
            if (ta == 0) {
                if (!wwait(&c->slot_free[kx ^ 1], (nkv - 1) & 1, abort)) break;
                load_slot(kx ^ 1, &tv, qa);
                ++nkv;
            }
            if (b_valid) {
                if (!wwait(&c->q_empty[(g + 1) & 1], (((g + 1) >> 1) - 1) & 1, abort)) break;
                load_q(bblock(), tb, g + 1);
                advance_b();
            }
        }
        // the consumers stop at -1: make sure one is published
        if (!ended && !abort->abort) {
            while (!ended && ok) {
                BItem nx = claim();
                if (nx.item >= 0) {  // cannot happen once b is exhausted; stop the sequence anyway
                    if (lane == 0) atomicOr(p.err, ERR_LAUNCH);
                    break;
                }
            }
        }
        if (leader) {
            // the copies in flight must land before the CTA exits (after an
            // abort, or when another role aborts after this loop ended; in a
            // normal run they have all landed and these waits return at once)
            if (nsl0 > 0) mbar_wait_drain(&c->slot_full[0], (nsl0 - 1) & 1);
            if (nsl1 > 0) mbar_wait_drain(&c->slot_full[1], (nsl1 - 1) & 1);
            if (nq0 > 0) mbar_wait_drain(&c->q_full[0], (nq0 - 1) & 1);
            if (nq1 > 0) mbar_wait_drain(&c->q_full[1], (nq1 - 1) & 1);
            if (nd > 0) mbar_wait_drain(&c->do_full, (nd - 1) & 1);
        }
    } else if (warp == kBwdMma) {
        const bool leader = elect_one();
        constexpr uint64_t KDESC = sdesc_sw128_base(16, 1024);       // K-major, 128-byte swizzle
        constexpr uint64_t MDESC = sdesc_sw128_base(C::BOX, 1024);   // MN-major: 64-element groups a box apart
        const uint64_t do_k = KDESC + (smem_u32(sDO) >> 4);
        const uint64_t ds_k = KDESC + (smem_u32(sDS) >> 4);
        const uint64_t p_m = MDESC + (smem_u32(sP) >> 4), ds_m = MDESC + (smem_u32(sDS) >> 4);
        const uint64_t do_m = MDESC + (smem_u32(sDO) >> 4);
        bool ok = true;
        int g = 0, u = 0;
        for (int k = 0; ok; ++k) {
            const int slot = k & 3;
            if (!wwait(&c->item_full[slot], (k >> 2) & 1, abort)) break;
            const int x = c->ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->item_empty[slot]);
            if (x < 0) break;
            const BItem it = bitem(p, x);
            // this block's K in slot u & 1, V in the other
            const int kx = u & 1;
            uint8_t* sKu = kx ? sV : sK;
            uint8_t* sVu = kx ? sK : sV;
            const uint64_t k_k = KDESC + (smem_u32(sKu) >> 4), v_k = KDESC + (smem_u32(sVu) >> 4);
            const uint64_t k_m = MDESC + (smem_u32(sKu) >> 4);
            if (!wwait(&c->slot_full[kx], u & 1, abort)) {
                ok = false;
                break;
            }
            // S = Q K^T of step gs (Q buffer gs & 1); K-major operands: 16
            // columns (32 bytes) per MMA inside a box, the next box every 4
            auto issue_s = [&](int gs) -> bool {
                if (!wwait(&c->q_full[gs & 1], (gs >> 1) & 1, abort)) return false;
                tc_fence_after();
                if (leader) {
                    const uint64_t qs = KDESC + (smem_u32(sQ + (gs & 1) * C::TILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                        mma_ss(tmem + C::C_S, qs + off, k_k + off, C::ID_S, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&c->s_full);
                }
                __syncwarp();
                return true;
            };
            for (int t = 0; t < it.n; ++t, ++g) {
                const int b = g & 1;
                const uint64_t q_m = MDESC + (smem_u32(sQ + b * C::TILE) >> 4);
                // S's columns were read before the previous step's P was
                // published; in the unpaired form a later step of the block
                // had its S issued during the previous step's row math
                if ((t == 0 || !SAHEAD) && !issue_s(g)) {
                    ok = false;
                    break;
                }
                // dP = dO V^T in two halves of 64 keys, each into the columns
                // that half h of dQ of step g - 1 occupied until its warpgroup
                // read it out (D = 64: half 1 holds no dQ)
                if (!wwait(&c->do_full, g & 1, abort) || (t == 0 && !wwait(&c->slot_full[kx ^ 1], u & 1, abort))) {
                    ok = false;
                    break;
                }
#pragma unroll 1
                for (int hh = 0; hh < 2 && ok; ++hh) {
                    if (g > 0 && hh < C::NQH && !wwait(&c->dq_free[hh], (g - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint64_t vh = (uint64_t)((hh * 64 * 128) >> 4);  // V rows (keys) 64 hh ..
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                            mma_ss(tmem + C::C_DP + hh * 64, do_k + off, v_k + vh + off, C::ID_S64, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&c->dp_full[hh]);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                // the block's last dP has read V: its slot takes the next block's K
                if (leader && t + 1 == it.n) mma_commit(&c->slot_free[kx ^ 1]);
                // S of the next step of this block, into S's columns as soon as
                // the row warps hold this step's S in registers: it runs while
                // they compute P and dS
                if (SAHEAD && t + 1 < it.n && (!wwait(&c->s_read, g & 1, abort) || !issue_s(g + 1))) {
                    ok = false;
                    break;
                }
                // unpaired form: dV as soon as P is written (the row warps
                // compute dS meanwhile), so dO is free for the next copy earlier
                if (!wwait(SAHEAD ? &c->p_full : &c->ps_full, g & 1, abort) ||
                    (t == 0 && u > 0 && !wwait(&c->acc_free, (u - 1) & 1, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader) {
                    // dV += P^T dO, dK += dS^T Q: the reduction runs over the 128 query
                    // rows, 16 (2048 bytes of every box) per MMA; the first step of a
                    // block overwrites the accumulators (the row warps have read the
                    // previous block's)
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq) {
                        const uint64_t off = (uint64_t)((kq * 2048) >> 4);
                        mma_ss(tmem + C::C_DV, p_m + off, do_m + off, C::ID_KV, (t > 0 || kq > 0) ? 1u : 0u);
                    }
                    mma_commit(&c->do_empty);
                }
                __syncwarp();
                if (SAHEAD) {
                    if (!wwait(&c->ds_full, g & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                if (leader) {
                    // dQ_i = dS K (the reduction runs over the 128 keys) before dK, so
                    // its read-out, which the next step's dP waits for, overlaps dK;
                    // in halves of 64 D columns (box hh of the K tile), each
                    // released to its warpgroup as soon as it is done
#pragma unroll
                    for (int hh = 0; hh < C::NQH; ++hh) {
                        const uint64_t kbox = (uint64_t)((hh * C::BOX) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t aoff = (uint64_t)(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4);
                            const uint64_t boff = (uint64_t)((kk * 2048) >> 4);
                            mma_ss(tmem + C::C_DQ + hh * 64, ds_k + aoff, k_m + kbox + boff, C::ID_Q64,
                                   kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&c->dq_full[hh]);
                    }
                    // the block's last dQ (after its last S) has read K: its
                    // slot takes the next block's V
                    if (t + 1 == it.n) mma_commit(&c->slot_free[kx]);
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq) {
                        const uint64_t off = (uint64_t)((kq * 2048) >> 4);
                        mma_ss(tmem + C::C_DK, ds_m + off, q_m + off, C::ID_KV, (t > 0 || kq > 0) ? 1u : 0u);
                    }
                    mma_commit(&c->q_empty[b]);
                }
                __syncwarp();
            }
            if (!ok) break;
            // every MMA of this block is done: dK and dV may be read out
            if (leader) mma_commit(&c->kv_done);
            __syncwarp();
            ++u;
        }
        if (leader) {
            mma_commit(&c->drain);
            mbar_wait_drain(&c->drain, 0);
        }
        __syncwarp();
    } else if (warp < kBwdRowWarps) {
        // Thread (warp w, lane l) owns query row r = 32 (w & 3) + l of each
        // step (TMEM lane r) and, at the end of a block, key row r.  Key
        // columns 64h .. 64h + 63 of S and dP (box h of the P and dS tiles)
        // are column half h; with eight row warps warpgroup w >> 2 takes half
        // w >> 2, with four each warp takes both.  The rows need no reduction
        // (the forward's LSE is given), so the halves are independent.
        // Paired form: rows 64 qh .. 64 qh + 63 (qh = r >> 6) are the step's
        // query block qh and column half h is key block h of the item, so a
        // warp's 32 x 64 share of a half is one (query block, key block) pair:
        // listed or not as a whole, by the union entry's membership bit.
        constexpr int NHG = kBwdRowWarps / 4;  // warpgroups splitting the column halves
        static_assert(NHG == 2, "one column half per warpgroup");
        const int wq = warp & 3, hlo = warp >> 2;
        const int r = wq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t xr = (uint32_t)(r & 7);
        const int qh = r >> 6;       // paired form: the step's query block of this row
        const int rt = r & (KB - 1);  // query token of this row inside its block
        bool ok = true;
        int g = 0, u = 0;
        for (int k = 0; ok; ++k) {
            const int slot = k & 3;
            if (!wwait(&c->item_full[slot], (k >> 2) & 1, abort)) break;
            const int x = c->ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->item_empty[slot]);
            if (x < 0) break;
            const BItem it = bitem(p, x);
            const int row0 = it.row0;
            for (int t = 0; t < it.n && ok; ++t, ++g) {
                // query block i of this row; member: bit h lists the pair (i, key block h)
                int i;
                bool valid;
                uint32_t member;
                if (PAIR) {
                    const int e = 2 * t + qh;
                    valid = e < it.cnt;
                    const uint32_t ue = valid ? bentry(p, it, e) : 0u;
                    i = (int)(ue & 0x3fffffffu);
                    member = ue >> 30;
                } else {
                    i = p.tci[it.beg + t];
                    valid = true;
                    member = 3u;  // one 128-token key block: both column halves
                }
                const int64_t row = (int64_t)row0 + (int64_t)i * KB + rt;
                const float lse2 = valid ? p.lse[row] * 1.4426950408889634f : 0.f;
                const float dv_row = valid ? p.dvec[row] : 0.f;
                const f2 sl2 = {p.scale_log2, p.scale_log2}, nl2 = {-lse2, -lse2}, ndv = {-dv_row, -dv_row};
                if constexpr (SAHEAD) {
                    // S of this warp's column half into registers first, so S's
                    // columns take the next step's S while the warp works; P =
                    // 2^(s scale log2 e - LSE log2 e) is taken before dP arrives
                    const int h = hlo;  // one column half per warpgroup
                    const int jk = PAIR && h ? it.jb : it.j;  // key block of column half h
                    const bool diag = i == jk && row_causal_b(p.causal, p.row_flags, (int64_t)it.bh * p.nb + i);
                    // warp-uniform: the warp's rows are one query block
                    const bool listed = __all_sync(0xffffffffu, valid && ((member >> h) & 1u));
                    if (!wwait(&c->s_full, g & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float pf[2][32];  // P of the warp's 64 columns, fp32
                    if (listed) {
                        uint32_t sv[2][32];
                        tmem_ld32(tmem + lane_base + C::C_S + (2 * h) * 32, sv[0]);
                        tmem_ld32(tmem + lane_base + C::C_S + (2 * h + 1) * 32, sv[1]);
                        tmem_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&c->s_read);
#pragma unroll
                        for (int cb = 0; cb < 2; ++cb) {
                            reg_fence(sv[cb]);
#pragma unroll
                            for (int xx = 0; xx < 16; ++xx) {
                                const int col = ((2 * h + cb) * 32 + 2 * xx) & (KB - 1);  // key token inside its block
                                const f2 tt =
                                    fma2({__uint_as_float(sv[cb][2 * xx]), __uint_as_float(sv[cb][2 * xx + 1])}, sl2, nl2);
                                float p0 = ex2_approx(tt.x), p1 = ex2_approx(tt.y);
                                if (diag && col > rt) p0 = 0.f;  // key token after the query token
                                if (diag && col + 1 > rt) p1 = 0.f;
                                pf[cb][2 * xx] = p0;
                                pf[cb][2 * xx + 1] = p1;
                            }
                        }
                    } else {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&c->s_read);
                    }
                    // P (bf16, [query][key], 128-byte swizzle, boxes of 64 keys)
                    // goes to the P tile before dP is awaited.  The tile is free:
                    // dV of the previous step has read it, this warp's dQ slabs
                    // of that step have been read (bulk wait), and at a block
                    // start the previous block's dK / dV store has read it.
                    if ((g > 0 && !wwait(&c->do_empty, (g - 1) & 1, abort)) ||
                        (t == 0 && u > 0 && !wwait(&c->st_read, (u - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    if (listed) {
#pragma unroll
                        for (int cb = 0; cb < 2; ++cb) {
                            const int ch = 2 * h + cb;
                            uint32_t pk[16];
#pragma unroll
                            for (int xx = 0; xx < 16; ++xx) pk[xx] = pack_bf16x2(pf[cb][2 * xx], pf[cb][2 * xx + 1]);
                            uint8_t* bp = sP + (ch >> 1) * C::BOX + r * 128;
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                const uint32_t sw = ((uint32_t)((ch & 1) * 4 + v4) ^ xr) << 4;
                                *reinterpret_cast<uint4*>(bp + sw) =
                                    make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                            }
                        }
                    } else {  // an unlisted pair (or no second query block): P = 0
                        uint8_t* bp = sP + h * C::BOX + r * 128;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *reinterpret_cast<uint4*>(bp + ((v ^ xr) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();  // P is read by the tensor cores
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c->p_full);
                    // dS = P (dP - Dv) into the dS tile, which dQ and dK of the
                    // previous step have read (they complete before this dP)
                    if (!wwait(&c->dp_full[hlo], g & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (listed) {
#pragma unroll
                        for (int cb = 0; cb < 2; ++cb) {
                            const int ch = 2 * h + cb;
                            uint32_t dpv[32];
                            tmem_ld32(tmem + lane_base + C::C_DP + ch * 32, dpv);
                            tmem_wait_ld();
                            reg_fence(dpv);
                            uint32_t dk[16];
#pragma unroll
                            for (int xx = 0; xx < 16; ++xx) {
                                const f2 ds = mul2({pf[cb][2 * xx], pf[cb][2 * xx + 1]},
                                                   add2({__uint_as_float(dpv[2 * xx]), __uint_as_float(dpv[2 * xx + 1])}, ndv));
                                dk[xx] = pack_bf16x2(ds.x, ds.y);
                            }
                            uint8_t* bd = sDS + (ch >> 1) * C::BOX + r * 128;
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                const uint32_t sw = ((uint32_t)((ch & 1) * 4 + v4) ^ xr) << 4;
                                *reinterpret_cast<uint4*>(bd + sw) =
                                    make_uint4(dk[4 * v4], dk[4 * v4 + 1], dk[4 * v4 + 2], dk[4 * v4 + 3]);
                            }
                        }
                    } else {  // dS = 0
                        uint8_t* bd = sDS + h * C::BOX + r * 128;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *reinterpret_cast<uint4*>(bd + ((v ^ xr) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                } else {
                    if (!wwait(&c->s_full, g & 1, abort) || !wwait(&c->dp_full[hlo], g & 1, abort) ||
                        (t == 0 && u > 0 && !wwait(&c->st_read, (u - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // this warp's rows of the P and dS boxes it writes held its dQ
                    // blocks of step g - 1 (and, at a block start, its share of the
                    // previous block's dK / dV, whose store has read them): the
                    // reductions must have read them
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll 1
                    for (int h = hlo; h < 2; h += NHG) {
                        const int jk = PAIR && h ? it.jb : it.j;  // key block of column half h
                        const bool diag = i == jk && row_causal_b(p.causal, p.row_flags, (int64_t)it.bh * p.nb + i);
                        // one 32-column chunk of S and dP -> P and dS (bf16, [query][key],
                        // 128-byte swizzle, boxes of 64 keys)
                        auto chunk = [&](const uint32_t (&sv)[32], const uint32_t (&dpv)[32], int ch) {
                            uint32_t pk[16], dk[16];
#pragma unroll
                            for (int xx = 0; xx < 16; ++xx) {
                                const int col = (ch * 32 + 2 * xx) & (KB - 1);  // key token inside its block
                                const f2 tt =
                                    fma2({__uint_as_float(sv[2 * xx]), __uint_as_float(sv[2 * xx + 1])}, sl2, nl2);
                                float p0 = ex2_approx(tt.x), p1 = ex2_approx(tt.y);
                                if (diag && col > rt) p0 = 0.f;  // key token after the query token
                                if (diag && col + 1 > rt) p1 = 0.f;
                                pk[xx] = pack_bf16x2(p0, p1);
                                const f2 ds = mul2(
                                    {p0, p1}, add2({__uint_as_float(dpv[2 * xx]), __uint_as_float(dpv[2 * xx + 1])}, ndv));
                                dk[xx] = pack_bf16x2(ds.x, ds.y);
                            }
                            uint8_t* bp = sP + (ch >> 1) * C::BOX + r * 128;
                            uint8_t* bd = sDS + (ch >> 1) * C::BOX + r * 128;
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                const uint32_t sw = ((uint32_t)((ch & 1) * 4 + v4) ^ xr) << 4;
                                *reinterpret_cast<uint4*>(bp + sw) =
                                    make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                                *reinterpret_cast<uint4*>(bd + sw) =
                                    make_uint4(dk[4 * v4], dk[4 * v4 + 1], dk[4 * v4 + 2], dk[4 * v4 + 3]);
                            }
                        };
                        // warp-uniform: the warp's rows are one query block
                        if (__all_sync(0xffffffffu, valid && ((member >> h) & 1u))) {
#pragma unroll 1
                            for (int cb = 0; cb < 2; ++cb) {
                                uint32_t sv[32], dpv[32];
                                tmem_ld32(tmem + lane_base + C::C_S + (2 * h + cb) * 32, sv);
                                tmem_ld32(tmem + lane_base + C::C_DP + (2 * h + cb) * 32, dpv);
                                tmem_wait_ld();
                                reg_fence(sv);
                                reg_fence(dpv);
                                chunk(sv, dpv, 2 * h + cb);
                            }
                        } else {  // an unlisted pair (or no second query block): P = dS = 0
                            uint8_t* bp = sP + h * C::BOX + r * 128;
                            uint8_t* bd = sDS + h * C::BOX + r * 128;
                            // the swizzled order: one store instruction covers all banks
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                *reinterpret_cast<uint4*>(bp + ((v ^ xr) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                                *reinterpret_cast<uint4*>(bd + ((v ^ xr) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                }
                fence_proxy_async_smem();  // P and dS are read by the tensor cores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(SAHEAD ? &c->ds_full : &c->ps_full);
                // dQ_i half hlo (D columns 64 hlo .. + 63, chunks 2 hlo, 2 hlo + 1;
                // D = 64: warpgroup 0 takes both chunks, warpgroup 1 none): each
                // 32-column chunk of this warp's 32 rows goes through a swizzled
                // slab (16-byte chunk c of slab row y at y * 128 + ((c ^ (y & 7)) << 4))
                // and is added to the fp32 buffer by one bulk tensor reduction,
                // so the L2 sees whole lines.  The slab is this warp's rows of
                // box hlo of the P tile, which dV (complete before dQ) has read
                // and which stays idle until the next step's row math (that
                // first waits for these reductions to have read it); the dS
                // tile is still being read by dK.  The rows of a missing second
                // query block add nothing.
                if (hlo < C::NQH) {
                    if (!wwait(&c->dq_full[hlo], g & 1, abort)) {
                        ok = false;
                        break;
                    }
                    if constexpr (SAHEAD) {
                        tc_fence_after();
                        uint32_t o[2][32];
                        if (valid) {
                            tmem_ld32(tmem + lane_base + C::C_DQ + hlo * 64, o[0]);
                            tmem_ld32(tmem + lane_base + C::C_DQ + hlo * 64 + 32, o[1]);
                            tmem_wait_ld();
                        }
                        // this warp's rows of dQ half hlo are in registers: half hlo
                        // of the next dP may overwrite the columns while they are
                        // staged and reduced
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&c->dq_free[hlo]);
                        if (valid) {
#pragma unroll
                            for (int y = 0; y < 2; ++y) {
                                const int ch = 2 * hlo + y;
                                reg_fence(o[y]);
                                uint8_t* slab = sP + hlo * C::BOX + wq * C::SLAB;
                                if (y > 0) {  // the previous chunk's reduction must have read the slab
                                    if (lane == 0) bulk_wait_read_all();
                                    __syncwarp();
                                }
#pragma unroll
                                for (int c4 = 0; c4 < 8; ++c4)
                                    *reinterpret_cast<uint4*>(slab + lane * 128 + ((c4 ^ (lane & 7)) << 4)) =
                                        make_uint4(o[y][4 * c4], o[y][4 * c4 + 1], o[y][4 * c4 + 2], o[y][4 * c4 + 3]);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_reduce_add_2d(&tdq, slab, ch * 32, row0 + i * KB + (wq * 32 & (KB - 1)));
                                    bulk_commit_group();
                                }
                            }
                        }
                    } else {
                        tc_fence_after();
                        if (valid) {
                            uint32_t o[2][32];
                            tmem_ld32(tmem + lane_base + C::C_DQ + hlo * 64, o[0]);
                            tmem_ld32(tmem + lane_base + C::C_DQ + hlo * 64 + 32, o[1]);
                            tmem_wait_ld();
#pragma unroll
                            for (int y = 0; y < 2; ++y) {
                                const int ch = 2 * hlo + y;
                                reg_fence(o[y]);
                                uint8_t* slab = sP + hlo * C::BOX + wq * C::SLAB;
                                if (y > 0) {  // the previous chunk's reduction must have read the slab
                                    if (lane == 0) bulk_wait_read_all();
                                    __syncwarp();
                                }
#pragma unroll
                                for (int c4 = 0; c4 < 8; ++c4)
                                    *reinterpret_cast<uint4*>(slab + lane * 128 + ((c4 ^ (lane & 7)) << 4)) =
                                        make_uint4(o[y][4 * c4], o[y][4 * c4 + 1], o[y][4 * c4 + 2], o[y][4 * c4 + 3]);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_reduce_add_2d(&tdq, slab, ch * 32, row0 + i * KB + (wq * 32 & (KB - 1)));
                                    bulk_commit_group();
                                }
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&c->dq_free[hlo]);
                    }
                }
            }
            if (!ok) break;
            // dK and dV of this item.  Thread r owns key row r: its rows of dK
            // (x scale) and dV are staged as bf16 in the 128-byte swizzled box
            // layout of the dK / dV tensor maps, and one thread writes them by
            // TMA stores (one per 64-column box and key block) while the next
            // item's copies and first products are under way.  D = 128: half h
            // is columns 64h .. 64h + 63, dK in box h of the P tile and dV in
            // box h of the dS tile.  D = 64: half h is columns 32h .. 32h + 31,
            // dK in box 0 and dV in box 1 of the dS tile.  Either way a warp
            // writes only rows whose dQ slabs were its own (its reductions
            // have read them) or held none.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if (!wwait(&c->kv_done, u & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint8_t* st_k = D == 128 ? sP : sDS;
            uint8_t* st_v = D == 128 ? sDS : sDS + C::BOX;
            if (!PAIR || qh == 0 || it.jb >= 0) {  // key row r: key block it.j (rows 0-63) or it.jb
#pragma unroll 1
                for (int h = hlo; h < 2; h += NHG) {
#pragma unroll 1
                    for (int y = 0; y < D / 64; ++y) {
                        const int ch = D == 128 ? 2 * h + y : h;
                        uint32_t a[32], b[32];
                        tmem_ld32(tmem + lane_base + C::C_DK + ch * 32, a);
                        tmem_ld32(tmem + lane_base + C::C_DV + ch * 32, b);
                        tmem_wait_ld();
                        reg_fence(a);
                        reg_fence(b);
                        const int off = (ch >> 1) * C::BOX + r * 128;
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint32_t ka[4], va[4];
#pragma unroll
                            for (int uu = 0; uu < 4; ++uu) {
                                const int xx = v4 * 8 + 2 * uu;
                                ka[uu] = pack_bf16x2(__uint_as_float(a[xx]) * p.scale,
                                                     __uint_as_float(a[xx + 1]) * p.scale);
                                va[uu] = pack_bf16x2(__uint_as_float(b[xx]), __uint_as_float(b[xx + 1]));
                            }
                            const int sw = (((ch & 1) * 4 + v4) ^ (int)xr) << 4;
                            *reinterpret_cast<uint4*>(st_k + off + sw) = make_uint4(ka[0], ka[1], ka[2], ka[3]);
                            *reinterpret_cast<uint4*>(st_v + off + sw) = make_uint4(va[0], va[1], va[2], va[3]);
                        }
                    }
                }
            }
            // the accumulators are read: the next item's first dV / dK may overwrite them
            tc_fence_before();
            fence_proxy_async_smem();  // the staging is read next by the TMA unit
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&c->acc_free);
                mbar_arrive(&c->staged);
            }
            if (warp == 0) {
                if (!wwait(&c->staged, u & 1, abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    if (!abort->abort) {
#pragma unroll
                        for (int xx = 0; xx < C::NBOX; ++xx) {
                            tma_store_2d(&tdk, st_k + xx * C::BOX, xx * 64, row0 + it.j * KB);
                            tma_store_2d(&tdv, st_v + xx * C::BOX, xx * 64, row0 + it.j * KB);
                            if (PAIR && it.jb >= 0) {
                                tma_store_2d(&tdk, st_k + xx * C::BOX + 64 * 128, xx * 64, row0 + it.jb * KB);
                                tma_store_2d(&tdv, st_v + xx * C::BOX + 64 * 128, xx * 64, row0 + it.jb * KB);
                            }
                        }
                        bulk_commit_group();
                    }
                    bulk_wait_read_all();
                    mbar_arrive(&c->st_read);  // P and dS may be rewritten
                }
                __syncwarp();
            }
            ++u;
        }
        if (lane == 0) bulk_wait_read_all();  // every bulk operation has read its staging
        __syncwarp();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && c->wf.abort) atomicOr(p.err, ERR_TIMEOUT);
}

}  // namespace

size_t bwd_workspace_bytes(int32_t BH, int32_t N, int32_t D, int32_t block, int32_t nb, int64_t col_capacity) {
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t R = (size_t)BH * nb;
    return a((R + 1) * 4) + a(R * 4) + a((size_t)col_capacity * 4 + 4) + a((size_t)BH * N * 4) +
           a((size_t)BH * N * D * 4) + a(R * 4) + 256 + (block == 64 ? pairing_workspace_bytes(BH, nb) : 0);
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
    w += a((size_t)rows * L.D * 4);
    int32_t* perm = reinterpret_cast<int32_t*>(w);  // key blocks, longest transposed list first
    w += a((size_t)R * 4);
    int32_t* counter = reinterpret_cast<int32_t*>(w);
    w += 256;
    const bool paired = L.block == 64;
    cudaError_t e;
    if ((e = cudaMemsetAsync(trp, 0, (size_t)(R + 1) * 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(cursor, 0, (size_t)R * 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dq_acc, 0, (size_t)rows * L.D * 4, s)) != cudaSuccess) return e;
    int64_t blocks = (R + 255) / 256;
    if (blocks > 8 * (int64_t)L.sm_count) blocks = 8 * (int64_t)L.sm_count;
    tcsr_count_kernel<<<(unsigned)blocks, 256, 0, s>>>(L.row_ptr, L.col_idx, R, L.nb, L.causal, L.row_flags, trp + 1,
                                                       L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_row_ptr_scan(trp + 1, R, trp, s)) != cudaSuccess) return e;
    tcsr_fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(L.row_ptr, L.col_idx, R, L.nb, L.causal, L.row_flags, trp,
                                                      cursor, tci, L.col_capacity, L.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the work items in claim order (the forward's stable longest-first sort,
    // on the transposed lists or the paired items' steps); zeroes the claim
    // counter.  64-token blocks: key blocks paired by their transposed lists
    // (the forward's pairing pass, rows = key blocks, entries = query blocks;
    // the causal cut is already applied).
    PairingBuffers pb{};
    if (paired) {
        pb = pairing_buffers(w, L.BH, L.nb);
        const PairGeom pg{L.nb, L.nb, 0, 0, nullptr, L.col_capacity};
        if ((e = launch_pairing(trp, tci, L.BH, pg, pb, L.err, L.sm_count, s)) != cudaSuccess) return e;
        // classes of 8 steps (measured 1.4 % faster here than one class of 32)
        if ((e = launch_schedule_lens(pb.item_len, pb.n_items, (int32_t)R, perm, counter, 3, s)) != cudaSuccess)
            return e;
    } else if ((e = launch_schedule(trp, (int32_t)R, perm, counter, s)) != cudaSuccess) {
        return e;
    }
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
    p.row_flags = L.row_flags;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(L.dk);
    p.dv = static_cast<__nv_bfloat16*>(L.dv);
    p.err = L.err;
    p.N = L.N;
    p.nb = L.nb;
    p.causal = L.causal;
    p.scale = L.scale;
    p.scale_log2 = L.scale * 1.4426950408889634f;
    p.wait_limit_ns = wait_limit_ns();
    p.n_items = (int32_t)R;
    p.perm = perm;
    p.counter = counter;
    p.item_a = paired ? pb.item_a : nullptr;
    p.item_b = pb.item_b;
    p.item_cnt = pb.item_cnt;
    p.slots = pb.slots;
    p.n_items_dev = pb.n_items;
    {
        int64_t zb = (R * L.block + 255) / 256;
        if (zb > 8 * (int64_t)L.sm_count) zb = 8 * (int64_t)L.sm_count;
        if (L.block == 128)
            L.D == 128 ? bwd_zero_kernel<128, 128><<<(unsigned)zb, 256, 0, s>>>(p)
                       : bwd_zero_kernel<64, 128><<<(unsigned)zb, 256, 0, s>>>(p);
        else
            L.D == 128 ? bwd_zero_kernel<128, 64><<<(unsigned)zb, 256, 0, s>>>(p)
                       : bwd_zero_kernel<64, 64><<<(unsigned)zb, 256, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    auto run = [&](auto kernel, int smem) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        // persistent: one CTA per SM, claiming key blocks until none is left
        const int64_t grid = R < (int64_t)L.sm_count ? R : (int64_t)L.sm_count;
        kernel<<<(unsigned)(grid > 0 ? grid : 1), kBwdThreads, smem, s>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, L.tdk,
                                                                           L.tdv, p);
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
