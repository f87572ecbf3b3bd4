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
// GB300 design: one CTA per SM, 15 warps, warp-specialised.
//   warp 14      claimer: claims work items (query-block rows) from a global
//                counter, scans the row's col_idx 32 entries at a time and
//                publishes its block count, diagonal position and extent in a
//                ring of 4 rows, ahead of the pipeline.
//   warp 12      producer: TMA-loads the Q tile (2 buffers) and the K_j / V_j
//                tiles of each claimed row into a ring of NT tiles.
//   warp 13      MMA (warp-wide loop, one elected lane issues): S_j = Q K_j^T
//                (both operands in shared memory, fp32 in TMEM, two S buffers)
//                and O += P_j V_j (P from TMEM, V MN-major from shared memory)
//                into one of two O accumulators, alternating per row so the
//                epilogue of a row overlaps the next row.  The issue order is
//                one flat stream across rows -- QK_0, QK_1, PV_0, QK_2, PV_1,
//                ... -- so the next row's first QK is queued behind the
//                current row's last PV.
//   warps 0-7    softmax: warpgroup h (warps 4h..4h+3) owns key columns
//                [h*BS/2, (h+1)*BS/2) of every S tile; thread t of a warpgroup
//                owns query row t.  The two warps holding the same rows swap
//                their half-row maxima each step (shared memory + mbarrier),
//                so both halves use one running max and one O accumulator;
//                each exponentiates its own half.  The running max is refreshed only
//                when it grows by more than 2^8, which keeps every exponent
//                <= 2^8 and is exact after the final division.  P (bf16)
//                overwrites the S columns it was computed from.
//   warps 8-11   epilogue: O / l (bf16) and LSE (fp32) for each finished row.
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
constexpr int kXchBytes = 2 * 2 * 128 * 4;  // per-step half-row maxima: [S buffer][half][row]
constexpr int kAlign = 1024;                // 128-byte swizzle atoms need 1024-byte alignment
constexpr int kThreads = 480;
constexpr int kSoftmaxWarps = 8;
constexpr int kEpiWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kClaimWarp = 14;
constexpr int kConsumerWarps = 1 + 1 + kSoftmaxWarps + 4;  // releases of an item slot (producer, MMA, softmax, epilogue)

template <int BS, int D>
struct Cfg {
    static constexpr int M = 128;                 // MMA rows (query rows; BS = 64 pads to 128)
    static constexpr int H2 = BS / 2;             // key columns per softmax half
    static constexpr int NBOX = D / 64;           // 64 bf16 = one 128-byte swizzled row per box
    static constexpr int Q_BOX = M * 128;         // bytes of one box of the Q tile
    static constexpr int Q_BYTES = NBOX * Q_BOX;
    static constexpr int T_BOX = BS * 128;        // bytes of one box of a K or V tile
    static constexpr int T_BYTES = NBOX * T_BOX;
    static constexpr int NQ = 2;
    // The dynamic shared memory must start 1024-byte aligned (checked at run
    // time); no slack is reserved for realigning it.
    static constexpr int NT_FIT = (kSmemLimit - kCtrlBytes - kXchBytes - NQ * Q_BYTES) / T_BYTES;
    static constexpr int NT = NT_FIT > 8 ? 8 : NT_FIT;
    static constexpr int SMEM = NQ * Q_BYTES + NT * T_BYTES + kCtrlBytes + kXchBytes;
    // TMEM columns: two S buffers (P_h written over the S columns of half h),
    // two O accumulators (row it uses O buffer it & 1).
    static constexpr int S_COL = 0;
    static constexpr int O_COL = 2 * BS;
    static constexpr int USED_COLS = 2 * BS + 2 * D;
    static constexpr int TMEM_COLS = USED_COLS <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(M, BS, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(M, D, true);
    static constexpr uint32_t TX_BYTES = BS * D * 2;
    // FP8 scores (D = 128): Q and K tiles are e4m3, one 128-byte row per
    // token, i.e. a single swizzled box; they fill the first half of the
    // (bf16-sized) Q buffers and K slots of the ring.
    static constexpr uint32_t TX_BYTES_F8 = BS * D;
    static constexpr uint32_t IDESC_QK_F8 = idesc_e4m3_f32(M, BS);
    // Per-row statistics handed from the softmax halves to the epilogue live
    // in the (consumed) Q tile of the row: float [5][128] = m, l_0, l_1,
    // lr_0, lr_1.
    static constexpr int STATS_BYTES = 5 * 128 * 4;
    static_assert(NT >= 2, "shared memory ring too small");
    static_assert(USED_COLS <= 512, "TMEM overflow");
    static_assert(SMEM <= kSmemLimit, "shared memory overflow");
    static_assert(STATS_BYTES <= BS * 128, "statistics must sit inside the TMA-written part of Q");
};

struct Ctrl {
    uint64_t item_full[4];
    uint64_t item_empty[4];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t t_full[8];
    uint64_t t_empty[8];
    uint64_t s_full[2];
    uint64_t p_full[2];     // [S buffer]: both softmax halves wrote P
    uint64_t mx_full[4][2]; // [warp pair][S buffer]: both warps of a pair posted their half-row max
    uint64_t pv_done[2];    // [S buffer]: the PV of the step in it has completed
    uint64_t o_full[2];     // [O buffer]: the last PV of the row in it has completed
    uint64_t stats_full[2];   // per Q buffer: the softmax halves posted (m, l, lr)
    uint64_t stats_empty[2];  // per Q buffer: the epilogue read them
    uint64_t o_free[2];     // [O buffer]: the epilogue has read it
    uint64_t ep_sync;       // the epilogue warps have read the row's statistics
    uint64_t o_staged;      // the epilogue warps have written the row's O into the Q tile
    uint64_t drain;
    // claimed item: {item, steps, position of the diagonal block among the valid
    // entries or -1, beg, end, CSR row of the (first) query block, second query
    // block or -1 (paired form), valid entries, causal cut of the first row,
    // then for a pair the softmax masks sel[qh][h] (4) and dsel[qh][h] (4)}
    int32_t ring[4][17];
    uint32_t tmem_base;
    WaitFlag wf;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile WaitFlag* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// Key block j is computed for query block i: inside the key blocks, and not
// after the query block (key position i + q_off) when the row is causal.
__device__ __forceinline__ bool block_ok(const FwdParams& p, int j, int i, bool crow) {
    return (unsigned)j < (unsigned)p.nbk && !(crow && j > i + p.q_off);
}

// The causal cut applies to CSR row r unless its row flag lifts it.
__device__ __forceinline__ bool row_causal(const FwdParams& p, int r) {
    return p.causal && !(p.row_flags && (p.row_flags[r] & 1));
}

// Bits k = 2e + h of x, packed to bit e.
__device__ __forceinline__ uint32_t even_bits(uint64_t x) {
    x &= 0x5555555555555555ull;
    x = (x | (x >> 1)) & 0x3333333333333333ull;
    x = (x | (x >> 2)) & 0x0f0f0f0f0f0f0f0full;
    x = (x | (x >> 4)) & 0x00ff00ff00ff00ffull;
    x = (x | (x >> 8)) & 0x0000ffff0000ffffull;
    x = (x | (x >> 16)) & 0x00000000ffffffffull;
    return (uint32_t)x;
}

// ---------------------------------------------------------------- claimer
// The whole warp claims the next row and scans its col_idx 32 entries at a
// time (count of processed blocks, position of the diagonal), running up to
// 4 rows ahead of the pipeline so these dependent global loads stay hidden.
template <bool PAIR>
__device__ void claimer(const FwdParams& p, Ctrl* c, volatile WaitFlag* abort) {
    const int lane = threadIdx.x & 31;
    // The schedule kernel writes perm and zeroes the counter; this kernel may
    // have started (dependent launch) before it finished.  Nothing else in the
    // kernel reads its outputs, and every other role waits on this warp.
    griddep_wait();
    // the paired form's item count is written by the pairing pass, which ran
    // before this launch on the same stream
    const int n_items = PAIR ? *p.n_items_dev : p.n_items;
    for (uint32_t it = 0;; ++it) {
        // Test hook of the hang detection: after stall_after items this warp
        // publishes nothing more, not even the end marker, so every other
        // role's next wait runs out.
        if (p.stall_after >= 0 && it >= (uint32_t)p.stall_after) break;
        const uint32_t slot = it & 3;
        if (!warp_wait(&c->item_empty[slot], ((it >> 2) & 1) ^ 1, abort)) break;
        int w = 0;
        if (lane == 0) w = atomicAdd(p.counter, 1);
        w = __shfl_sync(0xffffffffu, w, 0);
        const int item = w < n_items ? p.perm[w] : -1;
        int beg = 0, end = 0, nent = 0, diag = -1, ra = -1, ib = -1;
        bool crow = false;
        if (item >= 0) {
            ra = PAIR ? p.item_a[item] : item;
            ib = PAIR ? p.item_b[item] : -1;
            crow = row_causal(p, ra);
        }
        // a pair's softmax masks, per query half qh and column half h (entry
        // k = 2e + h of the union): sel bit e = entry listed for that query
        // block, dsel bit e = entry is its diagonal (causal).  Computed here,
        // rows ahead, so the union's entries are not read on the softmax's path.
        uint32_t psel[2][2] = {{0u, 0u}, {0u, 0u}}, pdsel[2][2] = {{0u, 0u}, {0u, 0u}};
        if (PAIR && ib >= 0) {
            // a pair: its union was built by the pairing pass
            nent = p.item_cnt[item];
            beg = item * kPairSlot;
            end = beg + nent;
            const uint32_t e0 = lane < nent ? p.slots[beg + lane] : 0u;
            const uint32_t e1 = 32 + lane < nent ? p.slots[beg + 32 + lane] : 0u;
#pragma unroll
            for (int qh = 0; qh < 2; ++qh) {
                const int i_my = qh ? ib : ra % p.nb;
                const bool ok0 = lane < nent && ((e0 >> (30 + qh)) & 1u);
                const bool ok1 = 32 + lane < nent && ((e1 >> (30 + qh)) & 1u);
                const uint64_t am = (uint64_t)__ballot_sync(0xffffffffu, ok0) |
                                    ((uint64_t)__ballot_sync(0xffffffffu, ok1) << 32);
                const uint64_t dm =
                    (uint64_t)__ballot_sync(0xffffffffu, ok0 && p.causal && (int)(e0 & 0x3fffffffu) == i_my + p.q_off) |
                    ((uint64_t)__ballot_sync(0xffffffffu, ok1 && p.causal && (int)(e1 & 0x3fffffffu) == i_my + p.q_off)
                     << 32);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    psel[qh][h] = even_bits(am >> h);
                    pdsel[qh][h] = even_bits(dm >> h);
                }
            }
        } else if (item >= 0) {
            const int i = ra % p.nb;
            beg = p.row_ptr[ra];
            end = p.row_ptr[ra + 1];
            if (end < beg) {
                if (lane == 0) atomicOr(p.err, ERR_BAD_ROW);
                end = beg;
            }
            for (int e0 = beg; e0 < end; e0 += 32) {
                const int e = e0 + lane;
                const int j = e < end ? p.col_idx[e] : -1;
                if (e < end && (unsigned)j >= (unsigned)p.nbk) atomicOr(p.err, ERR_BAD_COL);
                const unsigned vm = __ballot_sync(0xffffffffu, e < end && block_ok(p, j, i, crow));
                const unsigned dm = __ballot_sync(0xffffffffu, e < end && crow && j == i + p.q_off);
                if (diag < 0 && dm) diag = nent + __popc(vm & ((1u << (__ffs(dm) - 1)) - 1u));
                nent += __popc(vm);
            }
        }
        // one step per valid key block; the paired form takes two per step
        const int steps = PAIR ? (nent + 1) >> 1 : nent;
        if (lane == 0) {
            int32_t* r = c->ring[slot];
            r[0] = item;
            r[1] = steps;
            r[2] = diag;
            r[3] = beg;
            r[4] = end;
            r[5] = ra;
            r[6] = ib;
            r[7] = nent;
            r[8] = crow ? 1 : 0;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                r[9 + x] = (int32_t)psel[x >> 1][x & 1];
                r[13 + x] = (int32_t)pdsel[x >> 1][x & 1];
            }
            mbar_arrive(&c->item_full[slot]);
        }
        __syncwarp();
        if (item < 0) break;
    }
}

// ---------------------------------------------------------------- producer
// The whole warp runs this loop with identical values; one elected lane
// issues the copies.  The paired form (64-token blocks in a 128-row tile)
// loads each Q, K and V tile as two 64-row boxes: query blocks (a, b) and key
// blocks (j1, j2); a missing second block is read from outside the tensor,
// which the copy fills with zeros.
template <int BS, int D, bool PAIR, bool F8>
__device__ void producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const FwdParams& p,
                         uint8_t* sQ, uint8_t* sT, Ctrl* c, volatile WaitFlag* abort) {
    using C = Cfg<BS, D>;
    constexpr int KB = PAIR ? BS / 2 : BS;  // rows of one box (one key or query block)
    const int lane = threadIdx.x & 31;
    const bool leader = elect_one();
    uint32_t tt = 0, nq = 0;
    bool ok = true;
    for (uint32_t it = 0; ok; ++it) {
        const uint32_t slot = it & 3;
        if (!warp_wait(&c->item_full[slot], (it >> 2) & 1, abort)) break;
        const int item = c->ring[slot][0];
        const int beg = c->ring[slot][3], end = c->ring[slot][4];
        const int ra = c->ring[slot][5], ib = c->ring[slot][6];
        const bool crow = c->ring[slot][8] != 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->item_empty[slot]);
        if (item < 0) break;
        const int bh = ra / p.nb;
        const int i = ra - bh * p.nb;
        const int row0 = bh * p.N;      // query rows of this head
        const int krow0 = bh * p.Nk;    // key / value rows of this head
        const uint32_t qb = it & 1;
        if (!warp_wait(&c->q_empty[qb], ((it >> 1) & 1) ^ 1, abort)) break;
        if (leader) {
            mbar_arrive_expect_tx(&c->q_full[qb], F8 ? C::TX_BYTES_F8 : C::TX_BYTES);
#pragma unroll
            for (int b = 0; b < (F8 ? 1 : C::NBOX); ++b) {
                uint8_t* dst = sQ + qb * C::Q_BYTES + b * C::Q_BOX;
                tma_load_2d(dst, tq, &c->q_full[qb], b * 64, row0 + i * KB);
                if (PAIR) tma_load_2d(dst + KB * 128, tq, &c->q_full[qb], b * 64, ib >= 0 ? row0 + ib * KB : -KB);
            }
        }
        ++nq;
        // K and V tiles of key block j1 (and j2 in the paired form; -1: none)
        auto issue = [&](int j1, int j2) -> bool {
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t t = tt % C::NT;
                if (!warp_wait(&c->t_empty[t], ((tt / C::NT) & 1) ^ 1, abort)) return false;
                if (leader) {
                    const bool k8 = F8 && kv == 0;  // an e4m3 K tile: one box
                    mbar_arrive_expect_tx(&c->t_full[t], k8 ? C::TX_BYTES_F8 : C::TX_BYTES);
#pragma unroll
                    for (int b = 0; b < C::NBOX; ++b) {
                        if (k8 && b > 0) break;
                        uint8_t* dst = sT + t * C::T_BYTES + b * C::T_BOX;
                        tma_load_2d(dst, kv ? tv : tk, &c->t_full[t], b * 64, krow0 + j1 * KB);
                        if (PAIR)
                            tma_load_2d(dst + KB * 128, kv ? tv : tk, &c->t_full[t], b * 64,
                                        j2 >= 0 ? krow0 + j2 * KB : -KB);
                    }
                }
                ++tt;
            }
            return true;
        };
        int held = -1;  // paired form: first block of the next tile
        for (int e0 = beg; e0 < end && ok; e0 += 32) {
            const int e = e0 + lane;
            int j;
            unsigned vm;
            if (PAIR && ib >= 0) {
                // a pair's union: every entry is valid
                j = e < end ? (int)(p.slots[e] & 0x3fffffffu) : -1;
                vm = __ballot_sync(0xffffffffu, e < end);
            } else {
                j = e < end ? p.col_idx[e] : -1;
                vm = __ballot_sync(0xffffffffu, e < end && block_ok(p, j, i, crow));
            }
            while (vm) {
                const int src = __ffs(vm) - 1;
                vm &= vm - 1;
                const int jb = __shfl_sync(0xffffffffu, j, src);
                if (!PAIR) {
                    ok = issue(jb, -1);
                } else if (held < 0) {
                    held = jb;
                } else {
                    ok = issue(held, jb);
                    held = -1;
                }
                if (!ok) break;
            }
        }
        if (PAIR && ok && held >= 0) ok = issue(held, -1);
    }
    if (leader) {
        // The copies still in flight must land before the CTA exits: after an
        // abort, or when another role aborts after this loop ended.  (In a
        // normal run every one of them has landed and these waits return at
        // once.)
        for (uint32_t n = (tt > (uint32_t)C::NT ? tt - C::NT : 0); n < tt; ++n)
            mbar_wait_drain(&c->t_full[n % C::NT], (n / C::NT) & 1);
        for (uint32_t n = (nq > 2 ? nq - 2 : 0); n < nq; ++n) mbar_wait_drain(&c->q_full[n & 1], (n >> 1) & 1);
    }
}

// ---------------------------------------------------------------- MMA issuer
// The whole warp runs the loop (waits, descriptors); the elected lane issues
// the MMAs and the commits that track them.  The last PV of a row also
// signals its O buffer complete: the epilogue waits on that per-buffer
// barrier, not on the per-step one, whose phase may move on by two steps
// (the next row's) before an epilogue that lags behind gets to it.
template <int BS, int D>
__device__ bool issue_pv(uint8_t* sT, Ctrl* c, uint32_t tmem, volatile WaitFlag* abort, bool leader, uint32_t gp,
                         uint32_t vseq, bool first, bool last, uint32_t it) {
    using C = Cfg<BS, D>;
    constexpr uint64_t VDESC = sdesc_sw128_base(C::T_BOX, 1024);
    const uint32_t sb = gp & 1;
    const uint32_t vt = vseq % C::NT;
    const uint32_t ob = it & 1;
    if (!warp_wait(&c->t_full[vt], (vseq / C::NT) & 1, abort)) return false;
    // the first PV of a row overwrites its O buffer: the epilogue of the row
    // that used the buffer before must have read it
    if (first && it >= 2 && !warp_wait(&c->o_free[ob], ((it >> 1) & 1) ^ 1, abort)) return false;
    if (!warp_wait(&c->p_full[sb], (gp >> 1) & 1, abort)) return false;
    tc_fence_after();
    // V rows (keys) 16kk ..: MN-major B operand, 2 groups of 8 swizzled
    // 128-byte rows (SBO = 1024); the next 64 columns of D live in the next
    // box (LBO = box size).  P of key half h sits in the first BS/4 columns
    // of that half of the S buffer.
    const uint64_t vdesc = VDESC + (smem_u32(sT + vt * C::T_BYTES) >> 4);
    if (leader) {
#pragma unroll
        for (int kk = 0; kk < BS / 16; ++kk) {
            const int h = kk / (C::H2 / 16), k2 = kk % (C::H2 / 16);
            mma_ts(tmem + C::O_COL + ob * D, tmem + C::S_COL + sb * BS + h * C::H2 + k2 * 8,
                   vdesc + (uint64_t)((kk * 16 * 128) >> 4), C::IDESC_PV, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(&c->pv_done[sb]);
        mma_commit(&c->t_empty[vt]);
        if (last) mma_commit(&c->o_full[ob]);
    }
    __syncwarp();
    return true;
}

template <int BS, int D, bool F8>
__device__ void mma_issuer(const FwdParams& p, uint8_t* sQ, uint8_t* sT, Ctrl* c, uint32_t tmem,
                           volatile WaitFlag* abort) {
    using C = Cfg<BS, D>;
    // Q and K tiles are K-major with 128-byte swizzle: 16 columns (32 bytes)
    // per MMA inside a box, the next box every 4 steps.
    constexpr uint64_t KDESC = sdesc_sw128_base(16, 1024);
    const int lane = threadIdx.x & 31;
    const bool leader = elect_one();
    uint32_t g = 0, tt = 0;
    bool pend = false, pend_first = false, pend_last = false, ok = true;
    uint32_t pend_g = 0, pend_v = 0, pend_it = 0;
    for (uint32_t it = 0; ok; ++it) {
        const uint32_t slot = it & 3;
        if (!warp_wait(&c->item_full[slot], (it >> 2) & 1, abort)) {
            ok = false;
            break;
        }
        const int item = c->ring[slot][0];
        const uint32_t n = (uint32_t)c->ring[slot][1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->item_empty[slot]);
        if (item < 0) break;
        if (n == 0) continue;  // a row without blocks: the epilogue writes zeros
        const uint32_t qb = it & 1;
        // Q is awaited only by rows that use it: a row without blocks lets the
        // epilogue release its Q buffer at once.
        if (!warp_wait(&c->q_full[qb], (it >> 1) & 1, abort)) {
            ok = false;
            break;
        }
        const uint64_t qdesc = KDESC + (smem_u32(sQ + qb * C::Q_BYTES) >> 4);
        for (uint32_t e = 0; e < n; ++e) {
            const uint32_t kseq = tt, vseq = tt + 1;
            tt += 2;
            const uint32_t kt = kseq % C::NT;
            if (!warp_wait(&c->t_full[kt], (kseq / C::NT) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sb = g & 1;
            const uint64_t kdesc = KDESC + (smem_u32(sT + kt * C::T_BYTES) >> 4);
            if (leader) {
                if (F8) {
                    // e4m3: 32 elements (32 bytes) of the single 128-byte box per MMA
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk)
                        mma_ss_f8(tmem + C::S_COL + sb * BS, qdesc + (uint64_t)((kk * 32) >> 4),
                                  kdesc + (uint64_t)((kk * 32) >> 4), C::IDESC_QK_F8, kk > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t qoff = (uint64_t)(((kk >> 2) * C::Q_BOX + (kk & 3) * 32) >> 4);
                        const uint64_t koff = (uint64_t)(((kk >> 2) * C::T_BOX + (kk & 3) * 32) >> 4);
                        mma_ss(tmem + C::S_COL + sb * BS, qdesc + qoff, kdesc + koff, C::IDESC_QK,
                               kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&c->s_full[sb]);
                mma_commit(&c->t_empty[kt]);
            }
            __syncwarp();
            if (pend && !issue_pv<BS, D>(sT, c, tmem, abort, leader, pend_g, pend_v, pend_first, pend_last, pend_it)) {
                ok = false;
                break;
            }
            pend = true;
            pend_g = g;
            pend_v = vseq;
            pend_first = (e == 0);
            pend_last = (e + 1 == n);
            pend_it = it;
            ++g;
        }
    }
    if (ok && pend) issue_pv<BS, D>(sT, c, tmem, abort, leader, pend_g, pend_v, pend_first, pend_last, pend_it);
    // Every MMA this warp issued must finish before TMEM is freed.
    if (leader) {
        mma_commit(&c->drain);
        mbar_wait_drain(&c->drain, 0);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- softmax
// P = 2^(s * scale * log2(e) - m) for this thread's half row, written as bf16
// pairs over the S columns it came from (chunk c lands in columns
// [16c, 16c + 16) of the half); fp32 and bf16-rounded sums added to l2, lr2.
template <int NCH>
__device__ __forceinline__ void exp_store(const uint32_t (&sr)[NCH][32], f2 sl2, float m, uint32_t t_p, f2& l2,
                                          f2& lr2) {
    const f2 nm2 = {-m, -m};
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            const f2 sv = {__uint_as_float(sr[ch][2 * x]), __uint_as_float(sr[ch][2 * x + 1])};
            const f2 t = fma2(sv, sl2, nm2);
            const f2 pv = {ex2_approx(t.x), ex2_approx(t.y)};
            l2 = add2(l2, pv);
            pk[x] = pack_bf16x2(pv.x, pv.y);
            add_bf16x2_f32(pk[x], lr2.x, lr2.y);
        }
        tmem_st16(t_p + ch * 16, pk);
    }
}

// Multiply this thread's D/2 columns of an O row (TMEM) by alpha.
template <int D>
__device__ __forceinline__ void rescale_o_half(uint32_t t_o, float alpha) {
#pragma unroll 1
    for (int ch = 0; ch < D / 64; ++ch) {
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

// Warpgroup h, thread t: query row t, key columns [h*BS/2, (h+1)*BS/2).  In
// the paired form row t belongs to query block a (t < 64) or b, and column
// half h to the step's key block j_h: a key block absent from the row's list
// masks the whole half row.
// SC (FP8 scores with per-block scales): the logit scale of a step is
// scale * log2(e) * q_descale[query block of the row] * k_descale[key block of
// the thread's column half], so every thread follows the key blocks of its
// steps: the valid entries of the CSR row in order (a pair: the union's
// entries 2e + h), 32 at a time, their descale factors loaded by the lanes
// and handed out with a shuffle.
template <int BS, int D, bool PAIR, bool SC = false>
__device__ void softmax_role(const FwdParams& p, uint8_t* sQ, float* xch_base, Ctrl* c, uint32_t tmem,
                             volatile WaitFlag* abort) {
    using C = Cfg<BS, D>;
    constexpr int NCH = C::H2 / 32;  // 32-column chunks per half
    const int h = threadIdx.x >> 7;          // 0 or 1
    const int tid = threadIdx.x & 127;       // row in the tile = TMEM lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::S_COL + h * C::H2;         // my half of S
    const uint32_t t_o = tmem + lane_base + C::O_COL + h * (D / 2);       // my half of O's columns (+ buffer)
    const int col0 = h * C::H2;
    const f2 sl2 = {p.scale_log2, p.scale_log2};
    uint32_t g = 0;
    bool ok = true;
    // Rows of the unpaired bf16 / per-tensor FP8 form read the next claimed item one row ahead
    // (during the first step of the current row, where the warp would
    // otherwise wait for S), so that a row transition does not wait for the
    // ring (long_window_128k forward -1.8 %, window_16k -0.9 %).  The paired
    // form and per-block FP8 scales read each row's item at its start: holding
    // the next item's fields across the row spills registers there
    // (content_topk +3 %).
    constexpr bool AHEAD = !PAIR && !SC;
    struct RowItem {
        int item, diag, pbeg, pend, ra, ib, nent, rdsel;
        uint32_t n, rsel;
        bool crow;
    };
    auto read_item = [&](uint32_t k, RowItem& r) -> bool {
        const uint32_t slot = k & 3;
        if (!warp_wait(&c->item_full[slot], (k >> 2) & 1, abort)) return false;
        r.item = c->ring[slot][0];
        r.n = (uint32_t)c->ring[slot][1];
        r.diag = c->ring[slot][2];
        r.pbeg = c->ring[slot][3];
        r.pend = c->ring[slot][4];
        r.ra = c->ring[slot][5];
        r.ib = c->ring[slot][6];
        r.nent = c->ring[slot][7];
        r.crow = c->ring[slot][8] != 0;
        // a pair's masks for this thread's query half (tid >> 6) and column half
        r.rsel = PAIR ? (uint32_t)c->ring[slot][9 + 2 * (tid >> 6) + h] : 0u;
        r.rdsel = PAIR ? c->ring[slot][13 + 2 * (tid >> 6) + h] : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->item_empty[slot]);
        return true;
    };
    RowItem nxt;
    bool have_next = AHEAD ? read_item(0, nxt) : true;
    for (uint32_t it = 0; ok && have_next; ++it) {
        if (!AHEAD && !read_item(it, nxt)) break;
        const RowItem cur = nxt;
        if (cur.item < 0) break;
        bool fetched = !AHEAD;  // the next row's item (read one row ahead)
        const uint32_t n = cur.n;
        const int diag = cur.diag, pbeg = cur.pbeg, pend = cur.pend, ra = cur.ra, ib = cur.ib, nent = cur.nent;
        const bool crow = cur.crow;
        const uint32_t ring_sel = cur.rsel;
        const int ring_dsel = cur.rdsel;
        // Per-block FP8 scales: this thread's query-block factor, and the key
        // blocks of the coming steps (cursor over the valid entries).
        float qsl = 0.f;
        int cur_e0 = pbeg;
        unsigned cur_vm = 0u;
        float cur_kd = 0.f, pkd0 = 0.f, pkd1 = 0.f;
        const int bh_it = ra / p.nb;
        auto refill = [&]() {
            while (cur_vm == 0u && cur_e0 < pend) {
                const int e = cur_e0 + lane;
                const int j = e < pend ? p.col_idx[e] : -1;
                const bool okj = e < pend && block_ok(p, j, ra - bh_it * p.nb, crow);
                cur_vm = __ballot_sync(0xffffffffu, okj);
                cur_kd = okj ? p.k_descale[(size_t)bh_it * p.nbk + j] : 0.f;
                cur_e0 += 32;
            }
        };
        // Descale of the next valid entry; 1 when none is left (a masked half
        // then still multiplies -inf by a positive factor).
        auto next_kd = [&]() -> float {
            refill();
            const int src = cur_vm ? __ffs(cur_vm) - 1 : 0;
            const float v = __shfl_sync(0xffffffffu, cur_kd, src);
            const bool had = cur_vm != 0u;
            cur_vm &= cur_vm - 1u;
            return had ? v : 1.f;
        };
        if (SC) {
            const int qrow = (PAIR && (tid >> 6) && ib >= 0) ? bh_it * p.nb + ib : ra;
            qsl = p.q_descale[qrow] * p.scale_log2;
            if (PAIR && ib >= 0) {
                // a pair's union: lane l holds entries l and 32 + l
                const uint32_t u0 = lane < nent ? p.slots[pbeg + lane] : 0u;
                const uint32_t u1 = 32 + lane < nent ? p.slots[pbeg + 32 + lane] : 0u;
                pkd0 = lane < nent ? p.k_descale[(size_t)bh_it * p.nbk + (u0 & 0x3fffffffu)] : 1.f;
                pkd1 = 32 + lane < nent ? p.k_descale[(size_t)bh_it * p.nbk + (u1 & 0x3fffffffu)] : 1.f;
            } else {
                refill();
            }
        }
        // Paired form, per step e of this column half h (entry k = 2e + h):
        //   pair:   sel bit e = entry allowed for this row's query block,
        //           dsel bit e = entry is that block's diagonal (causal);
        //   single: sel = steps holding an entry (rows 64-127: none),
        //           dsel = step of the diagonal or -1.
        // A pair's union has at most 64 entries, so 32 steps fit the masks.
        const bool pair = PAIR && ib >= 0;
        uint32_t sel = 0;
        int dsel = -1;
        if (PAIR) {
            const int qh = tid >> 6;
            if (pair) {
                // the claimer's masks for this query half and column half
                sel = ring_sel;
                dsel = ring_dsel;
            } else {
                sel = qh == 0 ? (uint32_t)((nent - h + 1) >> 1) : 0u;
                dsel = (qh == 0 && diag >= 0 && (diag & 1) == h) ? diag >> 1 : -1;
            }
        }
        // l: fp32 sum of this half's exponentials (LSE).  lr: the same values
        // after rounding to bf16 -- the weights the PV MMA uses -- so that
        // O / lr is an exact convex combination of them.
        float m_used = -INFINITY;
        f2 l2 = {0.f, 0.f}, lr2 = {0.f, 0.f};
        uint32_t s = 0;
        for (uint32_t e = 0; e < n; ++e) {
            const uint32_t sb = g & 1;
            // this step's logit scale (log2 domain) for this thread's half
            float sl_e = p.scale_log2;
            if (SC) {
                float kd;
                if (PAIR && ib >= 0) {
                    const int k = 2 * (int)e + h;
                    const float a = __shfl_sync(0xffffffffu, pkd0, k & 31);
                    const float b = __shfl_sync(0xffffffffu, pkd1, k & 31);
                    kd = k < 32 ? a : b;
                } else if (PAIR) {
                    const float k0 = next_kd(), k1 = next_kd();
                    kd = h ? k1 : k0;
                } else {
                    kd = next_kd();
                }
                sl_e = qsl * kd;
            }
            const f2 sl2_e = {sl_e, sl_e};
            if (!fetched) {
                fetched = true;
                if (!(have_next = read_item(it + 1, nxt))) {
                    ok = false;
                    break;
                }
            }
            if (!warp_wait(&c->s_full[sb], (g >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            bool is_diag = (int)e == diag, masked = false;
            if (PAIR) {
                if (pair) {
                    masked = ((sel >> e) & 1u) == 0u;
                    is_diag = ((uint32_t)dsel >> e) & 1u;
                } else {
                    masked = e >= sel;
                    is_diag = (int)e == dsel;
                }
            }
            uint32_t sr[NCH][32];
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) tmem_ld32(t_s + sb * BS + ch * 32, sr[ch]);
            tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) reg_fence(sr[ch]);
            if (masked || is_diag) {
                // Columns x + 32 ch > lim of this half row are masked: all of
                // them for a key block the row does not list (lim = -1); in the
                // diagonal block the token-level causal mask, key column col0 +
                // 32 ch + x after query row tid (paired form: within the row's
                // own 64-token block, lim = tid mod 64).
                const int lim = masked ? -1 : (PAIR ? (tid & 63) : tid - col0);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const int k = lim - ch * 32;
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (x > k) sr[ch][x] = __float_as_uint(-INFINITY);
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float a = __uint_as_float(sr[ch][0]), b = __uint_as_float(sr[ch][1]);
#pragma unroll
                for (int x = 2; x < 32; x += 4) {
                    a = fmax3(a, __uint_as_float(sr[ch][x]), __uint_as_float(sr[ch][x + 1]));
                    b = fmax3(b, __uint_as_float(sr[ch][x + 2]), __uint_as_float(sr[ch][x + 3]));
                }
                mx = fmax3(mx, a, b);
            }
            // Publish this half's row max to the partner warp (same rows, other
            // half): both halves use one running max so they can share one O.
            // (per-block scales: the halves' factors differ, so the scaled max
            // is exchanged; the scale is positive, so scaling commutes with max)
            const float mxs = SC ? mx * sl_e : mx;
            float* xch = xch_base + sb * 256;
            xch[h * 128 + tid] = mxs;
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->mx_full[warp & 3][sb]);
            const float sl = p.scale_log2;
            const uint32_t t_p = t_s + sb * BS;
            const uint32_t t_oh = t_o + (it & 1) * D;
            // The running max changes only when the row max grows by more than
            // 2^8.  A warp none of whose rows grew here exponentiates at once
            // with the current max and checks the partner's max afterwards
            // (its own exponents stay <= 2^8 either way); otherwise it waits
            // for the exchange first.
            const bool exact_path = (s == 0) || __any_sync(0xffffffffu, (SC ? mxs : mx * sl) > m_used + 8.f);
            if (exact_path) {
                if (!warp_wait(&c->mx_full[warp & 3][sb], (g >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                // same value in both halves
                const float mtot = SC ? fmaxf(mxs, xch[(1 - h) * 128 + tid]) : fmaxf(mx, xch[(1 - h) * 128 + tid]) * sl;
                float alpha = 1.f;
                bool need = false;
                if (s == 0) {
                    m_used = mtot;
                } else if (mtot > m_used + 8.f) {
                    alpha = ex2_approx(m_used - mtot);
                    m_used = mtot;
                    const f2 a2 = {alpha, alpha};
                    l2 = mul2(l2, a2);
                    lr2 = mul2(lr2, a2);
                    need = true;
                }
                if (__any_sync(0xffffffffu, need)) {
                    // rescale this half's columns of O once PV_{g-1} has landed
                    const uint32_t gp = g - 1;
                    if (!warp_wait(&c->pv_done[gp & 1], (gp >> 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    rescale_o_half<D>(t_oh, alpha);
                }
                exp_store<NCH>(sr, SC ? sl2_e : sl2, m_used == -INFINITY ? 0.f : m_used, t_p, l2, lr2);
            } else {
                f2 ls2 = {0.f, 0.f}, lrs2 = {0.f, 0.f};
                // (a row with nothing allowed yet has no max: any finite reference works)
                exp_store<NCH>(sr, SC ? sl2_e : sl2, m_used == -INFINITY ? 0.f : m_used, t_p, ls2, lrs2);
                if (!warp_wait(&c->mx_full[warp & 3][sb], (g >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                const float mtot = SC ? fmaxf(mxs, xch[(1 - h) * 128 + tid]) : fmaxf(mx, xch[(1 - h) * 128 + tid]) * sl;
                const bool upd = mtot > m_used + 8.f;  // the partner's max grew
                if (__any_sync(0xffffffffu, upd)) {
                    // Rare: bring this step's P (already in TMEM), its sums, the
                    // earlier sums and this half of O to the new max.
                    const float alpha = upd ? ex2_approx(m_used - mtot) : 1.f;
                    if (upd) m_used = mtot;
                    tmem_wait_st();
                    const f2 a2 = {alpha, alpha};
                    lrs2 = {0.f, 0.f};
#pragma unroll 1
                    for (int ch = 0; ch < NCH; ++ch) {
                        uint32_t pk[16];
                        tmem_ld16(t_p + ch * 16, pk);
                        tmem_wait_ld();
                        reg_fence(pk);
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const f2 pv = mul2({__uint_as_float(pk[x] << 16), __uint_as_float(pk[x] & 0xffff0000u)}, a2);
                            pk[x] = pack_bf16x2(pv.x, pv.y);
                            add_bf16x2_f32(pk[x], lrs2.x, lrs2.y);
                        }
                        tmem_st16(t_p + ch * 16, pk);
                    }
                    ls2 = mul2(ls2, a2);
                    l2 = mul2(l2, a2);
                    lr2 = mul2(lr2, a2);
                    const uint32_t gp = g - 1;
                    if (!warp_wait(&c->pv_done[gp & 1], (gp >> 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    rescale_o_half<D>(t_oh, alpha);
                }
                l2 = add2(l2, ls2);
                lr2 = add2(lr2, lrs2);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->p_full[sb]);
            ++g;
            ++s;
        }
        if (!ok) break;
        if (!fetched && !(have_next = read_item(it + 1, nxt))) break;  // a row without steps
        // hand (m, l, lr) of this half to the epilogue through the consumed
        // Q tile of the row (its QK MMAs have all completed: S_last is full)
        const uint32_t qb = it & 1;
        if (!warp_wait(&c->stats_empty[qb], ((it >> 1) & 1) ^ 1, abort)) break;
        if (s > 0) {
            float* st = reinterpret_cast<float*>(sQ + qb * C::Q_BYTES);
            if (h == 0) st[tid] = m_used;
            st[(1 + h) * 128 + tid] = l2.x + l2.y;
            st[(3 + h) * 128 + tid] = lr2.x + lr2.y;
            fence_proxy_async_smem();  // this Q tile is later rewritten by TMA
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->stats_full[qb]);
    }
    // An abort can leave this warp's last P stores in flight: they must land
    // before TMEM is freed.
    tmem_wait_st();
}

// ---------------------------------------------------------------- epilogue
// Thread tid of the four epilogue warps owns query row tid of the tile.  O is
// divided by lr, rounded to bf16 and staged in the row's consumed Q tile in
// the 128-byte swizzled layout of the O tensor map (16-byte chunk c of row r
// at r * 128 + ((c ^ (r & 7)) << 4) within each 64-column box), then written
// by one TMA store, so the O traffic leaves the SM as whole lines instead of
// 32 scattered rows per store instruction.  The softmax statistics sit in
// the same tile: all four warps read theirs before any warp stages O.  In the
// paired form rows 0-63 belong to query block a and rows 64-127 to block b,
// stored by one 64-row box each.
template <int BS, int D, bool PAIR>
__device__ void epilogue_role(const CUtensorMap* to, const FwdParams& p, uint8_t* sQ, Ctrl* c, uint32_t tmem,
                              volatile WaitFlag* abort) {
    using C = Cfg<BS, D>;
    const int tid = threadIdx.x & 127;  // row in the tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_o0 = tmem + lane_base + C::O_COL;
    const bool storer = warp == kEpiWarp0;
    const bool leader = storer && elect_one();
    uint32_t o_phase = 0;  // bit b: parity of the next completion of O buffer b
    for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it & 3;
        if (!warp_wait(&c->item_full[slot], (it >> 2) & 1, abort)) break;
        const int item = c->ring[slot][0];
        const int n = c->ring[slot][1];
        const int ra = c->ring[slot][5], ib = c->ring[slot][6];
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->item_empty[slot]);
        if (item < 0) break;
        const int bh = ra / p.nb;
        const int i = ra - bh * p.nb;
        constexpr int KB = PAIR ? BS / 2 : BS;  // rows of one query block
        const int qh = PAIR ? tid >> 6 : 0;
        const int i_my = qh ? ib : i;
        const bool row_valid = PAIR ? (qh == 0 || ib >= 0) : tid < BS;
        const uint32_t qb = it & 1;
        uint8_t* stage = sQ + qb * C::Q_BYTES;
        if (!warp_wait(&c->q_full[qb], (it >> 1) & 1, abort)) break;
        if (!warp_wait(&c->stats_full[qb], (it >> 1) & 1, abort)) break;
        float m = 0.f, l = 0.f, lr = 1.f;
        if (n > 0) {
            const float* st = reinterpret_cast<const float*>(stage);
            m = st[tid];
            l = st[128 + tid] + st[256 + tid];
            lr = st[384 + tid] + st[512 + tid];
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&c->stats_empty[qb]);
            mbar_arrive(&c->ep_sync);
        }
        if (!warp_wait(&c->ep_sync, it & 1, abort)) break;
        const size_t row = (size_t)bh * p.N + (size_t)i_my * KB + (PAIR ? (tid & 63) : tid);
        float lse_v = -INFINITY;
        const uint32_t xr = (uint32_t)(tid & 7);
        uint8_t* my_row = stage + tid * 128;
        if (n > 0) {
            // rows without blocks issue no PV and leave their buffer's phase alone
            if (!warp_wait(&c->o_full[it & 1], (o_phase >> (it & 1)) & 1u, abort)) break;
            o_phase ^= 1u << (it & 1);
            tc_fence_after();
            // a row none of whose keys were allowed (possible in the paired
            // form) gets O = 0 and LSE = -inf
            const float inv = lr > 0.f ? 1.f / lr : 0.f;
            const f2 inv2 = {inv, inv};
            lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            const uint32_t t_o = t_o0 + (it & 1) * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(t_o + ch * 32, o);
                tmem_wait_ld();
                reg_fence(o);
                if (p.out_f32) {
                    // fp32 output (partial results that are merged later):
                    // the row's 32 values straight to global memory
                    if (row_valid) {
                        float4* dst = reinterpret_cast<float4*>(p.out_f32 + row * D + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4) {
                            const f2 a = mul2({__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1])}, inv2);
                            const f2 b = mul2({__uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3])}, inv2);
                            dst[v4] = make_float4(a.x, a.y, b.x, b.y);
                        }
                    }
                    continue;
                }
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const f2 u = {__uint_as_float(o[2 * x]), __uint_as_float(o[2 * x + 1])};
                    const f2 r = mul2(u, inv2);
                    pk[x] = pack_bf16x2(r.x, r.y);
                }
                if (row_valid) {
                    uint8_t* box = my_row + (ch >> 1) * C::Q_BOX;
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const uint32_t cidx = (uint32_t)((ch & 1) * 4 + v4);
                        *reinterpret_cast<uint4*>(box + ((cidx ^ xr) << 4)) =
                            make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
        } else if (row_valid) {
            if (p.out_f32) {
                float4* dst = reinterpret_cast<float4*>(p.out_f32 + row * D);
#pragma unroll 1
                for (int v4 = 0; v4 < D / 4; ++v4) dst[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
#pragma unroll 1
                for (int b = 0; b < C::NBOX; ++b)
#pragma unroll
                    for (int cidx = 0; cidx < 8; ++cidx)
                        *reinterpret_cast<uint4*>(my_row + b * C::Q_BOX + (cidx << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (row_valid) p.lse[row] = lse_v;
        // the staged O is read by the TMA (async proxy)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&c->o_free[it & 1]);
            mbar_arrive(&c->o_staged);
        }
        if (storer) {
            if (!warp_wait(&c->o_staged, it & 1, abort)) break;
            if (leader && !p.out_f32) {
                const int y = bh * p.N + i * KB;
#pragma unroll
                for (int b = 0; b < C::NBOX; ++b) {
                    tma_store_2d(to, stage + b * C::Q_BOX, b * 64, y);
                    if (PAIR && ib >= 0) tma_store_2d(to, stage + b * C::Q_BOX + KB * 128, b * 64, bh * p.N + ib * KB);
                }
                bulk_commit_group();
                bulk_wait_read_all();  // the Q tile may be reloaded now
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->q_empty[qb]);
        }
    }
    if (leader) bulk_wait_all();
}

// ---------------------------------------------------------------- kernel
// PAIR: the paired form for 64-token blocks, run on the 128-row geometry
// (BS = 128): two query blocks per tile, two key blocks per step.
// F8: Q and K are e4m3 (D = 128) and S = Q K^T runs as kind::f8f6f4; the
// descale factors of Q and K are folded into the score scale by the host.
template <int BS, int D, bool PAIR, bool F8 = false, bool SC = false>
__global__ void __launch_bounds__(kThreads, 1)
    bsa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                   const FwdParams p) {
    using C = Cfg<BS, D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & (kAlign - 1)) {
        // the swizzled tiles need a 1024-byte aligned base; fail loudly
        if (threadIdx.x == 0) atomicOr(p.err, ERR_LAUNCH);
        return;
    }
    uint8_t* sQ = smem_raw;
    uint8_t* sT = sQ + C::NQ * C::Q_BYTES;
    Ctrl* c = reinterpret_cast<Ctrl*>(sT + C::NT * C::T_BYTES);
    float* xch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(c) + kCtrlBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 4; ++x) {
            mbar_init(&c->item_full[x], 1);
            mbar_init(&c->item_empty[x], kConsumerWarps);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&c->q_full[x], 1);
            mbar_init(&c->q_empty[x], 1);
            mbar_init(&c->s_full[x], 1);
            mbar_init(&c->p_full[x], kSoftmaxWarps);
            mbar_init(&c->o_free[x], 4);
            mbar_init(&c->pv_done[x], 1);
            mbar_init(&c->o_full[x], 1);
            for (int w = 0; w < 4; ++w) mbar_init(&c->mx_full[w][x], 2);
        }
        for (int x = 0; x < C::NT; ++x) {
            mbar_init(&c->t_full[x], 1);
            mbar_init(&c->t_empty[x], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&c->stats_full[x], kSoftmaxWarps);
            mbar_init(&c->stats_empty[x], 4);
        }
        mbar_init(&c->ep_sync, 4);
        mbar_init(&c->o_staged, 4);
        mbar_init(&c->drain, 1);
        c->wf.abort = 0;
        c->wf.limit_ns = p.wait_limit_ns;
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
    if (warp == kMmaWarp) {
        tmem_alloc(&c->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == kEpiWarp0 && lane == 0) tma_prefetch_desc(&to);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c->tmem_base;
    volatile WaitFlag* abort = &c->wf;

    if (warp == kClaimWarp) {
        claimer<PAIR>(p, c, abort);
    } else if (warp == kProducerWarp) {
        producer<BS, D, PAIR, F8>(&tq, &tk, &tv, p, sQ, sT, c, abort);
    } else if (warp == kMmaWarp) {
        mma_issuer<BS, D, F8>(p, sQ, sT, c, tmem, abort);
    } else if (warp >= kEpiWarp0) {
        epilogue_role<BS, D, PAIR>(&to, p, sQ, c, tmem, abort);
    } else {
        softmax_role<BS, D, PAIR, SC>(p, sQ, xch, c, tmem, abort);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && c->wf.abort) atomicOr(p.err, ERR_TIMEOUT);
}

template <int BS, int D, bool PAIR = false, bool F8 = false, bool SC = false>
cudaError_t launch_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                        const FwdParams& p, int grid, cudaStream_t stream) {
    using C = Cfg<BS, D>;
    cudaError_t e = cudaFuncSetAttribute(bsa_fwd_kernel<BS, D, PAIR, F8, SC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // Dependent launch: the kernel's prologue (barriers, TMEM, descriptors)
    // overlaps the schedule kernel; its claimer waits for the schedule.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bsa_fwd_kernel<BS, D, PAIR, F8, SC>, tq, tk, tv, to, p);
}

// ---------------------------------------------------------------- schedule
constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kSchedBins = 64;  // length classes: 0..47 exact, then half octaves (48-63, 64-95, 96-127, ...)

__device__ __forceinline__ int sched_bin(int len) {
    int cls;
    if (len < 48) {
        cls = len < 0 ? 0 : len;
    } else {
        const int e = 31 - __clz(len);          // floor(log2 len) >= 5
        const int h = (len >> (e - 1)) & 1;     // upper half of the octave
        const int k = 2 * (e - 5) + h - 1;      // 48..63 -> 0, 64..95 -> 1, 96..127 -> 2, ...
        cls = 48 + (k < 15 ? k : 15);
    }
    return kSchedBins - 1 - cls;  // ascending bin = descending row length
}

// Longest-first, stable order of the R rows: a counting sort on the row
// length (exact below 48 blocks, half-octave classes above), ties kept in row
// order so the CTAs running at the same time share a head's K/V in L2.  One
// CTA; each warp owns a contiguous segment of rows, so the only shared state
// is a [warp][class] count table.  Row lengths are first staged in shared
// memory with coalesced loads when they fit (STAGED).  Also zeroes the
// forward kernel's work counter.
// LENS: lengths given directly (src = lens[0 .. *n_dev)) instead of as
// row_ptr differences, sorted in classes of 2^lens_shift steps (empty items in
// a class of their own, last): the paired form's items come from the pairing
// pass grouped by head, and a class keeps that order, so the CTAs running
// together share few heads' K/V in L2.
template <bool STAGED, bool LENS>
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const int32_t* __restrict__ src,
                                                                 const int32_t* __restrict__ n_dev, int32_t R,
                                                                 int32_t* __restrict__ perm, int32_t* counter,
                                                                 int lens_shift) {
    if (LENS) R = min(R, *n_dev);
    __shared__ int32_t cnt[kSchedWarps][kSchedBins];
    __shared__ int32_t bin_base[kSchedBins];
    extern __shared__ int32_t lens_s[];  // [R] when STAGED
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();  // the forward may set itself up meanwhile
    if (tid == 0) *counter = 0;
    for (int x = tid; x < kSchedWarps * kSchedBins; x += kSchedThreads) (&cnt[0][0])[x] = 0;
    auto src_len = [&](int r) { return LENS ? src[r] : src[r + 1] - src[r]; };
    if (STAGED)
        for (int r = tid; r < R; r += kSchedThreads) lens_s[r] = src_len(r);
    __syncthreads();
    auto row_len = [&](int r) {
        const int len = STAGED ? lens_s[r] : src_len(r);
        return LENS ? (len > 0 ? 1 + (len >> lens_shift) : 0) : len;
    };
    const int per = (R + kSchedWarps - 1) / kSchedWarps;
    const int r0 = warp * per, r1 = min(R, r0 + per);
    // 1. per-warp class counts (each class has one leader lane per group)
    for (int base = r0; base < r1; base += 32) {
        const int r = base + lane;
        const bool valid = r < r1;
        const int key = valid ? sched_bin(row_len(r)) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (valid && lane == __ffs(peers) - 1) cnt[warp][key] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // 2. class totals -> class bases (descending length), then per-warp
    //    offsets inside each class (exclusive over warps)
    if (warp == 0) {
        int tot[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = lane + 32 * u;
            int t = 0;
            for (int w = 0; w < kSchedWarps; ++w) t += cnt[w][b];
            tot[u] = t;
        }
        // exclusive scan over the 64 classes (two per lane: b = lane, lane + 32)
        int incl0 = tot[0];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl0, o);
            if (lane >= o) incl0 += y;
        }
        const int sum0 = __shfl_sync(0xffffffffu, incl0, 31);
        int incl1 = tot[1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl1, o);
            if (lane >= o) incl1 += y;
        }
        bin_base[lane] = incl0 - tot[0];
        bin_base[lane + 32] = sum0 + incl1 - tot[1];
    }
    __syncthreads();
    if (tid < kSchedBins) {
        int run = bin_base[tid];
        for (int w = 0; w < kSchedWarps; ++w) {
            const int c = cnt[w][tid];
            cnt[w][tid] = run;
            run += c;
        }
    }
    __syncthreads();
    // 3. scatter, stable inside each warp's segment
    for (int base = r0; base < r1; base += 32) {
        const int r = base + lane;
        const bool valid = r < r1;
        const int key = valid ? sched_bin(row_len(r)) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (valid) {
            const int pos = cnt[warp][key] + __popc(peers & ((1u << lane) - 1u));
            perm[pos] = r;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) cnt[warp][key] += __popc(peers);
        __syncwarp();
    }
    if (LENS) {
        // The final claims, longest first: classes keep the items' head order
        // for L2 locality, which leaves the end of the launch to whatever
        // lengths come last; the last min(R, kSchedThreads) entries are
        // re-sorted by length (descending, ties in their order) so the last
        // CTAs to finish get the shortest items.
        __shared__ uint64_t tkey[kSchedThreads];
        __shared__ int32_t tval[kSchedThreads];
        __syncthreads();  // this CTA's perm writes are visible to its threads
        const int T = min(R, kSchedThreads);
        const int base = R - T;
        int n2 = 1;
        while (n2 < T) n2 <<= 1;
        if (tid < n2) {
            uint64_t key = 0;  // padding: below every real key
            if (tid < T) {
                const int32_t item = perm[base + tid];
                const uint32_t len = (uint32_t)max(STAGED ? lens_s[item] : src_len(item), 0);
                tval[tid] = item;
                key = ((uint64_t)len << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)tid);
            }
            tkey[tid] = key;
        }
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                if (tid < n2) {
                    const int o = tid ^ j;
                    if (o > tid) {
                        const uint64_t x = tkey[tid], y = tkey[o];
                        const bool desc = (tid & k) == 0;
                        if (desc ? x < y : x > y) {
                            tkey[tid] = y;
                            tkey[o] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        if (tid < T) perm[base + tid] = tval[0xFFFFFFFFu - (uint32_t)tkey[tid]];
    }
}

}  // namespace

int fwd_smem_bytes(int block, int D, bool paired) {
    if (paired && block == 64 && D == 128) return Cfg<128, 128>::SMEM;
    if (paired && block == 64 && D == 64) return Cfg<128, 64>::SMEM;
    if (block == 128 && D == 128) return Cfg<128, 128>::SMEM;
    if (block == 128 && D == 64) return Cfg<128, 64>::SMEM;
    if (block == 64 && D == 128) return Cfg<64, 128>::SMEM;
    if (block == 64 && D == 64) return Cfg<64, 64>::SMEM;
    return 0;
}

cudaError_t launch_forward(int block, int D, bool paired, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int grid,
                           cudaStream_t stream) {
    if (paired && block == 64 && D == 128) return launch_impl<128, 128, true>(tq, tk, tv, to, p, grid, stream);
    if (paired && block == 64 && D == 64) return launch_impl<128, 64, true>(tq, tk, tv, to, p, grid, stream);
    if (block == 128 && D == 128) return launch_impl<128, 128>(tq, tk, tv, to, p, grid, stream);
    if (block == 128 && D == 64) return launch_impl<128, 64>(tq, tk, tv, to, p, grid, stream);
    if (block == 64 && D == 128) return launch_impl<64, 128>(tq, tk, tv, to, p, grid, stream);
    if (block == 64 && D == 64) return launch_impl<64, 64>(tq, tk, tv, to, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_forward_f8(int block, int D, bool paired, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int grid,
                              cudaStream_t stream) {
    if (D != 128) return cudaErrorInvalidValue;
    const bool sc = p.q_descale != nullptr;  // per-block scales
    if (paired && block == 64)
        return sc ? launch_impl<128, 128, true, true, true>(tq, tk, tv, to, p, grid, stream)
                  : launch_impl<128, 128, true, true>(tq, tk, tv, to, p, grid, stream);
    if (!paired && block == 128)
        return sc ? launch_impl<128, 128, false, true, true>(tq, tk, tv, to, p, grid, stream)
                  : launch_impl<128, 128, false, true>(tq, tk, tv, to, p, grid, stream);
    return cudaErrorInvalidValue;
}

template <bool LENS>
cudaError_t schedule_impl(const int32_t* src, const int32_t* n_dev, int32_t R, int32_t* perm, int32_t* counter,
                          int lens_shift, cudaStream_t stream) {
    constexpr int32_t kMaxStaged = 40960;  // 160 KB of row lengths
    if (R <= kMaxStaged) {
        const size_t smem = (size_t)R * sizeof(int32_t);
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(schedule_kernel<true, LENS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)(kMaxStaged * sizeof(int32_t)));
            if (e != cudaSuccess) return e;
        }
        schedule_kernel<true, LENS><<<1, kSchedThreads, smem, stream>>>(src, n_dev, R, perm, counter, lens_shift);
    } else {
        schedule_kernel<false, LENS><<<1, kSchedThreads, 0, stream>>>(src, n_dev, R, perm, counter, lens_shift);
    }
    return cudaGetLastError();
}

cudaError_t launch_schedule(const int32_t* row_ptr, int32_t R, int32_t* perm, int32_t* counter,
                            cudaStream_t stream) {
    return schedule_impl<false>(row_ptr, nullptr, R, perm, counter, 0, stream);
}

cudaError_t launch_schedule_lens(const int32_t* lens, const int32_t* n_dev, int32_t R_max, int32_t* perm,
                                 int32_t* counter, int lens_shift, cudaStream_t stream) {
    return schedule_impl<true>(lens, n_dev, R_max, perm, counter, lens_shift, stream);
}

}  // namespace bsa
