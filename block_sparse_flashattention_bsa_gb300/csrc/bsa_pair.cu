// bsa_pair.cu -- work items of the block-64 forward: query blocks in pairs.
//
// The tensor-core tile is 128 query rows x 128 keys.  With 64-token blocks a
// tile holds two query blocks (a pair) and two key blocks per step, taken from
// the union of the pair's key-block lists; each query half masks the key
// blocks its own list lacks.  Pairing rows whose lists overlap makes the union
// barely longer than either list, so the tile carries little masked work.
// Lists of block-sparse rows ("How Does Flash-MSA Sparse Attention Work?",
// "How Do Sparse Attention Kernels Work in GPU Clusters?", step 2) are sets:
// their order is free, so the union is taken as a set.
//
//   pair_plan_kernel   per (head, chunk of 8192 rows): rows with at most
//                      kPairRowMax raw entries are sorted by two MinHash
//                      values of their valid key blocks other than the
//                      diagonal (ties by row) and paired in that order;
//                      longer rows (and an odd one out) stay single.
//   pair_union_kernel  one warp per item: a pair's union, ascending and
//                      without repeats, with each entry's membership bits, in
//                      a fixed slot; a single's count of valid entries.
// A MinHash collision (same minimum of a random hash over the set) is likely
// exactly when the sets overlap a lot, so equal keys group similar rows; the
// diagonal block is left out because it is different for every row, and the
// second hash orders the rows inside a group of equal first hashes.  On the
// top-k workload this takes the tile steps from 86,516 (one hash, diagonal
// included) to 80,252, against 73,724 if every union were a single row.

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanRows = 8192;  // rows sorted together (64 KB of keys)

// Integer finalisers (xor-shift-multiply): fixed pseudo-random permutations
// of 32-bit values, two independent ones.
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}
__device__ __forceinline__ uint32_t mix32b(uint32_t x) {
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}

// Key block j counts for query block i: inside the key blocks, and not after
// the query block's key position i + q_off when the row is causal.
__device__ __forceinline__ bool key_ok(int j, int i, const PairGeom& g, bool crow) {
    return (unsigned)j < (unsigned)g.nbk && !(crow && j > i + g.q_off);
}
// Entries of row r below the capacity of col_idx (a malformed row_ptr may
// point past it; whoever built the lists has flagged that).
__device__ __forceinline__ int row_len(const int32_t* row_ptr, int64_t r, const PairGeom& g) {
    const int64_t beg = min((int64_t)row_ptr[r], g.col_cap), end = min((int64_t)row_ptr[r + 1], g.col_cap);
    return end > beg ? (int)(end - beg) : 0;
}
// A flagged row (causal cut lifted) is never paired: the tile's mask logic
// applies one causal rule to both halves of a pair.
__device__ __forceinline__ bool row_flagged(const PairGeom& g, int64_t r) {
    return g.causal && g.row_flags && (g.row_flags[r] & 1);
}

__global__ void __launch_bounds__(kPlanThreads) pair_plan_kernel(const int32_t* __restrict__ row_ptr,
                                                                 const int32_t* __restrict__ col_idx,
                                                                 const PairGeom g, int32_t* __restrict__ item_a,
                                                                 int32_t* __restrict__ item_b,
                                                                 int32_t* __restrict__ n_items) {
    extern __shared__ uint64_t key[];  // [kPlanRows]
    __shared__ int32_t n_cand, n_long, base;
    const int nb = g.nb;
    const int bh = blockIdx.y;
    const int i0 = blockIdx.x * kPlanRows;
    const int rows = min(kPlanRows, nb - i0);
    if (threadIdx.x == 0) {
        n_cand = 0;
        n_long = 0;
    }
    // sort only the next power of two above the chunk's rows
    int n2 = 32;
    while (n2 < rows) n2 <<= 1;
    __syncthreads();
    for (int x = threadIdx.x; x < n2; x += kPlanThreads) {
        uint64_t k = ~0ull;
        if (x < rows) {
            const int i = i0 + x;
            const int64_t r = (int64_t)bh * nb + i;
            const int beg = row_ptr[r];
            const int len = row_len(row_ptr, r, g);
            if (len <= kPairRowMax && !row_flagged(g, r)) {
                uint32_t h = 0xffffffffu, h2 = 0xffffffffu;
                for (int e = beg; e < beg + len; ++e) {
                    const int j = col_idx[e];
                    if (j != i + g.q_off && key_ok(j, i, g, g.causal != 0)) {
                        h = min(h, mix32((uint32_t)j));
                        h2 = min(h2, mix32b((uint32_t)j));
                    }
                }
                // 31 bits of the first hash, 19 of the second, 13 of row (below
                // 2^63, clear of the padding key)
                k = ((uint64_t)(h >> 1) << 32) | ((uint64_t)(h2 >> 13) << 13) | (uint64_t)x;
                atomicAdd(&n_cand, 1);
            } else {
                atomicAdd(&n_long, 1);
            }
        }
        key[x] = k;
    }
    __syncthreads();
    // bitonic sort, ascending
    for (int k = 2; k <= n2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int x = threadIdx.x; x < n2; x += kPlanThreads) {
                const int y = x ^ j;
                if (y > x) {
                    const uint64_t a = key[x], b = key[y];
                    const bool up = (x & k) == 0;
                    if ((a > b) == up) {
                        key[x] = b;
                        key[y] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    const int pairs = n_cand >> 1, odd = n_cand & 1;
    if (threadIdx.x == 0) base = atomicAdd(n_items, pairs + odd + n_long);
    __syncthreads();
    const int32_t rbase = bh * nb + i0;
    for (int t = threadIdx.x; t < pairs; t += kPlanThreads) {
        item_a[base + t] = rbase + (int32_t)(key[2 * t] & 8191u);
        item_b[base + t] = i0 + (int32_t)(key[2 * t + 1] & 8191u);
    }
    if (odd && threadIdx.x == 0) {
        item_a[base + pairs] = rbase + (int32_t)(key[n_cand - 1] & 8191u);
        item_b[base + pairs] = -1;
    }
    // long rows, in row order (one warp scans the chunk with ballots)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int out = base + pairs + odd;
        for (int x0 = 0; x0 < rows; x0 += 32) {
            const int x = x0 + lane;
            bool lng = false;
            if (x < rows) {
                const int64_t r = (int64_t)bh * nb + i0 + x;
                lng = row_len(row_ptr, r, g) > kPairRowMax || row_flagged(g, r);
            }
            const unsigned m = __ballot_sync(0xffffffffu, lng);
            if (lng) {
                item_a[out + __popc(m & ((1u << lane) - 1u))] = rbase + x;
                item_b[out + __popc(m & ((1u << lane) - 1u))] = -1;
            }
            out += __popc(m);
        }
    }
}

// One warp per item.  Pair: both rows have at most 32 raw entries; lane l
// holds entry l of each.  Candidates (j << 2 | membership) are ranked (ties by
// position, so ranks are distinct), placed in order in shared memory, equal
// blocks merged (their membership bits ORed), and the result compacted into
// the item's slot.  Single: count the row's valid entries.
__global__ void __launch_bounds__(256) pair_union_kernel(const int32_t* __restrict__ row_ptr,
                                                         const int32_t* __restrict__ col_idx, const PairGeom g,
                                                         const int32_t* __restrict__ item_a,
                                                         const int32_t* __restrict__ item_b,
                                                         const int32_t* __restrict__ n_items,
                                                         int32_t* __restrict__ item_cnt,
                                                         int32_t* __restrict__ item_len,
                                                         uint32_t* __restrict__ slots, int32_t* err) {
    __shared__ uint32_t buf[8][2 * 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = *n_items;
    const int nb = g.nb;
    for (int it = blockIdx.x * 8 + warp; it < n; it += gridDim.x * 8) {
        const int ra = item_a[it], ib = item_b[it];
        const int bh = ra / nb, ia = ra - bh * nb;
        int cnt = 0;
        if (ib < 0) {
            int beg = row_ptr[ra], end = row_ptr[ra + 1];
            if (end < beg) {
                if (lane == 0) atomicOr(err, ERR_BAD_ROW);
                end = beg;
            }
            end = beg + row_len(row_ptr, ra, g);
            const bool crow = g.causal && !row_flagged(g, ra);
            for (int e0 = beg; e0 < end; e0 += 32) {
                const int e = e0 + lane;
                const int j = e < end ? col_idx[e] : 0;
                if (e < end && (unsigned)j >= (unsigned)g.nbk) atomicOr(err, ERR_BAD_COL);
                cnt += __popc(__ballot_sync(0xffffffffu, e < end && key_ok(j, ia, g, crow)));
            }
        } else {
            const int64_t rb = (int64_t)bh * nb + ib;
            uint32_t cand[2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int64_t r = s ? rb : (int64_t)ra;
                const int i = s ? ib : ia;
                int beg = row_ptr[r], end = row_ptr[r + 1];
                if (end < beg) {
                    if (lane == 0) atomicOr(err, ERR_BAD_ROW);
                    end = beg;
                }
                end = beg + row_len(row_ptr, r, g);
                const int e = beg + lane;
                const int j = e < end ? col_idx[e] : 0;
                if (e < end && (unsigned)j >= (unsigned)g.nbk) atomicOr(err, ERR_BAD_COL);
                cand[s] = (e < end && key_ok(j, i, g, g.causal != 0)) ? ((uint32_t)j << 2) | (1u << s) : 0xffffffffu;
            }
            // rank among the 64 candidates (position p = 2 * lane + s)
            int rank[2] = {0, 0};
            for (int q = 0; q < 32; ++q) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint32_t y = __shfl_sync(0xffffffffu, cand[t], q);
                    const int py = 2 * q + t;
#pragma unroll
                    for (int s = 0; s < 2; ++s)
                        rank[s] += (y < cand[s] || (y == cand[s] && py < 2 * lane + s)) ? 1 : 0;
                }
            }
            buf[warp][rank[0]] = cand[0];
            buf[warp][rank[1]] = cand[1];
            __syncwarp();
            // sorted position p = 2 * lane + s: keep it when its block differs from p - 1
            uint32_t ent[2];
            bool keep[2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int pos = 2 * lane + s;
                const uint32_t x = buf[warp][pos];
                const uint32_t prev = pos > 0 ? buf[warp][pos - 1] : 0xffffffffu;
                const uint32_t next = pos < 63 ? buf[warp][pos + 1] : 0xffffffffu;
                keep[s] = x != 0xffffffffu && (pos == 0 || (prev >> 2) != (x >> 2));
                uint32_t m = x & 3u;
                if (next != 0xffffffffu && (next >> 2) == (x >> 2)) m |= next & 3u;
                ent[s] = (x >> 2) | ((m & 1u) << 30) | ((m >> 1) << 31);
            }
            __syncwarp();
            const unsigned k0 = __ballot_sync(0xffffffffu, keep[0]);
            const unsigned k1 = __ballot_sync(0xffffffffu, keep[1]);
            const unsigned below = (1u << lane) - 1u;
            // kept entries before position 2 * lane: both slots of every lower lane
            int out = __popc(k0 & below) + __popc(k1 & below);
            uint32_t* slot = slots + (size_t)it * kPairSlot;
            if (keep[0]) slot[out++] = ent[0];
            if (keep[1]) slot[out] = ent[1];
            cnt = __popc(k0) + __popc(k1);
        }
        if (lane == 0) {
            item_cnt[it] = cnt;
            item_len[it] = (cnt + 1) >> 1;
        }
    }
}

}  // namespace

size_t pairing_workspace_bytes(int32_t BH, int32_t nb) {
    const size_t n = (size_t)BH * nb;  // at most one item per row
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return 4 * a(n * sizeof(int32_t)) + a(64) + a(n * kPairSlot * sizeof(uint32_t));  // slots by item index
}

PairingBuffers pairing_buffers(void* ws, int32_t BH, int32_t nb) {
    const size_t n = (size_t)BH * nb;
    auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
    char* w = static_cast<char*>(ws);
    PairingBuffers b;
    b.item_a = reinterpret_cast<int32_t*>(w);
    w += a(n * sizeof(int32_t));
    b.item_b = reinterpret_cast<int32_t*>(w);
    w += a(n * sizeof(int32_t));
    b.item_cnt = reinterpret_cast<int32_t*>(w);
    w += a(n * sizeof(int32_t));
    b.item_len = reinterpret_cast<int32_t*>(w);
    w += a(n * sizeof(int32_t));
    b.n_items = reinterpret_cast<int32_t*>(w);
    w += a(64);
    b.slots = reinterpret_cast<uint32_t*>(w);
    return b;
}

cudaError_t launch_pairing(const int32_t* row_ptr, const int32_t* col_idx, int32_t BH, const PairGeom& g,
                           const PairingBuffers& b, int32_t* err, int sm_count, cudaStream_t stream) {
    const int32_t nb = g.nb;
    cudaError_t e = cudaMemsetAsync(b.n_items, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((nb + kPlanRows - 1) / kPlanRows), (unsigned)BH);
    const int smem = kPlanRows * (int)sizeof(uint64_t);
    e = cudaFuncSetAttribute(pair_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    pair_plan_kernel<<<grid, kPlanThreads, smem, stream>>>(row_ptr, col_idx, g, b.item_a, b.item_b, b.n_items);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t max_items = (int64_t)BH * nb;
    int64_t blocks = (max_items + 7) / 8;
    if (blocks > 8 * (int64_t)sm_count) blocks = 8 * (int64_t)sm_count;
    pair_union_kernel<<<(unsigned)blocks, 256, 0, stream>>>(row_ptr, col_idx, g, b.item_a, b.item_b, b.n_items,
                                                           b.item_cnt, b.item_len, b.slots, err);
    return cudaGetLastError();
}

}  // namespace bsa
