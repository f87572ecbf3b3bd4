// bsa_shard.cu -- the sequence-sharded forward's host planners and its two
// data-movement kernels.
//
// "How Do Sparse Attention Kernels Work in GPU Clusters?", section
// "Distributed Sparse Attention", names the ways to run block-sparse
// attention over a sequence split across GPUs.  Two are built here:
//
//   key/value exchange (the page's sparse all-to-all, indices first, then the
//   blocks): every rank lists the remote key blocks its rows need, fetches
//   them into its own memory, and runs the unchanged forward on its query
//   blocks against an extended key range -- received blocks before its own
//   shard, its own blocks, received blocks after it -- through a renumbered
//   CSR (bsa_shard_plan_kv);
//
//   local attention plus a merge of partial outputs: every rank computes its
//   query blocks against its own key blocks, and against each other rank's
//   key blocks at that rank (it ships the query blocks there); the partial
//   (O, LSE) pairs come back and are merged with the online-softmax rescale
//   (bsa_shard_plan_partial, bsa_merge_partial_blocks).
//
// Shards are contiguous: rank g of W owns query and key blocks
// [g * nb / W, (g + 1) * nb / W) of every (batch, head).  The plans are host
// work over the rank's own CSR rows (the mask does not change between steps
// of a fixed pattern, so a plan is made once and reused).  Moving blocks is
// device work: bsa_copy_blocks gathers or scatters whole blocks of rows, and
// the merge is one thread block per query block.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

struct Shard {
    int32_t first, count;
};

Shard shard_of(int32_t world, int32_t rank, int32_t nb) {
    const int64_t a = (int64_t)rank * nb / world, b = (int64_t)(rank + 1) * nb / world;
    return Shard{(int32_t)a, (int32_t)(b - a)};
}

int check_geometry(const bsa_shard_geometry* g) {
    if (!g) return BSA_ERR_INVALID_ARG;
    if (g->world < 1 || g->rank < 0 || g->rank >= g->world) return BSA_ERR_INVALID_ARG;
    if (g->n_blocks < g->world || g->BH < 1) return BSA_ERR_INVALID_ARG;
    if ((int64_t)g->BH * g->n_blocks > INT32_MAX) return BSA_ERR_INVALID_ARG;
    return BSA_OK;
}

// The local rows' CSR: BH * count rows, monotone row_ptr from 0.
int check_rows(const bsa_shard_geometry* g, const int32_t* row_ptr, const int32_t* col_idx, int64_t* nnz) {
    const Shard s = shard_of(g->world, g->rank, g->n_blocks);
    const int64_t R = (int64_t)g->BH * s.count;
    if (!row_ptr) return BSA_ERR_INVALID_ARG;
    if (row_ptr[0] != 0) return BSA_ERR_INVALID_ARG;
    for (int64_t r = 0; r < R; ++r)
        if (row_ptr[r + 1] < row_ptr[r]) return BSA_ERR_INVALID_ARG;
    *nnz = row_ptr[R];
    if (*nnz > 0 && !col_idx) return BSA_ERR_INVALID_ARG;
    return BSA_OK;
}

// ---------------------------------------------------------------- kernels
// dst block n (rows dst_row[n] .. + rows_per_block) = src block n (rows
// src_row[n] ..); 16-byte vectors, one CTA per block.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          const int64_t* __restrict__ src_row,
                                                          const int64_t* __restrict__ dst_row, int64_t n,
                                                          int32_t rows_per_block, int32_t vec_per_row) {
    const int64_t per = (int64_t)rows_per_block * vec_per_row;
    for (int64_t b = blockIdx.x; b < n; b += gridDim.x) {
        const uint4* s = src + src_row[b] * vec_per_row;
        uint4* d = dst + dst_row[b] * vec_per_row;
        for (int64_t x = threadIdx.x; x < per; x += blockDim.x) d[x] = s[x];
    }
}

// Merge a compact list of partial query blocks into the accumulated result:
// for each row, LSE = log(exp(LSE_acc) + exp(LSE_part)) and O = w_acc O_acc +
// w_part O_part with w = exp(LSE_x - LSE); one warp per row, fp32 throughout.
// A part with LSE = -inf leaves the row as it is.
__global__ void __launch_bounds__(256) merge_blocks_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                           const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           const int64_t* __restrict__ dst_row, int64_t n_rows,
                                                           int32_t rows_per_block, int32_t D) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t x = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); x < n_rows; x += warps) {
        const int64_t b = x / rows_per_block, t = x - b * rows_per_block;
        const int64_t row = dst_row[b] + t;
        const float la = lse_acc[row], lp = lse_part[x];
        if (lp == -INFINITY) continue;
        const float m = fmaxf(la, lp);
        const float wa = (la == -INFINITY) ? 0.f : expf(la - m);
        const float wp = expf(lp - m);
        const float tot = wa + wp;
        const float ca = wa / tot, cp = wp / tot;
        float* oa = o_acc + row * D;
        const float* op = o_part + x * D;
        for (int d = lane; d < D; d += 32) oa[d] = ca * oa[d] + cp * op[d];
        __syncwarp();
        if (lane == 0) lse_acc[row] = m + logf(tot);
    }
}

__global__ void __launch_bounds__(256) convert_f32_bf16_kernel(const float4* __restrict__ x, uint4* __restrict__ y,
                                                               int64_t n8) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = x[2 * t], b = x[2 * t + 1];
        __nv_bfloat162 r[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                               __floats2bfloat162_rn(b.x, b.y), __floats2bfloat162_rn(b.z, b.w)};
        y[t] = *reinterpret_cast<uint4*>(r);
    }
}

}  // namespace

extern "C" {

int bsa_shard_range(const bsa_shard_geometry* g, int32_t* first, int32_t* count) {
    int st = check_geometry(g);
    if (st != BSA_OK) return st;
    if (!first || !count) return BSA_ERR_INVALID_ARG;
    const Shard s = shard_of(g->world, g->rank, g->n_blocks);
    *first = s.first;
    *count = s.count;
    return BSA_OK;
}

int bsa_shard_plan_kv(const bsa_shard_geometry* g, const int32_t* row_ptr, const int32_t* col_idx,
                      int32_t* col_idx_ext, int32_t* need_bh, int32_t* need_j, int32_t* need_pos,
                      int64_t need_cap, int32_t* need_count_by_rank, int32_t* n_before_out,
                      int32_t* n_after_out) {
    int st = check_geometry(g);
    if (st != BSA_OK) return st;
    int64_t nnz = 0;
    if ((st = check_rows(g, row_ptr, col_idx, &nnz)) != BSA_OK) return st;
    if (!n_before_out || !n_after_out || !need_count_by_rank) return BSA_ERR_INVALID_ARG;
    const Shard s = shard_of(g->world, g->rank, g->n_blocks);
    const int32_t nb = g->n_blocks;
    // remote key blocks each head needs, before and after the shard (sorted, distinct)
    std::vector<std::vector<int32_t>> before(g->BH), after(g->BH);
    for (int32_t bh = 0; bh < g->BH; ++bh) {
        for (int32_t i = 0; i < s.count; ++i) {
            const int64_t r = (int64_t)bh * s.count + i;
            for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
                const int32_t j = col_idx[e];
                if (j < 0 || j >= nb) continue;
                if (j < s.first) before[bh].push_back(j);
                else if (j >= s.first + s.count) after[bh].push_back(j);
            }
        }
        for (auto* v : {&before[bh], &after[bh]}) {
            std::sort(v->begin(), v->end());
            v->erase(std::unique(v->begin(), v->end()), v->end());
        }
    }
    int32_t nbf = 0, naf = 0;
    int64_t total = 0;
    for (int32_t bh = 0; bh < g->BH; ++bh) {
        nbf = std::max<int32_t>(nbf, (int32_t)before[bh].size());
        naf = std::max<int32_t>(naf, (int32_t)after[bh].size());
        total += (int64_t)before[bh].size() + after[bh].size();
    }
    *n_before_out = nbf;
    *n_after_out = naf;
    if (!col_idx_ext) return BSA_OK;  // sizes only
    if (total > need_cap || (total > 0 && (!need_bh || !need_j || !need_pos))) return BSA_ERR_CAPACITY;
    // extended key position of every global key block a head uses: the
    // head's remote blocks before the shard end right where the shard starts
    // (position nbf), its remote blocks after the shard follow it
    auto ext_of = [&](int32_t bh, int32_t j) -> int32_t {
        if (j < 0 || j >= nb) return -1;  // out of range: stays invalid (skipped and flagged by the forward)
        if (j < s.first) {
            const auto& v = before[bh];
            const int32_t p = (int32_t)(std::lower_bound(v.begin(), v.end(), j) - v.begin());
            return nbf - (int32_t)v.size() + p;
        }
        if (j < s.first + s.count) return nbf + (j - s.first);
        const auto& v = after[bh];
        return nbf + s.count + (int32_t)(std::lower_bound(v.begin(), v.end(), j) - v.begin());
    };
    for (int32_t bh = 0; bh < g->BH; ++bh)
        for (int32_t i = 0; i < s.count; ++i) {
            const int64_t r = (int64_t)bh * s.count + i;
            for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) col_idx_ext[e] = ext_of(bh, col_idx[e]);
        }
    // requests sorted by owner, then head, then key block
    for (int32_t p = 0; p < g->world; ++p) need_count_by_rank[p] = 0;
    int64_t n = 0;
    for (int32_t p = 0; p < g->world; ++p) {
        if (p == g->rank) continue;
        const Shard sp = shard_of(g->world, p, nb);
        for (int32_t bh = 0; bh < g->BH; ++bh)
            for (const auto* v : {&before[bh], &after[bh]})
                for (int32_t j : *v) {
                    if (j < sp.first || j >= sp.first + sp.count) continue;
                    need_bh[n] = bh;
                    need_j[n] = j;
                    need_pos[n] = ext_of(bh, j);
                    ++n;
                    ++need_count_by_rank[p];
                }
    }
    return BSA_OK;
}

int bsa_shard_plan_partial(const bsa_shard_geometry* g, const int32_t* row_ptr, const int32_t* col_idx,
                           const uint8_t* row_flags, int32_t causal, int32_t* local_row_ptr,
                           int32_t* local_col_idx, int32_t* guest_q, int32_t* guest_ptr, int32_t* guest_col,
                           int64_t cap, int32_t* guest_rows_by_rank, int32_t* guest_entries_by_rank) {
    int st = check_geometry(g);
    if (st != BSA_OK) return st;
    int64_t nnz = 0;
    if ((st = check_rows(g, row_ptr, col_idx, &nnz)) != BSA_OK) return st;
    if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
    if (!local_row_ptr || !guest_rows_by_rank || !guest_entries_by_rank) return BSA_ERR_INVALID_ARG;
    if (nnz > cap || (nnz > 0 && (!local_col_idx || !guest_q || !guest_ptr || !guest_col)))
        return BSA_ERR_CAPACITY;
    const Shard s = shard_of(g->world, g->rank, g->n_blocks);
    const int32_t nb = g->n_blocks;
    const int64_t R = (int64_t)g->BH * s.count;
    // local part: own key blocks, renumbered to the shard
    int64_t nl = 0;
    local_row_ptr[0] = 0;
    for (int64_t r = 0; r < R; ++r) {
        for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
            const int32_t j = col_idx[e];
            if (j >= s.first && j < s.first + s.count) local_col_idx[nl++] = j - s.first;
        }
        local_row_ptr[r + 1] = (int32_t)nl;
    }
    // guest part, by owner: a query block goes to the owner of any of its
    // remote key blocks, with those blocks in the owner's numbering.  A causal
    // row sends only the blocks wholly before it (a block after it adds
    // nothing, its own block is local), so the owner computes the guest rows
    // without a causal cut.
    std::vector<int32_t> tmp;
    int64_t ng = 0, ne = 0;
    guest_ptr[0] = 0;
    for (int32_t p = 0; p < g->world; ++p) {
        guest_rows_by_rank[p] = 0;
        guest_entries_by_rank[p] = 0;
        if (p == g->rank) continue;
        const Shard sp = shard_of(g->world, p, nb);
        for (int64_t r = 0; r < R; ++r) {
            const int32_t i = s.first + (int32_t)(r % s.count);
            const bool crow = causal && !(row_flags && (row_flags[r] & 1));
            tmp.clear();
            for (int32_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
                const int32_t j = col_idx[e];
                if (j < sp.first || j >= sp.first + sp.count) continue;
                if (crow && j >= i) continue;
                tmp.push_back(j - sp.first);
            }
            if (tmp.empty()) continue;
            std::sort(tmp.begin(), tmp.end());
            tmp.erase(std::unique(tmp.begin(), tmp.end()), tmp.end());
            guest_q[ng] = (int32_t)r;  // local CSR row: bh * count + i_local
            for (int32_t x : tmp) guest_col[ne++] = x;
            guest_ptr[++ng] = (int32_t)ne;
            ++guest_rows_by_rank[p];
            guest_entries_by_rank[p] += (int32_t)tmp.size();
        }
    }
    return BSA_OK;
}

int bsa_copy_blocks(const void* src, void* dst, const int64_t* src_row, const int64_t* dst_row, int64_t n_blocks,
                    int32_t rows_per_block, int32_t row_bytes, bsa_stream_t stream) {
    if (n_blocks < 0 || rows_per_block <= 0 || row_bytes <= 0 || row_bytes % 16 != 0) return BSA_ERR_INVALID_ARG;
    if (n_blocks == 0) return BSA_OK;
    if (!src || !dst || !src_row || !dst_row) return BSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16) return BSA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
        return BSA_ERR_CUDA;
    const int64_t grid = std::min<int64_t>(n_blocks, 8LL * sms);
    copy_blocks_kernel<<<(unsigned)grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(src), static_cast<uint4*>(dst), src_row, dst_row, n_blocks, rows_per_block,
        row_bytes / 16);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

int bsa_merge_partial_blocks(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                             const int64_t* dst_row, int64_t n_blocks, int32_t rows_per_block, int32_t D,
                             bsa_stream_t stream) {
    if (n_blocks < 0 || rows_per_block <= 0 || D <= 0) return BSA_ERR_INVALID_ARG;
    if (n_blocks == 0) return BSA_OK;
    if (!o_acc || !lse_acc || !o_part || !lse_part || !dst_row) return BSA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
        return BSA_ERR_CUDA;
    const int64_t rows = n_blocks * rows_per_block;
    const int64_t grid = std::min<int64_t>((rows + 7) / 8, 16LL * sms);
    merge_blocks_kernel<<<(unsigned)grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        o_acc, lse_acc, o_part, lse_part, dst_row, rows, rows_per_block, D);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

int bsa_convert_f32_bf16(const float* x, void* y, int64_t n, bsa_stream_t stream) {
    if (n < 0 || n % 8 != 0) return BSA_ERR_INVALID_ARG;
    if (n == 0) return BSA_OK;
    if (!x || !y || (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16) return BSA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
        return BSA_ERR_CUDA;
    const int64_t n8 = n / 8;
    const int64_t grid = std::min<int64_t>((n8 + 255) / 256, 8LL * sms);
    convert_f32_bf16_kernel<<<(unsigned)grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(x), static_cast<uint4*>(y), n8);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // extern "C"
