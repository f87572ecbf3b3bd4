// bsa_mask.cu -- pattern -> block CSR on the device, and the debug CSR check.
//
// A pattern row i holds (ascending): the global key blocks below the window,
// the window [max(0, i - wl), min(nb - 1, i + wr)] (cut at i when causal), and
// the global key blocks above it; a global query row (when global rows attend
// to all) holds every block up to the causal limit.  Window: "Flash MSA Sparse
// Attention vs Full Attention", section "The Mechanics" (Mask[i][j] = 1 if
// |i - j| <= W, causal form j <= i); global tokens: same page, "Sparse
// Patterns Beyond Sliding Windows", "Global Tokens".  Each row is a list of
// active key-block indices ("How Do Sparse Attention Kernels Work in GPU
// Clusters?", section "How Does Flash-MSA Sparse Attention Work?", step 2),
// built on the GPU so a new mask never costs a host round trip (the same
// guide, "When Sparse Kernels Break", item 2, on mask rebuild overhead).

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

namespace {

struct RowDesc {
    int32_t full;     // global query row: every block 0..cap
    int32_t cap;      // last allowed key block (i when causal)
    int32_t lo, hi;   // window (never empty: lo <= i <= hi)
    int32_t n_below;  // global blocks < lo  (a prefix of the sorted globals)
    int32_t k_above;  // index of the first global > hi
    int32_t n_above;  // global blocks in (hi, cap]
    int32_t len;
};

__host__ __device__ inline RowDesc describe_row(const PatternDev& p, int32_t i) {
    RowDesc d{};
    d.cap = p.causal ? i : p.nb - 1;
    bool is_global = false;
    for (int g = 0; g < p.n_global; ++g) is_global |= (p.globals[g] == i);
    if (p.gra && is_global) {
        // a global query row: every block up to the causal limit, or every
        // block when global rows take no causal cut
        d.full = 1;
        d.len = (p.grnc ? p.nb - 1 : d.cap) + 1;
        return d;
    }
    d.lo = i - p.wl < 0 ? 0 : i - p.wl;
    d.hi = i + p.wr > p.nb - 1 ? p.nb - 1 : i + p.wr;
    if (d.hi > d.cap) d.hi = d.cap;
    d.k_above = p.n_global;
    for (int g = 0; g < p.n_global; ++g) {
        const int32_t x = p.globals[g];
        if (x < d.lo) {
            ++d.n_below;
        } else if (x > d.hi) {
            if (d.k_above == p.n_global) d.k_above = g;
            if (x <= d.cap) ++d.n_above;
        }
    }
    d.len = d.n_below + (d.hi - d.lo + 1) + d.n_above;
    return d;
}

__host__ __device__ inline int32_t row_elem(const PatternDev& p, const RowDesc& d, int32_t e) {
    if (d.full) return e;
    if (e < d.n_below) return p.globals[e];
    e -= d.n_below;
    const int32_t w = d.hi - d.lo + 1;
    if (e < w) return d.lo + e;
    return p.globals[d.k_above + (e - w)];
}

// One warp per CSR row r = bh * nb + i.  The row's offset inside its head
// is the sum of the lengths of rows 0..i-1, computed by the warp itself
// (lane-strided, then reduced), so one launch writes row_ptr and col_idx.
__global__ void __launch_bounds__(256) mask_kernel(const PatternDev p, int32_t BH, int32_t nnz_head,
                                                   int32_t* __restrict__ row_ptr, int32_t* __restrict__ col_idx) {
    const int lane = threadIdx.x & 31;
    const int64_t R = (int64_t)BH * p.nb;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < R; r += warps) {
        const int32_t bh = (int32_t)(r / p.nb);
        const int32_t i = (int32_t)(r - (int64_t)bh * p.nb);
        int32_t pre = 0;
        for (int32_t i2 = lane; i2 < i; i2 += 32) pre += describe_row(p, i2).len;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
        const RowDesc d = describe_row(p, i);
        const int32_t base = bh * nnz_head + pre;
        if (lane == 0) {
            row_ptr[r + 1] = base + d.len;
            if (r == 0) row_ptr[0] = 0;
        }
        for (int32_t e = lane; e < d.len; e += 32) col_idx[base + e] = row_elem(p, d, e);
    }
}

// Row flags of a pattern's CSR: bit 0 for the rows of non-causal global
// query blocks.  One thread per row.
__global__ void __launch_bounds__(256) row_flags_kernel(const PatternDev p, int64_t R, uint8_t* __restrict__ flags) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int32_t i = (int32_t)(r % p.nb);
        bool g = false;
        for (int x = 0; x < p.n_global; ++x) g |= (p.globals[x] == i);
        flags[r] = (p.gra && p.grnc && g) ? 1 : 0;
    }
}

constexpr int kScanThreads = 1024;

// Row lengths -> row_ptr (running sum), one CTA.  Rows are staged through
// shared memory in coalesced chunks of kScanThreads * 8; each thread scans 8
// consecutive rows, the CTA scans the thread totals, a running offset carries
// across chunks.  A chunk is read whole before any of it is written, so lens
// may be row_ptr + 1 (no __restrict__ for that reason).
__global__ void __launch_bounds__(kScanThreads) lens_scan_kernel(const int32_t* lens, int64_t R, int32_t* row_ptr) {
    constexpr int PER = 8;
    constexpr int CHUNK = kScanThreads * PER;
    __shared__ int32_t buf[CHUNK];
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        carry = 0;
        row_ptr[0] = 0;
    }
    for (int64_t c0 = 0; c0 < R; c0 += CHUNK) {
        __syncthreads();
        for (int x = tid; x < CHUNK; x += kScanThreads) buf[x] = (c0 + x < R) ? lens[c0 + x] : 0;
        __syncthreads();
        int v[PER], local = 0;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            v[u] = buf[tid * PER + u];
            local += v[u];
        }
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
        int run = carry + incl - local + warp_tot[warp];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            run += v[u];
            buf[tid * PER + u] = run;  // inclusive prefix of row tid*PER+u
        }
        __syncthreads();
        for (int x = tid; x < CHUNK; x += kScanThreads)
            if (c0 + x < R) row_ptr[c0 + x + 1] = buf[x];
        if (tid == kScanThreads - 1) carry = run;
        __syncthreads();
    }
}


// ---------------------------------------------------------------- per-head patterns
// Walks the key blocks of row i of pattern p in ascending order, each once,
// calling emit(j); returns how many.  Sources: each dilated window (an
// arithmetic progression clipped to [0, cap]), the strided progression
// j = i (mod stride) and the sorted global blocks; a k-way merge emits the
// smallest head and advances every source that holds it.  A global query row
// (when global rows attend to all) is 0 .. cap.
template <class Emit>
__host__ __device__ inline int32_t walk_row_ex(const PatternSetDev& s, const PatternExDev& p, int32_t i, Emit emit) {
    const int32_t cap = p.causal ? i : s.nb - 1;
    const int32_t* g = s.globals + p.g_off;
    bool is_global = false;
    for (int x = 0; x < p.g_cnt; ++x) is_global |= (g[x] == i);
    if (p.gra && is_global) {
        for (int32_t j = 0; j <= cap; ++j) emit(j);
        return cap + 1;
    }
    int32_t cur[kMaxWindows + 1], step[kMaxWindows + 1], last[kMaxWindows + 1];
    int ns = 0;
    for (int w = 0; w < p.n_win; ++w) {
        const int32_t d = p.wd[w];
        const int32_t tl = p.wl[w] < i / d ? p.wl[w] : i / d;
        const int32_t tr = p.wr[w] < (cap - i) / d ? p.wr[w] : (cap - i) / d;
        cur[ns] = i - d * tl;
        last[ns] = i + d * tr;
        step[ns] = d;
        ++ns;
    }
    if (p.stride > 0) {
        cur[ns] = i % p.stride;
        last[ns] = i + p.stride * ((cap - i) / p.stride);
        step[ns] = p.stride;
        ++ns;
    }
    int gi = 0;
    int32_t n = 0;
    for (;;) {
        int32_t m = INT32_MAX;
        for (int k = 0; k < ns; ++k)
            if (cur[k] <= last[k] && cur[k] < m) m = cur[k];
        if (gi < p.g_cnt && g[gi] <= cap && g[gi] < m) m = g[gi];
        if (m == INT32_MAX) break;
        emit(m);
        ++n;
        for (int k = 0; k < ns; ++k)
            if (cur[k] <= last[k] && cur[k] == m) cur[k] += step[k];
        if (gi < p.g_cnt && g[gi] == m) ++gi;
    }
    return n;
}

struct NoEmit {
    __host__ __device__ void operator()(int32_t) const {}
};

// One thread per CSR row r = (b * H + h) * nb + i: its length into
// row_ptr[r + 1] (scanned in place afterwards).
__global__ void __launch_bounds__(256) mask_ex_len_kernel(const PatternSetDev s, int64_t R, int32_t* row_ptr) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bhrow = r / s.nb;
        const int32_t i = (int32_t)(r - bhrow * s.nb);
        const int32_t h = (int32_t)(bhrow % s.H);
        row_ptr[r + 1] = walk_row_ex(s, s.pat[s.head_pat[h]], i, NoEmit{});
    }
}

// One thread per row: writes its entries at row_ptr[r].
__global__ void __launch_bounds__(256) mask_ex_fill_kernel(const PatternSetDev s, int64_t R,
                                                           const int32_t* __restrict__ row_ptr,
                                                           int32_t* __restrict__ col_idx) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bhrow = r / s.nb;
        const int32_t i = (int32_t)(r - bhrow * s.nb);
        const int32_t h = (int32_t)(bhrow % s.H);
        int32_t* out = col_idx + row_ptr[r];
        walk_row_ex(s, s.pat[s.head_pat[h]], i, [&](int32_t j) { *out++ = j; });
    }
}

__global__ void validate_kernel(int32_t R, int32_t nb, const int32_t* __restrict__ row_ptr,
                                const int32_t* __restrict__ col_idx, int32_t* d_err) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    int32_t bad = 0;
    if (r == 0 && row_ptr[0] != 0) bad |= 1;
    const int32_t beg = row_ptr[r], end = row_ptr[r + 1];
    if (end < beg) bad |= 1;
    for (int32_t e = beg; e < end; ++e) {
        const int32_t j = col_idx[e];
        if (j < 0 || j >= nb) bad |= 2;
        for (int32_t f = e + 1; f < end; ++f)
            if (col_idx[f] == j) bad |= 4;
    }
    if (bad) atomicOr(d_err, bad);
}

}  // namespace

int32_t pattern_row_len(const PatternDev& p, int32_t i) { return describe_row(p, i).len; }

cudaError_t launch_mask(const PatternDev& p, int32_t BH, int64_t nnz_head, int32_t* row_ptr, int32_t* col_idx,
                        cudaStream_t stream) {
    const int64_t R = (int64_t)BH * p.nb;
    int64_t blocks = (R + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    mask_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, BH, (int32_t)nnz_head, row_ptr, col_idx);
    return cudaGetLastError();
}

cudaError_t launch_row_flags(const PatternDev& p, int32_t BH, uint8_t* flags, cudaStream_t stream) {
    const int64_t R = (int64_t)BH * p.nb;
    int64_t blocks = (R + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    row_flags_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, R, flags);
    return cudaGetLastError();
}

int32_t pattern_ex_row_len(const PatternSetDev& s, const PatternExDev& p, int32_t i) {
    return walk_row_ex(s, p, i, NoEmit{});
}

cudaError_t launch_row_ptr_scan(const int32_t* lens, int64_t R, int32_t* row_ptr, cudaStream_t stream) {
    lens_scan_kernel<<<1, kScanThreads, 0, stream>>>(lens, R, row_ptr);
    return cudaGetLastError();
}

cudaError_t launch_mask_ex(const PatternSetDev& s, int32_t B, int32_t* row_ptr, int32_t* col_idx,
                           cudaStream_t stream) {
    const int64_t R = (int64_t)B * s.H * s.nb;
    int64_t blocks = (R + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    mask_ex_len_kernel<<<(unsigned)blocks, 256, 0, stream>>>(s, R, row_ptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = launch_row_ptr_scan(row_ptr + 1, R, row_ptr, stream)) != cudaSuccess) return e;
    mask_ex_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(s, R, row_ptr, col_idx);
    return cudaGetLastError();
}

cudaError_t launch_validate(int32_t R, int32_t nb, const int32_t* row_ptr, const int32_t* col_idx, int32_t* d_err,
                            cudaStream_t stream) {
    validate_kernel<<<(R + 255) / 256, 256, 0, stream>>>(R, nb, row_ptr, col_idx, d_err);
    return cudaGetLastError();
}

}  // namespace bsa
