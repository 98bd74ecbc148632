// dw_prep.cu -- preparation of the linear_logp weight gradient (dW).
//
// dW is a sum over tokens, the batch-dependent axis, so its bitwise
// invariance only makes sense over the same complete logical sample set
// reduced in one canonical order (issue #244 "[WS1 Test] ...", Workstream 3
// #153: fixed, batch-shape-independent reduction order; compare parameter
// gradients over the same complete sample set; restore packed/chunked
// results to canonical (sample_id, token_position) order).  These kernels
// put the active tokens into that order once:
//
//   compact  the caller's canonical row order (or rows 0..T-1) filtered to
//            the active rows, order kept (block counts, one scan of the
//            counts, then each block writes its rows at its offset);
//   gather   h, g, lse and the target of every canonical token into dense
//            buffers; positions past the active count hold zeros and target
//            -1, so a GEMM over all n positions adds exact zeros for them;
// After the dZ / dZ^T GEMM over the canonical tokens has filled each token's
// list of fp32 entries (the target column and the columns with p >= 1/64):
//   flatten  the lists in canonical token order (per-token counts, one scan);
//   sort     (column, flat index) pairs by column with a stable
//            least-significant-digit radix sort, kRadixBits per pass: a
//            digit histogram per tile, one scan of the histograms (digit
//            major, tile minor), then a stable scatter per tile; a column's
//            entries keep canonical token order;
//   bounds   the [begin, end) range of each column in the sorted list.
// A separate kernel sorts each row's own list by column (for the dh GEMM).
//
// Every step is deterministic: counts and prefix sums over integers, no
// floating-point atomics.
#include <algorithm>
#include <utility>

#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kRadixBits = 5;

// Exclusive prefix sum of one int per thread across the block; returns the
// prefix and writes the block total to *total.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t x, int64_t *total) {
    __shared__ int64_t warp_sums[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t w = (lane < kScanThreads / 32) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before_warp = (warp > 0) ? warp_sums[warp - 1] : 0;
    *total = warp_sums[kScanThreads / 32 - 1];
    __syncthreads();
    return before_warp + incl - x;
}

__device__ __forceinline__ int64_t candidate_row(const int64_t *order, int64_t i) {
    return order ? order[i] : i;
}

__device__ __forceinline__ bool candidate_active(const int64_t *order, int64_t i, int64_t T,
                                                 const int64_t *targets, const int32_t *cu,
                                                 int num_seqs, int64_t V) {
    const int64_t r = candidate_row(order, i);
    if (r < 0 || r >= T) return false;
    const int64_t t = targets[r];
    return row_active(r, t, cu, num_seqs) && t < V;
}

// Exclusive prefix sums over cnt[0..len) in place (one block); *total gets
// the sum when total is not null.
__global__ void __launch_bounds__(kScanThreads)
    scan_counts(int32_t *__restrict__ cnt, int64_t len, int64_t *__restrict__ total) {
    const int64_t per = (len + kScanThreads - 1) / kScanThreads;
    const int64_t b = (int64_t)threadIdx.x * per;
    const int64_t e = min(len, b + per);
    int64_t s = 0;
    for (int64_t i = b; i < e; ++i) s += cnt[i];
    int64_t all;
    int64_t pos = block_exclusive_scan(s, &all);
    for (int64_t i = b; i < e; ++i) {
        const int32_t c = cnt[i];
        cnt[i] = (int32_t)pos;
        pos += c;
    }
    if (total && threadIdx.x == 0) *total = all;
}

// Compaction, first half: the number of active candidates in each block of
// kScanThreads candidates.
__global__ void __launch_bounds__(kScanThreads)
    dw_compact_count(const int64_t *__restrict__ order, int64_t n, int64_t T,
                     const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                     int num_seqs, int64_t V, int32_t *__restrict__ block_cnt) {
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    const bool a = i < n && candidate_active(order, i, T, targets, cu, num_seqs, V);
    const int c = __syncthreads_count(a);
    if (threadIdx.x == 0) block_cnt[blockIdx.x] = c;
}

// Compaction, second half: crow[offset of the block + rank in the block] =
// physical row, ranks in candidate order.
__global__ void __launch_bounds__(kScanThreads)
    dw_compact_write(const int64_t *__restrict__ order, int64_t n, int64_t T,
                     const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                     int num_seqs, int64_t V, const int32_t *__restrict__ block_ofs,
                     int64_t *__restrict__ crow) {
    __shared__ int warp_cnt[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    const bool a = i < n && candidate_active(order, i, T, targets, cu, num_seqs, V);
    const unsigned m = __ballot_sync(0xffffffffu, a);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    if (a)
        crow[(int64_t)block_ofs[blockIdx.x] + before + __popc(m & ((1u << lane) - 1u))] =
            candidate_row(order, i);
}

// Canonical buffers: hc [n, H] bf16, gc / lsec fp32 [n], tgtc int64 [n].
__global__ void dw_gather(const uint16_t *__restrict__ h, const float *__restrict__ grad,
                          const float *__restrict__ lse, const int64_t *__restrict__ targets,
                          const int64_t *__restrict__ crow, const int64_t *__restrict__ n_active,
                          int64_t n, int64_t H, uint16_t *__restrict__ hc, float *__restrict__ gc,
                          float *__restrict__ lsec, int64_t *__restrict__ tgtc) {
    const int64_t c = blockIdx.x;
    if (c >= n) return;
    const int64_t na = *n_active;
    const bool live = c < na;
    const int64_t r = live ? crow[c] : 0;
    const uint4 *src = reinterpret_cast<const uint4 *>(h + r * H);
    uint4 *dst = reinterpret_cast<uint4 *>(hc + c * H);
    for (int64_t k = threadIdx.x; k < H / 8; k += blockDim.x)
        dst[k] = live ? src[k] : make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        gc[c] = live ? grad[r] : 0.f;
        lsec[c] = live ? lse[r] : 0.f;
        const int64_t t = live ? targets[r] : -1;
        tgtc[c] = t;
    }
}

constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;                         // consecutive items per thread
constexpr int kSortTile = kSortThreads * kSortItems;  // items per block
constexpr int kBins = 1 << kRadixBits;

// Radix pass, first half: hist[d * tiles + b] = number of items of tile b
// whose digit (key >> shift) & (kBins - 1) is d.
__global__ void __launch_bounds__(kSortThreads)
    radix_histogram(const int32_t *__restrict__ key, const int64_t *__restrict__ n_active,
                    int shift, int32_t *__restrict__ hist, int tiles) {
    __shared__ int cnt[kBins];
    if (threadIdx.x < kBins) cnt[threadIdx.x] = 0;
    __syncthreads();
    const int64_t n = *n_active;
    const int64_t base = (int64_t)blockIdx.x * kSortTile + (int64_t)threadIdx.x * kSortItems;
#pragma unroll
    for (int k = 0; k < kSortItems; ++k)
        if (base + k < n) atomicAdd(&cnt[(key[base + k] >> shift) & (kBins - 1)], 1);
    __syncthreads();
    if (threadIdx.x < kBins) hist[threadIdx.x * tiles + blockIdx.x] = cnt[threadIdx.x];
}

// Radix pass, second half (after the histograms are scanned): every item goes
// to hist[d * tiles + b] + (items of digit d earlier in the tile).  A thread's
// items are consecutive, so "earlier" = in an earlier thread, or earlier in
// the same thread: the scatter is stable.
__global__ void __launch_bounds__(kSortThreads)
    radix_scatter(const int32_t *__restrict__ ks, const int32_t *__restrict__ vs,
                  int32_t *__restrict__ kd, int32_t *__restrict__ vd,
                  const int64_t *__restrict__ n_active, int shift,
                  const int32_t *__restrict__ hist, int tiles) {
    __shared__ int S[kBins * kSortThreads];  // [digit][thread] counts, then offsets
    __shared__ int tile_base[kBins];
    __shared__ int part[kSortThreads];
    const int t = threadIdx.x;
    const int64_t n = *n_active;
    const int64_t base = (int64_t)blockIdx.x * kSortTile + (int64_t)t * kSortItems;
    int32_t k[kSortItems], v[kSortItems];
#pragma unroll
    for (int d = 0; d < kBins; ++d) S[d * kSortThreads + t] = 0;
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
        const bool live = base + i < n;
        k[i] = live ? ks[base + i] : 0;
        v[i] = live ? vs[base + i] : 0;
        if (live) ++S[((k[i] >> shift) & (kBins - 1)) * kSortThreads + t];
    }
    __syncthreads();
    // exclusive scan of S in (digit, thread) order: kBins entries per thread
    constexpr int kPer = kBins * kSortThreads / kSortThreads;
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) sum += S[t * kPer + j];
    part[t] = sum;
    __syncthreads();
    // Hillis-Steele inclusive scan of the per-thread sums
    for (int off = 1; off < kSortThreads; off <<= 1) {
        const int y = (t >= off) ? part[t - off] : 0;
        __syncthreads();
        part[t] += y;
        __syncthreads();
    }
    int run = part[t] - sum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int c = S[t * kPer + j];
        S[t * kPer + j] = run;
        run += c;
    }
    __syncthreads();
    if (t < kBins) tile_base[t] = S[t * kSortThreads];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
        if (base + i < n) {
            const int d = (k[i] >> shift) & (kBins - 1);
            const int64_t pos =
                (int64_t)hist[d * tiles + blockIdx.x] + (S[d * kSortThreads + t]++ - tile_base[d]);
            kd[pos] = k[i];
            vd[pos] = v[i];
        }
    }
}

// Each row's entry list sorted by column: entry i goes to the number of
// entries of the row with a smaller column (the columns of a row are
// distinct).  One warp per row.
constexpr int kSortRowsPerBlock = 8;
__global__ void __launch_bounds__(32 * kSortRowsPerBlock)
    sort_entries(const int32_t *__restrict__ ecount, int2 *__restrict__ ent, int64_t rows) {
    __shared__ int2 buf[kSortRowsPerBlock][kEntCap];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kSortRowsPerBlock + w;
    if (r >= rows) return;
    const int c = min(ecount[r], kEntCap);
    if (c <= 1) return;
    int2 *row = ent + r * kEntCap;
    for (int i = lane; i < c; i += 32) buf[w][i] = row[i];
    __syncwarp();
    for (int i = lane; i < c; i += 32) {
        const int2 e = buf[w][i];
        int pos = 0;
        for (int j = 0; j < c; ++j) pos += (buf[w][j].x < e.x) ? 1 : 0;
        row[pos] = e;
    }
}

// Per-token entry counts (capped) for the flat list.
__global__ void entries_count(const int32_t *__restrict__ ecount, int64_t n,
                              int32_t *__restrict__ eoff) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n;
         t += (int64_t)gridDim.x * blockDim.x)
        eoff[t] = min(ecount[t], kEntCap);
}

// The flat list: token t's entries at eoff[t] (exclusive prefix sums), as
// (column, flat index) sort pairs plus the token and w of each entry.
__global__ void entries_scatter(const int32_t *__restrict__ eoff, const int2 *__restrict__ ent,
                                int64_t n, int32_t *__restrict__ key, int32_t *__restrict__ val,
                                int32_t *__restrict__ ent_t, float *__restrict__ ent_w,
                                const int32_t *__restrict__ ecount) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int c = min(ecount[t], kEntCap);
        const int64_t o = eoff[t];
        for (int i = 0; i < c; ++i) {
            const int2 e = ent[t * kEntCap + i];
            key[o + i] = e.x;
            val[o + i] = (int32_t)(o + i);
            ent_t[o + i] = (int32_t)t;
            ent_w[o + i] = __int_as_float(e.y);
        }
    }
}

// begin/end (pre-zeroed, [V]) of each column's range in the sorted keys.
__global__ void dw_bounds(const int32_t *__restrict__ key, const int64_t *__restrict__ n_active,
                          int32_t *__restrict__ begin, int32_t *__restrict__ end) {
    const int64_t n = *n_active;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t k = key[i];
        if (i == 0 || key[i - 1] != k) begin[k] = (int32_t)i;
        if (i == n - 1 || key[i + 1] != k) end[k] = (int32_t)(i + 1);
    }
}

// Rows with entries, in ascending order: a segment of the sorted keys starts
// at i when i == 0 or key[i - 1] != key[i].  First half: segment starts per
// block of kScanThreads keys.
__global__ void __launch_bounds__(kScanThreads)
    seg_count(const int32_t *__restrict__ key, const int64_t *__restrict__ n_keys,
              int32_t *__restrict__ block_cnt) {
    const int64_t n = *n_keys;
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    const bool start = i < n && (i == 0 || key[i - 1] != key[i]);
    const int c = __syncthreads_count(start);
    if (threadIdx.x == 0) block_cnt[blockIdx.x] = c;
}

// Second half: rows[offset of the block + rank in the block] = the row.
__global__ void __launch_bounds__(kScanThreads)
    seg_write(const int32_t *__restrict__ key, const int64_t *__restrict__ n_keys,
              const int32_t *__restrict__ block_ofs, int32_t *__restrict__ rows) {
    __shared__ int warp_cnt[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n = *n_keys;
    const int64_t i = (int64_t)blockIdx.x * kScanThreads + threadIdx.x;
    const bool start = i < n && (i == 0 || key[i - 1] != key[i]);
    const unsigned m = __ballot_sync(0xffffffffu, start);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    if (start) rows[block_ofs[blockIdx.x] + before + __popc(m & ((1u << lane) - 1u))] = key[i];
}

// The fp32 term of dW, S[v, :] = sum over column v's entries e, in canonical
// token order, of w_e h_{t_e}: one block per (row with entries, 256-column
// slice of H), 128 threads with 2 columns each.  Entries go through shared
// memory 32 at a time so that the h loads of a batch overlap; the sum is one
// fmaf chain per column in entry order.  Written into dW, whose GEMM epilogue
// then subtracts the tensor-core part.  (A hot vocabulary row -- a token that
// thousands of canonical tokens target -- is a long loop here but only for
// its own 16 blocks; inside the GEMM epilogue it stalled whole tiles.)
constexpr int kSThreads = 128;
constexpr int kSCols = 2 * kSThreads;
__global__ void __launch_bounds__(kSThreads)
    dw_fp32_term(const int32_t *__restrict__ rows, const int64_t *__restrict__ n_rows,
                 const int32_t *__restrict__ begin, const int32_t *__restrict__ end,
                 const int32_t *__restrict__ idx, const int32_t *__restrict__ ent_t,
                 const float *__restrict__ ent_w, const uint16_t *__restrict__ hc, int64_t H,
                 float *__restrict__ dW) {
    __shared__ int32_t s_t[32];
    __shared__ float s_w[32];
    const int64_t ncb = (H + kSCols - 1) / kSCols;
    const int64_t items = *n_rows * ncb;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int32_t v = rows[it / ncb];
        const int64_t col = (it % ncb) * kSCols + 2 * threadIdx.x;  // H % 64 == 0: col + 1 < H
        const bool live = col < H;
        const int32_t b0 = begin[v], b1 = end[v];
        float s0 = 0.f, s1 = 0.f;
        for (int32_t i0 = b0; i0 < b1; i0 += 32) {
            const int m = min(32, b1 - i0);
            __syncthreads();
            if (threadIdx.x < m) {
                const int32_t e = idx[i0 + threadIdx.x];
                s_t[threadIdx.x] = ent_t[e];
                s_w[threadIdx.x] = ent_w[e];
            }
            __syncthreads();
            if (live) {
#pragma unroll 8
                for (int k = 0; k < m; ++k) {
                    const uint32_t hv =
                        *reinterpret_cast<const uint32_t *>(hc + (int64_t)s_t[k] * H + col);
                    const float w = s_w[k];
                    s0 = __fmaf_rn(w, bf16_lo(hv), s0);
                    s1 = __fmaf_rn(w, bf16_hi(hv), s1);
                }
            }
        }
        if (live) *reinterpret_cast<float2 *>(dW + (int64_t)v * H + col) = make_float2(s0, s1);
        __syncthreads();
    }
}

}  // namespace

int64_t dw_scan_entries(int64_t n) {
    const int64_t blocks = (n + kScanThreads - 1) / kScanThreads;
    const int64_t tiles = (n + kSortTile - 1) / kSortTile;
    return std::max<int64_t>(1, std::max(blocks, tiles * (int64_t)kBins));
}

int dw_sort_passes(int64_t V) {
    int bits = 1;
    while ((int64_t(1) << bits) < V) ++bits;
    return (bits + kRadixBits - 1) / kRadixBits;
}

cudaError_t launch_dw_prep(const uint16_t *h, const int64_t *targets, const int32_t *cu,
                           int num_seqs, int64_t T, int64_t H, int64_t V, const float *lse,
                           const float *grad, const int64_t *order, int64_t n, const DwBuffers &b,
                           const DeviceInfo &di, cudaStream_t st) {
    (void)di;
    const unsigned cblocks = (unsigned)((n + kScanThreads - 1) / kScanThreads);
    dw_compact_count<<<cblocks, kScanThreads, 0, st>>>(order, n, T, targets, cu, num_seqs, V,
                                                       b.scan);
    scan_counts<<<1, kScanThreads, 0, st>>>(b.scan, cblocks, b.n_active);
    dw_compact_write<<<cblocks, kScanThreads, 0, st>>>(order, n, T, targets, cu, num_seqs, V,
                                                       b.scan, b.crow);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dw_gather<<<(unsigned)n, 128, 0, st>>>(h, grad, lse, targets, b.crow, b.n_active, n, H, b.hc,
                                           b.gc, b.lsec, b.tgtc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the dZ / dZ^T GEMM appends to these lists
    return cudaMemsetAsync(b.ecount, 0, (size_t)n * sizeof(int32_t), st);
}

cudaError_t launch_dw_entries(int64_t n, int64_t V, const DwBuffers &b, const uint16_t *hc,
                              int64_t H, float *dW, const DeviceInfo &di, cudaStream_t st) {
    const unsigned grid_n =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)di.sm_count * 8));
    entries_count<<<grid_n, 256, 0, st>>>(b.ecount, n, b.eoff);
    scan_counts<<<1, kScanThreads, 0, st>>>(b.eoff, n, b.etotal);
    entries_scatter<<<grid_n, 256, 0, st>>>(b.eoff, b.ent, n, b.key0, b.val0, b.ent_t, b.ent_w,
                                            b.ecount);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t emax = n * (int64_t)kEntCap;
    const int passes = dw_sort_passes(V);
    const int tiles = (int)((emax + kSortTile - 1) / kSortTile);
    int32_t *ks = b.key0, *vs = b.val0, *kd = b.key1, *vd = b.val1;
    for (int p = 0; p < passes; ++p) {
        const int shift = p * kRadixBits;
        radix_histogram<<<tiles, kSortThreads, 0, st>>>(ks, b.etotal, shift, b.scan, tiles);
        scan_counts<<<1, kScanThreads, 0, st>>>(b.scan, (int64_t)tiles * kBins, nullptr);
        radix_scatter<<<tiles, kSortThreads, 0, st>>>(ks, vs, kd, vd, b.etotal, shift, b.scan,
                                                      tiles);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        std::swap(ks, kd);
        std::swap(vs, vd);
    }
    e = cudaMemsetAsync(b.begin, 0, (size_t)V * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.end, 0, (size_t)V * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((emax + 255) / 256, (int64_t)di.sm_count * 8));
    dw_bounds<<<grid, 256, 0, st>>>(ks, b.etotal, b.begin, b.end);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the rows with entries, then their fp32 term written into dW
    const unsigned sblocks = (unsigned)((emax + kScanThreads - 1) / kScanThreads);
    seg_count<<<sblocks, kScanThreads, 0, st>>>(ks, b.etotal, b.scan);
    scan_counts<<<1, kScanThreads, 0, st>>>(b.scan, sblocks, b.n_rows);
    seg_write<<<sblocks, kScanThreads, 0, st>>>(ks, b.etotal, b.scan, b.rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dw_fp32_term<<<(unsigned)di.sm_count * 16, kSThreads, 0, st>>>(
        b.rows, b.n_rows, b.begin, b.end, vs, b.ent_t, b.ent_w, hc, H, dW);
    return cudaGetLastError();
}

cudaError_t launch_sort_entries(int32_t *ecount, int2 *ent, int64_t rows, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + kSortRowsPerBlock - 1) / kSortRowsPerBlock);
    sort_entries<<<grid, 32 * kSortRowsPerBlock, 0, st>>>(ecount, ent, rows);
    return cudaGetLastError();
}

}  // namespace rk
