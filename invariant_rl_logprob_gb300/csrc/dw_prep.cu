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
//            the active rows, order kept (one block, chunked prefix sums);
//   gather   h, g, lse and the target of every canonical token into dense
//            buffers; positions past the active count hold zeros and target
//            -1, so a GEMM over all n positions adds exact zeros for them;
//   sort     (target, canonical index) pairs by target with a stable
//            one-bit LSD radix sort (one block): ties keep canonical order;
//   bounds   the [begin, end) range of each target in the sorted list.
//
// Every step is deterministic: counts and prefix sums over integers, no
// floating-point atomics.
#include <algorithm>

#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

constexpr int kScanThreads = 1024;

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

// crow[c] = physical row of canonical token c (c < n_active); *n_active.
__global__ void __launch_bounds__(kScanThreads)
    dw_compact(const int64_t *__restrict__ order, int64_t n, int64_t T,
               const int64_t *__restrict__ targets, const int32_t *__restrict__ cu, int num_seqs,
               int64_t V, int64_t *__restrict__ crow, int64_t *__restrict__ n_active) {
    const int64_t per = (n + kScanThreads - 1) / kScanThreads;
    const int64_t b = (int64_t)threadIdx.x * per;
    const int64_t e = min(n, b + per);
    int64_t cnt = 0;
    for (int64_t i = b; i < e; ++i)
        cnt += candidate_active(order, i, T, targets, cu, num_seqs, V) ? 1 : 0;
    int64_t total;
    int64_t pos = block_exclusive_scan(cnt, &total);
    for (int64_t i = b; i < e; ++i)
        if (candidate_active(order, i, T, targets, cu, num_seqs, V))
            crow[pos++] = candidate_row(order, i);
    if (threadIdx.x == 0) *n_active = total;
}

// Canonical buffers: hc [n, H] bf16, gc / lsec fp32 [n], tgtc int64 [n],
// key / val int32 [n] (sort input).
__global__ void dw_gather(const uint16_t *__restrict__ h, const float *__restrict__ grad,
                          const float *__restrict__ lse, const int64_t *__restrict__ targets,
                          const int64_t *__restrict__ crow, const int64_t *__restrict__ n_active,
                          int64_t n, int64_t H, uint16_t *__restrict__ hc, float *__restrict__ gc,
                          float *__restrict__ lsec, int64_t *__restrict__ tgtc,
                          int32_t *__restrict__ key, int32_t *__restrict__ val) {
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
        key[c] = (int32_t)t;
        val[c] = (int32_t)c;
    }
}

// Stable LSD radix sort of (key, val) over the first *n_active entries, one
// bit per pass, keys < 2^bits.  Result in (key0, val0) when bits is even,
// (key1, val1) when odd.
__global__ void __launch_bounds__(kScanThreads)
    dw_radix_sort(int32_t *__restrict__ key0, int32_t *__restrict__ val0,
                  int32_t *__restrict__ key1, int32_t *__restrict__ val1,
                  const int64_t *__restrict__ n_active, int bits) {
    const int64_t n = *n_active;
    const int64_t per = (n + kScanThreads - 1) / kScanThreads;
    const int64_t b = (int64_t)threadIdx.x * per;
    const int64_t e = min(n, b + per);
    int32_t *ks = key0, *vs = val0, *kd = key1, *vd = val1;
    for (int bit = 0; bit < bits; ++bit) {
        int64_t zeros = 0;
        for (int64_t i = b; i < e; ++i) zeros += ((ks[i] >> bit) & 1) ? 0 : 1;
        int64_t total_zeros;
        const int64_t zpos0 = block_exclusive_scan(zeros, &total_zeros);
        int64_t zpos = zpos0;
        int64_t opos = total_zeros + (b - zpos0);  // ones before this chunk = b - zeros before
        for (int64_t i = b; i < e; ++i) {
            const int32_t k = ks[i];
            if ((k >> bit) & 1) {
                kd[opos] = k;
                vd[opos] = vs[i];
                ++opos;
            } else {
                kd[zpos] = k;
                vd[zpos] = vs[i];
                ++zpos;
            }
        }
        __syncthreads();
        int32_t *t;
        t = ks; ks = kd; kd = t;
        t = vs; vs = vd; vd = t;
    }
}

// begin/end (pre-zeroed, [V]) of each target's range in the sorted keys.
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

}  // namespace

cudaError_t launch_dw_prep(const uint16_t *h, const int64_t *targets, const int32_t *cu,
                           int num_seqs, int64_t T, int64_t H, int64_t V, const float *lse,
                           const float *grad, const int64_t *order, int64_t n, const DwBuffers &b,
                           const DeviceInfo &di, cudaStream_t st) {
    dw_compact<<<1, kScanThreads, 0, st>>>(order, n, T, targets, cu, num_seqs, V, b.crow,
                                           b.n_active);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dw_gather<<<(unsigned)n, 128, 0, st>>>(h, grad, lse, targets, b.crow, b.n_active, n, H, b.hc,
                                           b.gc, b.lsec, b.tgtc, b.key0, b.val0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int bits = 1;
    while ((int64_t(1) << bits) < V) ++bits;
    dw_radix_sort<<<1, kScanThreads, 0, st>>>(b.key0, b.val0, b.key1, b.val1, b.n_active, bits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int32_t *sorted_key = (bits % 2 == 0) ? b.key0 : b.key1;
    e = cudaMemsetAsync(b.begin, 0, (size_t)V * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.end, 0, (size_t)V * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)di.sm_count * 4);
    if (grid == 0) grid = 1;
    dw_bounds<<<grid, 256, 0, st>>>(sorted_key, b.n_active, b.begin, b.end);
    return cudaGetLastError();
}

}  // namespace rk
