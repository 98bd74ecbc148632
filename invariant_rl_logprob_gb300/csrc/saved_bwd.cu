// saved_bwd.cu -- the two elementwise steps of the linear_logp backward that
// starts from the forward's saved state instead of recomputing z = h W^T
// (issue #244 "[WS1 Test] ...", Workstream 3 #153: fixed,
// batch-shape-independent order, no atomicAdd on values).
//
// The forward (tile mode kFwdS) saved, per row t and vocabulary tile j of 256
// columns, the tile maximum m_tj and e[t, v] = bf16(2^((z - m_tj) log2 e)).
// With lse from the forward and the upstream gradient g,
//   p[t, v] = e^(m_tj - lse_t) * e[t, v]
// is the row's softmax up to the bf16 rounding of e, and
//   stash_to_dz   rewrites e in place into dZ = bf16(g e^(m_tj - lse) e) on
//                 every column except the target and the columns with
//                 p >= 1/64, which it leaves as 0 and lists as the row's fp32
//                 entries (as the recompute path does);
//   stash_to_dz_canonical does the same for the canonical tokens of the dW
//                 backward, writing dZ in canonical order (transpose_dz then
//                 gives the dW GEMM its dZ^T);
//   exact_entries gives each listed column its fp32 weight
//                 w = g (onehot - p) from an exact z = h_t . W_v (fp32, one
//                 fixed order), so a peaked softmax never puts a rounded large
//                 term into dh.
// Each element and each entry depends only on its row, so a row's results do
// not depend on the batch around it.
#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvGroupsPerThread = 4;
constexpr int64_t kConvCols = (int64_t)kConvThreads * 8 * kConvGroupsPerThread;  // 8192 per block
constexpr int kTileCols = 256;  // the forward's vocabulary tile

// Elementwise max of two bf16 pairs (exact).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __noinline__ void list_entry(int64_t col, int32_t *count, int2 *list, unsigned *err) {
    const int slot = atomicAdd(count, 1);
    if (slot < kEntCap)
        list[slot] = make_int2((int)col, 0);
    else
        atomicOr(err, kErrLse);
}

// One group of 8 saved terms (columns [c0, c0 + 8) of a row with lse l,
// gradient g and target tgt, in the tile whose maximum is mt) -> dZ, with
// the target and p >= 1/64 columns left at 0 and listed.  The one function
// both conversion kernels use, so a row's dZ and entries do not depend on
// which of them ran.
__device__ __forceinline__ uint4 convert_group(uint4 w, int64_t c0, int64_t V, int64_t tgt, float mt,
                                               float l, float g, int32_t *count, int2 *list,
                                               unsigned *err) {
    const float f = ex2(__fmul_rn(__fsub_rn(mt, l), kLog2e));  // e^(m_tj - lse) <= 1
    const float c = __fmul_rn(g, f);
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[4];
    // The group's largest term decides, in one test, that no column of it
    // needs an fp32 entry (f e <= f max(e) by the monotonic rounding of the
    // product): the same decision as the per-column test below.
    const uint32_t mx = max_bf16x2(max_bf16x2(q[0], q[1]), max_bf16x2(q[2], q[3]));
    const bool plain = c0 + 8 <= V && !(tgt >= c0 && tgt < c0 + 8) &&
                       __fmul_rn(f, fmaxf(bf16_lo(mx), bf16_hi(mx))) < kEntTau;
    if (plain) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = pack_bf16x2(__fmul_rn(c, bf16_lo(q[k])), __fmul_rn(c, bf16_hi(q[k])));
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float d[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int64_t col = c0 + 2 * k + hh;
                const float e = hh ? bf16_hi(q[k]) : bf16_lo(q[k]);
                d[hh] = 0.f;
                if (col < V) {
                    if (col == tgt || __fmul_rn(f, e) >= kEntTau)
                        list_entry(col, count, list, err);
                    else
                        d[hh] = __fmul_rn(c, e);
                }
            }
            o[k] = pack_bf16x2(d[0], d[1]);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// grid (rows, ceil(V / kConvCols)): block (r, q) takes columns
// [q kConvCols, (q + 1) kConvCols) of row row0 + r, 8 consecutive columns per
// thread and group (a group of 8 never crosses a 256-column tile).
__global__ void __launch_bounds__(kConvThreads)
    stash_to_dz(uint16_t *__restrict__ dz, int64_t ldz, const float2 *__restrict__ part,
                int32_t num_n, const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                int num_seqs, int64_t row0, int64_t V, const float *__restrict__ lse,
                const float *__restrict__ grad, const uint8_t *__restrict__ live,
                int32_t *__restrict__ ecount, int2 *__restrict__ ent, unsigned *err) {
    const int64_t row = row0 + blockIdx.x;
    // a row block without active rows is skipped by the dh GEMM too
    if (live != nullptr && live[row / kLiveBlockRows] == 0) return;
    const int64_t tgt = targets[row];
    const bool active = row_active(row, tgt, cu, num_seqs) && tgt < V;
    uint16_t *drow = dz + row * ldz;
    const float g = active ? grad[row] : 0.f;
    const float l = active ? lse[row] : 0.f;
    // all of the thread's loads first, then the conversions (1.3 % faster
    // than loading each group just before converting it)
    uint4 w[kConvGroupsPerThread];
#pragma unroll
    for (int i = 0; i < kConvGroupsPerThread; ++i) {
        const int64_t c0 = (int64_t)blockIdx.y * kConvCols + (int64_t)i * (kConvThreads * 8) +
                           (int64_t)threadIdx.x * 8;
        // ldz % 8 == 0: 16-byte aligned
        if (active && c0 < V) w[i] = *reinterpret_cast<const uint4 *>(drow + c0);
    }
#pragma unroll
    for (int i = 0; i < kConvGroupsPerThread; ++i) {
        const int64_t c0 = (int64_t)blockIdx.y * kConvCols + (int64_t)i * (kConvThreads * 8) +
                           (int64_t)threadIdx.x * 8;
        if (c0 >= V) continue;
        uint4 *gp = reinterpret_cast<uint4 *>(drow + c0);
        if (!active) {
            *gp = make_uint4(0, 0, 0, 0);
            continue;
        }
        *gp = convert_group(w[i], c0, V, tgt, part[row * num_n + c0 / kTileCols].x, l, g,
                            ecount + row, ent + row * kEntCap, err);
    }
}

// The same conversion into canonical order: canonical token c (physical row
// crow[c], c < n_active; later positions are zero rows) takes the saved terms
// of its row and writes dZ row c of dzc and entry list c.  The row's lse, g
// and target come from the canonical copies.
__global__ void __launch_bounds__(kConvThreads)
    stash_to_dz_canonical(const uint16_t *__restrict__ terms, int64_t ldz,
                          const float2 *__restrict__ part, int32_t num_n,
                          const int64_t *__restrict__ crow, const int64_t *__restrict__ n_active,
                          const int64_t *__restrict__ tgtc, const float *__restrict__ lsec,
                          const float *__restrict__ gc, int64_t V, uint16_t *__restrict__ dzc,
                          int32_t *__restrict__ ecount, int2 *__restrict__ ent, unsigned *err) {
    const int64_t c = blockIdx.x;
    const bool live = c < *n_active;
    const int64_t row = live ? crow[c] : 0;
    const int64_t tgt = live ? tgtc[c] : -1;
    uint16_t *drow = dzc + c * ldz;
    const uint16_t *srow = terms + row * ldz;
#pragma unroll
    for (int i = 0; i < kConvGroupsPerThread; ++i) {
        const int64_t c0 = (int64_t)blockIdx.y * kConvCols + (int64_t)i * (kConvThreads * 8) +
                           (int64_t)threadIdx.x * 8;
        if (c0 >= V) continue;
        uint4 *gp = reinterpret_cast<uint4 *>(drow + c0);
        if (!live) {
            *gp = make_uint4(0, 0, 0, 0);
            continue;
        }
        *gp = convert_group(*reinterpret_cast<const uint4 *>(srow + c0), c0, V, tgt,
                            part[row * num_n + c0 / kTileCols].x, lsec[c], gc[c], ecount + c,
                            ent + c * kEntCap, err);
    }
}

// dZ^T [V][ldn] from dZ [n][ldz] (bf16), through 64 x 64 tiles in shared
// memory; token columns in [n, ldn) are written as 0.  Global memory moves in
// 16-byte vectors (8 bf16): ldz and ldn are multiples of 8.
constexpr int kTrTile = 64;
constexpr int kTrPitch = kTrTile;  // halfwords per shared row (16-byte aligned, swizzled groups)
__global__ void __launch_bounds__(256)
    transpose_dz(const uint16_t *__restrict__ dz, int64_t ldz, int64_t n, int64_t V,
                 uint16_t *__restrict__ dzt, int64_t ldn) {
    __shared__ __align__(16) uint16_t tile[kTrTile][kTrPitch];
    const int64_t t0 = (int64_t)blockIdx.x * kTrTile, v0 = (int64_t)blockIdx.y * kTrTile;
    // load: 64 token rows x 8 vectors of 8 vocabulary columns, 2 per thread
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int idx = threadIdx.x + 256 * j;
        const int r = idx >> 3, c8 = idx & 7;
        const int64_t t = t0 + r, v = v0 + c8 * 8;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (t < n && v < V) {
            if (v + 8 <= ldz) {
                x = *reinterpret_cast<const uint4 *>(dz + t * ldz + v);
            }
        }
        // 8-column group g of row r sits at group g ^ (r / 8): the reads below
        // (one column, 8 rows 8 apart) then fall in different banks
        *reinterpret_cast<uint4 *>(&tile[r][((c8 ^ (r >> 3)) & 7) * 8]) = x;
    }
    __syncthreads();
    // store: 64 vocabulary rows x 8 vectors of 8 tokens, 2 per thread
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int idx = threadIdx.x + 256 * j;
        const int r = idx >> 3, c8 = idx & 7;  // r: vocabulary row in the tile
        const int64_t v = v0 + r, t = t0 + c8 * 8;
        if (v >= V || t >= ldn) continue;
        // column r of rows c8 * 8 .. c8 * 8 + 7 (all with row / 8 == c8)
        const int pc = ((((r >> 3) ^ c8) & 7) * 8) + (r & 7);
        uint32_t q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            q[k] = (uint32_t)tile[c8 * 8 + 2 * k][pc] | ((uint32_t)tile[c8 * 8 + 2 * k + 1][pc] << 16);
        *reinterpret_cast<uint4 *>(dzt + v * ldn + t) = make_uint4(q[0], q[1], q[2], q[3]);
    }
}

// One warp per row: each listed column's exact z = h_t . W_v, summed in fp32
// with lane l taking the 8-element groups l, l + 32, ... (products exact in
// fp32, added in group order), then a fixed xor tree; w = g (onehot - p).
constexpr int kExactRowsPerBlock = 8;
__global__ void __launch_bounds__(32 * kExactRowsPerBlock)
    exact_entries(const uint16_t *__restrict__ h, const uint16_t *__restrict__ W, int64_t H,
                  const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                  int num_seqs, int64_t row0, int64_t row_end, int64_t V,
                  const float *__restrict__ lse, const float *__restrict__ grad,
                  const int32_t *__restrict__ ecount, int2 *__restrict__ ent) {
    const int64_t row = row0 + (int64_t)blockIdx.x * kExactRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= row_end) return;
    const int64_t tgt = targets[row];
    if (!row_active(row, tgt, cu, num_seqs) || tgt >= V) return;
    const int n = min(ecount[row], kEntCap);
    const float g = grad[row];
    const float l = lse[row];
    const uint4 *hr = reinterpret_cast<const uint4 *>(h + row * H);
    int2 *el = ent + row * kEntCap;
    for (int e = 0; e < n; ++e) {
        const int v = el[e].x;
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (int64_t)v * H);
        float acc = 0.f;
        for (int64_t k8 = lane; k8 < H / 8; k8 += 32) {
            const uint4 a = __ldg(hr + k8), b = __ldg(wr + k8);
            const uint32_t qa[4] = {a.x, a.y, a.z, a.w}, qb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc = __fmaf_rn(bf16_lo(qa[j]), bf16_lo(qb[j]), acc);
                acc = __fmaf_rn(bf16_hi(qa[j]), bf16_hi(qb[j]), acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        const float p = ex2(__fmul_rn(__fsub_rn(acc, l), kLog2e));
        const float w = __fmul_rn(g, __fsub_rn(v == tgt ? 1.f : 0.f, p));
        if (lane == 0) el[e].y = __float_as_int(w);
    }
}

}  // namespace

cudaError_t launch_stash_to_dz(uint16_t *dz, int64_t ldz, const float2 *part, int32_t num_n,
                               const int64_t *targets, const int32_t *cu, int num_seqs,
                               int64_t row0, int64_t rows, int64_t V, const float *lse,
                               const float *grad, const uint8_t *live, int32_t *ecount, int2 *ent,
                               const DeviceInfo &di, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int64_t segs = (V + kConvCols - 1) / kConvCols;
    if (segs > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)rows, (unsigned)segs);
    stash_to_dz<<<grid, kConvThreads, 0, st>>>(dz, ldz, part, num_n, targets, cu, num_seqs, row0, V,
                                              lse, grad, live, ecount, ent, di.err);
    return cudaGetLastError();
}

cudaError_t launch_stash_to_dz_canonical(const uint16_t *terms, int64_t ldz, const float2 *part,
                                         int32_t num_n, const int64_t *crow,
                                         const int64_t *n_active, const int64_t *tgtc,
                                         const float *lsec, const float *gc, int64_t n, int64_t V,
                                         uint16_t *dzc, int32_t *ecount, int2 *ent,
                                         const DeviceInfo &di, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t segs = (V + kConvCols - 1) / kConvCols;
    if (segs > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)n, (unsigned)segs);
    stash_to_dz_canonical<<<grid, kConvThreads, 0, st>>>(terms, ldz, part, num_n, crow, n_active,
                                                        tgtc, lsec, gc, V, dzc, ecount, ent,
                                                        di.err);
    return cudaGetLastError();
}

cudaError_t launch_transpose_dz(const uint16_t *dz, int64_t ldz, int64_t n, int64_t V,
                                uint16_t *dzt, int64_t ldn, cudaStream_t st) {
    if (n == 0 || V == 0) return cudaSuccess;
    const int64_t gy = (V + kTrTile - 1) / kTrTile;
    if (gy > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((ldn + kTrTile - 1) / kTrTile), (unsigned)gy);
    transpose_dz<<<grid, 256, 0, st>>>(dz, ldz, n, V, dzt, ldn);
    return cudaGetLastError();
}

cudaError_t launch_exact_entries(const uint16_t *h, const uint16_t *W, int64_t H,
                                 const int64_t *targets, const int32_t *cu, int num_seqs,
                                 int64_t row0, int64_t rows, int64_t V, const float *lse,
                                 const float *grad, const int32_t *ecount, int2 *ent,
                                 cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + kExactRowsPerBlock - 1) / kExactRowsPerBlock);
    exact_entries<<<grid, 32 * kExactRowsPerBlock, 0, st>>>(h, W, H, targets, cu, num_seqs, row0,
                                                           row0 + rows, V, lse, grad, ecount, ent);
    return cudaGetLastError();
}

}  // namespace rk
