// logits_logp.cu -- the logits path: selected-token logprob from materialised
// bf16 logits ("logp / batch_invariant_logp", RL-Kernel issue #101, maintainer
// comment, P0 operator list; chain index 8 of PR #264 "docs(ws1):
// batch-invariance contract RFC"), and its backward.
//
//   lse[t]  = log sum_v exp(logits[t, v])
//   logp[t] = logits[t, targets[t]] - lse[t]
//
// HBM-bound: every logit is read once (T*V*2 bytes), nothing else is large.
//
// Batch invariance by construction.  A row is reduced by four warps, i.e. 128
// "virtual lanes" vl = 32 * (warp of the row) + lane.  The columns are cut into
// groups of 8 (group g = columns [8g, 8g+8)); virtual lane vl owns groups
// vl, vl + 128, vl + 256, ... and folds them, in that order, in batches of 8
// groups: the batch maximum (exact, any order) updates the running max once,
// then the batch's 64 terms 2^((z - m) log2 e) are summed by a fixed pairwise
// tree and added to the running sum.  The 32 partials of a warp are merged by a
// fixed xor-shuffle tree, and the four warps' partials in warp order.  All of
// that depends only on V -- never on T, the row's index, the grid or the
// row's address: rows whose address allows 16-byte loads use them, others load
// 2-byte elements into the same groups (missing columns read as -inf) and run
// exactly the same floating-point operations.
//
// Four warps per row rather than fewer: with 64 values in flight per lane and
// one wave of rows, the extra warps hide the load latency behind the other
// warps' arithmetic, so the kernel stays at the memory's pace when the SM
// clock drops (about 1.5 GHz right after power-capped GEMMs: 24.3 us per
// T = 2048, V = 32000 call against 28.6 us with two warps per row).
#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

// forward: four warps per row; backward: two (each element is independent)
constexpr int kWarpsPerRow = 4;
constexpr int kLanesPerRow = 32 * kWarpsPerRow;
constexpr int kThreads = 128;
constexpr int kRowsPerBlock = kThreads / kLanesPerRow;
constexpr int kBwdWarpsPerRow = 2;
constexpr int kBwdLanesPerRow = 32 * kBwdWarpsPerRow;
constexpr int kBwdRowsPerBlock = kThreads / kBwdLanesPerRow;
constexpr int kBatch = 8;  // groups per batch (64 values)
constexpr uint32_t kNegInfPair = 0xFF80FF80u;  // two bf16 -inf

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch.  The logits kernels are launched so that
// their blocks may become resident while the previous kernel in the stream
// finishes; each block then waits (griddepcontrol.wait) until that kernel has
// completed and its writes are visible, before it reads anything.  Right after
// that wait it lets the next such launch start the same way.  Stream order is
// therefore unchanged; only launch latency overlaps.
__device__ __forceinline__ void wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Elementwise max of two bf16 pairs (exact).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Folds a batch of kBatch groups (8 bf16 each, packed as uint4) into (m, s).
__device__ __forceinline__ void fold_batch(const uint4 (&w)[kBatch], float &m, float &s) {
    uint32_t t[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        t[u] = max_bf16x2(max_bf16x2(w[u].x, w[u].y), max_bf16x2(w[u].z, w[u].w));
#pragma unroll
    for (int st = 1; st < kBatch; st *= 2)
#pragma unroll
        for (int u = 0; u + st < kBatch; u += 2 * st) t[u] = max_bf16x2(t[u], t[u + st]);
    const float bm = fmaxf(bf16_lo(t[0]), bf16_hi(t[0]));
    if (bm > m) {
        // ex2((m - bm) log2 e) == 1 exactly when bm == m, so skipping the
        // rescale when the maximum does not grow changes no bit.
        s = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, bm), kLog2e)));
        m = bm;
    }
    const float mb = __fmul_rn(-m, kLog2e);
    float l[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        float e[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            e[2 * j] = ex2(__fmaf_rn(bf16_lo(q[j]), kLog2e, mb));
            e[2 * j + 1] = ex2(__fmaf_rn(bf16_hi(q[j]), kLog2e, mb));
        }
        l[u] = __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3])),
                         __fadd_rn(__fadd_rn(e[4], e[5]), __fadd_rn(e[6], e[7])));
    }
#pragma unroll
    for (int st = 1; st < kBatch; st *= 2)
#pragma unroll
        for (int u = 0; u + st < kBatch; u += 2 * st) l[u] = __fadd_rn(l[u], l[u + st]);
    s = __fadd_rn(s, l[0]);
}

// Group g of a row as 4 packed bf16 pairs, from 2-byte loads (-inf past V).
__device__ __forceinline__ uint4 load_group_scalar(const uint16_t *zrow, int64_t g, int64_t V) {
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = (g << 3) + j;
        h[j] = (c < V) ? (uint32_t)__ldg(zrow + c) : 0xFF80u;
    }
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                      h[6] | (h[7] << 16));
}

// VEC: 16-byte loads (V % 8 == 0 and a 16-byte aligned base); otherwise
// 2-byte loads of the same groups.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    logits_logp_kernel(const uint16_t *__restrict__ logits, const int64_t *__restrict__ targets,
                       const int32_t *__restrict__ cu, int num_seqs, int64_t T, int64_t V,
                       float *__restrict__ logp, float *__restrict__ lse, unsigned *err) {
    __shared__ float sh_m[kThreads / 32], sh_s[kThreads / 32];
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wr = warp % kWarpsPerRow;
    const int vl = wr * 32 + lane;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + warp / kWarpsPerRow;
    const int64_t tgt = (row < T) ? targets[row] : -1;
    const bool active = row < T && row_active(row, tgt, cu, num_seqs);  // uniform per row
    const uint16_t *zrow = logits + row * V;
    const int64_t G = (V + 7) >> 3;

    float m = -INFINITY, s = 0.f;
    if (active) {
        const int64_t n_i = (G - vl + kLanesPerRow - 1) / kLanesPerRow;  // groups of this lane
        for (int64_t i0 = 0; i0 < n_i; i0 += kBatch) {
            uint4 w[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t i = i0 + u;
                const int64_t g = vl + (int64_t)kLanesPerRow * i;
                if (i < n_i)
                    w[u] = VEC ? ld_stream_v4(reinterpret_cast<const uint4 *>(zrow) + g)
                               : load_group_scalar(zrow, g, V);
                else
                    w[u] = make_uint4(kNegInfPair, kNegInfPair, kNegInfPair, kNegInfPair);
            }
            fold_batch(w, m, s);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        lse_merge(m, s, mo, so);
    }
    if (lane == 0) {
        sh_m[warp] = m;
        sh_s[warp] = s;
    }
    __syncthreads();
    if (row < T && wr == 0 && lane == 0) {
        if (!active) {
            logp[row] = 0.f;
            if (lse) lse[row] = 0.f;
        } else if (tgt < V) {
#pragma unroll
            for (int k = 1; k < kWarpsPerRow; ++k) lse_merge(m, s, sh_m[warp + k], sh_s[warp + k]);
            const float l = __fadd_rn(m, logf(s));
            logp[row] = __fsub_rn(bf16_bits_to_f32(zrow[tgt]), l);
            if (lse) lse[row] = l;
        } else {
            logp[row] = __int_as_float(0x7fc00000);
            if (lse) lse[row] = __int_as_float(0x7fc00000);
            atomicOr(err, kErrTargetRange);
        }
    }
}

// Logits-path backward: dlogits[t, v] = g[t] * (onehot(target_t)[v] - p[t, v]),
// p = 2^((z - lse) log2 e), written in fp32; each element is independent, so
// the result of a row depends only on that row, its lse and its g.  Two warps
// per row; virtual lane vl owns groups vl, vl + 64, ... of 8 columns.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    logits_bwd_kernel(const uint16_t *__restrict__ logits, const int64_t *__restrict__ targets,
                      const int32_t *__restrict__ cu, int num_seqs, int64_t T, int64_t V,
                      const float *__restrict__ lse, const float *__restrict__ grad,
                      float *__restrict__ dlogits, unsigned *err) {
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int vl = (warp % kBwdWarpsPerRow) * 32 + lane;
    const int64_t row = (int64_t)blockIdx.x * kBwdRowsPerBlock + warp / kBwdWarpsPerRow;
    if (row >= T) return;
    const int64_t tgt = targets[row];
    const bool active = row_active(row, tgt, cu, num_seqs);
    const bool bad = active && tgt >= V;
    if (bad && vl == 0) atomicOr(err, kErrTargetRange);
    const bool live = active && !bad;
    const float g = live ? grad[row] : 0.f;
    const float nl = live ? __fmul_rn(-lse[row], kLog2e) : 0.f;
    const float fill = bad ? __int_as_float(0x7fc00000) : 0.f;
    const uint16_t *zrow = logits + row * V;
    float *orow = dlogits + row * V;
    const int64_t G = (V + 7) >> 3;
#pragma unroll 4
    for (int64_t gi = vl; gi < G; gi += kBwdLanesPerRow) {
        const int64_t c0 = gi << 3;
        float z[8];
        if (VEC) {
            const uint4 w = live ? ld_stream_v4(reinterpret_cast<const uint4 *>(zrow) + gi)
                                 : make_uint4(0, 0, 0, 0);
            z[0] = bf16_lo(w.x);
            z[1] = bf16_hi(w.x);
            z[2] = bf16_lo(w.y);
            z[3] = bf16_hi(w.y);
            z[4] = bf16_lo(w.z);
            z[5] = bf16_hi(w.z);
            z[6] = bf16_lo(w.w);
            z[7] = bf16_hi(w.w);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                z[j] = (live && c0 + j < V) ? bf16_bits_to_f32(__ldg(zrow + c0 + j)) : 0.f;
        }
        float d[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p = ex2(__fmaf_rn(z[j], kLog2e, nl));
            const float oh = (c0 + j == tgt) ? 1.f : 0.f;
            d[j] = live ? __fmul_rn(g, __fsub_rn(oh, p)) : fill;
        }
        if (VEC) {
            // one 32-byte store per lane: a warp writes 1 KB contiguously
            asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(orow + c0),
                         "f"(d[0]), "f"(d[1]), "f"(d[2]), "f"(d[3]), "f"(d[4]), "f"(d[5]), "f"(d[6]),
                         "f"(d[7])
                         : "memory");
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (c0 + j < V) orow[c0 + j] = d[j];
        }
    }
}

// Launch configuration with programmatic stream serialisation (see
// wait_prior_grid).
void dependent_launch_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, unsigned grid,
                             cudaStream_t st) {
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(grid);
    cfg->blockDim = dim3(kThreads);
    cfg->dynamicSmemBytes = 0;
    cfg->stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

}  // namespace

cudaError_t launch_logits_bwd(const uint16_t *logits, const int64_t *targets, const int32_t *cu,
                              int num_seqs, int64_t T, int64_t V, const float *lse,
                              const float *grad, float *dlogits, const DeviceInfo &di,
                              cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((T + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock);
    // VEC: 16-byte loads and 32-byte stores (rows of V % 8 == 0 elements keep
    // both aligned)
    const bool vec = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0) &&
                     ((reinterpret_cast<uintptr_t>(dlogits) & 31u) == 0);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    dependent_launch_config(&cfg, attr, grid, st);
    if (vec)
        return cudaLaunchKernelEx(&cfg, logits_bwd_kernel<true>, logits, targets, cu, num_seqs, T,
                                  V, lse, grad, dlogits, di.err);
    return cudaLaunchKernelEx(&cfg, logits_bwd_kernel<false>, logits, targets, cu, num_seqs, T, V,
                              lse, grad, dlogits, di.err);
}

cudaError_t launch_logits_logp(const uint16_t *logits, const int64_t *targets, const int32_t *cu,
                               int num_seqs, int64_t T, int64_t V, float *logp, float *lse,
                               const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((T + kRowsPerBlock - 1) / kRowsPerBlock);
    const bool vec = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    dependent_launch_config(&cfg, attr, grid, st);
    if (vec)
        return cudaLaunchKernelEx(&cfg, logits_logp_kernel<true>, logits, targets, cu, num_seqs, T,
                                  V, logp, lse, di.err);
    return cudaLaunchKernelEx(&cfg, logits_logp_kernel<false>, logits, targets, cu, num_seqs, T, V,
                              logp, lse, di.err);
}

}  // namespace rk
