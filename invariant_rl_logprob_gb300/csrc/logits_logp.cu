// logits_logp.cu -- the logits path: selected-token logprob from materialised
// bf16 logits ("logp / batch_invariant_logp", RL-Kernel issue #101, maintainer
// comment, P0 operator list; chain index 8 of PR #264 "docs(ws1):
// batch-invariance contract RFC").
//
//   lse[t]  = log sum_v exp(logits[t, v])
//   logp[t] = logits[t, targets[t]] - lse[t]
//
// HBM-bound: every logit is read once (T*V*2 bytes), nothing else is large.
//
// Batch invariance by construction.  A row is reduced by one CTA; the columns
// are cut into groups of 8 (group g = columns [8g, 8g+8)); thread i of the
// CTA folds groups i, i+NT, i+2NT, ... in ascending order into a running
// (max, sum-exp); the NT partials are merged by a fixed xor-shuffle tree and
// a fixed cross-warp tree.  That order depends only on V -- never on T, the
// row's index, the grid size or the row's address alignment: rows whose
// address allows 16-byte loads use them, others load 2-byte elements, and both
// evaluate exactly the same sequence of floating-point operations.
#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

constexpr int kThreads = 256;           // threads per row (fixed for every T)
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;              // groups in flight per thread
constexpr int kBlocksPerSm = 4;

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Folds one group of 8 values (invalid columns hold -inf) into (m, s).
__device__ __forceinline__ void fold_group(const float (&x)[8], float &m, float &s) {
    float gm = x[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) gm = fmaxf(gm, x[j]);
    if (gm > m) {
        // ex2((m - gm) * log2e) == 1 exactly when gm == m, so skipping the
        // rescale when the maximum does not grow changes no bit.
        s = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(m, gm), kLog2e)));
        m = gm;
    }
    const float mb = __fmul_rn(-m, kLog2e);
    float e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = ex2(__fmaf_rn(x[j], kLog2e, mb));
    const float local = __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3])),
                                  __fadd_rn(__fadd_rn(e[4], e[5]), __fadd_rn(e[6], e[7])));
    s = __fadd_rn(s, local);
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&x)[8]) {
    x[0] = bf16_lo(v.x);
    x[1] = bf16_hi(v.x);
    x[2] = bf16_lo(v.y);
    x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z);
    x[5] = bf16_hi(v.z);
    x[6] = bf16_lo(v.w);
    x[7] = bf16_hi(v.w);
}

// VEC: 16-byte loads (V % 8 == 0 and a 16-byte aligned base); otherwise
// 2-byte loads of the same groups.
template <bool VEC>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
    logits_logp_kernel(const uint16_t *__restrict__ logits, const int64_t *__restrict__ targets,
                       const int32_t *__restrict__ cu, int num_seqs, int64_t T, int64_t V,
                       float *__restrict__ logp, float *__restrict__ lse, unsigned *err) {
    __shared__ float sm_m[kWarps];
    __shared__ float sm_s[kWarps];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t G = (V + 7) >> 3;

    for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
        const int64_t tgt = targets[row];
        const bool active = row_active(row, tgt, cu, num_seqs);
        if (!active) {  // uniform across the block
            if (tid == 0) {
                logp[row] = 0.f;
                if (lse) lse[row] = 0.f;
            }
            continue;
        }
        const uint16_t *zrow = logits + row * V;
        const bool tgt_ok = tgt < V;
        float zt = 0.f;
        if (tid == 0 && tgt_ok) zt = bf16_bits_to_f32(zrow[tgt]);

        float m = -INFINITY, s = 0.f;
        if (VEC) {
            const uint4 *rv = reinterpret_cast<const uint4 *>(zrow);
            for (int64_t g0 = tid; g0 < G; g0 += (int64_t)kThreads * kUnroll) {
                uint4 v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t g = g0 + (int64_t)u * kThreads;
                    if (g < G) v[u] = ld_stream_v4(rv + g);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t g = g0 + (int64_t)u * kThreads;
                    if (g < G) {
                        float x[8];
                        unpack8(v[u], x);
                        fold_group(x, m, s);
                    }
                }
            }
        } else {
            for (int64_t g = tid; g < G; g += kThreads) {
                float x[8];
                const int64_t c0 = g << 3;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t c = c0 + j;
                    x[j] = (c < V) ? bf16_bits_to_f32(__ldg(zrow + c)) : -INFINITY;
                }
                fold_group(x, m, s);
            }
        }

#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, off);
            const float so = __shfl_xor_sync(0xffffffffu, s, off);
            lse_merge(m, s, mo, so);
        }
        if (lane == 0) {
            sm_m[warp] = m;
            sm_s[warp] = s;
        }
        __syncthreads();
        if (warp == 0) {
            m = (lane < kWarps) ? sm_m[lane] : -INFINITY;
            s = (lane < kWarps) ? sm_s[lane] : 0.f;
#pragma unroll
            for (int off = kWarps / 2; off > 0; off >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, m, off);
                const float so = __shfl_xor_sync(0xffffffffu, s, off);
                lse_merge(m, s, mo, so);
            }
            if (lane == 0) {
                if (tgt_ok) {
                    const float l = __fadd_rn(m, logf(s));
                    logp[row] = __fsub_rn(zt, l);
                    if (lse) lse[row] = l;
                } else {
                    logp[row] = __int_as_float(0x7fc00000);
                    if (lse) lse[row] = __int_as_float(0x7fc00000);
                    atomicOr(err, kErrTargetRange);
                }
            }
        }
        __syncthreads();  // sm_m / sm_s are reused by the next row
    }
}

}  // namespace

cudaError_t launch_logits_logp(const uint16_t *logits, const int64_t *targets, const int32_t *cu,
                               int num_seqs, int64_t T, int64_t V, float *logp, float *lse,
                               const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int64_t max_grid = (int64_t)di.sm_count * kBlocksPerSm;
    const unsigned grid = (unsigned)(T < max_grid ? T : max_grid);
    const bool vec = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
    if (vec)
        logits_logp_kernel<true><<<grid, kThreads, 0, st>>>(logits, targets, cu, num_seqs, T, V,
                                                            logp, lse, di.err);
    else
        logits_logp_kernel<false><<<grid, kThreads, 0, st>>>(logits, targets, cu, num_seqs, T, V,
                                                             logp, lse, di.err);
    return cudaGetLastError();
}

}  // namespace rk
