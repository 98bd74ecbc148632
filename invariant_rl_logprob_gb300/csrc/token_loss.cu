// token_loss.cu -- per-token GRPO loss on selected logprobs ("grpo_loss,
// ratio_kl", RL-Kernel issue #101, maintainer comment, P0 operator list;
// chain index 9 of PR #264 "docs(ws1): batch-invariance contract RFC", the
// end of the chain where drift is amplified into the policy ratio).
//
// Per active token t (no batch-level normalisation, so every output depends
// only on that token's inputs and the caller's scalars):
//   ratio = exp(logp - logp_old)
//   surr  = min(ratio * A, clip(ratio, 1 - eps_low, 1 + eps_high) * A)
//   kl    = exp(logp_ref - logp) - (logp_ref - logp) - 1      (0 without logp_ref)
//   loss  = scale * (-surr + beta * kl)
//   grad  = d loss / d logp  (the g that feeds the linear_logp backward)
// Inactive tokens get 0.  HBM-bound: about 28 bytes per token.
#include "rk_device.cuh"
#include "rk_internal.h"

namespace rk {
namespace {

__global__ void __launch_bounds__(256)
    grpo_token_kernel(const float *__restrict__ logp, const float *__restrict__ logp_old,
                      const float *__restrict__ logp_ref, const float *__restrict__ adv,
                      const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                      int num_seqs, int64_t T, float eps_low, float eps_high, float beta,
                      float scale, float *__restrict__ loss, float *__restrict__ grad,
                      float *__restrict__ ratio_out, float *__restrict__ kl_out) {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        if (!row_active(t, targets[t], cu, num_seqs)) {
            loss[t] = 0.f;
            grad[t] = 0.f;
            if (ratio_out) ratio_out[t] = 0.f;
            if (kl_out) kl_out[t] = 0.f;
            continue;
        }
        const float lp = logp[t];
        const float a = adv[t];
        const float ratio = ex2(__fmul_rn(__fsub_rn(lp, logp_old[t]), kLog2e));
        const float lo = 1.f - eps_low, hi = 1.f + eps_high;
        const float clipped = fminf(fmaxf(ratio, lo), hi);
        const float s1 = __fmul_rn(ratio, a), s2 = __fmul_rn(clipped, a);
        float surr, dsurr;
        if (s1 <= s2) {
            surr = s1;
            dsurr = s1;
        } else {
            surr = s2;
            dsurr = (ratio > lo && ratio < hi) ? s1 : 0.f;
        }
        float kl = 0.f, dkl = 0.f;
        if (logp_ref) {
            const float d = __fsub_rn(logp_ref[t], lp);
            const float e = ex2(__fmul_rn(d, kLog2e));
            kl = __fsub_rn(__fsub_rn(e, d), 1.f);
            dkl = __fsub_rn(1.f, e);
        }
        loss[t] = __fmul_rn(scale, __fmaf_rn(beta, kl, -surr));
        grad[t] = __fmul_rn(scale, __fmaf_rn(beta, dkl, -dsurr));
        if (ratio_out) ratio_out[t] = ratio;
        if (kl_out) kl_out[t] = kl;
    }
}

}  // namespace

cudaError_t launch_grpo_token(const float *logp, const float *logp_old, const float *logp_ref,
                              const float *adv, const int64_t *targets, const int32_t *cu,
                              int num_seqs, int64_t T, float eps_low, float eps_high, float beta,
                              float scale, float *loss, float *grad, float *ratio, float *kl,
                              const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    int64_t blocks = (T + 255) / 256;
    const int64_t cap = (int64_t)di.sm_count * 8;
    if (blocks > cap) blocks = cap;
    grpo_token_kernel<<<(unsigned)blocks, 256, 0, st>>>(logp, logp_old, logp_ref, adv, targets, cu,
                                                        num_seqs, T, eps_low, eps_high, beta,
                                                        scale, loss, grad, ratio, kl);
    return cudaGetLastError();
}

}  // namespace rk
