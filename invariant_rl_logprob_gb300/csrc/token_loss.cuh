// token_loss.cuh -- the per-token GRPO loss of one token, shared by the
// standalone kernel (token_loss.cu) and the forward merge that can apply it
// to the logprob it has just produced (linear_logp_tc.cu): the same
// arithmetic in both places, so both give the same bits.
//
// Per active token t ("grpo_loss, ratio_kl", RL-Kernel issue #101,
// maintainer comment, P0 operator list; chain index 9 of PR #264
// "docs(ws1): batch-invariance contract RFC"):
//   ratio = exp(logp - logp_old)
//   surr  = min(ratio * A, clip(ratio, 1 - eps_low, 1 + eps_high) * A)
//   kl    = exp(logp_ref - logp) - (logp_ref - logp) - 1      (0 without logp_ref)
//   loss  = scale * (-surr + beta * kl)
//   grad  = d loss / d logp  (the g that feeds the linear_logp backward)
// At the clip kinks the gradient is the one-sided value of the term min picks.
#pragma once

#include "rk_device.cuh"

namespace rk {

struct GrpoArgs {
    const float *logp_old;
    const float *logp_ref;  // or null: no KL term
    const float *adv;
    float eps_low, eps_high, beta, scale;
    float *loss;
    float *grad;
    float *ratio;  // or null
    float *kl;     // or null
};

__device__ __forceinline__ void grpo_token_inactive(const GrpoArgs &p, int64_t t) {
    p.loss[t] = 0.f;
    p.grad[t] = 0.f;
    if (p.ratio) p.ratio[t] = 0.f;
    if (p.kl) p.kl[t] = 0.f;
}

__device__ __forceinline__ void grpo_token(const GrpoArgs &p, int64_t t, float lp) {
    const float a = p.adv[t];
    const float ratio = ex2(__fmul_rn(__fsub_rn(lp, p.logp_old[t]), kLog2e));
    const float lo = 1.f - p.eps_low, hi = 1.f + p.eps_high;
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
    if (p.logp_ref) {
        const float d = __fsub_rn(p.logp_ref[t], lp);
        const float e = ex2(__fmul_rn(d, kLog2e));
        kl = __fsub_rn(__fsub_rn(e, d), 1.f);
        dkl = __fsub_rn(1.f, e);
    }
    p.loss[t] = __fmul_rn(p.scale, __fmaf_rn(p.beta, kl, -surr));
    p.grad[t] = __fmul_rn(p.scale, __fmaf_rn(p.beta, dkl, -dsurr));
    if (p.ratio) p.ratio[t] = ratio;
    if (p.kl) p.kl[t] = kl;
}

}  // namespace rk
