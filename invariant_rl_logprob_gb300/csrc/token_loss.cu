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
// (arithmetic in token_loss.cuh).  Inactive tokens get 0.  HBM-bound: about
// 28 bytes per token.
#include "rk_internal.h"
#include "token_loss.cuh"

namespace rk {
namespace {

__global__ void __launch_bounds__(256)
    grpo_token_kernel(const float *__restrict__ logp, const int64_t *__restrict__ targets,
                      const int32_t *__restrict__ cu, int num_seqs, int64_t T, GrpoArgs p) {
    // Launched with programmatic stream serialisation: the blocks may become
    // resident while the previous kernel in the stream finishes, and wait here
    // until it has completed and its writes (e.g. logp) are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        if (!row_active(t, targets[t], cu, num_seqs))
            grpo_token_inactive(p, t);
        else
            grpo_token(p, t, logp[t]);
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
    const GrpoArgs p{logp_old, logp_ref, adv, eps_low, eps_high, beta, scale, loss, grad, ratio, kl};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grpo_token_kernel, logp, targets, cu, num_seqs, T, p);
}

}  // namespace rk
