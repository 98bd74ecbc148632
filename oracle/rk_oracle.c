/*
 * rk_oracle.c -- plain fp64 CPU oracle for the selected-token logprob path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; it exists so that tests, the smoke check and the CPU
 * baseline of the benchmark can compare the CUDA kernels against a slow,
 * obviously correct definition.  It shares no code, header or constant with
 * the CUDA library.
 *
 * What is computed (the plain definition; the method reaches it up to
 * rounding order, so the oracle is that definition written out):
 *
 *   linear_logp  -- the "linear_logp" operator of the P0 suite
 *                   (RL-Kernel issue #101 "[RFC] Batch-Invariant RL Kernel
 *                   Suite for Train-Inference Consistency", maintainer comment,
 *                   P0 operator list; chain index 7 in PR #264 "docs(ws1):
 *                   batch-invariance contract RFC", First-Divergence
 *                   Localization chain listing):
 *                      z[v]  = sum_k h[k] * W[v,k]        (z = h . W^T)
 *                      lse   = log sum_v exp(z[v])
 *                      logp  = z[target] - lse
 *   logits path  -- "logp / batch_invariant_logp" (same P0 list; chain
 *                   index 8): the same with z given directly.
 *   backward     -- the gradient of logp with respect to h, made a
 *                   first-class property in issue #244 "[WS1 Test] ...",
 *                   Workstream 3 (#153 Backward-pass consistency):
 *                      p[v]  = exp(z[v] - lse)
 *                      dh[k] = g * (W[target,k] - sum_v p[v] * W[v,k])
 *
 * Precision: every input element is upcast exactly to double (a bf16 value is
 * a float with the low 16 bits zero, and every float is a double), every
 * product of two bf16 values is exact in double, and all sums run
 * sequentially in ascending index order in double.  Issue #244, Workstream 1
 * (#154 dtype coverage), Scope table: the reference path is the higher
 * precision one; fp64 is used here so that the oracle's own error is far below
 * any tolerance applied to the GPU.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off (no reassociation, no
 * fused multiply-add), so the summation order written here is the one run.
 *
 * Row selection: every function takes a list of row indices and computes only
 * those rows, so that large workloads can be checked on a seeded sample.
 * Which rows are active (masking) is decided by the caller (oracle/__init__.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element kinds accepted for matrix inputs. */
enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *base, int kind, int64_t i)
{
    if (kind == ORACLE_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[i]);
    return ((const double *)base)[i];
}

/* z[v] = sum_{k=0}^{H-1} h[row,k] * W[v,k], k ascending. */
static void logits_of_row(const void *h, int h_kind, int64_t row,
                          const void *W, int w_kind, int64_t H, int64_t V,
                          double *hrow, double *z)
{
    for (int64_t k = 0; k < H; ++k)
        hrow[k] = elem(h, h_kind, row * H + k);
    for (int64_t v = 0; v < V; ++v) {
        double acc = 0.0;
        const int64_t base = v * H;
        for (int64_t k = 0; k < H; ++k)
            acc += hrow[k] * elem(W, w_kind, base + k);
        z[v] = acc;
    }
}

/* log sum_v exp(z[v]), written with the usual shift by the maximum so that
 * the exponentials cannot overflow: lse = m + log(sum_v exp(z[v] - m)). */
static double log_sum_exp(const double *z, int64_t V)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (z[v] > m)
            m = z[v];
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v)
        s += exp(z[v] - m);
    return m + log(s);
}

/*
 * linear_logp forward on the listed rows.
 *   h: [T,H] (kind h_kind), W: [V,H] row-major (kind w_kind),
 *   targets: [T] int64, each listed row must have 0 <= target < V,
 *   rows: n_rows indices into [0,T),
 *   logp, lse: [n_rows] outputs (may be NULL).
 * Returns 0, or -1 if a scratch allocation failed or a target is out of range.
 */
int oracle_linear_logp(const void *h, int h_kind, const void *W, int w_kind,
                       const int64_t *targets, const int64_t *rows,
                       int64_t n_rows, int64_t H, int64_t V,
                       double *logp, double *lse)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!hrow || !z) {
        free(hrow);
        free(z);
        return -1;
    }
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t t = targets[r];
        if (t < 0 || t >= V) {
            rc = -1;
            break;
        }
        logits_of_row(h, h_kind, r, W, w_kind, H, V, hrow, z);
        const double l = log_sum_exp(z, V);
        if (lse)
            lse[i] = l;
        if (logp)
            logp[i] = z[t] - l;
    }
    free(hrow);
    free(z);
    return rc;
}

/*
 * Logits path on the listed rows: z = logits[r, :] (row stride V).
 * Same output and error conventions as oracle_linear_logp.
 */
int oracle_logp_from_logits(const void *logits, int kind,
                            const int64_t *targets, const int64_t *rows,
                            int64_t n_rows, int64_t V,
                            double *logp, double *lse)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!z)
        return -1;
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t t = targets[r];
        if (t < 0 || t >= V) {
            rc = -1;
            break;
        }
        for (int64_t v = 0; v < V; ++v)
            z[v] = elem(logits, kind, r * V + v);
        const double l = log_sum_exp(z, V);
        if (lse)
            lse[i] = l;
        if (logp)
            logp[i] = z[t] - l;
    }
    free(z);
    return rc;
}

/*
 * linear_logp backward on the listed rows:
 *   dh[i,k] = g[r] * (W[target_r,k] - sum_v p[v] * W[v,k]),
 *   p[v] = exp(z[v] - lse), z and lse recomputed here from h and W.
 *   grad_logp: [T] doubles (the upstream gradient g of each row's logp),
 *   dh: [n_rows, H] output.
 * The sum over v runs in ascending v for every k.
 */
int oracle_linear_logp_bwd(const void *h, int h_kind, const void *W, int w_kind,
                           const int64_t *targets, const double *grad_logp,
                           const int64_t *rows, int64_t n_rows,
                           int64_t H, int64_t V, double *dh)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!hrow || !acc || !z) {
        free(hrow);
        free(acc);
        free(z);
        return -1;
    }
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t t = targets[r];
        if (t < 0 || t >= V) {
            rc = -1;
            break;
        }
        logits_of_row(h, h_kind, r, W, w_kind, H, V, hrow, z);
        const double l = log_sum_exp(z, V);
        for (int64_t k = 0; k < H; ++k)
            acc[k] = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            const double p = exp(z[v] - l);
            const int64_t base = v * H;
            for (int64_t k = 0; k < H; ++k)
                acc[k] += p * elem(W, w_kind, base + k);
        }
        const double g = grad_logp[r];
        for (int64_t k = 0; k < H; ++k)
            dh[i * H + k] = g * (elem(W, w_kind, t * H + k) - acc[k]);
    }
    free(hrow);
    free(acc);
    free(z);
    return rc;
}

/*
 * lm_head on the listed rows: z[i, v] = sum_k h[r,k] W[v,k] in fp64 (the
 * dense path's logits before any rounding; chain index 6 "lm_head" of PR #264
 * "docs(ws1): batch-invariance contract RFC").  z: [n_rows, V].
 */
int oracle_lm_head(const void *h, int h_kind, const void *W, int w_kind,
                   const int64_t *rows, int64_t n_rows, int64_t H, int64_t V, double *z)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!hrow)
        return -1;
    for (int64_t i = 0; i < n_rows; ++i)
        logits_of_row(h, h_kind, rows[i], W, w_kind, H, V, hrow, z + i * V);
    free(hrow);
    return 0;
}

/*
 * Logits-path backward on the listed rows: the gradient of g * logp with
 * respect to the logits, dz[i, v] = g[r] * (onehot(target_r)[v] - p[v]),
 * p = softmax(logits[r, :]) (the "dense vs indexed selected-logprob paths" of
 * issue #101 "[RFC] Batch-Invariant RL Kernel Suite ...", Scope, with the
 * backward made first-class in issue #244, Workstream 3).  dz: [n_rows, V].
 */
int oracle_logits_bwd(const void *logits, int kind, const int64_t *targets,
                      const double *grad_logp, const int64_t *rows, int64_t n_rows,
                      int64_t V, double *dz)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!z)
        return -1;
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t t = targets[r];
        if (t < 0 || t >= V) {
            rc = -1;
            break;
        }
        for (int64_t v = 0; v < V; ++v)
            z[v] = elem(logits, kind, r * V + v);
        const double l = log_sum_exp(z, V);
        const double g = grad_logp[r];
        for (int64_t v = 0; v < V; ++v)
            dz[i * V + v] = g * ((v == t ? 1.0 : 0.0) - exp(z[v] - l));
    }
    free(z);
    return rc;
}

/*
 * Per-token GRPO loss ("grpo_loss, ratio_kl", issue #101 P0 list; chain index
 * 9 of PR #264).  The pages name the operator, not its formula; this is the
 * clipped-surrogate objective with a KL penalty to a reference policy, per
 * token (no batch-level normalisation; a caller-given scale multiplies it):
 *   ratio = exp(logp - logp_old)
 *   surr  = min(ratio * A, clip(ratio, 1 - eps_low, 1 + eps_high) * A)
 *   kl    = exp(logp_ref - logp) - (logp_ref - logp) - 1     (0 without logp_ref)
 *   loss  = scale * (-surr + beta * kl)
 *   grad  = d loss / d logp
 *         = scale * (-A * ratio * [unclipped term selected or ratio inside the
 *                                  clip range] + beta * (1 - exp(logp_ref - logp)))
 * where the unclipped term is selected when ratio * A <= clip(ratio) * A.
 * All n elements (the caller passes only active tokens).
 */
void oracle_grpo_token(const double *logp, const double *logp_old, const double *logp_ref,
                       const double *adv, int64_t n, double eps_low, double eps_high,
                       double beta, double scale, double *loss, double *grad,
                       double *ratio_out, double *kl_out)
{
    for (int64_t i = 0; i < n; ++i) {
        const double ratio = exp(logp[i] - logp_old[i]);
        const double a = adv[i];
        const double lo = 1.0 - eps_low, hi = 1.0 + eps_high;
        const double clipped = ratio < lo ? lo : (ratio > hi ? hi : ratio);
        const double s1 = ratio * a, s2 = clipped * a;
        const double surr = s1 <= s2 ? s1 : s2;
        /* d surr / d logp: ratio * a through the unclipped term; through the
         * clipped term only while ratio is inside [lo, hi] (there it equals s1) */
        double dsurr;
        if (s1 <= s2)
            dsurr = ratio * a;
        else
            dsurr = (ratio > lo && ratio < hi) ? ratio * a : 0.0;
        double kl = 0.0, dkl = 0.0;
        if (logp_ref) {
            const double d = logp_ref[i] - logp[i];
            const double e = exp(d);
            kl = e - d - 1.0;
            dkl = 1.0 - e;
        }
        loss[i] = scale * (-surr + beta * kl);
        grad[i] = scale * (-dsurr + beta * dkl);
        if (ratio_out)
            ratio_out[i] = ratio;
        if (kl_out)
            kl_out[i] = kl;
    }
}

/*
 * Greedy decoding step on the listed rows: the token with the largest logit
 * z = h . W^T (the lowest index among equal maxima) and its logprob
 * z[token] - logsumexp(z).  This is the decode side of issue #244, Workstream 2
 * (#152 "Generate-then-re-score"): a later prefill scoring of the same tokens
 * must give the same selected logprobs.
 */
int oracle_linear_greedy(const void *h, int h_kind, const void *W, int w_kind,
                         const int64_t *rows, int64_t n_rows, int64_t H, int64_t V,
                         int64_t *token, double *logp, double *zmax)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!hrow || !z) {
        free(hrow);
        free(z);
        return -1;
    }
    for (int64_t i = 0; i < n_rows; ++i) {
        logits_of_row(h, h_kind, rows[i], W, w_kind, H, V, hrow, z);
        int64_t best = 0;
        for (int64_t v = 1; v < V; ++v)
            if (z[v] > z[best])
                best = v;
        const double l = log_sum_exp(z, V);
        token[i] = best;
        logp[i] = z[best] - l;
        if (zmax)
            zmax[i] = z[best];
    }
    free(hrow);
    free(z);
    return 0;
}

/*
 * linear_logp backward with respect to W over the listed rows (dW, a
 * parameter gradient: a sum over tokens, issue #244 "[WS1 Test] ...",
 * Workstream 3 #153 -- "GEMM dW", fixed batch-shape-independent order, and
 * "compare parameter gradients over the same complete logical sample set"):
 *   dW[v, k] = sum_i g[r_i] * (onehot(target_{r_i})[v] - p_{r_i}[v]) * h[r_i, k]
 * with p = softmax(h . W^T) recomputed here; rows are summed in the listed
 * order.  dW: [V, H] (overwritten).
 */
int oracle_linear_logp_dw(const void *h, int h_kind, const void *W, int w_kind,
                          const int64_t *targets, const double *grad_logp,
                          const int64_t *rows, int64_t n_rows, int64_t H, int64_t V, double *dW)
{
    double *hrow = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!hrow || !z) {
        free(hrow);
        free(z);
        return -1;
    }
    for (int64_t i = 0; i < V * H; ++i)
        dW[i] = 0.0;
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int64_t t = targets[r];
        if (t < 0 || t >= V) {
            rc = -1;
            break;
        }
        logits_of_row(h, h_kind, r, W, w_kind, H, V, hrow, z);
        const double l = log_sum_exp(z, V);
        const double g = grad_logp[r];
        for (int64_t v = 0; v < V; ++v) {
            const double c = g * ((v == t ? 1.0 : 0.0) - exp(z[v] - l));
            double *out = dW + v * H;
            for (int64_t k = 0; k < H; ++k)
                out[k] += c * hrow[k];
        }
    }
    free(hrow);
    free(z);
    return rc;
}
