/*
 * rk.h -- C ABI of the batch-invariant selected-token logprob library (librk).
 *
 * The operators are the selected-logprob members of the P0 kernel suite named
 * in RL-Kernel issue #101 "[RFC] Batch-Invariant RL Kernel Suite for
 * Train-Inference Consistency" (maintainer comment, P0 operator list:
 * "lm_head, linear_logp, logp/batch_invariant_logp") and ordered in the
 * forward chain of PR #264 "docs(ws1): batch-invariance contract RFC"
 * (First-Divergence Localization: 6 lm_head, 7 linear_logp, 8 logp).
 *
 * Contract every entry point keeps (issue #101, maintainer comment, relation
 * table; PR #264, relation I): for a given logical token row, the outputs are
 * bitwise identical whatever the batch around it -- batch size (T1), the row's
 * position (T2), the content of other rows (T3), padding (T4) and varlen
 * packing or selection (T6).  The kernels use one tile shape and one
 * reduction order per (H, V) for every T, and no atomics in any result.
 *
 * Conventions shared by all entry points
 *  - All tensor pointers are DEVICE pointers, owned by the caller, contiguous
 *    row-major.  The library never allocates device memory; scratch space is
 *    passed in as `workspace`.  Outputs must not alias inputs or each other.
 *  - Workspace contents on entry are ignored.  Besides intermediates, every
 *    workspace holds the counter from which the tile kernel's CTA pairs take
 *    their tiles (the call zeroes it), so calls that may run at the same time
 *    (other streams, other host threads) need separate workspaces.
 *  - bf16 tensors are passed as `const uint16_t*` (IEEE bfloat16 bit patterns).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous and stream-ordered; none synchronises the host.
 *  - Active rows.  Row t is active iff targets[t] >= 0 and, when cu_seqlens is
 *    not NULL, cu_seqlens[0] <= t < cu_seqlens[num_seqs].  Inactive rows get
 *    logp = lse = 0 and dh = 0, and their inputs (even NaN) never reach an
 *    active row.  (Issue #244 "[WS1 Test] #154 dtype pin + #152 KV path + #153
 *    bwd invariance + #150 chain gate", Workstream 3, Logical-workload
 *    identity: padding is excluded from outputs and gradients.)
 *    cu_seqlens (int32, num_seqs + 1 ascending offsets) only bounds the active
 *    range; the operators are per token.
 *  - A target >= V on an active row is an input error found on the device:
 *    that row's outputs become NaN and the device error word gets
 *    RK_DEVERR_TARGET_RANGE (read it with rk_get_device_error).  Nothing traps.
 *  - Precision (issue #244, Workstream 1 #154, Scope table: bf16 inputs,
 *    fp32 accumulation): bf16 inputs, fp32 tensor-core accumulation, fp32
 *    outputs.  Results match the fp64 definition within
 *    |d logp| <= 1e-3 + 1e-3 |logp| and |d dh| <= 1e-3 + 1e-3 max|dh|.
 *  - Argument errors return a status before anything is launched.  Launch
 *    failures return RK_ERR_CUDA (the CUDA error is left for
 *    cudaGetLastError / rk_last_cuda_error).
 *  - Thread safety: entry points may be called from several host threads.
 *    Shared state: the CUDA driver's tensor-map encoder, looked up once; per
 *    device, the SM count and the device addresses of the library's static
 *    device variables (the error word, rk_linear_logp_noalloc's array), looked
 *    up on the first call on that device; the rk_set_row_blocks setting.
 *  - Contexts: those cached addresses belong to the device's primary context
 *    (the one the CUDA runtime uses).  After cudaDeviceReset, or with another
 *    context current, they no longer point at this library's variables:
 *    reload the library (a new process) before calling it again.
 */
#ifndef RK_H
#define RK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RK_OK = 0,
    RK_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad cu_seqlens count, ... */
    RK_ERR_UNSUPPORTED = 2,  /* shape outside the supported set (e.g. H % 64 != 0) */
    RK_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than the *_workspace_size query */
    RK_ERR_CUDA = 4          /* a CUDA runtime call or launch failed */
} rk_status;

/* Device error word bits (rk_get_device_error). */
#define RK_DEVERR_TARGET_RANGE 0x1  /* an active row had target >= V */
#define RK_DEVERR_TIMEOUT 0x2       /* a pipeline wait gave up after its time limit */
#define RK_DEVERR_LSE 0x4           /* a backward row had more than 64 columns with
                                       p >= 1/64: the lse passed in does not belong
                                       to these inputs (results unspecified) */

/*
 * Bytes of workspace rk_linear_logp needs for T rows (>= 0).  The layout is
 * private: per-row, per-vocab-tile (max, sum-exp) partials, the target logit
 * of every row, a flag per block of 256 rows telling whether it holds an
 * active row (blocks without one get no tensor work: padding is free), and
 * the counter from which the tile kernel's CTA pairs take their tiles.
 * Returns 0 if T == 0.  Calls running at the same time need separate
 * workspaces.
 */
size_t rk_linear_logp_workspace_size(int64_t T, int64_t H, int64_t V);

/*
 * linear_logp forward: for every active row t,
 *     z[t, v]  = sum_k h[t, k] * W[v, k]            (z = h . W^T, fp32 accumulation)
 *     lse[t]   = log sum_v exp(z[t, v])
 *     logp[t]  = z[t, targets[t]] - lse[t]
 * without writing z to memory (issue #101, maintainer comment, P0 list
 * "linear_logp"; PR #264 chain index 7).
 *
 *   h         bf16 [T, H]   hidden states, row-major, 16-byte aligned
 *   W         bf16 [V, H]   lm_head weight (row v is the weight of token v), 16-byte aligned
 *   targets   int64 [T]     selected token of each row (< 0: row inactive)
 *   cu_seqlens int32 [num_seqs + 1] or NULL
 *   logp      fp32 [T]      output
 *   lse       fp32 [T]      output (log-sum-exp of each row), or NULL
 *   workspace device scratch of >= rk_linear_logp_workspace_size(T, H, V) bytes,
 *             256-byte aligned; contents on entry are ignored.
 * Supported: H % 64 == 0, H <= 65536; 1 <= V < 2^31; 0 <= T < 2^31 (T == 0 is a no-op).
 */
rk_status rk_linear_logp(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                         const int32_t *cu_seqlens, int32_t num_seqs,
                         int64_t T, int64_t H, int64_t V,
                         float *logp, float *lse,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Logits path ("logp / batch_invariant_logp", issue #101 P0 list; PR #264 chain
 * index 8): from materialised logits,
 *     lse[t]  = log sum_v exp(logits[t, v]),   logp[t] = logits[t, targets[t]] - lse[t].
 *
 *   logits    bf16 [T, V], row stride V elements; any 2-byte alignment (the
 *             reduction order depends on column indices only, never on the
 *             address, so a row's result does not depend on where it sits)
 *   targets, cu_seqlens, num_seqs, logp, lse: as for rk_linear_logp (lse may be NULL)
 * Supported: 1 <= V < 2^31, 0 <= T.  Needs no workspace.
 */
rk_status rk_logp_from_logits(const uint16_t *logits, const int64_t *targets,
                              const int32_t *cu_seqlens, int32_t num_seqs,
                              int64_t T, int64_t V, float *logp, float *lse, void *stream);

/*
 * Bytes of workspace rk_linear_logp_bwd needs to process all T rows in one
 * pass (one bf16 [T, V] buffer of g * softmax probabilities, rounded up, the
 * rows' fp32 entry lists, a flag per 256-row block and 256 bytes for the
 * tile and round counters).
 * A smaller workspace (but at least rk_linear_logp_bwd_min_workspace_size)
 * makes the call process the rows in chunks; the results do not change.
 */
size_t rk_linear_logp_bwd_workspace_size(int64_t T, int64_t H, int64_t V);
size_t rk_linear_logp_bwd_min_workspace_size(int64_t H, int64_t V);

/*
 * linear_logp backward with respect to h (issue #244, Workstream 3 #153:
 * fixed, batch-shape-independent reduction order, no atomicAdd):
 *     p[t, v]  = exp(z[t, v] - lse[t])
 *     dh[t, :] = g[t] * (W[targets[t], :] - sum_v p[t, v] * W[v, :])
 * for every active row (dh = 0 on inactive rows).
 *
 *   h, W, targets, cu_seqlens, num_seqs: as for rk_linear_logp
 *   lse        fp32 [T]  the lse output of rk_linear_logp on the same inputs
 *   grad_logp  fp32 [T]  upstream gradient g of each row's logp
 *   dh         fp32 [T, H] output
 *   workspace  >= rk_linear_logp_bwd_min_workspace_size(H, V) bytes, 256-byte aligned
 * The sum over v runs in one fixed ascending order for every row (no split of
 * V across blocks, no atomic additions of values).  Per row, the target
 * column and every column with p >= 1/64 (at most 65 columns) are handled in
 * fp32: w = g (onehot - p), summed over those columns in ascending column
 * order.  All other probabilities enter a tensor-core sum rounded to bf16,
 * where each carries at most 1/64 of the row's mass.  So a peaked softmax (a
 * confident policy, p_target near 1) does not turn dh = g (1 - p_t) (...)
 * into a small difference of large bf16-rounded terms.  An lse that does not
 * belong to the inputs can make more than 64 columns qualify: the extra ones
 * are dropped and RK_DEVERR_LSE is set.
 */
rk_status rk_linear_logp_bwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                             const int32_t *cu_seqlens, int32_t num_seqs,
                             int64_t T, int64_t H, int64_t V,
                             const float *lse, const float *grad_logp, float *dh,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * The same forward and backward with the softmax terms kept between them, so
 * that the backward need not recompute z = h W^T with a second GEMM (HBM is
 * large enough to hold them: 16.8 GB for T = 65536, V = 128256).
 *
 * rk_linear_logp_fwd_saved is rk_linear_logp that also writes, into `saved`,
 * every row's per-tile softmax terms e[t, v] = exp(z[t, v] - m), in bf16, with
 * m the row's maximum over the 256-column vocabulary tile holding v, next to
 * the tiles' (max, sum) partials.  Its logp and lse are bitwise those of
 * rk_linear_logp.
 *
 * rk_linear_logp_bwd_saved computes dh as rk_linear_logp_bwd defines it
 * (issue #244, Workstream 3 #153: fixed, batch-shape-independent order, no
 * atomicAdd), from `saved` instead of a z recompute:
 *   p[t, v]  = exp(m - lse[t]) * e[t, v],   dZ = g p rounded to bf16,
 *   dh[t, :] = sum over the row's fp32 entries of w W[v, :] - dZ[t, :] W
 * where the entries are the target column and the columns with p >= 1/64,
 * whose w = g (onehot - p) uses an exact fp32 z = h[t] . W[v] (one fixed
 * order).  dZ carries two bf16 roundings (of e, then of g p) where the
 * recompute path carries one; the fp32 entries keep peaked softmaxes exact.
 * The bits differ from rk_linear_logp_bwd's; they are again a function of
 * the row alone (bitwise batch-invariant) and within the same tolerance.
 * The call turns the terms in `saved` into dZ in place, so a saved state
 * serves one backward.
 *
 *   saved      >= rk_linear_logp_saved_size(T, H, V) bytes, 256-byte aligned
 *              (caller-owned; written by the forward, consumed by the backward)
 *   workspace  >= rk_linear_logp_bwd_saved_workspace_size(T, H, V) bytes
 *              (tile counter, the rows' entry counts and lists), 16-byte aligned
 *   h, W, targets, cu_seqlens, lse, grad_logp, dh: as for rk_linear_logp_bwd
 *              (same h, W, targets, cu_seqlens as the forward that filled `saved`)
 * Supported: as rk_linear_logp, and V < 65535 * 8192.
 */
size_t rk_linear_logp_saved_size(int64_t T, int64_t H, int64_t V);
rk_status rk_linear_logp_fwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t T, int64_t H, int64_t V, float *logp, float *lse,
                                   void *saved, size_t saved_bytes, void *stream);
size_t rk_linear_logp_bwd_saved_workspace_size(int64_t T, int64_t H, int64_t V);
rk_status rk_linear_logp_bwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t T, int64_t H, int64_t V,
                                   const float *lse, const float *grad_logp,
                                   void *saved, size_t saved_bytes, float *dh,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * The dense path's lm_head (chain index 6 of PR #264; "dense vs indexed
 * selected-logprob paths", issue #101, Scope): logits[t, v] = bf16(sum_k
 * h[t, k] * W[v, k]) with fp32 accumulation and one rounding to bf16, using the
 * same tensor-core tiles as rk_linear_logp (one fixed tile shape and K order
 * for every T, so a row's logits do not depend on the batch).
 *   h bf16 [T, H], W bf16 [V, H] (16-byte aligned), logits bf16 [T, ld_logits]
 *   (16-byte aligned, ld_logits >= V and a multiple of 8; columns >= V untouched).
 *   workspace  NULL, or >= rk_lm_head_workspace_size() bytes (16-byte aligned):
 *              with it, the tile kernel's CTA pairs take their tiles from a
 *              counter there, in the order they become free, which keeps the
 *              pairs in step and L2 reuse high; without it each pair works
 *              through a fixed list of tiles.  The logits are the same bits
 *              either way.  Contents on entry are ignored.
 * Supported: as rk_linear_logp.  Every row is computed (no mask).
 */
size_t rk_lm_head_workspace_size(void);
rk_status rk_lm_head(const uint16_t *h, const uint16_t *W, int64_t T, int64_t H, int64_t V,
                     uint16_t *logits, int64_t ld_logits, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * Logits-path backward (the gradient of the dense path, issue #244 Workstream
 * 3: backward as a first-class property): for every active row,
 *     dlogits[t, v] = g[t] * (onehot(targets[t])[v] - exp(logits[t, v] - lse[t]))
 * in fp32 (0 on inactive rows; NaN and RK_DEVERR_TARGET_RANGE for targets >= V).
 *   logits bf16 [T, V], lse fp32 [T] (from rk_logp_from_logits), grad_logp
 *   fp32 [T], dlogits fp32 [T, V].  Each element is computed independently.
 */
rk_status rk_logp_from_logits_bwd(const uint16_t *logits, const int64_t *targets,
                                  const int32_t *cu_seqlens, int32_t num_seqs,
                                  int64_t T, int64_t V, const float *lse,
                                  const float *grad_logp, float *dlogits, void *stream);

/*
 * Per-token GRPO loss on selected logprobs ("grpo_loss, ratio_kl", issue #101
 * P0 list; chain index 9 of PR #264, whose review asks for per-token outputs
 * or a fixed normalisation before bitwise invariance can be required; this
 * operator is per token, with a caller-given `scale` standing for the
 * caller's fixed denominator).  For every active row t:
 *     ratio = exp(logp - logp_old)
 *     surr  = min(ratio * A, clip(ratio, 1 - eps_low, 1 + eps_high) * A)
 *     kl    = exp(logp_ref - logp) - (logp_ref - logp) - 1   (0 if logp_ref is NULL)
 *     loss  = scale * (-surr + beta * kl)
 *     grad_logp = d loss / d logp   (the g for rk_linear_logp_bwd)
 * Inactive rows get 0 in every output.  All arrays fp32 [T]; logp_ref, ratio
 * and kl may be NULL.  Requires 0 <= eps_low < 1, eps_high >= 0, beta >= 0.
 */
rk_status rk_grpo_token_loss(const float *logp, const float *logp_old, const float *logp_ref,
                             const float *advantages, const int64_t *targets,
                             const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                             float eps_low, float eps_high, float beta, float scale,
                             float *loss, float *grad_logp, float *ratio, float *kl,
                             void *stream);

/*
 * rk_linear_logp followed by rk_grpo_token_loss on its logp, in one call: the
 * forward's final merge applies the per-token loss to each logp it has just
 * produced, so the logprobs never make a second trip through memory and one
 * launch is saved.  Every output (logp, lse, loss, grad_logp, ratio, kl) is
 * bitwise identical to the two separate calls on the same inputs.
 *   h, W, targets, cu_seqlens, num_seqs, T, H, V, logp, lse, workspace,
 *   workspace_bytes: as for rk_linear_logp (workspace >=
 *   rk_linear_logp_workspace_size(T, H, V));
 *   logp_old, logp_ref, advantages, eps_low, eps_high, beta, scale, loss,
 *   grad_logp, ratio, kl: as for rk_grpo_token_loss.
 * Rows whose target is >= V get NaN logp, and the loss arithmetic then runs on
 * that NaN, as it would in the separate call.
 */
rk_status rk_linear_logp_grpo(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu_seqlens, int32_t num_seqs,
                              int64_t T, int64_t H, int64_t V,
                              const float *logp_old, const float *logp_ref,
                              const float *advantages, float eps_low, float eps_high,
                              float beta, float scale,
                              float *logp, float *lse, float *loss, float *grad_logp,
                              float *ratio, float *kl,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Greedy decoding step fused with its selected logprob: for every row (rows
 * outside [cu_seqlens[0], cu_seqlens[num_seqs]) when cu_seqlens is given get
 * token -1 and logp = lse = 0),
 *     token[t] = argmax_v z[t, v]   (z = h . W^T; the lowest v among equal maxima)
 *     logp[t]  = z[t, token[t]] - logsumexp_v z[t, v]
 * with exactly the arithmetic of rk_linear_logp, so that scoring the generated
 * tokens again later (rk_linear_logp with targets = token) reproduces logp and
 * lse bit for bit (issue #244, Workstream 2 #152: generate-then-re-score
 * selected-logprob equivalence).
 *   workspace >= rk_linear_greedy_workspace_size(T, H, V) bytes, 16-byte aligned.
 */
size_t rk_linear_greedy_workspace_size(int64_t T, int64_t H, int64_t V);
rk_status rk_linear_greedy(const uint16_t *h, const uint16_t *W, const int32_t *cu_seqlens,
                           int32_t num_seqs, int64_t T, int64_t H, int64_t V,
                           int64_t *token, float *logp, float *lse,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Weight gradient of linear_logp (issue #244 "[WS1 Test] ...", Workstream 3
 * #153: "GEMM dW", fixed batch-shape-independent reduction order, no
 * atomicAdd; parameter gradients are compared "over the same complete
 * logical sample set", with packed/chunked results restored to canonical
 * (sample_id, token_position) order):
 *     dW[v, :] = sum over canonical tokens i of g_i * (onehot(target_i)[v] - p_i[v]) * h_i
 * with p_i = softmax(h_i . W^T) recomputed from lse.  The canonical tokens are
 * the active rows among `row_order[0..n_order)` (physical row indices, in the
 * caller's canonical order; out-of-range entries are skipped), or among rows
 * 0..T-1 in ascending order when row_order is NULL.  The sum runs over the
 * canonical tokens in that order: the same tokens in the same canonical
 * order give a bitwise identical dW whatever their physical layout
 * (padding, packing, permutation, batch composition).
 *   h, W, targets, cu_seqlens, num_seqs, T, H, V: as for rk_linear_logp
 *   lse, grad_logp fp32 [T]; dW fp32 [V, H] output (16-byte aligned);
 *   workspace >= rk_linear_logp_dw_workspace_size(n, H, V) bytes, where n is
 *   n_order (or T): canonical copies of h and of g * softmax (bf16 [n, V]).
 * As in rk_linear_logp_bwd, each token's target column and its columns with
 * p >= 1/64 are handled in fp32: per vocabulary row, the fp32 terms
 * g (onehot - p) h_i are summed over those tokens in canonical order.  The
 * remaining g p h_i terms are a tensor-core GEMM with K = the canonical
 * tokens in one ascending pass.  An lse that does not belong to the inputs
 * sets RK_DEVERR_LSE as in rk_linear_logp_bwd.
 */
size_t rk_linear_logp_dw_workspace_size(int64_t n, int64_t H, int64_t V);
rk_status rk_linear_logp_dw(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                            const int32_t *cu_seqlens, int32_t num_seqs,
                            int64_t T, int64_t H, int64_t V,
                            const float *lse, const float *grad_logp,
                            const int64_t *row_order, int64_t n_order, float *dW,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * The whole backward of linear_logp in one call: dh (as rk_linear_logp_bwd)
 * and dW (as rk_linear_logp_dw) from one shared g * softmax over the
 * canonical tokens, so z is recomputed once instead of twice (8*T*H*V flop
 * for forward + this call instead of 10*T*H*V).  dh is bitwise identical to
 * rk_linear_logp_bwd's and dW to rk_linear_logp_dw's for the same inputs:
 * each dh row is computed over the canonical rows and stored at its physical
 * row; rows outside the canonical set get 0, active rows with targets >= V
 * get NaN and RK_DEVERR_TARGET_RANGE.
 *   arguments: as rk_linear_logp_dw, plus dh fp32 [T, H] (16-byte aligned);
 *   workspace >= rk_linear_logp_bwd_full_workspace_size(n, H, V) bytes (it
 *   holds g * softmax both as [n, V] for dh and as [V, n] for dW).
 */
size_t rk_linear_logp_bwd_full_workspace_size(int64_t n, int64_t H, int64_t V);
rk_status rk_linear_logp_bwd_full(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                  const int32_t *cu_seqlens, int32_t num_seqs,
                                  int64_t T, int64_t H, int64_t V,
                                  const float *lse, const float *grad_logp,
                                  const int64_t *row_order, int64_t n_order,
                                  float *dh, float *dW,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * rk_linear_logp_bwd_full from the forward's saved terms: dh and dW of the
 * same canonical tokens, with dZ converted from `saved` (as
 * rk_linear_logp_bwd_saved converts it) instead of recomputed, so the call
 * runs two GEMMs (dh, dW) instead of three.  dh is bitwise that of
 * rk_linear_logp_bwd_saved on the same saved state; dW is bitwise the same
 * for the same tokens in the same canonical order, whatever their layout, and
 * within the gradient tolerance of rk_linear_logp_dw.  `saved` is only read
 * (it can serve this call and then rk_linear_logp_bwd_saved, or be reused).
 *   arguments: as rk_linear_logp_bwd_full, plus saved / saved_bytes from
 *   rk_linear_logp_fwd_saved on the same h, W, targets, cu_seqlens (same T);
 *   workspace >= rk_linear_logp_bwd_full_workspace_size(n, H, V) bytes.
 */
rk_status rk_linear_logp_bwd_full_saved(const uint16_t *h, const uint16_t *W,
                                        const int64_t *targets, const int32_t *cu_seqlens,
                                        int32_t num_seqs, int64_t T, int64_t H, int64_t V,
                                        const float *lse, const float *grad_logp,
                                        const void *saved, size_t saved_bytes,
                                        const int64_t *row_order, int64_t n_order,
                                        float *dh, float *dW,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * rk_linear_logp without a workspace argument, for callers that cannot
 * allocate device memory.  (No counterpart in the pages: this is an interface
 * convenience, not part of the method.)  Such callers include programs whose
 * device memory belongs to a fixed-budget arena or pool, where an extra
 * cudaMalloc would fail against the budget, fragment the pool or stall the
 * device (cudaMalloc and cudaFree may synchronise), and plugin-style hosts
 * that hand over only input/output pointers and a stream.
 *
 * Same arguments, results and errors as rk_linear_logp, minus the workspace:
 * the scratch lives in a fixed 32 MiB array inside the library (static device
 * memory; every GPU on which the library is used keeps it until the process
 * exits).  The call allocates nothing.
 *  - Size limit: returns RK_ERR_WORKSPACE, before launching anything, when
 *    rk_linear_logp_workspace_size(T, H, V) > 32 MiB (33554432 bytes), i.e.
 *    about T * ceil(V/256) * 8 + T * 4 bytes; e.g. at most 8363 rows for
 *    V = 128256 and 33420 rows for V = 32000.
 *  - The first call on each device looks up that device's array address
 *    (with that device current) and keeps it for the life of the process (see
 *    "Contexts" above); make that first call before any stream capture.
 *  - All calls on a device share the one array and nothing in it needs to
 *    start at zero; calls that overlap on the GPU (several streams, or
 *    several host threads at once) race on it and must be serialised.
 */
rk_status rk_linear_logp_noalloc(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                 const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t T, int64_t H, int64_t V,
                                 float *logp, float *lse, void *stream);

/*
 * Reads and clears the device error word of the current device after
 * synchronising `stream`.  *err receives an OR of RK_DEVERR_* bits (0 = none).
 * For tests and debugging; it is the only call that synchronises.
 */
rk_status rk_get_device_error(void *stream, int32_t *err);

/*
 * Self-test of the failure path that every pipeline wait in the library
 * shares: one kernel waits on an mbarrier that is never completed, gives up
 * after `limit_ns` (1 ns .. 10 s) and sets RK_DEVERR_TIMEOUT in the device
 * error word, leaving the context usable.  (Issue #244, Workstream 4 #150
 * chain gate: a path that quietly falls back counts as a failure, so a
 * stalled pipeline has to come back as an error rather than a hang.)
 * Asynchronous; read the result with rk_get_device_error.
 */
rk_status rk_selftest_wait_timeout(int64_t limit_ns, void *stream);

/*
 * Diagnostics of the two backward GEMMs that sum over a long K axis: dh
 * (K = vocabulary; rk_linear_logp_bwd, rk_linear_logp_bwd_full) and dW
 * (K = canonical tokens; rk_linear_logp_dw, rk_linear_logp_bwd_full).  Each
 * runs with one or two 256-row blocks per 256-column tile.  Two blocks share
 * every B slice between both TMEM accumulators (half the B traffic) and are
 * picked automatically for long K loops (>= 256 stages of 64) with enough
 * tiles (about 8 per resident CTA pair).  Every accumulator sees the same MMA
 * sequence in either form, so the choice never changes a bit of dh or dW.
 *
 * rk_set_row_blocks(n): n = 0 automatic (the default), 1 or 2 forces that
 * form for every later launch in the process (so that tests can run either
 * form on shapes of their choice).  RK_ERR_INVALID_ARG for other n.
 * rk_last_row_blocks(gemm): blocks per tile of the last such GEMM launched
 * on the calling host thread: gemm 0 = dh, 1 = dW.  Returns 1 or 2, 0 before
 * the first launch, -1 for another gemm value.
 */
rk_status rk_set_row_blocks(int32_t n);
int32_t rk_last_row_blocks(int32_t gemm);

/*
 * Tile order of the same GEMMs.  Long K loops (>= 256 stages) take their
 * tiles in rounds: with P resident CTA pairs, pair p computes tiles p, p + P,
 * ... and starts round r only once every pair has issued the copies of round
 * r - 1, so the pairs that share a dZ row block or a W slice stay in step and
 * share it through L2 (the dh GEMM's DRAM reads at T = 65536, V = 128256 fell
 * from 115 to 84 GB).  That launch is cooperative (all pairs resident); if it
 * is refused, or the stream is being captured into a graph, the tiles are
 * taken from a counter in the order the pairs become free.  The order never
 * changes a bit.
 * rk_last_tile_order(gemm): 2 rounds, 1 counter, for the last such GEMM on
 * the calling host thread (gemm 0 = dh, 1 = dW); 0 before the first launch,
 * -1 for another gemm value.
 */
int32_t rk_last_tile_order(int32_t gemm);

/* Human-readable name of a status code (static string). */
const char *rk_status_string(rk_status s);

/* The CUDA error code behind the last RK_ERR_CUDA returned on this host thread. */
int rk_last_cuda_error(void);

/* Library version, e.g. "rk 0.1.0 sm_103a". */
const char *rk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RK_H */
