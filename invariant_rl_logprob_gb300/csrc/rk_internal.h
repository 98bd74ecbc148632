// rk_internal.h -- host-side declarations shared by the librk translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "rk.h"

namespace rk {

// Per-device facts the launchers need (cached by rk_api.cu).
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    unsigned *err = nullptr;  // device address of this device's error word
};

// Argument checks shared by the entry points.
inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
// targets is required; cu_seqlens, when given, needs num_seqs >= 0.
inline rk_status check_rows(const int64_t *targets, const int32_t *cu, int32_t num_seqs) {
    if (!targets) return RK_ERR_INVALID_ARG;
    if (cu && num_seqs < 0) return RK_ERR_INVALID_ARG;
    return RK_OK;
}

// Records the CUDA error behind an RK_ERR_CUDA for rk_last_cuda_error().
void record_cuda_error(int e);

// Fills `di` for the current device (first call per device does the lookups).
cudaError_t current_device_info(DeviceInfo *di);

// Encodes a 2-D bf16 TMA descriptor over a row-major [outer, inner] matrix
// with the given row stride (bytes) and box; 128-byte swizzle when `sw128`.
// Returns false if the CUDA driver rejects it.
bool encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                         bool sw128);
// The same with 64-byte swizzle (boxes whose rows are at most 64 bytes).
bool encode_tmap_bf16_2d_sw64(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// ---- logits path (logits_logp.cu) ----
cudaError_t launch_logits_logp(const uint16_t *logits, const int64_t *targets, const int32_t *cu,
                               int num_seqs, int64_t T, int64_t V, float *logp, float *lse,
                               const DeviceInfo &di, cudaStream_t st);

// ---- linear_logp forward (linear_logp_tc.cu) ----
struct GrpoArgs;  // token_loss.cuh
size_t linear_fwd_workspace_bytes(int64_t T, int64_t V);
// With `loss`, the merge also applies the per-token GRPO loss to each logp.
cudaError_t launch_linear_fwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                              float *logp, float *lse, void *workspace, const DeviceInfo &di,
                              cudaStream_t st, const GrpoArgs *loss = nullptr);

// ---- greedy step and dense lm_head (linear_logp_tc.cu) ----
size_t linear_greedy_workspace_bytes(int64_t T, int64_t V);
cudaError_t launch_linear_greedy(const uint16_t *h, const uint16_t *W, const int32_t *cu,
                                 int num_seqs, int64_t T, int64_t H, int64_t V, int64_t *token,
                                 float *logp, float *lse, void *workspace, const DeviceInfo &di,
                                 cudaStream_t st);
cudaError_t launch_lm_head(const uint16_t *h, const uint16_t *W, int64_t T, int64_t H, int64_t V,
                           uint16_t *logits, int64_t ld, unsigned *tile_counter,
                           const DeviceInfo &di, cudaStream_t st);

// ---- logits-path backward (logits_logp.cu) ----
cudaError_t launch_logits_bwd(const uint16_t *logits, const int64_t *targets, const int32_t *cu,
                              int num_seqs, int64_t T, int64_t V, const float *lse,
                              const float *grad, float *dlogits, const DeviceInfo &di,
                              cudaStream_t st);

// ---- per-token GRPO loss (token_loss.cu) ----
cudaError_t launch_grpo_token(const float *logp, const float *logp_old, const float *logp_ref,
                              const float *adv, const int64_t *targets, const int32_t *cu,
                              int num_seqs, int64_t T, float eps_low, float eps_high, float beta,
                              float scale, float *loss, float *grad, float *ratio, float *kl,
                              const DeviceInfo &di, cudaStream_t st);

// ---- backward: columns handled exactly in fp32 ----
// In every backward row, the target column and every column with
// p = exp(z - lse) >= kEntTau leave the bf16 g*softmax matrix (they are
// stored there as 0).  Their contribution w = g*(onehot - p) is kept in fp32
// as a per-row list of (column, w) entries, at most kEntCap of them (at most
// 1/kEntTau columns can reach kEntTau since the p of a row sum to 1, plus the
// target).  The lists are filled in any order and then sorted by column, so
// every later sum over them runs in one fixed order.
constexpr int kEntCap = 65;
// Rows per block of the live flags (one tile row of the CTA-pair kernel).
constexpr int kLiveBlockRows = 256;
constexpr float kEntTau = 1.0f / 64.0f;
// Sorts each of the first `rows` lists by column (one warp per row).
cudaError_t launch_sort_entries(int32_t *ecount, int2 *ent, int64_t rows, cudaStream_t st);

// ---- linear_logp weight gradient (dw_prep.cu, linear_logp_tc.cu) ----
struct DwBuffers {
    int64_t *crow;      // [n] physical row of each canonical token
    int64_t *n_active;  // [1] number of canonical tokens
    uint16_t *hc;       // [n, H] bf16 canonical h (zeros past n_active)
    float *gc;          // [n] canonical upstream gradient (0 past n_active)
    float *lsec;        // [n] canonical lse
    int64_t *tgtc;      // [n] canonical targets (-1 past n_active)
    int32_t *ecount;    // [n] entries of each canonical token
    int2 *ent;          // [n][kEntCap] (column, w bits) of each canonical token
    int32_t *eoff;      // [n] offset of each token's entries in the flat list
    int64_t *etotal;    // [1] entries in the flat list
    int32_t *ent_t;     // [n*kEntCap] flat list: token of each entry
    float *ent_w;       // [n*kEntCap] flat list: w of each entry
    int32_t *key0, *val0, *key1, *val1;  // [n*kEntCap] sort buffers (column, flat index)
    int32_t *begin, *end;                // [V] each column's range in the sorted list
    int32_t *rows;      // [V] the columns (rows of dW) with entries, ascending
    int64_t *n_rows;    // [1] how many
    int32_t *scan;      // [dw_scan_entries(n*kEntCap)] block counts and digit histograms
    uint16_t *dz;       // [n, ldz] bf16 canonical g * softmax
    int64_t ldz;
};
size_t linear_dw_workspace_bytes(int64_t n, int64_t H, int64_t V);
int64_t dw_scan_entries(int64_t n);
// radix passes of the column sort: the sorted list ends in (key0, val0) when
// even, in (key1, val1) when odd
int dw_sort_passes(int64_t V);
size_t linear_bwd_full_workspace_bytes(int64_t n, int64_t H, int64_t V);
cudaError_t launch_dw_prep(const uint16_t *h, const int64_t *targets, const int32_t *cu,
                           int num_seqs, int64_t T, int64_t H, int64_t V, const float *lse,
                           const float *grad, const int64_t *order, int64_t n, const DwBuffers &b,
                           const DeviceInfo &di, cudaStream_t st);
// After the dZ (or dZ^T) GEMM over the canonical tokens has filled the entry
// lists: flatten them in canonical token order, sort the flat list by column
// (stable, so each column's entries stay in token order) and find each
// column's [begin, end) range.
// Also writes each row's fp32 term S (the sum of its entries' w * h, in
// canonical token order) into dW, for the dW GEMM epilogue to complete.
cudaError_t launch_dw_entries(int64_t n, int64_t V, const DwBuffers &b, const uint16_t *hc,
                              int64_t H, float *dW, const DeviceInfo &di, cudaStream_t st);
cudaError_t launch_linear_dw(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                             const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                             const float *lse, const float *grad, const int64_t *order, int64_t n,
                             float *dW, void *workspace, const DeviceInfo &di, cudaStream_t st);
// With `saved` (the state of launch_linear_fwd_saved; read only), dZ comes
// from the saved terms instead of a z recompute.
cudaError_t launch_linear_bwd_full(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                                   const float *lse, const float *grad, const int64_t *order,
                                   int64_t n, float *dh, float *dW, void *workspace,
                                   const DeviceInfo &di, cudaStream_t st,
                                   const void *saved = nullptr);

// ---- dh / dW GEMM form (linear_logp_tc.cu) ----
// Both GEMMs run with one or two 256-row blocks per tile; the form never
// changes a bit.  0 = automatic, 1 or 2 = forced (process-wide).
enum class RowGemm { kDhGemm = 0, kDwGemm = 1 };
void set_row_blocks_override(int n);
// Blocks per tile of the last dh / dW GEMM launched on this host thread (0: none yet).
int last_row_blocks(RowGemm which);
// Tile order of the last dh / dW GEMM launched on this host thread: 1 tiles
// from a counter, 2 rounds started together (0: none yet).
int last_tile_order(RowGemm which);

// ---- forward that saves its exponentials; backward from them ----
// (linear_logp_tc.cu; the elementwise steps in saved_bwd.cu)
size_t linear_fwd_saved_bytes(int64_t T, int64_t V);
size_t linear_bwd_saved_workspace_bytes(int64_t T);
cudaError_t launch_linear_fwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                    const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                    int64_t V, float *logp, float *lse, void *saved,
                                    const DeviceInfo &di, cudaStream_t st);
cudaError_t launch_linear_bwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                    const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                    int64_t V, const float *lse, const float *grad, void *saved,
                                    float *dh, void *workspace, const DeviceInfo &di,
                                    cudaStream_t st);
// The elementwise steps over rows [row0, row0 + rows).  live (or null) flags
// the kLiveBlockRows-row blocks, counted from row 0, that hold an active row;
// the rows of other blocks are left untouched.
cudaError_t launch_stash_to_dz(uint16_t *dz, int64_t ldz, const float2 *part, int32_t num_n,
                               const int64_t *targets, const int32_t *cu, int num_seqs,
                               int64_t row0, int64_t rows, int64_t V, const float *lse,
                               const float *grad, const uint8_t *live, int32_t *ecount, int2 *ent,
                               const DeviceInfo &di, cudaStream_t st);
// Conversion into canonical order (the dW backward) and dZ -> dZ^T.
cudaError_t launch_stash_to_dz_canonical(const uint16_t *terms, int64_t ldz, const float2 *part,
                                         int32_t num_n, const int64_t *crow,
                                         const int64_t *n_active, const int64_t *tgtc,
                                         const float *lsec, const float *gc, int64_t n, int64_t V,
                                         uint16_t *dzc, int32_t *ecount, int2 *ent,
                                         const DeviceInfo &di, cudaStream_t st);
cudaError_t launch_transpose_dz(const uint16_t *dz, int64_t ldz, int64_t n, int64_t V,
                                uint16_t *dzt, int64_t ldn, cudaStream_t st);
cudaError_t launch_exact_entries(const uint16_t *h, const uint16_t *W, int64_t H,
                                 const int64_t *targets, const int32_t *cu, int num_seqs,
                                 int64_t row0, int64_t rows, int64_t V, const float *lse,
                                 const float *grad, const int32_t *ecount, int2 *ent,
                                 cudaStream_t st);

// ---- linear_logp backward (linear_logp_tc.cu) ----
size_t linear_bwd_chunk_bytes(int64_t rows, int64_t V);
int64_t linear_bwd_chunk_quantum();
cudaError_t launch_linear_bwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                              const float *lse, const float *grad, float *dh, void *workspace,
                              size_t workspace_bytes, const DeviceInfo &di, cudaStream_t st);

}  // namespace rk
