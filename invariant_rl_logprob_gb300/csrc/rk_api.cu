// rk_api.cu -- the extern "C" entry points declared in include/rk.h:
// argument validation (before any launch), per-device lookups, TMA descriptor
// encoding, and dispatch to the kernels' launchers.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "rk.h"
#include "rk_device.cuh"
#include "rk_internal.h"
#include "token_loss.cuh"

// One error word per device (the module is loaded per device context).
__device__ unsigned int g_rk_device_error = 0u;

namespace rk {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

thread_local int g_last_cuda_error = 0;

void load_encode() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, uint32_t esize, const void *base,
               uint64_t inner, uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
               uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    (void)esize;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

rk_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return RK_ERR_CUDA;
}

}  // namespace

bool encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                         bool sw128) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer,
                     row_stride_bytes, box_inner, box_outer,
                     sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_tmap_bf16_2d_sw64(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer,
                     row_stride_bytes, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_64B);
}

void record_cuda_error(int e) { g_last_cuda_error = e; }

cudaError_t current_device_info(DeviceInfo *di) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev_ready[dev]) {
            *di = g_dev[dev];
            return cudaSuccess;
        }
    }
    DeviceInfo d;
    d.device = dev;
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_rk_device_error);
    if (e != cudaSuccess) return e;
    d.err = static_cast<unsigned *>(p);
    std::lock_guard<std::mutex> lk(g_mu);
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
    *di = d;
    return cudaSuccess;
}

}  // namespace rk

using rk::DeviceInfo;

namespace {

// One thread waits on an mbarrier that nothing ever arrives on, through the
// same bounded wait the pipelines use; it gives up after `limit_ns`.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned *err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        rk::mbar_init(rk::smem_u32(&bar), 1);
        abort_flag = 0;
        rk::fence_mbar_init();
        (void)rk::mbar_wait_limit(rk::smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    }
}

using rk::aligned;
using rk::check_rows;

}  // namespace

extern "C" {

const char *rk_status_string(rk_status s) {
    switch (s) {
        case RK_OK: return "RK_OK";
        case RK_ERR_INVALID_ARG: return "RK_ERR_INVALID_ARG";
        case RK_ERR_UNSUPPORTED: return "RK_ERR_UNSUPPORTED";
        case RK_ERR_WORKSPACE: return "RK_ERR_WORKSPACE";
        case RK_ERR_CUDA: return "RK_ERR_CUDA";
    }
    return "RK_ERR_UNKNOWN";
}

int rk_last_cuda_error(void) { return rk::g_last_cuda_error; }

const char *rk_version(void) { return "rk 0.1.0 sm_103a"; }

size_t rk_linear_logp_workspace_size(int64_t T, int64_t H, int64_t V) {
    (void)H;
    if (T <= 0 || V <= 0) return 0;
    return rk::linear_fwd_workspace_bytes(T, V);
}

rk_status rk_linear_logp(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                         const int32_t *cu_seqlens, int32_t num_seqs, int64_t T, int64_t H,
                         int64_t V, float *logp, float *lse, void *workspace,
                         size_t workspace_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !logp) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16)) return RK_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < rk::linear_fwd_workspace_bytes(T, V))
        return RK_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_fwd(h, W, targets, cu_seqlens, num_seqs, T, H, V, logp, lse, workspace,
                              di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_linear_logp_grpo(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu_seqlens, int32_t num_seqs, int64_t T, int64_t H,
                              int64_t V, const float *logp_old, const float *logp_ref,
                              const float *advantages, float eps_low, float eps_high, float beta,
                              float scale, float *logp, float *lse, float *loss, float *grad_logp,
                              float *ratio, float *kl, void *workspace, size_t workspace_bytes,
                              void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !logp || !logp_old || !advantages || !loss || !grad_logp)
        return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (!(eps_low >= 0.f && eps_low < 1.f) || !(eps_high >= 0.f) || !(beta >= 0.f))
        return RK_ERR_INVALID_ARG;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16)) return RK_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < rk::linear_fwd_workspace_bytes(T, V))
        return RK_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    const rk::GrpoArgs p{logp_old, logp_ref, advantages, eps_low, eps_high, beta, scale,
                         loss, grad_logp, ratio, kl};
    e = rk::launch_linear_fwd(h, W, targets, cu_seqlens, num_seqs, T, H, V, logp, lse, workspace,
                              di, static_cast<cudaStream_t>(stream), &p);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_logp_saved_size(int64_t T, int64_t H, int64_t V) {
    (void)H;
    if (T <= 0 || V <= 0) return 0;
    return rk::linear_fwd_saved_bytes(T, V);
}

rk_status rk_linear_logp_fwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                                   int64_t H, int64_t V, float *logp, float *lse, void *saved,
                                   size_t saved_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !logp) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16)) return RK_ERR_UNSUPPORTED;
    if (!saved || saved_bytes < rk::linear_fwd_saved_bytes(T, V)) return RK_ERR_WORKSPACE;
    if (!aligned(saved, 256)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_fwd_saved(h, W, targets, cu_seqlens, num_seqs, T, H, V, logp, lse, saved,
                                    di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_logp_bwd_saved_workspace_size(int64_t T, int64_t H, int64_t V) {
    (void)H;
    if (T <= 0 || V <= 0) return 0;
    return rk::linear_bwd_saved_workspace_bytes(T);
}

rk_status rk_linear_logp_bwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                                   int64_t H, int64_t V, const float *lse,
                                   const float *grad_logp, void *saved, size_t saved_bytes,
                                   float *dh, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !lse || !grad_logp || !dh) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if ((V + 8191) / 8192 > 65535) return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dh, 16)) return RK_ERR_UNSUPPORTED;
    if (!saved || saved_bytes < rk::linear_fwd_saved_bytes(T, V)) return RK_ERR_WORKSPACE;
    if (!aligned(saved, 256)) return RK_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < rk::linear_bwd_saved_workspace_bytes(T))
        return RK_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_bwd_saved(h, W, targets, cu_seqlens, num_seqs, T, H, V, lse, grad_logp,
                                    saved, dh, workspace, di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_logp_from_logits(const uint16_t *logits, const int64_t *targets,
                              const int32_t *cu_seqlens, int32_t num_seqs, int64_t T, int64_t V,
                              float *logp, float *lse, void *stream) {
    if (T < 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!logits || !logp) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (V >= (int64_t(1) << 31)) return RK_ERR_UNSUPPORTED;
    if (!aligned(logits, 2)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_logits_logp(logits, targets, cu_seqlens, num_seqs, T, V, logp, lse, di,
                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_logp_bwd_workspace_size(int64_t T, int64_t H, int64_t V) {
    (void)H;
    if (T <= 0 || V <= 0) return 0;
    const int64_t q = rk::linear_bwd_chunk_quantum();
    return rk::linear_bwd_chunk_bytes((T + q - 1) / q * q, V);
}

size_t rk_linear_logp_bwd_min_workspace_size(int64_t H, int64_t V) {
    (void)H;
    if (V <= 0) return 0;
    return rk::linear_bwd_chunk_bytes(rk::linear_bwd_chunk_quantum(), V);
}

rk_status rk_linear_logp_bwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                             const int32_t *cu_seqlens, int32_t num_seqs, int64_t T, int64_t H,
                             int64_t V, const float *lse, const float *grad_logp, float *dh,
                             void *workspace, size_t workspace_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !lse || !grad_logp || !dh) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dh, 16)) return RK_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < rk_linear_logp_bwd_min_workspace_size(H, V))
        return RK_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_bwd(h, W, targets, cu_seqlens, num_seqs, T, H, V, lse, grad_logp, dh,
                              workspace, workspace_bytes, di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_lm_head_workspace_size(void) { return 256; }

rk_status rk_lm_head(const uint16_t *h, const uint16_t *W, int64_t T, int64_t H, int64_t V,
                     uint16_t *logits, int64_t ld_logits, void *workspace,
                     size_t workspace_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !logits || ld_logits < V) return RK_ERR_INVALID_ARG;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16) || !aligned(logits, 16) || ld_logits % 8 != 0)
        return RK_ERR_UNSUPPORTED;
    if (workspace && (workspace_bytes < rk_lm_head_workspace_size() || !aligned(workspace, 16)))
        return RK_ERR_WORKSPACE;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_lm_head(h, W, T, H, V, logits, ld_logits, static_cast<unsigned *>(workspace), di,
                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_logp_from_logits_bwd(const uint16_t *logits, const int64_t *targets,
                                  const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                                  int64_t V, const float *lse, const float *grad_logp,
                                  float *dlogits, void *stream) {
    if (T < 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!logits || !lse || !grad_logp || !dlogits) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (V >= (int64_t(1) << 31)) return RK_ERR_UNSUPPORTED;
    if (!aligned(logits, 2) || !aligned(dlogits, 4)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_logits_bwd(logits, targets, cu_seqlens, num_seqs, T, V, lse, grad_logp, dlogits,
                              di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_grpo_token_loss(const float *logp, const float *logp_old, const float *logp_ref,
                             const float *advantages, const int64_t *targets,
                             const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                             float eps_low, float eps_high, float beta, float scale, float *loss,
                             float *grad_logp, float *ratio, float *kl, void *stream) {
    if (T < 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!logp || !logp_old || !advantages || !loss || !grad_logp) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (!(eps_low >= 0.f && eps_low < 1.f) || !(eps_high >= 0.f) || !(beta >= 0.f))
        return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_grpo_token(logp, logp_old, logp_ref, advantages, targets, cu_seqlens, num_seqs,
                              T, eps_low, eps_high, beta, scale, loss, grad_logp, ratio, kl, di,
                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_greedy_workspace_size(int64_t T, int64_t H, int64_t V) {
    (void)H;
    if (T <= 0 || V <= 0) return 0;
    return rk::linear_greedy_workspace_bytes(T, V);
}

rk_status rk_linear_greedy(const uint16_t *h, const uint16_t *W, const int32_t *cu_seqlens,
                           int32_t num_seqs, int64_t T, int64_t H, int64_t V, int64_t *token,
                           float *logp, float *lse, void *workspace, size_t workspace_bytes,
                           void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !token || !logp) return RK_ERR_INVALID_ARG;
    if (cu_seqlens && num_seqs < 0) return RK_ERR_INVALID_ARG;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(W, 16)) return RK_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < rk::linear_greedy_workspace_bytes(T, V))
        return RK_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_greedy(h, W, cu_seqlens, num_seqs, T, H, V, token, logp, lse, workspace,
                                 di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_logp_dw_workspace_size(int64_t n, int64_t H, int64_t V) {
    if (n <= 0 || H <= 0 || V <= 0) return 0;
    return rk::linear_dw_workspace_bytes(n, H, V);
}

rk_status rk_linear_logp_dw(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                            const int32_t *cu_seqlens, int32_t num_seqs, int64_t T, int64_t H,
                            int64_t V, const float *lse, const float *grad_logp,
                            const int64_t *row_order, int64_t n_order, float *dW,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (!dW || !W) return RK_ERR_INVALID_ARG;
    const int64_t n = row_order ? n_order : T;
    if (n < 0) return RK_ERR_INVALID_ARG;
    if (n > 0 && (!h || !lse || !grad_logp)) return RK_ERR_INVALID_ARG;
    rk_status st = check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK && n > 0) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) ||
        n >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if ((h && !aligned(h, 16)) || !aligned(W, 16) || !aligned(dW, 16)) return RK_ERR_UNSUPPORTED;
    if (n > 0 && (!workspace || workspace_bytes < rk::linear_dw_workspace_bytes(n, H, V)))
        return RK_ERR_WORKSPACE;
    if (n > 0 && !aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_dw(h, W, targets, cu_seqlens, num_seqs, T, H, V, lse, grad_logp,
                             row_order, n, dW, workspace, di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

size_t rk_linear_logp_bwd_full_workspace_size(int64_t n, int64_t H, int64_t V) {
    if (n <= 0 || H <= 0 || V <= 0) return 0;
    return rk::linear_bwd_full_workspace_bytes(n, H, V);
}

rk_status rk_linear_logp_bwd_full(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                  const int32_t *cu_seqlens, int32_t num_seqs, int64_t T,
                                  int64_t H, int64_t V, const float *lse, const float *grad_logp,
                                  const int64_t *row_order, int64_t n_order, float *dh, float *dW,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (!dW || !W || (T > 0 && !dh)) return RK_ERR_INVALID_ARG;
    const int64_t n = row_order ? n_order : T;
    if (n < 0) return RK_ERR_INVALID_ARG;
    if ((n > 0 || T > 0) && (!h || !lse || !grad_logp)) return RK_ERR_INVALID_ARG;
    if (T > 0 || n > 0) {
        rk_status st = check_rows(targets, cu_seqlens, num_seqs);
        if (st != RK_OK) return st;
    }
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) ||
        n >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if ((h && !aligned(h, 16)) || !aligned(W, 16) || !aligned(dW, 16) || (dh && !aligned(dh, 16)))
        return RK_ERR_UNSUPPORTED;
    if (n > 0 && (!workspace || workspace_bytes < rk::linear_bwd_full_workspace_bytes(n, H, V)))
        return RK_ERR_WORKSPACE;
    if (n > 0 && !aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_bwd_full(h, W, targets, cu_seqlens, num_seqs, T, H, V, lse, grad_logp,
                                   row_order, n, dh, dW, workspace, di,
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_set_row_blocks(int32_t n) {
    if (n < 0 || n > 2) return RK_ERR_INVALID_ARG;
    rk::set_row_blocks_override((int)n);
    return RK_OK;
}

int32_t rk_last_row_blocks(int32_t gemm) {
    if (gemm != 0 && gemm != 1) return -1;
    return (int32_t)rk::last_row_blocks(gemm == 0 ? rk::RowGemm::kDhGemm : rk::RowGemm::kDwGemm);
}

int32_t rk_last_tile_order(int32_t gemm) {
    if (gemm != 0 && gemm != 1) return -1;
    return (int32_t)rk::last_tile_order(gemm == 0 ? rk::RowGemm::kDhGemm : rk::RowGemm::kDwGemm);
}

rk_status rk_linear_logp_bwd_full_saved(const uint16_t *h, const uint16_t *W,
                                        const int64_t *targets, const int32_t *cu_seqlens,
                                        int32_t num_seqs, int64_t T, int64_t H, int64_t V,
                                        const float *lse, const float *grad_logp,
                                        const void *saved, size_t saved_bytes,
                                        const int64_t *row_order, int64_t n_order, float *dh,
                                        float *dW, void *workspace, size_t workspace_bytes,
                                        void *stream) {
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (!dW || !W || (T > 0 && !dh)) return RK_ERR_INVALID_ARG;
    const int64_t n = row_order ? n_order : T;
    if (n < 0) return RK_ERR_INVALID_ARG;
    if ((n > 0 || T > 0) && (!h || !lse || !grad_logp)) return RK_ERR_INVALID_ARG;
    if (T > 0 || n > 0) {
        rk_status st = check_rows(targets, cu_seqlens, num_seqs);
        if (st != RK_OK) return st;
    }
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) ||
        n >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if ((V + 8191) / 8192 > 65535 || (V + 63) / 64 > 65535) return RK_ERR_UNSUPPORTED;
    if ((h && !aligned(h, 16)) || !aligned(W, 16) || !aligned(dW, 16) || (dh && !aligned(dh, 16)))
        return RK_ERR_UNSUPPORTED;
    if (T > 0 && (!saved || saved_bytes < rk::linear_fwd_saved_bytes(T, V)))
        return RK_ERR_WORKSPACE;
    if (saved && !aligned(saved, 256)) return RK_ERR_INVALID_ARG;
    if (n > 0 && (!workspace || workspace_bytes < rk::linear_bwd_full_workspace_bytes(n, H, V)))
        return RK_ERR_WORKSPACE;
    if (n > 0 && !aligned(workspace, 16)) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = rk::launch_linear_bwd_full(h, W, targets, cu_seqlens, num_seqs, T, H, V, lse, grad_logp,
                                   row_order, n, dh, dW, workspace, di,
                                   static_cast<cudaStream_t>(stream), T > 0 ? saved : nullptr);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_selftest_wait_timeout(int64_t limit_ns, void *stream) {
    if (limit_ns <= 0 || limit_ns > 10000000000ll) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns, di.err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return rk::cuda_fail(e);
    return RK_OK;
}

rk_status rk_get_device_error(void *stream, int32_t *err) {
    if (!err) return RK_ERR_INVALID_ARG;
    DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    e = cudaMemcpyAsync(&v, di.err, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    e = cudaMemsetAsync(di.err, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return rk::cuda_fail(e);
    *err = (int32_t)v;
    return RK_OK;
}

}  // extern "C"
