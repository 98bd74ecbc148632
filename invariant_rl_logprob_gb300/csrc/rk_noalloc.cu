// rk_noalloc.cu -- rk_linear_logp_noalloc: the linear_logp forward for callers
// that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a host program
// whose device memory is owned by a fixed-budget arena or pool (an extra
// cudaMalloc would fail against the budget, fragment the pool, or stall the
// device in the middle of a latency-critical loop, since cudaMalloc/cudaFree
// may synchronise), or a plugin-style interface that passes only input and
// output pointers plus a stream, with no allocator at hand.  For them the
// forward's scratch (the per-row, per-vocabulary-tile softmax partials and the
// target logits) lives in the fixed array below instead of a caller workspace.
// The kernels are the same as rk_linear_logp's, so the results are identical.
#include <mutex>

#include "rk.h"
#include "rk_internal.h"

namespace {

// Fixed scratch for rk_linear_logp_noalloc: 32 MiB per device.  It is part of
// the library's device image, so every GPU on which the library is used keeps
// it until the process exits.  Device code could name it directly; host code
// only ever passes its device address, looked up per device below.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array.  Done once per device, with
// that device current (the device the call runs on).
cudaError_t scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" rk_status rk_linear_logp_noalloc(const uint16_t *h, const uint16_t *W,
                                            const int64_t *targets, const int32_t *cu_seqlens,
                                            int32_t num_seqs, int64_t T, int64_t H, int64_t V,
                                            float *logp, float *lse, void *stream) {
    // the same checks, in the same order, as rk_linear_logp
    if (T < 0 || H <= 0 || V <= 0) return RK_ERR_INVALID_ARG;
    if (T == 0) return RK_OK;
    if (!h || !W || !logp) return RK_ERR_INVALID_ARG;
    const rk_status st = rk::check_rows(targets, cu_seqlens, num_seqs);
    if (st != RK_OK) return st;
    if (H % 64 != 0 || H > 65536 || V >= (int64_t(1) << 31) || T >= (int64_t(1) << 31))
        return RK_ERR_UNSUPPORTED;
    if (!rk::aligned(h, 16) || !rk::aligned(W, 16)) return RK_ERR_UNSUPPORTED;
    // The scratch this call needs must fit the fixed array; larger requests are
    // refused here, before anything runs.
    if (rk::linear_fwd_workspace_bytes(T, V) > kNoAllocScratchBytes) return RK_ERR_WORKSPACE;

    rk::DeviceInfo di;
    cudaError_t e = rk::current_device_info(&di);
    if (e != cudaSuccess) {
        rk::record_cuda_error((int)e);
        return RK_ERR_CUDA;
    }
    if (di.device < 0 || di.device >= kMaxDevices) return RK_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    e = scratch_address(di.device, &scratch);
    if (e != cudaSuccess) {
        rk::record_cuda_error((int)e);
        return RK_ERR_CUDA;
    }
    // Nothing in the scratch has to start at zero: every partial the merge
    // reads is written earlier in the same call.
    e = rk::launch_linear_fwd(h, W, targets, cu_seqlens, num_seqs, T, H, V, logp, lse, scratch,
                              di, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        rk::record_cuda_error((int)e);
        return RK_ERR_CUDA;
    }
    return RK_OK;
}
