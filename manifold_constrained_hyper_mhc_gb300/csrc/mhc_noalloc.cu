// mhc_shifted_post_pre_noalloc: the fused post+pre call for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the op: code
// that runs inside an allocator-less runtime (a host framework that owns all
// device memory and hands out only the tensors it manages), a plugin that may
// not grow the process's memory footprint, or a hot path where an allocation
// would synchronise the device.  This entry point takes only inputs and
// outputs; the scratch memory the kernels need lives in a file-scope device
// array of fixed size that every GPU loading this library holds until the
// process exits.
//
// The array is not reachable from host code by its name: on the host,
// `g_noalloc_scratch` is only a stand-in symbol, and handing it to a kernel
// would fault (or, where the GPU can reach host memory, use the wrong memory).
// Its device address is looked up once per device with cudaGetSymbolAddress,
// with that device current, and that address is what the kernels receive.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "mhc.h"

namespace mhc {
void set_last_error(const char *msg);  // mhc_api.cu: the text mhc_last_error() returns
}

namespace {

// 4 MiB: enough for the decode-sized calls this path is meant for (at H = 7168,
// up to 1170 tokens); the limit is checked on every call.
constexpr size_t kScratchBytes = size_t(4) << 20;

// Zero-initialised when the module loads, which is the state the op's
// workspace contract asks for before first use; every call that completes
// leaves it in a state the next call can use, whatever its T and H.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" MHC_API mhc_status mhc_shifted_post_pre_noalloc(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
    float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *stream) {
    if (T < 0 || H < 0) {
        mhc::set_last_error("mhc_shifted_post_pre_noalloc: T and H must not be negative");
        return MHC_ERR_INVALID_ARG;
    }
    const size_t need = mhc_workspace_size(T, H);
    if (need > kScratchBytes) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "mhc_shifted_post_pre_noalloc: T=%lld, H=%lld needs %zu bytes of scratch, "
                      "more than the %zu-byte static scratch",
                      (long long)T, (long long)H, need, kScratchBytes);
        mhc::set_last_error(msg);
        return MHC_ERR_INVALID_ARG;
    }
    if (T == 0) return MHC_OK;
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "mhc_shifted_post_pre_noalloc: cudaGetSymbolAddress: %s",
                      cudaGetErrorString(e));
        mhc::set_last_error(msg);
        return MHC_ERR_CUDA;
    }
    return mhc_shifted_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias,
                                mix_scales, rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps,
                                hc_post_scale, sinkhorn_eps, sinkhorn_iters, residual_out,
                                layer_in_out, pre_mix_out, post_mix_out, comb_res_mix_out, scratch,
                                kScratchBytes, stream);
}

// The static scratch holds a control block like any workspace: a status word that a
// bounded device-side wait sets when it gives up, and the grid barrier's word.  Callers of
// the allocation-free entry point never see the array's address, so this reads (and, after
// a timeout, clears) that block for them, as mhc_check_status does for a workspace.
extern "C" MHC_API mhc_status mhc_noalloc_check_status(void *stream) {
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "mhc_noalloc_check_status: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        mhc::set_last_error(msg);
        return MHC_ERR_CUDA;
    }
    return mhc_check_status(scratch, stream);
}
