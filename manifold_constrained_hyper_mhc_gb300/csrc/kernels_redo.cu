// The layer input of tokens whose streams cancel in X, recomputed with a direct square sum.
//
// The ws schedule forms sum_h X^2 (the statistic of the combine's RMSNorm, step (4)) as
// pre^T G pre from the Gram matrix of the four streams.  When the streams cancel in
// X = sum_i pre_i R'_i that is a small difference of large terms (gram_cancels in
// mhc_device.cuh), so the kernel's owner puts such a token on a list in the workspace (its
// length in control-block word kRedoCountWord).  When ws runs alone, this kernel follows it on
// the same stream and rewrites those tokens' layer input (redo_token: X again from R' with the
// combine's fp32 expression, sum_h X^2 summed directly in a fixed order, the RMSNorm with that
// rstd, and the MXFP8 form when the call asked for it).  (With the token-tile kernel beside ws, or
// alone, the tile kernel does the same in its tail and this kernel is not launched.)  One CTA per
// listed token (grid-stride over a small grid); with an empty list every CTA reads one word and
// exits, otherwise the last CTA to finish sets the list length back to zero.
//
// It is launched with programmatic dependent launch: its CTAs may be resident before the main
// kernel ends, and wait (griddepcontrol.wait) for the main kernel's completion before reading
// anything it wrote.
#include <cstdint>

#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace mhc {

namespace {

// One warp per CTA: small enough to be resident beside the main kernel (a ws CTA leaves 4096
// registers of its SM free), so the grid is in place, waiting, when the main kernel ends.
constexpr int kRT = 32;            // threads per CTA
constexpr int64_t kRedoCtas = 32;  // CTAs of the grid (grid-stride over the listed tokens)

__global__ void __launch_bounds__(kRT, 1)
redo_kernel(const uint16_t *__restrict__ Rp, const uint16_t *__restrict__ gamma, float rmsnorm_eps, int64_t T, int H,
            const float *__restrict__ pre_out, uint16_t *__restrict__ X_out, MxOut mx, unsigned int *ctrl,
            const unsigned int *__restrict__ list) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the main kernel is complete, its writes visible
    // what follows on the stream may launch now; it waits for this grid before it reads
    asm volatile("griddepcontrol.launch_dependents;");
    const int tid = threadIdx.x;
    // (a list longer than the call's tokens can only be left over from an aborted call)
    const unsigned int n0 = *reinterpret_cast<volatile unsigned int *>(ctrl + kRedoCountWord);
    const unsigned int n = n0 < (unsigned int)T ? n0 : (unsigned int)T;
    for (unsigned int i = blockIdx.x; i < n; i += gridDim.x)
        redo_token(Rp, gamma, rmsnorm_eps, H, pre_out, X_out, mx, (int64_t)list[i]);
    if (n0 == 0) return;  // nothing listed: the list is already empty for the next call
    // the last CTA to get here clears the list for the next call
    __syncwarp();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(ctrl + kRedoDoneWord, 1u) == gridDim.x - 1) {
            ctrl[kRedoCountWord] = 0u;
            ctrl[kRedoDoneWord] = 0u;
        }
    }
}

}  // namespace

cudaError_t launch_redo(const uint16_t *Rp, const uint16_t *gamma, float rmsnorm_eps, int64_t T, int H,
                        const float *pre_out, uint16_t *X_out, const MxOut &mx, unsigned int *ctrl,
                        const unsigned int *list, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // resident before the main kernel ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // a small grid: CTAs that find the list empty only read its length, and a full list (every
    // token's streams cancelling) still spreads over kRedoCtas SMs
    const int64_t g = T < kRedoCtas ? T : kRedoCtas;
    cfg.gridDim = dim3((unsigned)(g > 0 ? g : 1));
    cfg.blockDim = dim3(kRT);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, redo_kernel, Rp, gamma, rmsnorm_eps, T, H, pre_out, X_out, mx, ctrl, list);
}

}  // namespace mhc
