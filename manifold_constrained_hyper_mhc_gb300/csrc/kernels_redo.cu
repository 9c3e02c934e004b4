// The layer input of tokens whose streams cancel in X, recomputed with a direct square sum.
//
// The ws schedule forms sum_h X^2 (the statistic of the combine's RMSNorm, step (4)) as
// pre^T G pre from the Gram matrix of the four streams.  When the streams cancel in
// X = sum_i pre_i R'_i that is a small difference of large terms (gram_cancels in
// mhc_device.cuh), so the kernel's owner puts such a token on a list in the workspace (its
// length in control-block word kRedoCountWord).  This kernel follows the main kernel on the same
// stream and rewrites those tokens' layer input: X again from R' (same fp32 expression as the
// combine), sum_h X^2 summed directly in a fixed order, the RMSNorm with that rstd, and the MXFP8
// form when the call asked for it.  One CTA per listed token (grid-stride over a small grid);
// with an empty list every CTA reads one word and exits, otherwise the last CTA to finish sets
// the list length back to zero.
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
    const int nb32 = (H + 31) / 32;  // blocks of 32 values: block b holds vectors 4b .. 4b+3
    const float inv_h = 1.f / (float)H;
    for (unsigned int i = blockIdx.x; i < n; i += gridDim.x) {
        const int64_t t = list[i];
        const uint16_t *row = Rp + t * kHC * (int64_t)H;
        const float4 p4 = *reinterpret_cast<const float4 *>(pre_out + t * 4);
        const float pre[kHC] = {p4.x, p4.y, p4.z, p4.w};
        // X of one vector, as the combine computes it
        auto xvec = [&](int v, float (&x)[8]) {
            float rf[kHC][8];
#pragma unroll
            for (int j = 0; j < kHC; ++j) unpack8(ld_ro(row + (int64_t)j * H + v * kVec), rf[j]);
            combine_vec8_x2(rf, pre, x);
        };
        // sum_h X^2: each lane its blocks in order, then an xor tree
        float a = 0.f;
        for (int b = tid; b < nb32; b += kRT) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = 4 * b + k;
                if (v * kVec < H) {
                    float x[8];
                    xvec(v, x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) a = fmaf(x[e], x[e], a);
                }
            }
        }
        a = warp_sum(a);
        const float rstd = __frsqrt_rn(fmaxf(a, 0.f) * inv_h + rmsnorm_eps);
        for (int b = tid; b < nb32; b += kRT) {
            uint4 ob[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = 4 * b + k;
                ob[k] = make_uint4(0u, 0u, 0u, 0u);
                if (v * kVec < H) {
                    float x[8];
                    xvec(v, x);
                    ob[k] = norm_vec8(x, rstd, ld_ro(gamma + v * kVec));
                    if (X_out != nullptr) st_stream(X_out + t * (int64_t)H + v * kVec, ob[k]);
                }
            }
            if (mx.q != nullptr) {  // H % 32 == 0: the block is whole
                const int jj[4] = {0, 1, 2, 3};
                mx_quantize_block(ob, jj, mx.mode, mx.q + t * (int64_t)H + 32 * b, mx.scale + mx_scale_offset(t, b, H));
            }
        }
    }
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
