// The mHC post (step (1)) with the layer output given as int8 codes and one fp32 scale per
// token, and/or with the fused square sum of the updated streams: the post kernels of
// "[SM80] Backport mHC fused post + int8 all-reduce; fixes #28, #29", "What this fixes"
// (VLLM_MHC_AR_INT8 consumers, VLLM_MHC_POST_FUSE_SQRSUM).
//
// One CTA per token: it streams the token's 4 x H residual and its layer output once, writes
// R' (the same fp32 expression and rounding as every other post), and, for the square sum,
// adds R'^2 of the bf16-rounded values in a fixed order (per thread in vector order, then an
// xor tree within each warp, then the warps in order), so the result is deterministic.
#include <cstdint>

#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace mhc {

namespace {

constexpr int kPT = 256;  // threads per CTA

template <bool kInt8, bool kSq>
__global__ void __launch_bounds__(kPT)
post_ex_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y, const int8_t *__restrict__ Yq,
               const float *__restrict__ x_scales, const float *__restrict__ prev_post,
               const float *__restrict__ prev_comb, int H, uint16_t *__restrict__ R_out,
               float *__restrict__ sqrsum) {
    __shared__ float sMix[20];  // comb [4][4], post [4]
    __shared__ float sWarp[kPT / 32];
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid < 16) sMix[tid] = __ldg(prev_comb + t * 16 + tid);
    else if (tid < 20) sMix[tid] = __ldg(prev_post + t * 4 + (tid - 16));
    __syncthreads();
    const float xs = kInt8 ? __ldg(x_scales + t) : 0.f;
    const int nvec = H / kVec;
    float ss = 0.f;
    for (int v = tid; v < nvec; v += kPT) {
        const int64_t base = t * kHC * (int64_t)H + (int64_t)v * kVec;
        uint4 r[kHC];
#pragma unroll
        for (int j = 0; j < kHC; ++j) r[j] = ld_stream(R + base + (int64_t)j * H);
        float y[8];
        if (kInt8) {
            const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(Yq + t * (int64_t)H + (int64_t)v * kVec));
            const uint32_t w[2] = {q.x, q.y};
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = (float)(int8_t)(w[e >> 2] >> (8 * (e & 3))) * xs;
        } else {
            unpack8(ld_stream(Y + t * (int64_t)H + (int64_t)v * kVec), y);
        }
        uint4 o[kHC];
        float rf[kHC][8];
        post_vec8_yf(r, y, sMix, sMix + 16, o, rf);
#pragma unroll
        for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
        if (kSq) {
#pragma unroll
            for (int i = 0; i < kHC; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(rf[i][e], rf[i][e], ss);
        }
    }
    if (kSq) {
        ss = warp_sum(ss);
        if ((tid & 31) == 0) sWarp[tid >> 5] = ss;
        __syncthreads();
        if (tid == 0) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kPT / 32; ++w) a += sWarp[w];
            sqrsum[t] = a;
        }
    }
}

// The first layer's residual: four copies of the (T, H) input, R[t][j] = x[t] (plain stores:
// a following pre reads them back, from L2 when they fit).
__global__ void __launch_bounds__(kPT)
broadcast4_kernel(const uint16_t *__restrict__ x, int64_t n_vec, int nvec_row, int H, uint16_t *__restrict__ R) {
    for (int64_t i = (int64_t)blockIdx.x * kPT + threadIdx.x; i < n_vec; i += (int64_t)gridDim.x * kPT) {
        const int64_t t = i / nvec_row;
        const int v = (int)(i % nvec_row);
        const uint4 a = ld_stream(x + t * (int64_t)H + (int64_t)v * kVec);
        uint16_t *dst = R + t * kHC * (int64_t)H + (int64_t)v * kVec;
#pragma unroll
        for (int j = 0; j < kHC; ++j) *reinterpret_cast<uint4 *>(dst + (int64_t)j * H) = a;
    }
}

// The MXFP8 form of a bf16 layer input already in HBM: a thread takes two blocks of 32 values
// per step (eight 16-byte loads in flight), quantizes them as the epilogues do and stores each
// block's 32 codes as two 16-byte stores.
__global__ void __launch_bounds__(kPT)
mx_quantize_kernel(const uint16_t *__restrict__ X, int64_t n_blk, int blk_row, int H, int mode,
                   uint8_t *__restrict__ q, uint8_t *__restrict__ scale) {
    // may start while the kernel before it (which wrote X) still runs: wait for its results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t stride = (int64_t)gridDim.x * kPT;
    for (int64_t i0 = (int64_t)blockIdx.x * kPT + threadIdx.x; i0 < n_blk; i0 += 2 * stride) {
        uint4 o[2][4];
        int64_t t[2];
        int k[2];
        bool on[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int64_t i = i0 + b * stride;
            on[b] = i < n_blk;
            t[b] = on[b] ? i / blk_row : 0;
            k[b] = on[b] ? (int)(i % blk_row) : 0;
            const uint16_t *src = X + t[b] * (int64_t)H + (int64_t)k[b] * 32;
#pragma unroll
            for (int j = 0; j < 4; ++j) o[b][j] = on[b] ? ld_stream(src + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            if (!on[b]) continue;
            uint32_t w[8];
            const uint8_t sb = mx_quantize_block32(o[b], mode, w);
            uint4 *dst = reinterpret_cast<uint4 *>(q + t[b] * (int64_t)H + (int64_t)k[b] * 32);
            __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
            __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
            scale[mx_scale_offset(t[b], k[b], H)] = sb;
        }
    }
}

}  // namespace

cudaError_t launch_mx_quantize(const uint16_t *X, int64_t T, int H, const MxOut &mx, int num_sms, cudaStream_t stream) {
    const int blk_row = H / 32;
    const int64_t n = T * blk_row;
    const int64_t want = (n + kPT - 1) / kPT, cap = (int64_t)num_sms * 8;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap its launch with the tail before it
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
    cfg.blockDim = dim3(kPT);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mx_quantize_kernel, X, n, blk_row, H, mx.mode, mx.q, mx.scale);
}

cudaError_t launch_broadcast4(const uint16_t *x, int64_t T, int H, uint16_t *R_out, int num_sms, cudaStream_t stream) {
    const int nvec = H / kVec;
    const int64_t n = T * nvec;
    const int64_t want = (n + kPT - 1) / kPT, cap = (int64_t)num_sms * 8;
    broadcast4_kernel<<<(unsigned)(want < cap ? want : cap), kPT, 0, stream>>>(x, n, nvec, H, R_out);
    return cudaGetLastError();
}

cudaError_t launch_post_ex(const uint16_t *R, const uint16_t *Y, const int8_t *Yq, const float *x_scales,
                           const float *prev_post, const float *prev_comb, int64_t T, int H, uint16_t *R_out,
                           float *sqrsum, cudaStream_t stream) {
    const bool i8 = Yq != nullptr, sq = sqrsum != nullptr;
    auto kern = i8 ? (sq ? post_ex_kernel<true, true> : post_ex_kernel<true, false>)
                   : (sq ? post_ex_kernel<false, true> : post_ex_kernel<false, false>);
    mark_main_kernel(stream, true);
    kern<<<(unsigned)T, kPT, 0, stream>>>(R, Y, Yq, x_scales, prev_post, prev_comb, H, R_out, sqrsum);
    mark_main_kernel(stream, false);
    return cudaGetLastError();
}

}  // namespace mhc
