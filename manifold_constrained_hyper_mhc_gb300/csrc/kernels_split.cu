// Split schedule: the mHC post+pre step as three launches.
//
//   1. split_partials_kernel: post (optional) + per-chunk square sum and the
//      24 projection partial sums, for 16 tokens x 256 hidden elements per CTA.
//   2. split_mix_kernel: one warp per token sums the chunk partials in a fixed
//      order, then the sigmoid heads and the Sinkhorn residual mix.
//   3. split_combine_kernel: one CTA per token, combine with pre_mix and RMSNorm.
//
// It re-reads R' once (28H bytes per token instead of 20H), so it is the
// simple, fully general schedule; every reduction runs in a fixed order, so the
// results do not depend on timing and the fused call equals post followed by
// pre bit for bit.  Also hosts the standalone post kernel.
#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace mhc {

namespace {

constexpr int kThreads = 256;

template <bool kPost>
__global__ void __launch_bounds__(kThreads)
split_partials_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y,
                      const float *__restrict__ prev_post, const float *__restrict__ prev_comb,
                      const float *__restrict__ phi, int64_t T, int H, uint16_t *__restrict__ R_out,
                      float *__restrict__ part) {
    __shared__ __align__(16) uint16_t sR[kSplitTok][kHC][kSplitH];  // 32 KB of R'
    __shared__ float sSS[kSplitTok][kSplitH / kVec];
    __shared__ float sMix[kSplitTok][20];  // comb[16] then post[4]

    const int tid = threadIdx.x;
    const int nchunk = gridDim.y;
    const int chunk = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * kSplitTok;
    const int h0 = chunk * kSplitH;
    const int hv = min(kSplitH, H - h0);

    if (kPost) {
        for (int idx = tid; idx < kSplitTok * 20; idx += kThreads) {
            const int g = idx / 20, m = idx % 20;
            const int64_t t = t0 + g;
            float v = 0.f;
            if (t < T) v = m < 16 ? prev_comb[t * 16 + m] : prev_post[t * 4 + (m - 16)];
            sMix[g][m] = v;
        }
        __syncthreads();
    }

    // Phase 1: R' for 16 tokens x 256 hidden x 4 streams, square sums per vector.
    for (int item = tid; item < kSplitTok * (kSplitH / kVec); item += kThreads) {
        const int g = item / (kSplitH / kVec), v = item % (kSplitH / kVec);
        const int h = v * kVec;
        const int64_t t = t0 + g;
        uint4 o[kHC] = {};
        float ss = 0.f;
        if (t < T && h < hv) {
            float rf[kHC][8];
            const int64_t base = t * kHC * (int64_t)H + h0 + h;
            if (kPost) {
                uint4 r[kHC];
#pragma unroll
                for (int j = 0; j < kHC; ++j) r[j] = ld_stream(R + base + (int64_t)j * H);
                const uint4 y = ld_stream(Y + t * (int64_t)H + h0 + h);
                post_vec8(r, y, &sMix[g][0], &sMix[g][16], o, rf);
#pragma unroll
                for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
            } else {
#pragma unroll
                for (int i = 0; i < kHC; ++i) {
                    o[i] = ld_stream(R + base + (int64_t)i * H);
                    unpack8(o[i], rf[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < kHC; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(rf[i][e], rf[i][e], ss);
        }
#pragma unroll
        for (int i = 0; i < kHC; ++i) *reinterpret_cast<uint4 *>(&sR[g][i][h]) = o[i];
        sSS[g][v] = ss;
    }
    __syncthreads();

    // Phase 2: projection partials.  Thread = (token g, lane l of 16); lane l
    // takes the flattened indices kl = l, l+16, ... of this chunk.
    const int g = tid >> 4, l = tid & 15;
    const int64_t t = t0 + g;
    float acc[kNumMix];
#pragma unroll
    for (int n = 0; n < kNumMix; ++n) acc[n] = 0.f;
    for (int kl = l; kl < kHC * kSplitH; kl += 16) {
        const int i = kl / kSplitH, h = kl % kSplitH;
        if (h >= hv) continue;
        const float x = __uint_as_float((uint32_t)sR[g][i][h] << 16);
        const float4 *prow = reinterpret_cast<const float4 *>(phi + ((int64_t)i * H + h0 + h) * kNumMix);
#pragma unroll
        for (int q = 0; q < kNumMix / 4; ++q) {
            const float4 p = __ldg(prow + q);
            acc[4 * q + 0] = fmaf(x, p.x, acc[4 * q + 0]);
            acc[4 * q + 1] = fmaf(x, p.y, acc[4 * q + 1]);
            acc[4 * q + 2] = fmaf(x, p.z, acc[4 * q + 2]);
            acc[4 * q + 3] = fmaf(x, p.w, acc[4 * q + 3]);
        }
    }
#pragma unroll
    for (int n = 0; n < kNumMix; ++n) {
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], o);
    }
    if (t < T) {
        float *dst = part + (t * nchunk + chunk) * kPartStride;
        // every lane of the 16 holds all 24 sums; lane l writes l and l + 16
#pragma unroll
        for (int n = 0; n < kNumMix; ++n)
            if (n == l || n == l + 16) dst[n] = acc[n];
        if (l == 0) {
            float ss = 0.f;
            for (int v = 0; v < kSplitH / kVec; ++v) ss += sSS[g][v];
            dst[kNumMix] = ss;
        }
    }
}

__global__ void __launch_bounds__(128)
split_mix_kernel(const float *__restrict__ part, int nchunk, const float *__restrict__ bias,
                 const float *__restrict__ mix_scales, Scalars s, int64_t T, int H, float *__restrict__ pre_out,
                 float *__restrict__ post_out, float *__restrict__ res_out) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t >= T) return;
    float acc = 0.f;
    if (lane <= kNumMix)
        for (int c = 0; c < nchunk; ++c) acc += part[(t * nchunk + c) * kPartStride + lane];
    const float ss = __shfl_sync(0xffffffffu, acc, kNumMix);
    const float r = 1.f / sqrtf(ss / (float)(kHC * H) + s.hc_norm_eps);
    const float v = heads_and_sinkhorn(r * acc, bias, mix_scales, s);
    if (lane < 4) pre_out[t * 4 + lane] = v;
    else if (lane < 8) post_out[t * 4 + lane - 4] = v;
    else if (lane < 24) res_out[t * 16 + lane - 8] = v;
}

__global__ void __launch_bounds__(kThreads)
split_combine_kernel(const uint16_t *__restrict__ Rp, const uint16_t *__restrict__ gamma,
                     const float *__restrict__ pre_mix, float rmsnorm_eps, int H,
                     uint16_t *__restrict__ X_out) {
    __shared__ float sWarp[kThreads / 32];
    __shared__ float sRstd;
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    float pre[kHC];
#pragma unroll
    for (int i = 0; i < kHC; ++i) pre[i] = pre_mix[t * 4 + i];
    const uint16_t *row = Rp + t * kHC * (int64_t)H;
    const int nv = H / kVec;

    float sx = 0.f;
    for (int v = tid; v < nv; v += kThreads) {
        float rf[kHC][8], x[8];
#pragma unroll
        for (int i = 0; i < kHC; ++i) unpack8(ld_ro(row + (int64_t)i * H + v * kVec), rf[i]);
        combine_vec8(rf, pre, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) sx = fmaf(x[e], x[e], sx);
    }
    sx = warp_sum(sx);
    if ((tid & 31) == 0) sWarp[tid >> 5] = sx;
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) a += sWarp[w];
        sRstd = 1.f / sqrtf(a / (float)H + rmsnorm_eps);
    }
    __syncthreads();
    const float rstd = sRstd;
    for (int v = tid; v < nv; v += kThreads) {
        float rf[kHC][8], x[8];
#pragma unroll
        for (int i = 0; i < kHC; ++i) unpack8(ld_stream(row + (int64_t)i * H + v * kVec), rf[i]);
        combine_vec8(rf, pre, x);
        st_stream(X_out + t * (int64_t)H + v * kVec, norm_vec8(x, rstd, ld_ro(gamma + v * kVec)));
    }
}

__global__ void __launch_bounds__(kThreads)
post_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y,
            const float *__restrict__ prev_post, const float *__restrict__ prev_comb, int64_t T,
            int H, uint16_t *__restrict__ R_out) {
    const int nv = H / kVec;
    const int64_t items = T * nv;
    for (int64_t it = (int64_t)blockIdx.x * kThreads + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * kThreads) {
        const int64_t t = it / nv;
        const int h = (int)(it % nv) * kVec;
        float comb[16], post[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 c = __ldg(reinterpret_cast<const float4 *>(prev_comb + t * 16) + q);
            comb[4 * q] = c.x; comb[4 * q + 1] = c.y; comb[4 * q + 2] = c.z; comb[4 * q + 3] = c.w;
        }
        const float4 p = __ldg(reinterpret_cast<const float4 *>(prev_post + t * 4));
        post[0] = p.x; post[1] = p.y; post[2] = p.z; post[3] = p.w;
        const int64_t base = t * kHC * (int64_t)H + h;
        uint4 r[kHC], o[kHC];
        float rf[kHC][8];
#pragma unroll
        for (int j = 0; j < kHC; ++j) r[j] = ld_stream(R + base + (int64_t)j * H);
        const uint4 y = ld_stream(Y + t * (int64_t)H + h);
        post_vec8(r, y, comb, post, o, rf);
#pragma unroll
        for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
    }
}

}  // namespace

cudaError_t launch_split(const SplitArgs &a, cudaStream_t stream) {
    const int nchunk = (a.H + kSplitH - 1) / kSplitH;
    const unsigned tblocks = (unsigned)((a.T + kSplitTok - 1) / kSplitTok);
    dim3 g1(tblocks, nchunk);
    mark_main_kernel(stream, true);  // the main span: all three kernels
    if (a.R_out != nullptr)
        split_partials_kernel<true><<<g1, kThreads, 0, stream>>>(
            a.R, a.Y, a.prev_post, a.prev_comb, a.phi, a.T, a.H, a.R_out, a.part);
    else
        split_partials_kernel<false><<<g1, kThreads, 0, stream>>>(
            a.R, nullptr, nullptr, nullptr, a.phi, a.T, a.H, nullptr, a.part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    split_mix_kernel<<<(unsigned)((a.T + 3) / 4), 128, 0, stream>>>(
        a.part, nchunk, a.bias, a.mix_scales, a.s, a.T, a.H, a.pre_out, a.post_out, a.res_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    split_combine_kernel<<<(unsigned)a.T, kThreads, 0, stream>>>(
        a.R_out != nullptr ? a.R_out : a.R, a.gamma, a.pre_out, a.s.rmsnorm_eps, a.H, a.X_out);
    mark_main_kernel(stream, false);
    return cudaGetLastError();
}

cudaError_t launch_post(const uint16_t *R, const uint16_t *Y, const float *prev_post,
                        const float *prev_comb, int64_t T, int H, uint16_t *R_out,
                        int num_sms, cudaStream_t stream) {
    const int64_t items = T * (H / kVec);
    int64_t blocks = (items + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap) blocks = cap;
    mark_main_kernel(stream, true);
    post_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(R, Y, prev_post, prev_comb, T, H, R_out);
    mark_main_kernel(stream, false);
    return cudaGetLastError();
}

}  // namespace mhc
