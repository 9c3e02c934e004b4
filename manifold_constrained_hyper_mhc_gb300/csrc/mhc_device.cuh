// Device-side building blocks shared by every schedule of the mHC post+pre
// kernels.  Each schedule computes the same fp32 expressions in the same order
// through these helpers, so the post (residual update) and the combine are bit
// for bit the same whichever schedule runs them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace mhc {

constexpr int kHC = 4;      // hc_mult: residual streams per token
constexpr int kNumMix = 24; // 4 pre + 4 post + 16 residual-mix logits
constexpr int kVec = 8;     // bf16 elements per 16-byte vector

struct Scalars {
    float hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps;
    int sinkhorn_iters;
};

// ---- 16-byte vector access ------------------------------------------------

// Streaming load of data that is read once (evict-first in L1/L2).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
// Load through the read-only path (data reused across CTAs, e.g. weights).
__device__ __forceinline__ uint4 ld_ro(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(w[q] << 16);
        f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ uint4 pack8_rn(const float (&f)[8]) {
    return make_uint4(pack2_rn(f[0], f[1]), pack2_rn(f[2], f[3]), pack2_rn(f[4], f[5]),
                      pack2_rn(f[6], f[7]));
}

// ---- step (1): post --------------------------------------------------------
// R'[i][h] = post[i] * Y[h] + sum_{j=0..3} comb[j][i] * R[j][h], fp32 fma chain
// in this order, then round to nearest even bf16.  out[i] is the rounded
// stream i as bf16 bits; rf[i][e] the rounded values widened back to fp32.
__device__ __forceinline__ void post_vec8(const uint4 (&r)[kHC], uint4 y, const float *comb /*[4][4]*/,
                                          const float *post /*[4]*/, uint4 (&out)[kHC],
                                          float (&rf)[kHC][8]) {
    float R[kHC][8], Y[8];
#pragma unroll
    for (int j = 0; j < kHC; ++j) unpack8(r[j], R[j]);
    unpack8(y, Y);
#pragma unroll
    for (int i = 0; i < kHC; ++i) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = post[i] * Y[e];
#pragma unroll
        for (int j = 0; j < kHC; ++j) {
            const float c = comb[j * kHC + i];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(c, R[j][e], acc[e]);
        }
        out[i] = pack8_rn(acc);
        unpack8(out[i], rf[i]);
    }
}

// Same arithmetic as post_vec8 on packed fp32 pairs (__fmul2_rn/__ffma2_rn), with the
// layer output given as 8 fp32 values: each half of a packed operation is the same IEEE
// operation, so the results are bit-identical to post_vec8; half the instructions.
__device__ __forceinline__ void post_vec8_yf(const uint4 (&r)[kHC], const float (&Y)[8], const float *comb,
                                             const float *post, uint4 (&out)[kHC], float (&rf)[kHC][8]) {
    float R[kHC][8];
#pragma unroll
    for (int j = 0; j < kHC; ++j) unpack8(r[j], R[j]);
#pragma unroll
    for (int i = 0; i < kHC; ++i) {
        float acc[8];
        const float2 p2 = make_float2(post[i], post[i]);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float2 a2 = __fmul2_rn(p2, make_float2(Y[e], Y[e + 1]));
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                const float c = comb[j * kHC + i];
                a2 = __ffma2_rn(make_float2(c, c), make_float2(R[j][e], R[j][e + 1]), a2);
            }
            acc[e] = a2.x;
            acc[e + 1] = a2.y;
        }
        out[i] = pack8_rn(acc);
        unpack8(out[i], rf[i]);
    }
}
__device__ __forceinline__ void post_vec8_x2(const uint4 (&r)[kHC], uint4 y, const float *comb,
                                             const float *post, uint4 (&out)[kHC], float (&rf)[kHC][8]) {
    float Y[8];
    unpack8(y, Y);
    post_vec8_yf(r, Y, comb, post, out, rf);
}

// ---- step (4): combine ------------------------------------------------------
// X[h] = sum_i pre[i] * R'[i][h], fp32: pre0*R0, then fma with i = 1, 2, 3.
__device__ __forceinline__ void combine_vec8(const float (&rf)[kHC][8], const float (&pre)[kHC],
                                             float (&x)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float a = pre[0] * rf[0][e];
        a = fmaf(pre[1], rf[1][e], a);
        a = fmaf(pre[2], rf[2][e], a);
        a = fmaf(pre[3], rf[3][e], a);
        x[e] = a;
    }
}

// combine_vec8 on packed fp32 pairs; bit-identical to combine_vec8.
__device__ __forceinline__ void combine_vec8_x2(const float (&rf)[kHC][8], const float (&pre)[kHC],
                                                float (&x)[8]) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float2 a = __fmul2_rn(make_float2(pre[0], pre[0]), make_float2(rf[0][e], rf[0][e + 1]));
        a = __ffma2_rn(make_float2(pre[1], pre[1]), make_float2(rf[1][e], rf[1][e + 1]), a);
        a = __ffma2_rn(make_float2(pre[2], pre[2]), make_float2(rf[2][e], rf[2][e + 1]), a);
        a = __ffma2_rn(make_float2(pre[3], pre[3]), make_float2(rf[3][e], rf[3][e + 1]), a);
        x[e] = a.x;
        x[e + 1] = a.y;
    }
}

// out[h] = bf16((X[h] * rstd) * gamma[h])
__device__ __forceinline__ uint4 norm_vec8(const float (&x)[8], float rstd, uint4 g) {
    float G[8], o[8];
    unpack8(g, G);
    // packed fp32 multiplies: each half is the same IEEE product as the scalar form
    const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 v = __fmul2_rn(__fmul2_rn(make_float2(x[e], x[e + 1]), r2), make_float2(G[e], G[e + 1]));
        o[e] = v.x;
        o[e + 1] = v.y;
    }
    return pack8_rn(o);
}

// ---- MXFP8 form of the layer input -----------------------------------------
// Blocks of 32 consecutive hidden values of a token: E4M3 codes of x / 2^E and the
// scale byte E + 127, with E from the block's largest magnitude (mode 0:
// floor(log2 amax) - 8; mode 1: the smallest E with amax <= 448 * 2^E; zero or
// subnormal amax: -127).  The values quantized are the bf16 outputs.
struct MxOut {
    uint8_t *q;      // [T][H] E4M3 codes (nullptr: no MXFP8 output)
    uint8_t *scale;  // scale bytes in the 128 x 4 tile layout
    int mode;
};

__device__ __forceinline__ int mx_exp(float amax, int mode) {
    const uint32_t u = __float_as_uint(amax);
    const int ef = (int)((u >> 23) & 0xFFu);
    if (ef == 0) return -127;
    int E = ef - 127 - 8;
    if (mode == 1 && (u & 0x7FFFFFu) > 0x600000u) E += 1;  // significand above 1.75
    return E < -127 ? -127 : (E > 127 ? 127 : E);
}

// Byte offset of (token m, block k) in the 128 x 4 tile layout of the scales, as the sum of
// a token part and a block part.
__device__ __forceinline__ int64_t mx_scale_row(int64_t m, int H) {
    const int kt = (H / 32 + 3) / 4;
    return (m / 128) * kt * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4;
}
__device__ __forceinline__ int mx_scale_col(int k) { return (k / 4) * 512 + (k % 4); }
__device__ __forceinline__ int64_t mx_scale_offset(int64_t m, int k, int H) {
    return mx_scale_row(m, H) + mx_scale_col(k);
}

// Quantizes the 8 bf16 outputs `o` held by this lane; the four lanes lane ^ 1, lane ^ 2 of
// an aligned group of four hold one block (consecutive vectors).  Every lane of the warp
// must call it (inactive lanes with active = false).  Writes the 8 codes at q_dst and, from
// the group's first lane, the scale byte at scale_dst.
__device__ __forceinline__ void mx_quantize8(uint4 o, bool active, int mode, uint8_t *q_dst,
                                             uint8_t *scale_dst) {
    float x[8];
    unpack8(o, x);
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    if (!active) amax = 0.f;
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!active) return;
    const int E = mx_exp(amax, mode);
    const float m = __uint_as_float((uint32_t)(127 - E) << 23);  // 2^-E (E <= 120 for finite bf16)
    const float2 m2 = make_float2(m, m);
    uint32_t w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)  // exact products (a power of two), then one rounding to E4M3
        w[p] = (uint32_t)__nv_cvt_float2_to_fp8x2(__fmul2_rn(make_float2(x[2 * p], x[2 * p + 1]), m2),
                                                   __NV_SATFINITE, __NV_E4M3);
    __stcs(reinterpret_cast<uint2 *>(q_dst), make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16)));
    if (((threadIdx.x & 31) & 3) == 0) *scale_dst = (uint8_t)(E + 127);
}

// One block of 32 as four vectors o[0..3]: its 32 E4M3 codes in 8 words (vector k in words
// 2k, 2k + 1) and, returned, the scale byte.
__device__ __forceinline__ uint8_t mx_quantize_block32(const uint4 (&o)[4], int mode, uint32_t (&w)[8]) {
    float x[4][8];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        unpack8(o[k], x[k]);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[k][e]));
    }
    const int E = mx_exp(amax, mode);
    const float m = __uint_as_float((uint32_t)(127 - E) << 23);
    const float2 m2 = make_float2(m, m);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t h[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            h[p] = (uint32_t)__nv_cvt_float2_to_fp8x2(__fmul2_rn(make_float2(x[k][2 * p], x[k][2 * p + 1]), m2),
                                                       __NV_SATFINITE, __NV_E4M3);
        w[2 * k] = h[0] | (h[1] << 16);
        w[2 * k + 1] = h[2] | (h[3] << 16);
    }
    return (uint8_t)(E + 127);
}

// One block of 32 held by one lane as four vectors o[k] (vector j[k] of the block, any
// order): E4M3 codes to q_block + 8 * j[k], scale byte to *scale_dst.
__device__ __forceinline__ void mx_quantize_block(const uint4 (&o)[4], const int (&j)[4], int mode,
                                                  uint8_t *q_block, uint8_t *scale_dst) {
    uint32_t w[8];
    const uint8_t sb = mx_quantize_block32(o, mode, w);
#pragma unroll
    for (int k = 0; k < 4; ++k) __stcs(reinterpret_cast<uint2 *>(q_block + 8 * j[k]), make_uint2(w[2 * k], w[2 * k + 1]));
    *scale_dst = sb;
}

// ---- step (3): heads and Sinkhorn, one warp per token -----------------------
// pre[i] = sigmoid(alpha_pre * z[i] + bias[i]), the product-add fused.
__device__ __forceinline__ float pre_value(float z, float alpha_pre, float b) {
    return 1.f / (1.f + expf(-fmaf(alpha_pre, z, b)));
}
// Input: lane n holds the finished logit z[n] for n = 0..23 (other lanes are
// ignored).  pre_head: lanes 0-3 return pre[lane] (the rest 0).
__device__ __forceinline__ float pre_head(float z, const float *bias, const float *mix_scales) {
    const int lane = threadIdx.x & 31;
    return lane < 4 ? pre_value(z, mix_scales[0], bias[lane]) : 0.f;
}
// r = 1 / sqrt(mean of the 4H squares + eps) from the square sum.
__device__ __forceinline__ float hc_rsqrt(float sumsq, int H, float eps) {
    return 1.f / sqrtf(sumsq / (float)(kHC * H) + eps);
}

// Hardware reciprocal approximation (rcp.approx.ftz.f32, within 1 ulp).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sinkhorn normalisation of one positive 4x4 matrix held in registers
// (row-major M[4a+c]): sinkhorn_iters times, each row then each column is
// multiplied by the reciprocal of (sum + sinkhorn_eps); sums are taken in the
// order ((m0 + m1) + (m2 + m3)).  The hardware reciprocal keeps the dependent
// chain short (the correctly rounded one is a long instruction sequence); its
// error is within 1 ulp per step.
__device__ __forceinline__ void sinkhorn16(float (&M)[16], const Scalars &s) {
    for (int it = 0; it < s.sinkhorn_iters; ++it) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float inv = rcp_approx(((M[4 * a] + M[4 * a + 1]) + (M[4 * a + 2] + M[4 * a + 3])) + s.sinkhorn_eps);
#pragma unroll
            for (int c = 0; c < 4; ++c) M[4 * a + c] *= inv;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float inv = rcp_approx(((M[c] + M[4 + c]) + (M[8 + c] + M[12 + c])) + s.sinkhorn_eps);
#pragma unroll
            for (int a = 0; a < 4; ++a) M[4 * a + c] *= inv;
        }
    }
}

// post and residual-mix heads.  Lanes 4-7 return post[lane-4]; lanes 8-23
// return the Sinkhorn-normalised residual mix entry e = lane - 8 (row a = e/4,
// column c = e%4).  Every lane gathers the 16 logits and runs sinkhorn16 on
// the whole 4x4 matrix in registers.
__device__ __forceinline__ float post_and_sinkhorn(float z, const float *bias, const float *mix_scales,
                                                   const Scalars &s) {
    const int lane = threadIdx.x & 31;
    const float a_res = mix_scales[2];
    float M[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float ze = __shfl_sync(0xffffffffu, z, 8 + e);
        M[e] = expf(a_res * ze + bias[8 + e]);
    }
    sinkhorn16(M, s);
    float v = 0.f;
    if (lane >= 4 && lane < 8) v = s.hc_post_scale / (1.f + expf(-(mix_scales[1] * z + bias[lane])));
#pragma unroll
    for (int e = 0; e < 16; ++e)
        if (lane == 8 + e) v = M[e];
    return v;
}

// All three heads: lanes 0-3 pre, 4-7 post, 8-23 residual mix.
__device__ __forceinline__ float heads_and_sinkhorn(float z, const float *bias, const float *mix_scales,
                                                    const Scalars &s) {
    const int lane = threadIdx.x & 31;
    const float p = pre_head(z, bias, mix_scales);
    const float q = post_and_sinkhorn(z, bias, mix_scales, s);
    return lane < 4 ? p : q;
}

// ---- step (4): the square sum of X from the Gram matrix --------------------
// The fused schedules take sum_h X^2 as pre^T G pre, G the Gram matrix of the four bf16
// streams (G_ij = sum_h R'_i[h] R'_j[h], accumulated in fp32).  Its rounding error is a
// small multiple k of 2^-24 * sum_ij pre_i pre_j |G_ij| <= (sum_i pre_i sqrt(G_ii))^2
// <= 4 D, D = sum_i pre_i^2 G_ii (Cauchy-Schwarz twice).  When the streams cancel in X
// (anti-correlated streams with similar pre weights) pre^T G pre is a small difference of such
// terms and loses its accuracy; gram_cancels() flags a token whose result is below D / 16, and
// the schedules then sum X^2 over the combined row directly.  Above the threshold the relative
// error of the Gram form stays below 64 k 2^-24 (far below a bf16 ulp of the output).
// Independent streams give pre^T G pre / D ~ 1 (up to O(H^-1/2)), identical ones >= 1.  No
// square root: the test sits on the latency-bound path of the small schedule.
constexpr float kGramCancel = 1.f / 16.f;
__device__ __forceinline__ bool gram_cancels(float sx, const float (&pre)[kHC], const float *G /*diagonal 0..3*/) {
    const float d = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] + pre[3] * pre[3] * G[3];
    return sx < kGramCancel * d;
}

// Deterministic warp sum (fixed xor-tree order).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The layer input of token t redone with a direct square sum (the fix-up of a token whose streams
// cancel in X, see gram_cancels), by one warp: X from the updated residual Rp (the combine's fp32
// expression), sum_h X^2 summed by each lane over its blocks of 32 values in order and then an
// xor tree, the RMSNorm with that rstd, the bf16 row (when X_out is given) and its MXFP8 form (when
// mx.q is given; H % 32 == 0).
__device__ __forceinline__ void redo_token(const uint16_t *__restrict__ Rp, const uint16_t *__restrict__ gamma,
                                           float rmsnorm_eps, int H, const float *__restrict__ pre_out,
                                           uint16_t *__restrict__ X_out, const MxOut &mx, int64_t t) {
    const int lane = threadIdx.x & 31;
    const int nb32 = (H + 31) / 32;  // blocks of 32 values: block b holds vectors 4b .. 4b+3
    // R' and pre through L2 only (the token-tile kernel redoes tokens whose R' and pre other CTAs of
    // its own grid wrote)
    const uint16_t *row = Rp + t * kHC * (int64_t)H;
    const float4 p4 = __ldcg(reinterpret_cast<const float4 *>(pre_out + t * 4));
    const float pre[kHC] = {p4.x, p4.y, p4.z, p4.w};
    auto xvec = [&](int v, float (&x)[8]) {
        float rf[kHC][8];
#pragma unroll
        for (int j = 0; j < kHC; ++j) unpack8(__ldcg(reinterpret_cast<const uint4 *>(row + (int64_t)j * H + v * kVec)), rf[j]);
        combine_vec8_x2(rf, pre, x);
    };
    float a = 0.f;
    for (int b = lane; b < nb32; b += 32) {
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
    const float rstd = __frsqrt_rn(fmaxf(a, 0.f) * (1.f / (float)H) + rmsnorm_eps);
    for (int b = lane; b < nb32; b += 32) {
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

}  // namespace mhc
