// Small-T schedule (schedule "small"): the whole mHC post+pre step in one
// launch for decode-sized calls (T <= 128 while the shared memory fits: eight 16-token
// tiles for the eight warps of the projection), built for latency rather than bandwidth.
//
// The hidden dimension is split across up to one CTA per SM (slices of Hs
// values, a multiple of 8; Hs = 64 at H = 7168, 112 CTAs).  CTA c:
//   1. post: R' of its slice for all T tokens (same fp32 expression as every
//      other schedule), kept in shared memory and written to HBM; its slice of
//      phi (fp32, 4*Hs rows), of gamma and the previous mixes arrive by bulk
//      copies issued first;
//   2. per token, the 24 projection partials over the slice on the tensor
//      cores (mma.sync bf16: R' is exact in bf16, phi is split into a bf16 high
//      part and a bf16 remainder, fp32 accumulation), and the 10 Gram-matrix
//      partials R'_i . R'_j in fp32, to workspace records;
//   3. grid barrier (bounded in time; the launch is cooperative, so every CTA
//      is resident);
//   4. every CTA bulk-copies the pre-logit and Gram part of every record into
//      shared memory and sums it over the CTAs in one fixed order, so all CTAs
//      hold identical r, pre and rstd (sum_h X^2 = pre^T G pre);
//   5. combine + RMSNorm of its slice from the R' in shared memory;
//   meanwhile warp 0 of CTA c < T bulk-copies token c's other 20 logits and sums
//   them; below 16 tokens it computes r and takes the pre logits from phase 4's sums
//   (signalled as soon as they are in, before the workers' rstd), from 16 tokens it
//   sums the token's heads itself in phase 4's order (the same bits, without waiting
//   for phase 4's sums over every token); then it finishes its mixes (pre, post,
//   Sinkhorn residual mix), so the Sinkhorn runs beside phase 5.
// phi is used in fp32 directly (no packing launch) and nothing is re-read from
// HBM, so a call is a single launch.
//
// Workspace records, token-major so that one bulk copy fetches a token's (or a
// token chunk's) records of every CTA:
//   heads [T][nc][16]: pre logits 0..3, Gram entries (0,0) (1,1) (2,2) (3,3)
//                      (0,1) (0,2) (0,3) (1,2) (1,3) (2,3), two zeros;
//   tails [T][nc][24]: logits 4..23, four zeros;
//   then [T][nc] floats: each CTA's share of sum_h X^2 for tokens whose streams cancel in X
//   (written and read only when gram_cancels flags a token).
#include <cstdint>

#include "mhc_device.cuh"
#include "mhc_kernels.h"
#include "sm100_ptx.cuh"

namespace mhc {

namespace {

using namespace ptx;

constexpr int kSNT = 256;  // threads per CTA
constexpr int kHead = 16, kTail = 24;  // floats per record head / tail
constexpr uint64_t kSpinLimitNs = 1000000000ull;
constexpr int kBigBytes = 100 * 1024;  // shared memory for one token chunk of record heads
constexpr size_t kSmallSmemLimit = 227 * 1024;
// From this many tokens the owner warp sums its token's heads itself (graph-replayed, H = 7168:
// T = 32 12.4 us against 14.0 us taking the workers' sums; T = 6 9.1 against 8.7 us).
constexpr int kOwnHeadsMinT = 16;
constexpr int kMaxCtas = 160;  // CTAs at most (one per SM)

// Tokens per chunk of the phase-4 reduction (the heads of nc records each), at most 16.
__host__ __device__ inline int small_chunk(int T, int nc) {
    int tc = kBigBytes / (nc * kHead * 4);
    if (tc < 1) tc = 1;
    if (tc > 16) tc = 16;
    return tc < T ? tc : T;
}

struct SmallSmem {
    int T, Hs, nc;
    __host__ __device__ int tpad() const { return (T + 15) / 16 * 16; }
    __host__ __device__ int rs() const { return kHC * Hs + 8; }  // R' row stride (elements), padded
    __host__ __device__ size_t bar_off() const { return 0; }      // 4 mbarriers
    __host__ __device__ size_t comb_off() const { return 64; }    // [T][16] fp32
    __host__ __device__ size_t post_off() const { return comb_off() + (size_t)T * 64; }  // [T][4]
    __host__ __device__ size_t rp_off() const { return post_off() + (size_t)T * 16; }    // [tpad][rs] bf16
    __host__ __device__ size_t phi_off() const { return rp_off() + (size_t)tpad() * rs() * 2; }    // [4Hs][24] fp32
    __host__ __device__ size_t gam_off() const { return phi_off() + (size_t)kHC * Hs * kNumMix * 4; }  // [Hs] bf16
    __host__ __device__ size_t pp_off() const { return gam_off() + (size_t)Hs * 2; }         // [8 warps][16][24]
    __host__ __device__ size_t gram_off() const { return pp_off() + 8 * 16 * kNumMix * 4; }  // [T][10]
    __host__ __device__ size_t big_off() const {  // [tc][nc][16]
        return gram_off() + (((size_t)T * 10 * 4 + 15) & ~size_t(15));
    }
    __host__ __device__ size_t ownt_off() const {  // [nc][24]
        return big_off() + (size_t)small_chunk(T, nc) * nc * kHead * 4;
    }
    __host__ __device__ size_t ownh_off() const { return ownt_off() + (size_t)nc * kTail * 4; }  // [nc][16]
    __host__ __device__ size_t sums_off() const { return ownh_off() + (size_t)nc * kHead * 4; }  // [T][16]
    __host__ __device__ size_t st_off() const { return sums_off() + (size_t)T * 16 * 4; }        // [T][8]
    __host__ __device__ size_t tl_off() const { return st_off() + (size_t)T * 8 * 4; }           // [32]
    __host__ __device__ size_t flag_off() const { return tl_off() + 32 * 4; }
    __host__ __device__ size_t bytes() const { return flag_off() + 16; }
};

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
// Two fp32 values -> bf16 high parts (low half = first) and bf16 remainders.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack2_rn(x0, x1);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
    lo = pack2_rn(x0 - h0, x1 - h1);
}

// Warp-wide sum over the CTAs of 16 adjacent values, src[q * stride + 0..15] for CTA
// q < nc (16-byte aligned rows).  Lane (quad j4 = lane & 3, group g = lane >> 2) adds
// CTAs q = g, g + 8, g + 16, ... in that order from zero (its loads issued together,
// slots past the last CTA adding zero); then an xor tree over the eight groups.  Every
// lane returns the total of its quad, bit-identical across the lanes that share the quad
// (each tree step adds the same two values) and across CTAs.  quads < 4 limits the
// quads read.
__device__ __forceinline__ float4 warp_cta_sum16(const float *src, int stride, int nc, int quads) {
    const int lane = threadIdx.x & 31, j4 = lane & 3, g = lane >> 2;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kPer = kMaxCtas / 8, kHalf = kPer / 2;
#pragma unroll
    for (int h = 0; h < kPer; h += kHalf) {
        float4 v[kHalf];
#pragma unroll
        for (int i = 0; i < kHalf; ++i) {
            const int q = g + 8 * (h + i);
            v[i] = q < nc && j4 < quads ? *reinterpret_cast<const float4 *>(src + (size_t)q * stride + 4 * j4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kHalf; ++i) a = add4(a, v[i]);
    }
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
        float4 o;
        o.x = __shfl_xor_sync(0xffffffffu, a.x, m);
        o.y = __shfl_xor_sync(0xffffffffu, a.y, m);
        o.z = __shfl_xor_sync(0xffffffffu, a.z, m);
        o.w = __shfl_xor_sync(0xffffffffu, a.w, m);
        a = add4(a, o);
    }
    return a;
}

template <bool kPost, bool kMx>
__global__ void __launch_bounds__(kSNT, 1)
small_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y, const float *__restrict__ prev_post,
             const float *__restrict__ prev_comb, const float *__restrict__ phi, const float *__restrict__ bias,
             const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma, Scalars sc, int T, int H,
             int Hs, uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out, float *__restrict__ pre_out,
             float *__restrict__ post_out, float *__restrict__ res_out, float *__restrict__ part,
             unsigned int *__restrict__ ctrl, MxOut mx, int split) {
    extern __shared__ __align__(128) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, nc = gridDim.x;
    const SmallSmem L{T, Hs, nc};
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar_off());  // 0 mixes+gamma, 1 phi, 2 heads, 3 owner
    float *sComb = reinterpret_cast<float *>(sm + L.comb_off());
    float *sPost = reinterpret_cast<float *>(sm + L.post_off());
    uint16_t *sRp = reinterpret_cast<uint16_t *>(sm + L.rp_off());
    float *sPhi = reinterpret_cast<float *>(sm + L.phi_off());
    uint16_t *sGam = reinterpret_cast<uint16_t *>(sm + L.gam_off());
    float *sPP = reinterpret_cast<float *>(sm + L.pp_off());
    float *sGram = reinterpret_cast<float *>(sm + L.gram_off());
    float *sBig = reinterpret_cast<float *>(sm + L.big_off());
    float *sOwnT = reinterpret_cast<float *>(sm + L.ownt_off());
    float *sOwnH = reinterpret_cast<float *>(sm + L.ownh_off());
    float *sSums = reinterpret_cast<float *>(sm + L.sums_off());
    float *sSt = reinterpret_cast<float *>(sm + L.st_off());
    float *sTl = reinterpret_cast<float *>(sm + L.tl_off());
    int *sFlag = reinterpret_cast<int *>(sm + L.flag_off());
    const int RS = L.rs();
    const int h0 = c * Hs;
    const int nvec = Hs / kVec;
    const int hv = H - h0 < Hs ? H - h0 : Hs;  // valid hidden values of the slice (> 0, a multiple of 8)
    float *heads = part;                           // [T][nc][16]
    float *tails = part + (size_t)T * nc * kHead;  // [T][nc][24]
    bool dead = false;

    // ---- bulk copies: mixes + gamma (barrier 0), phi slice rows j*H + h0 .. (barrier 1)
    if (tid == 0) {
        sFlag[1] = 0;  // tokens flagged by gram_cancels
#pragma unroll
        for (int b = 0; b < 4; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], (kPost ? T * 80u : 0u) + hv * 2u);
        if (kPost) {
            bulk_g2s(sComb, prev_comb, T * 64u, &bars[0]);
            bulk_g2s(sPost, prev_post, T * 16u, &bars[0]);
        }
        bulk_g2s(sGam, gamma + h0, hv * 2u, &bars[0]);
        mbar_arrive_expect_tx(&bars[1], kHC * hv * 96u);
#pragma unroll
        for (int j = 0; j < kHC; ++j)
            bulk_g2s(sPhi + (size_t)j * Hs * kNumMix, phi + ((size_t)j * H + h0) * kNumMix, hv * 96u, &bars[1]);
    }
    if (hv < Hs)  // rows of the last slice beyond H: zero
        for (int i = tid; i < kHC * (Hs - hv) * 6; i += kSNT) {
            const int j = i / ((Hs - hv) * 6), r = i % ((Hs - hv) * 6);
            *reinterpret_cast<float4 *>(sPhi + ((size_t)j * Hs + hv) * kNumMix + 4 * r) =
                make_float4(0.f, 0.f, 0.f, 0.f);
        }

    // ---- 1. R' of the slice (zero beyond H), to shared memory and HBM.  The first item's rows
    // are loaded before waiting for the mixes.
    {
        uint4 r4[kHC], y4 = make_uint4(0u, 0u, 0u, 0u);
        const bool first_valid = tid < T * nvec && (tid % nvec) * kVec < hv;
        if (first_valid) {
            const int t = tid / nvec, v = tid % nvec;
            const size_t base = (size_t)t * kHC * H + h0 + v * kVec;
#pragma unroll
            for (int j = 0; j < kHC; ++j) r4[j] = ld_stream(R + base + (size_t)j * H);
            if (kPost) y4 = ld_stream(Y + (size_t)t * H + h0 + v * kVec);
        }
        __syncthreads();  // barrier initialisation visible to every thread
        mbar_wait_timed(&bars[0], 0, dead, kSpinLimitNs);
        for (int item = tid; item < T * nvec; item += kSNT) {
            const int t = item / nvec, v = item % nvec;
            const size_t base = (size_t)t * kHC * H + h0 + v * kVec;
            uint4 o[kHC];
            if (v * kVec < hv) {
                if (item != tid) {
#pragma unroll
                    for (int j = 0; j < kHC; ++j) r4[j] = ld_stream(R + base + (size_t)j * H);
                    if (kPost) y4 = ld_stream(Y + (size_t)t * H + h0 + v * kVec);
                }
                if (kPost) {
                    float rf[kHC][8];
                    post_vec8_x2(r4, y4, sComb + t * 16, sPost + t * 4, o, rf);
#pragma unroll
                    for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (size_t)i * H, o[i]);
                } else {
#pragma unroll
                    for (int j = 0; j < kHC; ++j) o[j] = r4[j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < kHC; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < kHC; ++j)
                *reinterpret_cast<uint4 *>(sRp + (size_t)t * RS + j * Hs + v * kVec) = o[j];
        }
        mbar_wait_timed(&bars[1], 0, dead, kSpinLimitNs);
        __syncthreads();
    }

    // ---- 2a. projection partials on the tensor cores: warp w takes m-tile (16 tokens) w / KW and
    // the K-steps (16 rows of the 4*Hs) of share w % KW; its 16 x 24 result goes to sPP[w].
    const int n_mt = (T + 15) / 16, KW = 8 / n_mt;
    {
        const int mt = warp / KW, kw = warp % KW;
        if (mt < n_mt) {
            const int nks = Hs / 4;  // 4*Hs / 16
            const int k0 = kw * nks / KW, k1 = (kw + 1) * nks / KW;
            float acc[3][4];
#pragma unroll
            for (int n = 0; n < 3; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
            const uint16_t *arow = sRp + (size_t)(mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 8 * (lane >> 4);
            const int kr = (lane & 3) * 2, nn = lane >> 2;
#pragma unroll 2
            for (int ks = k0; ks < k1; ++ks) {
                uint32_t a[4];
                ldsm_x4(arow + ks * 16, a);
                const float *pb = sPhi + (size_t)(ks * 16 + kr) * kNumMix + nn;
                float b[3][4];
#pragma unroll
                for (int n = 0; n < 3; ++n) {
                    b[n][0] = pb[8 * n];
                    b[n][1] = pb[kNumMix + 8 * n];
                    b[n][2] = pb[8 * kNumMix + 8 * n];
                    b[n][3] = pb[9 * kNumMix + 8 * n];
                }
#pragma unroll
                for (int n = 0; n < 3; ++n) {
                    uint32_t h01, l01, h89, l89;
                    split2(b[n][0], b[n][1], h01, l01);
                    split2(b[n][2], b[n][3], h89, l89);
                    mma16816(acc[n], a, h01, h89);
                    mma16816(acc[n], a, l01, l89);
                }
            }
            float *dst = sPP + (size_t)warp * 16 * kNumMix;
#pragma unroll
            for (int n = 0; n < 3; ++n) {
                const int col = 8 * n + kr;
                *reinterpret_cast<float2 *>(dst + nn * kNumMix + col) = make_float2(acc[n][0], acc[n][1]);
                *reinterpret_cast<float2 *>(dst + (nn + 8) * kNumMix + col) = make_float2(acc[n][2], acc[n][3]);
            }
        }
    }
    // ---- 2b. Gram partials in fp32: items (t, entry e), spread over the warps
    {
        constexpr uint64_t kIa = 0x2110003210ull, kIb = 0x3323213210ull;  // entry e -> (ia, ib), nibble e
        for (int p = lane * 8 + warp; p < T * 10; p += kSNT) {
            const int t = p / 10, e = p % 10;
            const int ia = (int)(kIa >> (4 * e)) & 15, ib = (int)(kIb >> (4 * e)) & 15;
            const uint16_t *ri = sRp + (size_t)t * RS + ia * Hs, *rj = sRp + (size_t)t * RS + ib * Hs;
            float2 acc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
            for (int u0 = 0; u0 < nvec; u0 += 4) {  // four vectors' loads issued together
                uint4 va[4], vb[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool in = u0 + k < nvec;
                    va[k] = in ? *reinterpret_cast<const uint4 *>(ri + 8 * (u0 + k)) : make_uint4(0u, 0u, 0u, 0u);
                    vb[k] = in ? *reinterpret_cast<const uint4 *>(rj + 8 * (u0 + k)) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float a[8], b[8];
                    unpack8(va[k], a);
                    unpack8(vb[k], b);
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        acc[k] = __ffma2_rn(make_float2(a[e], a[e + 1]), make_float2(b[e], b[e + 1]), acc[k]);
                }
            }
            sGram[p] = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
        }
    }
    __syncthreads();
    // ---- 2c. this CTA's records: K-shares of the projection in order, Gram entries
    for (int i = tid; i < T * 40; i += kSNT) {
        const int t = i / 40, s = i % 40;
        float a = 0.f;
        int n = -1;  // logit held in this slot
        if (s < 4) n = s;
        else if (s >= 16 && s < 36) n = s - 12;
        if (n >= 0) {  // the K-shares in order (loads issued together; shares past KW add zero)
            const int mt = t >> 4, row = t & 15;
            float v[8];
#pragma unroll
            for (int kw = 0; kw < 8; ++kw) v[kw] = kw < KW ? sPP[((size_t)(mt * KW + kw) * 16 + row) * kNumMix + n] : 0.f;
#pragma unroll
            for (int kw = 0; kw < 8; ++kw) a += v[kw];
        } else if (s >= 4 && s < 14) {
            a = sGram[t * 10 + s - 4];
        }
        if (s < kHead) heads[((size_t)t * nc + c) * kHead + s] = a;
        else tails[((size_t)t * nc + c) * kTail + s - kHead] = a;
    }

    // ---- 3. every CTA's records are in
    __syncthreads();
    if (tid == 0)
        sFlag[0] = grid_barrier(reinterpret_cast<unsigned long long *>(ctrl + kSmallBarrierWord), (unsigned int)nc,
                                kSpinLimitNs) ? 1 : 0;
    __syncthreads();
    if (!sFlag[0]) {
        if (tid == 0) atomicOr(ctrl, 1u);
        return;
    }

    // split: no owner warps; the post and residual mixes are left to small_tail_kernel
    const bool owner_cta = !split && c < T;
    // the owner warp sums its token's heads itself from kOwnHeadsMinT tokens on; with fewer, the
    // workers' sums over every token are done sooner than its own copy, and it takes theirs
    const bool own_heads = T >= kOwnHeadsMinT;
    if (owner_cta && warp == 0) {
        // ---- token c (and c + nc, ...): its records summed over the CTAs here (the heads in the
        // workers' order and arithmetic, so r and the pre logits are the same bits as theirs,
        // without waiting for their sums over every token); heads and the Sinkhorn mix.
        int it = 0;
        for (int t = c; t < T; t += nc, ++it) {
            if (lane == 0) {
                fence_proxy_async_global();
                if (it > 0) fence_proxy_async_smem();  // the previous token's reads of the buffer are done
                mbar_arrive_expect_tx(&bars[3], nc * (own_heads ? kTail + kHead : kTail) * 4u);
                bulk_g2s(sOwnT, tails + (size_t)t * nc * kTail, nc * kTail * 4u, &bars[3]);
                if (own_heads) bulk_g2s(sOwnH, heads + (size_t)t * nc * kHead, nc * kHead * 4u, &bars[3]);
            }
            mbar_wait_timed(&bars[3], it & 1, dead, kSpinLimitNs);
            float zpre = 0.f, r = 0.f;
            {
                const float4 a = warp_cta_sum16(sOwnT, kTail, nc, 4);       // logits 4..19
                const float4 b = warp_cta_sum16(sOwnT + 16, kTail, nc, 1);  // logits 20..23
                if (lane < 4) *reinterpret_cast<float4 *>(sTl + 4 * lane) = a;
                if (lane == 0) *reinterpret_cast<float4 *>(sTl + 16) = b;
                if (own_heads) {
                    // lane j holds quad j: pre logits (quad 0), Gram diagonal (quad 1)
                    const float4 h = warp_cta_sum16(sOwnH, kHead, nc, 2);
                    const float g0 = __shfl_sync(0xffffffffu, h.x, 1), g1 = __shfl_sync(0xffffffffu, h.y, 1),
                                g2 = __shfl_sync(0xffffffffu, h.z, 1), g3 = __shfl_sync(0xffffffffu, h.w, 1);
                    r = hc_rsqrt((g0 + g1) + (g2 + g3), H, sc.hc_norm_eps);
                    const float p0 = __shfl_sync(0xffffffffu, h.x, 0), p1 = __shfl_sync(0xffffffffu, h.y, 0),
                                p2 = __shfl_sync(0xffffffffu, h.z, 0), p3 = __shfl_sync(0xffffffffu, h.w, 0);
                    zpre = lane == 0 ? p0 : (lane == 1 ? p1 : (lane == 2 ? p2 : p3));
                }
            }
            __syncwarp();
            const float tl = lane >= 4 && lane < kNumMix ? sTl[lane - 4] : 0.f;  // lane n: logit n
            if (!own_heads) {
                if (it == 0) asm volatile("bar.sync 2, %0;" ::"r"(kSNT) : "memory");  // workers' sums are in
                // r as the workers compute it, from the same sums (the same bits)
                const float *sm16 = sSums + t * 16;
                r = hc_rsqrt((sm16[4] + sm16[5]) + (sm16[6] + sm16[7]), H, sc.hc_norm_eps);
                zpre = lane < 4 ? sm16[lane] : 0.f;
            }
            const float z = r * (lane < 4 ? zpre : tl);
            const float v = heads_and_sinkhorn(z, bias, mix_scales, sc);
            if (lane < 4) pre_out[(size_t)t * 4 + lane] = v;
            else if (lane < 8) post_out[(size_t)t * 4 + lane - 4] = v;
            else if (lane < kNumMix) res_out[(size_t)t * 16 + lane - 8] = v;
            __syncwarp();
        }
        if (dead && lane == 0) atomicOr(ctrl, 1u);
        return;
    }

    // ---- 4. workers (every warp but an owner CTA's warp 0): pre logits and Gram entries of every
    // token summed over the CTAs, in token chunks whose record heads are bulk-copied into shared
    // memory first.
    const int wbase = owner_cta ? 32 : 0, nwork = kSNT - wbase, wt = tid - wbase;
    auto wsync = [&]() { asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory"); };
    {
        const int TC = small_chunk(T, nc);
        int it = 0;
        for (int tc0 = 0; tc0 < T; tc0 += TC, ++it) {
            const int tcn = T - tc0 < TC ? T - tc0 : TC;
            if (wt == 0) {
                fence_proxy_async_global();
                if (it > 0) fence_proxy_async_smem();  // the previous chunk's reads of sBig are done
                mbar_arrive_expect_tx(&bars[2], tcn * nc * kHead * 4u);
                bulk_g2s(sBig, heads + (size_t)tc0 * nc * kHead, tcn * nc * kHead * 4u, &bars[2]);
            }
            mbar_wait_timed(&bars[2], it & 1, dead, kSpinLimitNs);
            // one warp per token of the chunk
            for (int tt = wt >> 5; tt < tcn; tt += nwork >> 5) {
                const float4 a = warp_cta_sum16(sBig + (size_t)tt * nc * kHead, kHead, nc, 4);
                if (lane < 4) *reinterpret_cast<float4 *>(sSums + (tc0 + tt) * 16 + 4 * lane) = a;
            }
            wsync();
        }
    }
    // the owner warp needs only these sums (r and the pre logits), not the workers' rstd below
    if (owner_cta && !own_heads) asm volatile("bar.arrive 2, %0;" ::"r"(kSNT) : "memory");  // sums -> owner warp
    // r, pre and rstd of every token, one thread per token (identical in every CTA)
    for (int t = wt; t < T; t += nwork) {
        const float *s = sSums + t * 16;
        float G[10];
#pragma unroll
        for (int e = 0; e < 10; ++e) G[e] = s[4 + e];
        const float r = hc_rsqrt((G[0] + G[1]) + (G[2] + G[3]), H, sc.hc_norm_eps);
        const float a_pre = mix_scales[0];
        float pre[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pre[i] = pre_value(r * s[i], a_pre, bias[i]);
        float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] + pre[3] * pre[3] * G[3];
        sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                     pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
        const float rstd = 1.f / sqrtf(fmaxf(sx, 0.f) / (float)H + sc.rmsnorm_eps);
        *reinterpret_cast<float4 *>(sSt + t * 8) = make_float4(pre[0], pre[1], pre[2], pre[3]);
        sSt[t * 8 + 4] = rstd;
        const bool fix = gram_cancels(sx, pre, G);
        sSt[t * 8 + 6] = fix ? 1.f : 0.f;
        if (fix) atomicAdd(&sFlag[1], 1);
        if (split && c == 0) *reinterpret_cast<float4 *>(pre_out + (size_t)t * 4) = make_float4(pre[0], pre[1], pre[2], pre[3]);
    }
    wsync();

    // ---- 4b. tokens whose streams cancel in X (gram_cancels): sum_h X^2 summed directly.  Every
    // CTA flags the same tokens (it holds the same sums), so all of them take this branch or
    // none does.  Each CTA's share over its slice goes to the workspace (one warp per token:
    // lane v takes vector v, then an xor tree), a second grid barrier, then every CTA adds the
    // shares in one fixed order and replaces the token's rstd.
    if (sFlag[1] > 0) {
        float *fixrec = part + (size_t)T * nc * (kHead + kTail);  // [T][nc]
        for (int t = wt >> 5; t < T; t += nwork >> 5) {
            if (sSt[t * 8 + 6] == 0.f) continue;
            const float4 p4 = *reinterpret_cast<const float4 *>(sSt + t * 8);
            const float pre[kHC] = {p4.x, p4.y, p4.z, p4.w};
            float a = 0.f;
            for (int v = lane; v < nvec && v * kVec < hv; v += 32) {
                float rf[kHC][8], x[8];
#pragma unroll
                for (int j = 0; j < kHC; ++j)
                    unpack8(*reinterpret_cast<const uint4 *>(sRp + (size_t)t * RS + j * Hs + v * kVec), rf[j]);
                combine_vec8_x2(rf, pre, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(x[e], x[e], a);
            }
            a = warp_sum(a);
            if (lane == 0) fixrec[(size_t)t * nc + c] = a;
        }
        wsync();
        if (wt == 0)
            sFlag[2] = grid_barrier(reinterpret_cast<unsigned long long *>(ctrl + kSmallBarrierWord + 2),
                                    (unsigned int)nc, kSpinLimitNs) ? 1 : 0;
        wsync();
        if (!sFlag[2]) {
            if (wt == 0) atomicOr(ctrl, 1u);
            return;
        }
        for (int t = wt >> 5; t < T; t += nwork >> 5) {
            if (sSt[t * 8 + 6] == 0.f) continue;
            float a = 0.f;
            for (int q = lane; q < nc; q += 32) a += fixrec[(size_t)t * nc + q];
            a = warp_sum(a);
            if (lane == 0) sSt[t * 8 + 4] = 1.f / sqrtf(fmaxf(a, 0.f) / (float)H + sc.rmsnorm_eps);
        }
        wsync();
    }

    // ---- 5. combine + RMSNorm of the slice.  Warp-uniform loop: with the MXFP8 output, the four
    // lanes 4a .. 4a+3 hold one block of 32 (nvec is then a multiple of 4).
    for (int base = wt - lane; base < T * nvec; base += nwork) {
        const int item = base + lane;
        const int t = item / nvec, v = item % nvec;
        const bool act = item < T * nvec && v * kVec < hv;
        uint4 ob = make_uint4(0u, 0u, 0u, 0u);
        if (act) {
            const float4 p4 = *reinterpret_cast<const float4 *>(sSt + t * 8);
            const float pre[kHC] = {p4.x, p4.y, p4.z, p4.w};
            float rf[kHC][8], x[8];
#pragma unroll
            for (int j = 0; j < kHC; ++j)
                unpack8(*reinterpret_cast<const uint4 *>(sRp + (size_t)t * RS + j * Hs + v * kVec), rf[j]);
            combine_vec8_x2(rf, pre, x);
            ob = norm_vec8(x, sSt[t * 8 + 4], *reinterpret_cast<const uint4 *>(sGam + v * kVec));
            if (!kMx || X_out != nullptr) st_stream(X_out + (size_t)t * H + h0 + v * kVec, ob);
        }
        if (kMx)
            mx_quantize8(ob, act, mx.mode, mx.q + (size_t)t * H + h0 + v * kVec,
                         mx.scale + mx_scale_offset(t, (h0 + v * kVec) / 32, H));
    }
    if (dead && wt == 0) atomicOr(ctrl, 1u);
}

// The post and residual mixes of token blockIdx.x from the records a split small_kernel left
// in the workspace: the same sums in the same order as the kernel's owner warp (so the
// same bits), then the heads and the Sinkhorn.  One warp per token.
__global__ void __launch_bounds__(32)
small_tail_kernel(const float *__restrict__ part, int T, int nc, int H, const float *__restrict__ bias,
                  const float *__restrict__ mix_scales, Scalars sc, float *__restrict__ post_out,
                  float *__restrict__ res_out) {
    __shared__ __align__(16) float sv[28];  // head slots 0..7, then logits 4..23
    const int t = blockIdx.x, lane = threadIdx.x;
    const float *heads = part + (size_t)t * nc * kHead;
    const float *tails = part + (size_t)T * nc * kHead + (size_t)t * nc * kTail;
    const float4 h4 = warp_cta_sum16(heads, kHead, nc, 2);        // pre logits, Gram diagonal
    const float4 ta = warp_cta_sum16(tails, kTail, nc, 4);        // logits 4..19
    const float4 tb = warp_cta_sum16(tails + 16, kTail, nc, 1);   // logits 20..23
    if (lane < 2) *reinterpret_cast<float4 *>(sv + 4 * lane) = h4;
    if (lane < 4) *reinterpret_cast<float4 *>(sv + 8 + 4 * lane) = ta;
    if (lane == 0) *reinterpret_cast<float4 *>(sv + 24) = tb;
    __syncwarp();
    const float r = hc_rsqrt((sv[4] + sv[5]) + (sv[6] + sv[7]), H, sc.hc_norm_eps);
    const float z = r * (lane < 4 ? sv[lane] : (lane < kNumMix ? sv[lane + 4] : 0.f));
    const float v = heads_and_sinkhorn(z, bias, mix_scales, sc);
    if (lane >= 4 && lane < 8) post_out[(size_t)t * 4 + lane - 4] = v;
    else if (lane >= 8 && lane < kNumMix) res_out[(size_t)t * 16 + lane - 8] = v;
}

}  // namespace

int small_ctas(int H, int num_sms) {
    const int n = (H + 63) / 64;
    return n < num_sms ? n : num_sms;
}
int small_slice(int H, int num_sms, int align) {
    const int n = small_ctas(H, num_sms);
    return ((H + n - 1) / n + align - 1) / align * align;
}
bool small_supported(int64_t T, int H, int num_sms, bool mx) {
    if (T < 1 || T > kSmallMaxT || num_sms < 1) return false;
    const int Hs = small_slice(H, num_sms, mx ? 32 : 8);
    const int n = (H + Hs - 1) / Hs;
    if (n > kMaxCtas) return false;
    return SmallSmem{(int)T, Hs, n}.bytes() <= kSmallSmemLimit;
}
size_t small_workspace_bytes(int64_t T, int H) {
    if (T < 1 || T > kSmallMaxT) return 0;
    return (size_t)((H + 63) / 64) * (size_t)T * (kHead + kTail + 1) * sizeof(float);
}

cudaError_t launch_small(const SplitArgs &a, unsigned int *ctrl, int num_sms, cudaStream_t stream) {
    const bool mxo = a.mx.q != nullptr;
    if (!small_supported(a.T, a.H, num_sms, mxo)) return cudaErrorInvalidValue;
    const int Hs = small_slice(a.H, num_sms, mxo ? 32 : 8);  // MXFP8: slices hold whole blocks of 32
    const int n = (a.H + Hs - 1) / Hs;  // every CTA holds at least one vector of the slice
    const bool post = a.R_out != nullptr;
    auto kern = post ? (mxo ? small_kernel<true, true> : small_kernel<true, false>)
                     : (mxo ? small_kernel<false, true> : small_kernel<false, false>);
    const size_t smem = SmallSmem{(int)a.T, Hs, n}.bytes();
    cudaError_t e;
    if (smem > 48 * 1024 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
                                cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barrier cannot deadlock
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)n);
    cfg.blockDim = dim3(kSNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    mark_main_kernel(stream, true);
    e = cudaLaunchKernelEx(&cfg, kern, a.R, a.Y, a.prev_post, a.prev_comb, a.phi, a.bias, a.mix_scales, a.gamma,
                           a.s, (int)a.T, a.H, Hs, a.R_out, a.X_out, a.pre_out, a.post_out, a.res_out, a.part,
                           ctrl, a.mx, a.side != nullptr ? 1 : 0);
    mark_main_kernel(stream, false);
    if (e != cudaSuccess || a.side == nullptr) return e;
    // split: the mixes on the side stream, after the records are in
    if ((e = cudaEventRecord(a.side->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(a.side->stream, a.side->fork, 0)) != cudaSuccess) return e;
    small_tail_kernel<<<(unsigned)a.T, 32, 0, a.side->stream>>>(a.part, (int)a.T, n, a.H, a.bias, a.mix_scales, a.s,
                                                                a.post_out, a.res_out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return cudaEventRecord(a.side->join, a.side->stream);
}

}  // namespace mhc
