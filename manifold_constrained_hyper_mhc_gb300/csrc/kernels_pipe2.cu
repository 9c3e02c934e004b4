// Pipelined cluster schedule with the projection on tcgen05 (schedule "pipe2").
//
// A cluster of 16 CTAs (one per SM) owns groups of G = 8 tokens; CTA c owns
// the hidden slice [c*Hs, (c+1)*Hs) of each token (Hs a multiple of 64, at
// most 480).  The CTA-local flattened index is k = j*Hs + h (stream j, hidden
// h of the slice), K = 4*Hs, split into two halves k < 2*Hs (streams 0, 1) and
// k >= 2*Hs (streams 2, 3).
//
// Projection on the tensor cores: one tcgen05.mma kind::f16 per 16 values of
// k, M = 128, N = 16, accumulating in tensor memory.
//   A (tensor memory, resident for the whole kernel): 128 lanes x Hs columns,
//     lane m holds row m, two bf16 values of k per 32-bit column.  Rows 0-23
//     are the bf16 "hi" parts of phi^T for the first half of k, rows 24-47
//     the "lo" parts (phi - hi), rows 64-87 and 88-111 the same for the second
//     half; the other rows are zero.
//   B (shared memory): the 8 tokens' R' for the first half (columns 0-7) and
//     the second half (columns 8-15), read straight from the TMA-written R'
//     tile, which is a K-major 128-byte-swizzled operand; the two 8-row groups
//     are 2048 bytes apart.
//   D (tensor memory, double-buffered): 128 x 16 fp32.  The logits of token
//     t are z[n] = D[n][t] + D[24+n][t] + D[64+n][8+t] + D[88+n][8+t].
// So the cross terms of the two halves are computed and ignored; the tensor
// core sums over all of K itself.
//
// Warps: 16 workers, a producer warp (TMA copies and the MMAs) and an owner
// warp (per-token reductions).  Per group k:
//   workers : post in shared memory (R' overwrites R), R' to HBM, Gram matrix;
//             release the tile to the MMA; combine + RMSNorm of group k-1;
//             read D of group k and send each token's record (24 logits + 10
//             Gram entries) to the token's owner CTA (st.async).
//   producer: 2*Hs/16 MMAs of group k once the tile is written, commit to an
//             mbarrier; TMA copies of group k+2 into the triple buffer.
//   owner   : for the token this CTA owns in group k: sum the 16 records,
//             r, the pre and post heads, rstd from the Gram matrix
//             (sum_h X^2 = pre^T G pre), (pre, rstd) to all 16 CTAs; the 16
//             residual-mix logits are kept for the end of the kernel, where all
//             warps run the Sinkhorn normalisations, one token per lane.
//
// Every mbarrier wait is bounded: on a timeout the CTA sets bit 0 of the
// status word and stops waiting (later waits give up at once), still meets
// the cluster barrier at the end, frees its tensor memory and exits.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "mhc_device.cuh"
#include "mhc_kernels.h"
#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace mhc {

namespace {

using namespace ptx;

constexpr int kC = 16;
constexpr int kG = 8;
constexpr int kWorkers = 16;
constexpr int kProducer = kWorkers;
constexpr int kOwner = kWorkers + 1;
constexpr int kNT = (kWorkers + 2) * 32;
constexpr int kNBuf = 3;
constexpr int kRec = 36;
constexpr int kTmemCols = 512;
constexpr int kMaxHs = kTmemCols - 32;  // A needs Hs columns, D two buffers of 16
constexpr uint32_t kWaitLimit = 1u << 25;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 16);

struct Layout {
    int nHB;
    __host__ __device__ size_t rbuf() const { return (size_t)nHB * 4096; }
    __host__ __device__ size_t ybuf() const { return (size_t)nHB * 1024; }
    __host__ __device__ size_t r_off(int b) const { return (size_t)b * rbuf(); }
    __host__ __device__ size_t y_off(int b) const { return kNBuf * rbuf() + (size_t)b * ybuf(); }
    __host__ __device__ size_t comb_off(int b) const { return y_off(kNBuf) + (size_t)b * 512; }
    __host__ __device__ size_t post_off(int b) const { return comb_off(kNBuf) + (size_t)b * 128; }
    __host__ __device__ size_t d_off() const { return post_off(kNBuf); }                    // [128][16] f32
    __host__ __device__ size_t gram_off() const { return d_off() + 128 * 16 * 4; }          // [16][12]
    __host__ __device__ size_t rec_off() const { return gram_off() + kWorkers * 12 * 4; }   // [8][36]
    __host__ __device__ size_t recv_off() const { return rec_off() + kG * kRec * 4; }       // [16][36]
    __host__ __device__ size_t prein_off() const { return recv_off() + kC * kRec * 4; }     // [2][8][8]
    __host__ __device__ size_t gam_off() const { return prein_off() + 2 * kG * 8 * 4; }     // [Hs] bf16
    __host__ __device__ size_t bar_off() const { return gam_off() + (size_t)nHB * 128; }
    // full[3] free[3] part_full pre_full[2] p1done[2] mma_done[2] d_free[2]
    __host__ __device__ size_t tmem_off() const { return bar_off() + 15 * 8; }
    __host__ __device__ size_t bytes() const { return tmem_off() + 8; }
};

// R' tile of one group: nHB boxes of [stream 4][token 8][64 hidden] bf16 with
// the 128-byte swizzle (16-byte chunk index XOR row % 8, row = j*8 + t).
__device__ __forceinline__ uint32_t r_swz(int hb, int t, int j, int c16) {
    const int row = j * 8 + t;
    return (uint32_t)(hb * 4096 + row * 128 + ((c16 ^ t) << 4));
}
__device__ __forceinline__ uint32_t y_swz(int hb, int t, int c16) {
    return (uint32_t)(hb * 1024 + t * 128 + ((c16 ^ t) << 4));
}

// Gram index order: (0,0) (1,1) (2,2) (3,3) (0,1) (0,2) (0,3) (1,2) (1,3) (2,3).
__device__ __forceinline__ void gram_acc(const float (&rf)[kHC][8], float2 (&gm)[10]) {
    constexpr int ia[10] = {0, 1, 2, 3, 0, 0, 0, 1, 1, 2}, ib[10] = {0, 1, 2, 3, 1, 2, 3, 2, 3, 3};
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
#pragma unroll
        for (int q = 0; q < 10; ++q)
            gm[q] = __ffma2_rn(make_float2(rf[ia[q]][e], rf[ia[q]][e + 1]),
                               make_float2(rf[ib[q]][e], rf[ib[q]][e + 1]), gm[q]);
    }
}

struct Maps {
    CUtensorMap R, Y, comb, post;
};

template <bool kPost>
__global__ void __launch_bounds__(kNT, 1)
pipe2_kernel(const __grid_constant__ Maps maps, const uint4 *__restrict__ a_pack,
             const float *__restrict__ bias, const float *__restrict__ mix_scales,
             const uint16_t *__restrict__ gamma, Scalars sc, int64_t T, int H, int Hs,
             uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out, float *__restrict__ pre_out,
             float *__restrict__ post_out, float *__restrict__ res_out, float *__restrict__ zstash,
             unsigned int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nHB = Hs / 64;
    const Layout L{nHB};
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float *sD = reinterpret_cast<float *>(smem + L.d_off());
    float *sGram = reinterpret_cast<float *>(smem + L.gram_off());
    float *sRec = reinterpret_cast<float *>(smem + L.rec_off());
    float *sRecv = reinterpret_cast<float *>(smem + L.recv_off());
    float *sPreIn = reinterpret_cast<float *>(smem + L.prein_off());
    unsigned char *sGam = smem + L.gam_off();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off());
    uint64_t *full = bars, *freeb = bars + 3, *part_full = bars + 6, *pre_full = bars + 7, *p1done = bars + 9,
             *mma_done = bars + 11, *d_free = bars + 13;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.tmem_off());

    const int h0 = c * Hs;
    const int nvec = Hs / kVec;  // <= 60
    const int nsteps = 2 * Hs / 16;
    const int64_t ngroups = (T + kG - 1) / kG;
    const int nclusters = gridDim.x / kC;
    const int cid = blockIdx.x / kC;
    const int n_it = cid < ngroups ? (int)((ngroups - cid + nclusters - 1) / nclusters) : 0;
    auto group_t0 = [&](int it) { return (int64_t)(cid + (int64_t)it * nclusters) * kG; };
    // token t of iteration `it` is owned by CTA (t + 8*(it&1)); the token this CTA owns:
    auto owned_token = [&](int it) { return c - 8 * (it & 1); };  // valid if in [0, 8)
    bool dead = false;

    // ---- set-up
    if (warp == kProducer) {
        if (lane == 0) {
            for (int i = 0; i < 3; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&freeb[i], kWorkers);
            }
            mbar_init(part_full, 1);
            for (int i = 0; i < 2; ++i) {
                mbar_init(&pre_full[i], 1);
                mbar_init(&p1done[i], kWorkers);
                mbar_init(&mma_done[i], 1);
                mbar_init(&d_free[i], 4);
            }
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *sTmem;
    if (warp < kWorkers) {
        for (int v = tid; v < nvec; v += kWorkers * 32) {
            const int h = h0 + v * kVec;
            *reinterpret_cast<uint4 *>(sGam + v * 16) = h < H ? ld_ro(gamma + h) : make_uint4(0u, 0u, 0u, 0u);
        }
        // A operand into tensor memory: warp w fills lane quarter w % 4,
        // columns [(w/4) * Hs/4, (w/4 + 1) * Hs/4) in 16-column pieces
        const int q = warp & 3, u = warp >> 2;
        const int per = Hs / 4 / 16;
        for (int i = 0; i < per; ++i) {
            const int cc = u * per + i;  // 16-column piece
            const uint4 *src = a_pack + (((size_t)c * (Hs / 16) + cc) * 128 + 32 * q + lane) * 4;
            uint32_t r[16];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint4 v = __ldg(src + x);
                r[4 * x] = v.x; r[4 * x + 1] = v.y; r[4 * x + 2] = v.z; r[4 * x + 3] = v.w;
            }
            tmem_st16(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(cc * 16), r);
        }
        tmem_wait_st();
    }
    if (warp == kOwner && lane == 0) {
        int first_owned = -1;
        for (int it = 0; it < n_it && first_owned < 0; ++it)
            if (owned_token(it) >= 0 && owned_token(it) < kG) first_owned = it;
        if (first_owned >= 0) mbar_arrive_expect_tx(part_full, kC * kRec * 4);
        if (n_it > 0) mbar_arrive_expect_tx(&pre_full[0], kG * 32);
        if (n_it > 1) mbar_arrive_expect_tx(&pre_full[1], kG * 32);
    }
    tmem_fence_before();
    cluster.sync();  // barriers of every CTA exist before any message; A is in TMEM
    tmem_fence_after();

    if (warp == kProducer) {
        // ======================== producer: TMA copies and MMAs
        const uint32_t expect_bytes = (uint32_t)nHB * (4096 + (kPost ? 1024 : 0)) + (kPost ? 512 + 128 : 0);
        auto issue = [&](int it) {
            const int b = it % kNBuf;
            const int t0 = (int)group_t0(it);
            mbar_arrive_expect_tx(&full[b], expect_bytes);
            for (int hb = 0; hb < nHB; ++hb) {
                tma_load_3d(smem + L.r_off(b) + hb * 4096, &maps.R, h0 + hb * 64, t0, 0, &full[b]);
                if (kPost) tma_load_2d(smem + L.y_off(b) + hb * 1024, &maps.Y, h0 + hb * 64, t0, &full[b]);
            }
            if (kPost) {
                tma_load_2d(smem + L.comb_off(b), &maps.comb, 0, t0, &full[b]);
                tma_load_2d(smem + L.post_off(b), &maps.post, 0, t0, &full[b]);
            }
        };
        if (lane == 0)
            for (int it = 0; it < kNBuf - 1 && it < n_it; ++it) issue(it);
        for (int it = 0; it < n_it; ++it) {
            const int db = it & 1;
            mbar_wait(&p1done[db], (uint32_t)((it >> 1) & 1), dead, kWaitLimit);
            if (it >= 2) mbar_wait(&d_free[db], (uint32_t)(((it - 2) >> 1) & 1), dead, kWaitLimit);
            tmem_fence_after();
            if (lane == 0) {
                const uint32_t rb = smem_u32(smem + L.r_off(it % kNBuf));
                const uint32_t dt = tbase + (uint32_t)(Hs + 16 * db);
                for (int s = 0; s < nsteps; ++s) {
                    const int kl = 16 * s;
                    const int j = kl >= Hs ? 1 : 0, h = kl - j * Hs;
                    const uint32_t sa = rb + (uint32_t)((h >> 6) * 4096 + j * 1024 + (h & 63) * 2);
                    umma_tmemA(dt, tbase + (uint32_t)(s * 8), sdesc_kmajor_sw128(sa, 2048), kIdesc, s > 0 ? 1u : 0u);
                }
                umma_commit(&mma_done[db]);
            }
            __syncwarp();
            const int nxt = it + kNBuf - 1;
            if (nxt < n_it) {
                if (it >= 1) mbar_wait(&freeb[(it - 1) % kNBuf], (uint32_t)(((it - 1) / kNBuf) & 1), dead, kWaitLimit);
                if (lane == 0) issue(nxt);
                __syncwarp();
            }
        }
    } else if (warp == kOwner) {
        // ======================== owner: per-token reductions and heads
        int owned_done = 0;
        for (int it = 0; it < n_it; ++it) {
            const int g = owned_token(it);
            if (g < 0 || g >= kG) continue;
            const int64_t t = group_t0(it) + g;
            mbar_wait(part_full, (uint32_t)(owned_done & 1), dead, kWaitLimit);
            ++owned_done;
            float a = 0.f, a2 = 0.f;
            for (int q = 0; q < kC; ++q) {
                a += sRecv[q * kRec + lane];
                if (lane < 2) a2 += sRecv[q * kRec + 32 + lane];
            }
            __syncwarp();
            if (lane == 0 && it + 2 < n_it) mbar_arrive_expect_tx(part_full, kC * kRec * 4);
            float G[10];
#pragma unroll
            for (int e = 0; e < 8; ++e) G[e] = __shfl_sync(0xffffffffu, a, 24 + e);
            G[8] = __shfl_sync(0xffffffffu, a2, 0);
            G[9] = __shfl_sync(0xffffffffu, a2, 1);
            const float ss = (G[0] + G[1]) + (G[2] + G[3]);
            const float r = 1.f / sqrtf(ss / (float)(kHC * H) + sc.hc_norm_eps);
            const float z = r * a;
            const float p = pre_head(z, bias, mix_scales);
            float pre[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pre[i] = __shfl_sync(0xffffffffu, p, i);
            float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] +
                       pre[3] * pre[3] * G[3];
            sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                         pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
            const float rstd = 1.f / sqrtf(fmaxf(sx, 0.f) / (float)H + sc.rmsnorm_eps);
            if (lane < kC) {
                const int sl = it & 1;
                const uint32_t raddr = mapa(smem_u32(sPreIn + ((size_t)sl * kG + g) * 8), (uint32_t)lane);
                const uint32_t rbar = mapa(smem_u32(&pre_full[sl]), (uint32_t)lane);
                st_async16(raddr, rbar, make_uint4(__float_as_uint(pre[0]), __float_as_uint(pre[1]),
                                                   __float_as_uint(pre[2]), __float_as_uint(pre[3])));
                st_async16(raddr + 16, rbar, make_uint4(__float_as_uint(rstd), 0u, 0u, 0u));
            }
            if (t < T) {
                if (lane < 4) pre_out[t * 4 + lane] = p;
                else if (lane < 8) post_out[t * 4 + lane - 4] = sc.hc_post_scale / (1.f + expf(-(mix_scales[1] * z + bias[lane])));
                else if (lane < 24) zstash[t * 16 + lane - 8] = z;
            }
        }
    } else {
        // ======================== workers
        const int t_p1 = warp >> 1, half = warp & 1;
        auto combine = [&](int it) {
            const int b = it % kNBuf, sl = it & 1;
            mbar_wait(&pre_full[sl], (uint32_t)((it >> 1) & 1), dead, kWaitLimit);
            if (tid == 0 && it + 2 < n_it) mbar_arrive_expect_tx(&pre_full[sl], kG * 32);
            const int64_t t0 = group_t0(it);
            const unsigned char *rb = smem + L.r_off(b);
            for (int item = tid; item < kG * nvec; item += kWorkers * 32) {
                const int t = item / nvec, v = item % nvec;
                const int h = h0 + v * kVec;
                if (t0 + t >= T || h >= H) continue;
                const float4 pv = *reinterpret_cast<const float4 *>(sPreIn + ((size_t)sl * kG + t) * 8);
                const float rstd = sPreIn[((size_t)sl * kG + t) * 8 + 4];
                const float pre[kHC] = {pv.x, pv.y, pv.z, pv.w};
                float rf[kHC][8], x[8];
#pragma unroll
                for (int j = 0; j < kHC; ++j)
                    unpack8(*reinterpret_cast<const uint4 *>(rb + r_swz(v >> 3, t, j, v & 7)), rf[j]);
                combine_vec8_x2(rf, pre, x);
                st_stream(X_out + (t0 + t) * (int64_t)H + h,
                          norm_vec8(x, rstd, *reinterpret_cast<const uint4 *>(sGam + v * 16)));
            }
            fence_proxy_async_smem();  // the tile is refilled by TMA after this
            __syncwarp();
            if (lane == 0) mbar_arrive(&freeb[b]);
        };

        for (int it = 0; it < n_it; ++it) {
            const int b = it % kNBuf, db = it & 1;
            const int64_t t0 = group_t0(it);
            mbar_wait(&full[b], (uint32_t)((it / kNBuf) & 1), dead, kWaitLimit);
            unsigned char *rb = smem + L.r_off(b);

            // ---- P1: warp w takes token w/2, half w%2 of the slice's vectors
            {
                const int t = t_p1;
                const int nh = (nvec + 1) >> 1;
                const int v = half * nh + lane;
                float2 gm2[10];
#pragma unroll
                for (int e = 0; e < 10; ++e) gm2[e] = make_float2(0.f, 0.f);
                if (lane < nh && v < nvec) {
                    const int hb = v >> 3, ch = v & 7;
                    float rf[kHC][8];
                    if (kPost) {
                        uint4 r4[kHC], o[kHC];
#pragma unroll
                        for (int j = 0; j < kHC; ++j) r4[j] = *reinterpret_cast<const uint4 *>(rb + r_swz(hb, t, j, ch));
                        const uint4 y = *reinterpret_cast<const uint4 *>(smem + L.y_off(b) + y_swz(hb, t, ch));
                        float cm[16], pm[4];
                        const float4 *cb = reinterpret_cast<const float4 *>(smem + L.comb_off(b)) + t * 4;
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const float4 f = cb[x];
                            cm[4 * x] = f.x; cm[4 * x + 1] = f.y; cm[4 * x + 2] = f.z; cm[4 * x + 3] = f.w;
                        }
                        const float4 pf = reinterpret_cast<const float4 *>(smem + L.post_off(b))[t];
                        pm[0] = pf.x; pm[1] = pf.y; pm[2] = pf.z; pm[3] = pf.w;
                        post_vec8_x2(r4, y, cm, pm, o, rf);
#pragma unroll
                        for (int j = 0; j < kHC; ++j) *reinterpret_cast<uint4 *>(rb + r_swz(hb, t, j, ch)) = o[j];
                        const int h = h0 + v * kVec;
                        if (t0 + t < T && h < H) {
                            const int64_t base = (t0 + t) * kHC * (int64_t)H + h;
#pragma unroll
                            for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kHC; ++j)
                            unpack8(*reinterpret_cast<const uint4 *>(rb + r_swz(hb, t, j, ch)), rf[j]);
                    }
                    gram_acc(rf, gm2);
                }
                float gm[10];
#pragma unroll
                for (int e = 0; e < 10; ++e) gm[e] = warp_sum(gm2[e].x + gm2[e].y);
                if (lane == 0) {
#pragma unroll
                    for (int e = 0; e < 10; ++e) sGram[warp * 12 + e] = gm[e];
                }
            }
            fence_proxy_async_smem();  // R' is read by the tensor core (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(&p1done[db]);

            if (it >= 1) combine(it - 1);

            // ---- D of this group -> shared memory (warps 0-3, one lane quarter each)
            mbar_wait(&mma_done[db], (uint32_t)((it >> 1) & 1), dead, kWaitLimit);
            tmem_fence_after();
            if (warp < 4) {
                uint32_t d[16];
                tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)(Hs + 16 * db), d);
                tmem_wait_ld();
                float4 *dst = reinterpret_cast<float4 *>(sD + (32 * warp + lane) * 16);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    dst[x] = make_float4(__uint_as_float(d[4 * x]), __uint_as_float(d[4 * x + 1]),
                                         __uint_as_float(d[4 * x + 2]), __uint_as_float(d[4 * x + 3]));
                tmem_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_free[db]);
            }
            named_sync(1, kWorkers * 32);

            // ---- records: logits from D, Gram entries from the two P1 warps of the token
            for (int idx = tid; idx < kG * kRec; idx += kWorkers * 32) {
                const int t = idx / kRec, n = idx % kRec;
                float v = 0.f;
                if (n < kNumMix) {
                    v = (sD[n * 16 + t] + sD[(24 + n) * 16 + t]) + (sD[(64 + n) * 16 + 8 + t] + sD[(88 + n) * 16 + 8 + t]);
                } else if (n < kNumMix + 10) {
                    v = sGram[(2 * t) * 12 + (n - kNumMix)] + sGram[(2 * t + 1) * 12 + (n - kNumMix)];
                }
                sRec[idx] = v;
            }
            named_sync(1, kWorkers * 32);
            if (tid < kG * (kRec / 4)) {
                const int t = tid / (kRec / 4), q = tid % (kRec / 4);
                const uint32_t owner = (uint32_t)(t + 8 * (it & 1));
                const uint4 val = *reinterpret_cast<const uint4 *>(sRec + t * kRec + 4 * q);
                st_async16(mapa(smem_u32(sRecv + c * kRec + 4 * q), owner), mapa(smem_u32(part_full), owner), val);
            }
        }
        if (n_it >= 1) combine(n_it - 1);
    }

    cluster.sync();  // every message delivered; the residual-mix logits are stashed

    // ---- Sinkhorn of the tokens this CTA owned, one token per thread
    {
        const int first = c >= 8 ? 1 : 0;  // owned iterations are first, first + 2, ...
        const int nown = n_it > first ? (n_it - first + 1) / 2 : 0;
        for (int k = tid; k < nown; k += kNT) {
            const int it = first + 2 * k;
            const int64_t t = group_t0(it) + (c - 8 * (it & 1));
            if (t >= T) continue;
            float M[16];
            const float4 *zs = reinterpret_cast<const float4 *>(zstash + t * 16);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float4 f = zs[x];
                M[4 * x] = f.x; M[4 * x + 1] = f.y; M[4 * x + 2] = f.z; M[4 * x + 3] = f.w;
            }
            const float a_res = mix_scales[2];
#pragma unroll
            for (int e = 0; e < 16; ++e) M[e] = expf(a_res * M[e] + bias[8 + e]);
            sinkhorn16(M, sc);
            float4 *ro = reinterpret_cast<float4 *>(res_out + t * 16);
#pragma unroll
            for (int x = 0; x < 4; ++x) ro[x] = make_float4(M[4 * x], M[4 * x + 1], M[4 * x + 2], M[4 * x + 3]);
        }
    }

    const bool any_dead = __any_sync(0xffffffffu, dead);
    if (any_dead && lane == 0) atomicOr(status, 1u);
    tmem_fence_before();
    __syncthreads();
    if (warp == kProducer) tmem_dealloc(tbase, kTmemCols);
}

// phi [4H][24] fp32 -> the A operand of every CTA in tensor-memory order:
// out[c][piece cc][row m][16 words], column = cc*16 + word, each word two bf16
// values of A[m][k] for k = 2*column and 2*column + 1 (low half first), with
// A as described at the top of this file.
__global__ void __launch_bounds__(256)
pack_a_kernel(const float *__restrict__ phi, int H, int Hs, uint32_t *__restrict__ out) {
    const int64_t total = (int64_t)kC * Hs * 128;  // words
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int w = (int)(idx & 15);
    const int m = (int)((idx >> 4) & 127);
    const int64_t rest = idx >> 11;
    const int cc = (int)(rest % (Hs / 16));
    const int c = (int)(rest / (Hs / 16));
    const int col = cc * 16 + w;
    const int r = m >= 64 ? 1 : 0, mm = m - 64 * r;
    float v[2] = {0.f, 0.f};
    if (mm < 2 * kNumMix) {
        const int n = mm % kNumMix;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int kl = 2 * col + e + r * 2 * Hs;
            const int j = kl / Hs, hg = c * Hs + kl % Hs;
            if (hg < H) {
                const float x = phi[((int64_t)j * H + hg) * kNumMix + n];
                const float hi = __bfloat162float(__float2bfloat16_rn(x));
                v[e] = mm < kNumMix ? hi : x - hi;
            }
        }
    }
    out[idx] = pack2_rn(v[0], v[1]);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

cudaError_t get_encode(EncodeTiledFn &fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    fn = g_encode;
    return cudaSuccess;
}

cudaError_t encode(EncodeTiledFn fn, CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr,
                   const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swz) {
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};  // one per dimension, up to rank 5
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

int pipe2_slice(int H) { return ((H + 64 * kC - 1) / (64 * kC)) * 64; }

bool pipe2_supported(int H) {
    const int Hs = pipe2_slice(H);
    return Hs <= kMaxHs && Hs % 64 == 0 && Layout{Hs / 64}.bytes() + 1024 <= 227 * 1024;
}

size_t pipe2_pack_bytes(int H) { return (size_t)kC * pipe2_slice(H) * 128 * 4; }
size_t pipe2_stash_bytes(int64_t T) { return (size_t)T * 16 * 4; }

cudaError_t launch_pipe2(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream) {
    if (!pipe2_supported(a.H)) return cudaErrorInvalidValue;
    const int Hs = pipe2_slice(a.H);
    const bool post = a.R_out != nullptr;
    EncodeTiledFn fn;
    cudaError_t e = get_encode(fn);
    if (e != cudaSuccess) return e;
    Maps maps;
    std::memset(&maps, 0, sizeof maps);
    const cuuint64_t H = (cuuint64_t)a.H, T = (cuuint64_t)a.T;
    {   // R [T][4][H] as (h, t, j): box 64 x 8 x 4 lands as [stream][token][64]
        const cuuint64_t dims[3] = {H, T, 4}, strides[2] = {H * 8, H * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kG, 4};
        if ((e = encode(fn, &maps.R, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    if (post) {
        const cuuint64_t dy[2] = {H, T}, sy[1] = {H * 2};
        const cuuint32_t by[2] = {64, (cuuint32_t)kG};
        if ((e = encode(fn, &maps.Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Y, dy, sy, by, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            cudaSuccess)
            return e;
        const cuuint64_t dc[2] = {16, T}, scm[1] = {64};
        const cuuint32_t bc[2] = {16, (cuuint32_t)kG};
        if ((e = encode(fn, &maps.comb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.prev_comb, dc, scm, bc,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
        const cuuint64_t dp[2] = {4, T}, sp[1] = {16};
        const cuuint32_t bp[2] = {4, (cuuint32_t)kG};
        if ((e = encode(fn, &maps.post, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.prev_post, dp, sp, bp,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
    }

    const int64_t words = (int64_t)kC * Hs * 128;
    pack_a_kernel<<<(unsigned)((words + 255) / 256), 256, 0, stream>>>(a.phi, a.H, Hs,
                                                                        reinterpret_cast<uint32_t *>(a.phi_pack));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    auto kern = post ? pipe2_kernel<true> : pipe2_kernel<false>;
    const size_t smem = Layout{Hs / 64}.bytes() + 1024;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static int max_clusters[64][2];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kNT);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.stream = stream;
    // one CTA per SM (the kernel takes all 512 TMEM columns)
    cfg.dynamicSmemBytes = std::max<size_t>(smem, 227 * 1024 / 2 + 1024);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int &mc = max_clusters[dev][post ? 1 : 0];
        if (mc == 0) {
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)) != cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
                return e;
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3(kC);
            int n = 0;
            if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &q)) != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
            mc = n;
        }
        cfg.gridDim = dim3((unsigned)(std::min<int64_t>((a.T + kG - 1) / kG, mc) * kC));
    }
    return cudaLaunchKernelEx(&cfg, kern, maps, (const uint4 *)a.phi_pack, a.bias, a.mix_scales, a.gamma, a.s, a.T,
                              a.H, Hs, a.R_out, a.X_out, a.pre_out, a.post_out, a.res_out, zstash, status);
}

}  // namespace mhc
