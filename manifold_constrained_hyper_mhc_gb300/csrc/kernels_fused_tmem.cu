// Cluster schedule with the projection weights resident in tensor memory.
//
// Same one-pass algorithm as kernels_fused.cu (clusters split the hidden
// dimension; R' stays in shared memory between the post and the combine;
// cluster reductions through distributed shared memory), with two changes
// that remove the per-group traffic and latency of the projection weights and
// keep HBM busy while a group is being reduced:
//
//   * phi, packed into mma.m16n8k16 A fragments (bf16 hi and lo parts), is
//     copied once per CTA into tensor memory (TMEM, 512 columns x 128 lanes x
//     32 bits per SM).  Warp w stores exactly the fragments of its own k16
//     steps at its own TMEM lanes (lane quarter w % 4), and reads them back
//     with tcgen05.ld for every token group.  With 16 CTAs per cluster a CTA's
//     slice of phi is 4*H/16 rows, 172 KB at H = 7168.
//   * R, Y and the previous mixes of group k+1 are fetched with bulk async
//     copies (cp.async.bulk, completion on an mbarrier) into the second half
//     of a double buffer while group k is being computed.  P1 then reads R
//     from shared memory and overwrites it in place with R'.
//
// Every wait on an mbarrier is bounded: after kWaitLimit polls the CTA sets
// bit 0 of the device status word, stops waiting and carries on through the
// cluster barriers (so no CTA of the cluster is left waiting), and the host
// reports MHC_ERR_DEVICE_TIMEOUT from mhc_check_status.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>

#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace cg = cooperative_groups;

namespace mhc {

namespace {

constexpr int kC = 16;             // CTAs per cluster
constexpr int kG = 16;             // tokens per group
constexpr int kNW = 16;            // warps per CTA
constexpr int kNT = kNW * 32;
constexpr int kTmemCols = 512;     // whole TMEM of the SM (one CTA per SM)
constexpr int kColsPerStep = 16;   // 12 fragment words + 4 unused per k16 step
constexpr uint32_t kWaitLimit = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier and bulk copies ------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; returns false if the limit was reached.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// ---- tensor memory -------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

// Shared memory layout (bytes), for slice width Hs.
struct Layout {
    int Hs;
    __host__ __device__ size_t rowb() const { return (size_t)kHC * Hs * 2 + 16; }   // R' row, padded
    __host__ __device__ size_t ybytes() const { return (size_t)Hs * 2; }
    __host__ __device__ size_t r_off(int b) const { return (size_t)b * kG * rowb(); }
    __host__ __device__ size_t y_off(int b) const { return 2 * kG * rowb() + (size_t)b * kG * ybytes(); }
    __host__ __device__ size_t comb_off(int b) const { return y_off(2) + (size_t)b * kG * 64; }   // [G][16] f32
    __host__ __device__ size_t post_off(int b) const { return comb_off(2) + (size_t)b * kG * 16; }  // [G][4] f32
    __host__ __device__ size_t z_off() const { return post_off(2); }                              // [NW][G][24]
    __host__ __device__ size_t part_off() const { return z_off() + (size_t)kNW * kG * kNumMix * 4; }  // [G][32]
    __host__ __device__ size_t ss_off() const { return part_off() + (size_t)kG * 32 * 4; }
    __host__ __device__ size_t pre_off() const { return ss_off() + (size_t)kG * 4; }   // [G][4]
    __host__ __device__ size_t xsq_off() const { return pre_off() + (size_t)kG * 16; }
    __host__ __device__ size_t bar_off() const { return (xsq_off() + (size_t)kG * 4 + 7) & ~size_t(7); }
    __host__ __device__ size_t tmem_off() const { return bar_off() + 16; }
    __host__ __device__ size_t bytes() const { return tmem_off() + 16; }
};

template <bool kPost>
__global__ void __launch_bounds__(kNT, 1)
fused_tmem_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y,
                  const float *__restrict__ prev_post, const float *__restrict__ prev_comb,
                  const uint4 *__restrict__ phi_pack, const float *__restrict__ bias,
                  const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma, Scalars sc,
                  int64_t T, int H, int Hs, uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out,
                  float *__restrict__ pre_out, float *__restrict__ post_out, float *__restrict__ res_out,
                  unsigned int *__restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout L{Hs};
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;

    float *sZ = reinterpret_cast<float *>(smem + L.z_off());
    float *sPart = reinterpret_cast<float *>(smem + L.part_off());
    float *sSS = reinterpret_cast<float *>(smem + L.ss_off());
    float *sPre = reinterpret_cast<float *>(smem + L.pre_off());
    float *sXsq = reinterpret_cast<float *>(smem + L.xsq_off());
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off());
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.tmem_off());

    const int h0 = c * Hs;
    const int hv = max(0, min(Hs, H - h0));
    const int nvec = Hs / kVec, nvec_valid = hv / kVec;
    const int S = kHC * Hs / 16;                       // k16 steps of the slice
    const int spw = (S + kNW - 1) / kNW;               // steps per warp (<= 8, checked on the host)
    const int s_begin = min(S, spw * warp), s_end = min(S, spw * (warp + 1));
    const int64_t ngroups = (T + kG - 1) / kG;
    const int nclusters = gridDim.x / kC;
    const int cid = blockIdx.x / kC;
    const size_t rowb = L.rowb();

    // ---- set-up: mbarriers, TMEM, phi fragments into TMEM
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *sTmem;
    // this warp's TMEM lanes (lane quarter warp % 4) and column block (warp / 4)
    const uint32_t tw = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * spw * kColsPerStep);
    {
        const uint4 *pack = phi_pack + (size_t)c * S * 96;
        for (int s = s_begin; s < s_end; ++s) {
            uint32_t r[16];
#pragma unroll
            for (int mt = 0; mt < 3; ++mt) {
                const uint4 a = __ldg(pack + ((size_t)s * 3 + mt) * 32 + lane);
                r[4 * mt] = a.x; r[4 * mt + 1] = a.y; r[4 * mt + 2] = a.z; r[4 * mt + 3] = a.w;
            }
            r[12] = r[13] = r[14] = r[15] = 0u;
            tmem_st16(tw + (uint32_t)((s - s_begin) * kColsPerStep), r);
        }
        tmem_wait_st();
    }

    // producer: warp 0 issues the bulk copies of group `grp` into buffer b
    auto issue = [&](int64_t grp, int b) {
        const int64_t t0 = grp * kG;
        const int gv = (int)(T - t0 < kG ? T - t0 : kG);
        const uint32_t rb = (uint32_t)hv * 2;
        const uint32_t bytes = (uint32_t)gv * rb * (kPost ? 5u : 4u) + (kPost ? (uint32_t)gv * 80u : 0u);
        if (lane == 0) mbar_arrive_expect_tx(&bars[b], bytes);
        __syncwarp();
        if (rb != 0) {
            const int ncopy = gv * (kPost ? 5 : 4);
            for (int q = lane; q < ncopy; q += 32) {
                const int g = q / (kPost ? 5 : 4), j = q % (kPost ? 5 : 4);
                const int64_t t = t0 + g;
                if (j < kHC)
                    bulk_g2s(smem + L.r_off(b) + g * rowb + (size_t)j * Hs * 2,
                             R + (t * kHC + j) * (int64_t)H + h0, rb, &bars[b]);
                else
                    bulk_g2s(smem + L.y_off(b) + g * L.ybytes(), Y + t * (int64_t)H + h0, rb, &bars[b]);
            }
        }
        if (kPost && lane == 0) {
            bulk_g2s(smem + L.comb_off(b), prev_comb + t0 * 16, (uint32_t)gv * 64u, &bars[b]);
            bulk_g2s(smem + L.post_off(b), prev_post + t0 * 4, (uint32_t)gv * 16u, &bars[b]);
        }
    };

    uint32_t phase[2] = {0u, 0u};
    bool pending[2] = {false, false};  // a phase was issued and not yet waited for successfully
    bool timed_out = false;
    if (warp == 0 && cid < ngroups) issue(cid, 0);
    pending[0] = cid < ngroups;

    int it = 0;
    for (int64_t grp = cid; grp < ngroups; grp += nclusters, ++it) {
        const int b = it & 1;
        const int64_t t0 = grp * kG;
        const int gv = (int)(T - t0 < kG ? T - t0 : kG);
        // prefetch the next group of this cluster into the other buffer (free
        // since the end of the previous group)
        if (grp + nclusters < ngroups) {
            if (warp == 0) issue(grp + nclusters, b ^ 1);
            pending[b ^ 1] = true;
        }
        if (mbar_wait(&bars[b], phase[b])) {
            pending[b] = false;
            phase[b] ^= 1u;
        } else {
            timed_out = true;
        }

        unsigned char *sRb = smem + L.r_off(b);
        const unsigned char *sYb = smem + L.y_off(b);
        const float *sComb = reinterpret_cast<const float *>(smem + L.comb_off(b));
        const float *sPost = reinterpret_cast<const float *>(smem + L.post_off(b));

        // ---- P1: post in shared memory (R -> R' in place), R' to HBM, square sums
        for (int g = warp; g < kG; g += kNW) {
            float ss = 0.f;
            if (g < gv) {
                const int64_t t = t0 + g;
                const int64_t rbase = t * kHC * (int64_t)H + h0;
                unsigned char *row = sRb + g * rowb;
                for (int v = lane; v < nvec; v += 32) {
                    uint4 o[kHC] = {};
                    if (v < nvec_valid) {
                        float rf[kHC][8];
                        if (kPost) {
                            uint4 r4[kHC];
#pragma unroll
                            for (int j = 0; j < kHC; ++j)
                                r4[j] = *reinterpret_cast<const uint4 *>(row + ((size_t)j * Hs + v * kVec) * 2);
                            const uint4 y = *reinterpret_cast<const uint4 *>(sYb + g * L.ybytes() + v * 16);
                            post_vec8(r4, y, sComb + g * 16, sPost + g * 4, o, rf);
#pragma unroll
                            for (int i = 0; i < kHC; ++i) st_stream(R_out + rbase + (int64_t)i * H + v * kVec, o[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < kHC; ++i) {
                                o[i] = *reinterpret_cast<const uint4 *>(row + ((size_t)i * Hs + v * kVec) * 2);
                                unpack8(o[i], rf[i]);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < kHC; ++i)
#pragma unroll
                            for (int e = 0; e < 8; ++e) ss = fmaf(rf[i][e], rf[i][e], ss);
                    }
                    if (kPost || v >= nvec_valid) {
#pragma unroll
                        for (int i = 0; i < kHC; ++i)
                            *reinterpret_cast<uint4 *>(row + ((size_t)i * Hs + v * kVec) * 2) = o[i];
                    }
                }
            }
            ss = warp_sum(ss);
            if (lane == 0) sSS[g] = ss;
        }
        __syncthreads();

        // ---- P2: projection partials; A fragments from TMEM, B from shared memory
        {
            float acc[2][3][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[nt][mt][q] = 0.f;
            const int ltok = 8 * ((lane >> 4) & 1) + (lane & 7);
            const int lk = 8 * ((lane >> 3) & 1);
            const uint32_t sR_u32 = smem_u32(sRb);
            for (int s = s_begin; s < s_end; ++s) {
                uint32_t a[16];
                tmem_ld16(tw + (uint32_t)((s - s_begin) * kColsPerStep), a);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(sR_u32 + (uint32_t)(ltok * rowb + (size_t)(16 * s + lk) * 2), b0, b1, b2, b3);
                tmem_wait_ld();
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) {
                    mma_bf16(acc[0][mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], b0, b1);
                    mma_bf16(acc[1][mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], b2, b3);
                }
            }
            float *zw = sZ + (size_t)warp * kG * kNumMix;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int g = nt * 8 + 2 * tig + e;
                    zw[g * kNumMix + gid] = acc[nt][0][e] + acc[nt][1][2 + e];
                    zw[g * kNumMix + gid + 8] = acc[nt][0][2 + e] + acc[nt][2][e];
                    zw[g * kNumMix + gid + 16] = acc[nt][1][e] + acc[nt][2][2 + e];
                }
            }
        }
        __syncthreads();
        for (int idx = tid; idx < kG * 32; idx += kNT) {
            const int g = idx >> 5, n = idx & 31;
            float v = 0.f;
            if (n < kNumMix) {
                for (int w = 0; w < kNW; ++w) v += sZ[((size_t)w * kG + g) * kNumMix + n];
            } else if (n == kNumMix) {
                v = sSS[g];
            }
            sPart[idx] = v;
        }
        cluster.sync();  // #1

        // ---- P3: the owner CTA of token g (g % 16 == c) reduces; pre pushed to all CTAs
        float zkeep = 0.f;
        const int g3 = c;  // 16 tokens, 16 CTAs: one token per CTA, handled by warp 0
        const bool owner = warp == 0 && g3 < gv;
        if (owner) {
            float acc = 0.f;
            if (lane <= kNumMix) {
                float v[kC];
#pragma unroll
                for (int q = 0; q < kC; ++q) v[q] = cluster.map_shared_rank(sPart, q)[g3 * 32 + lane];
#pragma unroll
                for (int q = 0; q < kC; ++q) acc += v[q];
            }
            const float ss = __shfl_sync(0xffffffffu, acc, kNumMix);
            const float r = 1.f / sqrtf(ss / (float)(kHC * H) + sc.hc_norm_eps);
            zkeep = r * acc;
            const float p = pre_head(zkeep, bias, mix_scales);
            if (lane < 4) {
                pre_out[(t0 + g3) * 4 + lane] = p;
#pragma unroll
                for (int q = 0; q < kC; ++q) cluster.map_shared_rank(sPre, q)[g3 * 4 + lane] = p;
            }
        }
        cluster_arrive();  // #2: pre of every token is in every CTA
        if (owner) {
            const float v = post_and_sinkhorn(zkeep, bias, mix_scales, sc);
            const int64_t t = t0 + g3;
            if (lane >= 4 && lane < 8) post_out[t * 4 + lane - 4] = v;
            else if (lane >= 8 && lane < 24) res_out[t * 16 + lane - 8] = v;
        }
        cluster_wait();

        // ---- P4: combine and square sum of X per token
        for (int g = warp; g < gv; g += kNW) {
            const float pre[kHC] = {sPre[g * 4], sPre[g * 4 + 1], sPre[g * 4 + 2], sPre[g * 4 + 3]};
            const unsigned char *row = sRb + g * rowb;
            float sx = 0.f;
            for (int v = lane; v < nvec_valid; v += 32) {
                float rf[kHC][8], x[8];
#pragma unroll
                for (int i = 0; i < kHC; ++i)
                    unpack8(*reinterpret_cast<const uint4 *>(row + ((size_t)i * Hs + v * kVec) * 2), rf[i]);
                combine_vec8(rf, pre, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) sx = fmaf(x[e], x[e], sx);
            }
            sx = warp_sum(sx);
            if (lane == 0) sXsq[g] = sx;
        }
        cluster.sync();  // #3

        for (int g = warp; g < gv; g += kNW) {
            float tot = 0.f;
            {
                float v[kC];
#pragma unroll
                for (int q = 0; q < kC; ++q) v[q] = cluster.map_shared_rank(sXsq, q)[g];
#pragma unroll
                for (int q = 0; q < kC; ++q) tot += v[q];
            }
            const float rstd = 1.f / sqrtf(tot / (float)H + sc.rmsnorm_eps);
            const float pre[kHC] = {sPre[g * 4], sPre[g * 4 + 1], sPre[g * 4 + 2], sPre[g * 4 + 3]};
            const unsigned char *row = sRb + g * rowb;
            const int64_t t = t0 + g;
            for (int v = lane; v < nvec_valid; v += 32) {
                float rf[kHC][8], x[8];
#pragma unroll
                for (int i = 0; i < kHC; ++i)
                    unpack8(*reinterpret_cast<const uint4 *>(row + ((size_t)i * Hs + v * kVec) * 2), rf[i]);
                combine_vec8(rf, pre, x);
                st_stream(X_out + t * (int64_t)H + h0 + v * kVec, norm_vec8(x, rstd, ld_ro(gamma + h0 + v * kVec)));
            }
        }
        // buffer b is refilled by bulk copies (async proxy) after the generic
        // writes above: order them, then release the buffer to warp 0
        fence_proxy_async_smem();
        __syncthreads();
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
    // a timed-out wait may leave copies in flight: wait for them once more (bounded)
#pragma unroll
    for (int b = 0; b < 2; ++b)
        if (pending[b] && !mbar_wait(&bars[b], phase[b])) timed_out = true;
    if (timed_out && lane == 0) atomicOr(status, 1u);
    tmem_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

std::mutex g_mu;

}  // namespace

int fused_tmem_slice(int H) { return ((H + 16 * kC - 1) / (16 * kC)) * 16; }

bool fused_tmem_supported(int H) {
    const int Hs = fused_tmem_slice(H);
    const int S = kHC * Hs / 16;
    const int spw = (S + kNW - 1) / kNW;
    return 4 * spw * kColsPerStep <= kTmemCols && Layout{Hs}.bytes() <= 227 * 1024;
}

size_t fused_tmem_pack_bytes(int H) {
    const int Hs = fused_tmem_slice(H);
    return (size_t)kC * (kHC * Hs / 16) * 96 * 16;
}

cudaError_t launch_fused_tmem(const FusedArgs &a, unsigned int *status, cudaStream_t stream) {
    const int Hs = fused_tmem_slice(a.H);
    if (!fused_tmem_supported(a.H)) return cudaErrorInvalidValue;
    const int64_t total = (int64_t)kC * (kHC * Hs / 16) * 96;
    launch_pack_phi(a.phi, a.H, kC, Hs, a.phi_pack, total, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const bool post = a.R_out != nullptr;
    auto kern = post ? fused_tmem_kernel<true> : fused_tmem_kernel<false>;
    const size_t smem = Layout{Hs}.bytes();
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
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int &mc = max_clusters[dev][post ? 1 : 0];
        if (mc == 0) {
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)) != cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
                return e;
            cfg.gridDim = dim3(kC);
            cfg.dynamicSmemBytes = 227 * 1024;  // one CTA per SM: TMEM is allocated whole
            int n = 0;
            if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
            mc = n;
        }
        cfg.gridDim = dim3((unsigned)(std::min<int64_t>((a.T + kG - 1) / kG, mc) * kC));
    }
    // one CTA per SM is required (the kernel allocates all 512 TMEM columns):
    // request the full shared memory so no second CTA fits.
    cfg.dynamicSmemBytes = std::max<size_t>(smem, 227 * 1024 / 2 + 1024);
    return cudaLaunchKernelEx(&cfg, kern, a.R, a.Y, a.prev_post, a.prev_comb, (const uint4 *)a.phi_pack, a.bias,
                              a.mix_scales, a.gamma, a.s, a.T, a.H, Hs, a.R_out, a.X_out, a.pre_out, a.post_out,
                              a.res_out, status);
}

}  // namespace mhc
