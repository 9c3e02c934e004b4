// The first layer's pre from its (T, H) input x ("mhc_pre_broadcast" with a (T, H) input, in
// "Paths on current main that still call DeepGEMM on SM12x"): the residual is four copies of x,
// so the whole step can be computed from x alone.  With R'_i = x for every stream i:
//
//   sum_{i,h} R'_i[h]^2            = 4 sum_h x[h]^2
//   flat(R') . phi[:, n]           = sum_h x[h] * phi_sum[h][n],  phi_sum[h][n] = sum_i phi[i*H + h][n]
//   X = sum_i pre_i R'_i           = sum_i pre_i x   (summed in the same order as the other schedules)
//   sum_h X^2 = pre^T G pre,         every G_ij = sum_h x^2
//
// One persistent kernel, one CTA per SM, walks tiles of 8 tokens.  A tile is read twice, as
// chunks of 8 tokens x 512 hidden values, through a ring of shared-memory buffers that one
// producer thread fills by TMA, in the order pass 1 (tile 0), then pass 1 (tile k) and pass 2
// (tile k - 1) for k = 1, 2, ..., then pass 2 (last tile), so a tile's heads are computed while
// the warps already run the previous tile's pass 2:
//   pass 1: a storer thread writes the chunk back out by TMA as the four residual streams (the
//           next layer's post reads them), and eight warps project it onto phi_sum (mma.sync
//           bf16: A = phi_sum^T split into bf16 hi + lo parts, pre-packed in fragment order by
//           pack_phisum_kernel; B = the chunk, tokens on the N = 8 side; fp32 accumulate) and
//           take the square sums (one more MMA: x times its own transpose, diagonal kept);
//   heads:  r, the pre and post heads and rstd per token; the residual-mix logits wait in the
//           workspace for the Sinkhorn pass at the end of the kernel;
//   pass 2: X = sum_i pre_i x, RMSNorm * gamma, bf16 to HBM.
// Pass 1 reads x with the L2 evict-last policy and the residual stores use evict-first, so pass 2
// finds the tile in L2: HBM moves 12H bytes per token (x once, the residual 8H, the layer input
// 2H) instead of the 20H of a materialised residual read back by the pre.
//
// Every mbarrier wait is bounded (1 s): on a timeout the thread sets bit 0 of the status word
// and stops waiting (later waits give up at once), and the producer waits (again bounded) for
// its copies in flight before the CTA exits.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "mhc_device.cuh"
#include "mhc_kernels.h"
#include "sm100_ptx.cuh"
#include "tma_encode.h"

namespace mhc {

namespace {

using namespace ptx;

constexpr int kTT = 8;                      // tokens per tile
constexpr int kCW = 512;                    // hidden values per chunk
constexpr int kCHB = kCW / 64;              // 64-wide blocks per chunk (one TMA box)
constexpr int kChunkBytes = kTT * kCW * 2;  // 8 KB
constexpr int kNCh = 6;                     // ring depth: a small ring leaves L1 to the fragment loads
constexpr int kCons = 8;                    // projection / combine warps
constexpr int kWProd = kCons, kWStore = kCons + 1;
constexpr int kNT = (kCons + 2) * 32;
constexpr int kKS = kCW / 16;               // k16 steps per chunk
constexpr int kKSW = kKS / kCons;           // k16 steps per warp and chunk
constexpr int kPart = 25;                   // floats per (warp, token) partial: 24 logits, square sum
constexpr uint64_t kWaitNs = 1000000000ull;
static_assert(kKS % kCons == 0, "whole k16 steps per warp");

__device__ __forceinline__ void bwait(uint64_t *bar, uint32_t parity, bool &dead) {
    mbar_wait_timed(bar, parity, dead, kWaitNs);
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory: the ring, the warps' partials, the heads of the tile, the barriers.
struct BLayout {
    __host__ __device__ static constexpr size_t ring() { return 0; }
    // [2][kCons][kTT][kPart] floats (by tile parity)
    __host__ __device__ static constexpr size_t part() { return (size_t)kNCh * kChunkBytes; }
    // [2][kTT][8] floats: pre 0-3, rstd (by tile parity)
    __host__ __device__ static constexpr size_t head() { return part() + (size_t)2 * kCons * kTT * kPart * 4; }
    // full[kNCh], empty[kNCh]
    __host__ __device__ static constexpr size_t bars() { return head() + (size_t)2 * kTT * 8 * 4; }
    __host__ __device__ static constexpr size_t bytes() { return bars() + (size_t)2 * kNCh * 8; }
};

struct BcastMaps {
    CUtensorMap x;  // x [T][H] as (h % 64, t, h / 64): box {64, 8, 8}
    CUtensorMap R;  // residual [T][4][H] as (h % 64, t, h / 64, stream): box {64, 8, 8, 1}
};

// phi_sum^T split into bf16 hi + lo, in the A-fragment order of mma m16n8k16 (rows = logits n,
// columns = hidden k; rows 24-31 are zero): per k16 step s and lane (gid = lane / 4, tig = lane % 4)
// three uint4, [s][j][lane]:
//   j = 0: rows 0-15 hi   {(gid, k0) (gid+8, k0) (gid, k0+8) (gid+8, k0+8)}, k0 = 16 s + 2 tig,
//          each a pair of consecutive k packed as bf16x2
//   j = 1: rows 0-15 lo   (same positions)
//   j = 2: rows 16-23     {hi (16+gid, k0), hi (16+gid, k0+8), lo (16+gid, k0), lo (16+gid, k0+8)}
// phi_sum is summed over the streams in fp32 in stream order; hi = bf16(v), lo = bf16(v - hi);
// zero for k >= H.
__global__ void __launch_bounds__(256)
pack_phisum_kernel(const float *__restrict__ phi, int H, int nks, uint4 *__restrict__ out) {
    // the main kernel, launched after this one with programmatic stream serialization, may
    // start now; it waits for this grid's results before reading them
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)nks * 96) return;
    const int lane = (int)(idx & 31), j = (int)((idx >> 5) % 3), s = (int)(idx / 96);
    const int gid = lane >> 2, tig = lane & 3;
    auto sum = [&](int n, int k) -> float {
        if (k >= H) return 0.f;
        float v = phi[(int64_t)k * kNumMix + n];
#pragma unroll
        for (int i = 1; i < kHC; ++i) v += phi[((int64_t)i * H + k) * kNumMix + n];
        return v;
    };
    auto part = [&](int n, int k, bool lo) -> float {
        const float v = sum(n, k);
        const float hi = __bfloat162float(__float2bfloat16_rn(v));
        return lo ? v - hi : hi;
    };
    const int k0 = 16 * s + 2 * tig;
    uint4 v;
    if (j < 2) {
        const bool lo = j == 1;
        v.x = pack2_rn(part(gid, k0, lo), part(gid, k0 + 1, lo));
        v.y = pack2_rn(part(gid + 8, k0, lo), part(gid + 8, k0 + 1, lo));
        v.z = pack2_rn(part(gid, k0 + 8, lo), part(gid, k0 + 9, lo));
        v.w = pack2_rn(part(gid + 8, k0 + 8, lo), part(gid + 8, k0 + 9, lo));
    } else {
        const int n = 16 + gid;
        v.x = pack2_rn(part(n, k0, false), part(n, k0 + 1, false));
        v.y = pack2_rn(part(n, k0 + 8, false), part(n, k0 + 9, false));
        v.z = pack2_rn(part(n, k0, true), part(n, k0 + 1, true));
        v.w = pack2_rn(part(n, k0 + 8, true), part(n, k0 + 9, true));
    }
    out[idx] = v;
}

__global__ void __launch_bounds__(kNT, 1)
bcast_pre_kernel(const __grid_constant__ BcastMaps maps, const uint4 *__restrict__ pack,
                 const float *__restrict__ bias, const float *__restrict__ mix_scales,
                 const uint16_t *__restrict__ gamma, Scalars sc, int64_t T, int H, uint16_t *__restrict__ X_out,
                 float *__restrict__ pre_out, float *__restrict__ post_out, float *__restrict__ res_out,
                 float *__restrict__ zstash, unsigned int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzled TMA boxes need a 1024-byte aligned base (1 KB of slack is allocated)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *ring = smem + BLayout::ring();
    float *sPart = reinterpret_cast<float *>(smem + BLayout::part());
    float *sHead = reinterpret_cast<float *>(smem + BLayout::head());
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + BLayout::bars());
    uint64_t *empty = full + kNCh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (T + kTT - 1) / kTT;
    const int nch = (H + kCW - 1) / kCW;
    const int nks = (H + 15) / 16;
    const int my_tiles = (int64_t)blockIdx.x < ntiles ? (int)((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    auto tile_t0 = [&](int k) { return ((int64_t)blockIdx.x + (int64_t)k * gridDim.x) * kTT; };
    bool dead = false;

    if (tid == 0) {
        for (int i = 0; i < kNCh; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCons + 1);  // the consumer warps and the storer
        }
        fence_mbar_init();
    }
    __syncthreads();

    // Every role walks the same sequence of chunks (pass 1 of tile k before pass 2 of tile k - 1);
    // chunk number seq sits in ring buffer seq % kNCh.  f(tile k, pass, chunk c, seq) per chunk.
    auto walk = [&](auto &&f) {
        int64_t seq = 0;
        for (int k = 0; k <= my_tiles; ++k) {
            if (k < my_tiles)
                for (int c = 0; c < nch; ++c, ++seq) f(k, 0, c, seq);
            if (k >= 1)
                for (int c = 0; c < nch; ++c, ++seq) f(k - 1, 1, c, seq);
        }
    };
    if (warp == kWProd) {
        // ================================ producer: TMA loads into the ring
        if (lane == 0) {
            const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
            int64_t n_issued = 0;
            walk([&](int k, int pass, int c, int64_t seq) {
                const int buf = (int)(seq % kNCh);
                if (seq >= kNCh) bwait(&empty[buf], (uint32_t)(((seq / kNCh) - 1) & 1), dead);
                if (dead) return;
                mbar_arrive_expect_tx(&full[buf], kChunkBytes);
                tma_load_3d_hint(ring + (size_t)buf * kChunkBytes, &maps.x, 0, (int)tile_t0(k), c * kCHB, &full[buf],
                                 pass == 0 ? keep : drop);
                n_issued = seq + 1;
            });
            // the copies issued last have landed (already true unless a wait timed out)
            bool drained = false;
            for (int64_t q = n_issued > kNCh ? n_issued - kNCh : 0; q < n_issued; ++q)
                mbar_wait_timed(&full[q % kNCh], (uint32_t)((q / kNCh) & 1), drained, kWaitNs);
            dead = dead || drained;
        }
    } else if (warp == kWStore) {
        // ================================ storer: pass-1 chunks back out as the four residual streams
        if (lane == 0) {
            const uint64_t drop = l2_policy_evict_first();
            // buffers whose stores may still read them, oldest first; a buffer is released to the
            // producer once its stores have read it (at most two outstanding chunks)
            int pend0 = -1, pend1 = -1;
            walk([&](int k, int pass, int c, int64_t seq) {
                const int buf = (int)(seq % kNCh);
                bwait(&full[buf], (uint32_t)((seq / kNCh) & 1), dead);
                if (pass == 1 || dead) {
                    // nothing to store; release what is outstanding too, so no pass-1 buffer is
                    // held while the producer needs it for the chunks that follow
                    if (pend0 >= 0) {
                        bulk_wait_read<0>();
                        mbar_arrive(&empty[pend0]);
                        if (pend1 >= 0) mbar_arrive(&empty[pend1]);
                        pend0 = pend1 = -1;
                    }
                    mbar_arrive(&empty[buf]);
                    return;
                }
                const unsigned char *src = ring + (size_t)buf * kChunkBytes;
#pragma unroll
                for (int i = 0; i < kHC; ++i) tma_store_4d_hint(&maps.R, src, 0, (int)tile_t0(k), c * kCHB, i, drop);
                bulk_commit();
                if (pend1 >= 0) {
                    bulk_wait_read<2>();  // the oldest of the three outstanding groups is done reading
                    mbar_arrive(&empty[pend0]);
                    pend0 = pend1;
                    pend1 = buf;
                } else if (pend0 >= 0) {
                    pend1 = buf;
                } else {
                    pend0 = buf;
                }
            });
            bulk_wait_read<0>();
            if (pend0 >= 0) mbar_arrive(&empty[pend0]);
            if (pend1 >= 0) mbar_arrive(&empty[pend1]);
            bulk_wait<0>();  // the residual writes are complete before the CTA exits
        }
    } else {
        // ================================ consumers: projection + square sums, heads, combine
        const int gid = lane >> 2, tig = lane & 3;
        // the lanes holding a diagonal entry of the square-sum tile: token gid, when gid / 2 == tig
        const bool gdiag = (gid >> 1) == tig;
        const int gsel = gid & 1;
        // ldmatrix.x2: lanes 0-7 address token row lane & 7 at k 0-7 of the step, lanes 8-15 at k 8-15
        const int lt = lane & 7, lk = (lane >> 3) & 1;
        const float a_pre = mix_scales[0], a_post = mix_scales[1];
        // the mean and the reciprocal square roots as in the ws schedule: a reciprocal multiply and
        // the correctly rounded rsqrt / rcp
        const float inv_kh = 1.f / (float)(kHC * H), inv_h = 1.f / (float)H;
        // the packed phi_sum comes from the launch before this one (programmatic dependent launch)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int64_t seq = 0;
        // phi_sum fragments of this warp's k16 steps in chunk c (independent of the chunk's data)
        auto load_fr = [&](int c, uint4 (&f)[kKSW][3]) {
#pragma unroll
            for (int s = 0; s < kKSW; ++s) {
                const int ks = c * kKS + warp * kKSW + s;
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    f[s][j] = ks < nks ? __ldg(pack + ((size_t)ks * 3 + j) * 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        for (int k = 0; k <= my_tiles; ++k) {
            if (k < my_tiles) {
                // ---- pass 1 of tile k
                float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f}, gq[4] = {0.f, 0.f, 0.f, 0.f};
                auto chunk = [&](const uint4 (&fr)[kKSW][3]) {
                    const int buf = (int)(seq % kNCh);
                    bwait(&full[buf], (uint32_t)((seq / kNCh) & 1), dead);
                    const uint32_t base = smem_u32(ring + (size_t)buf * kChunkBytes);
#pragma unroll
                    for (int s = 0; s < kKSW; ++s) {
                        const int st = warp * kKSW + s;  // k16 step within the chunk
                        const int hb = st >> 2, g16 = (st & 3) * 2 + lk;
                        uint32_t b0, b1;
                        ldmatrix_x2(base + (uint32_t)(hb * 1024 + lt * 128 + ((g16 ^ lt) << 4)), b0, b1);
                        const uint4 h0 = fr[s][0], l0 = fr[s][1], m1 = fr[s][2];
                        mma16816(acc0, h0.x, h0.y, h0.z, h0.w, b0, b1);
                        mma16816(acc0, l0.x, l0.y, l0.z, l0.w, b0, b1);
                        mma16816(acc1, m1.x, 0u, m1.y, 0u, b0, b1);
                        mma16816(acc1, m1.z, 0u, m1.w, 0u, b0, b1);
                        // square sums: A = x (tokens in rows 0-7 and again in rows 8-15), B = x^T
                        mma16816(gq, b0, b0, b1, b1, b0, b1);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[buf]);
                    ++seq;
                };
                // the next chunk's fragments are in flight while this chunk is worked on
                uint4 fa[kKSW][3], fb[kKSW][3];
                load_fr(0, fa);
                for (int c = 0; c < nch; c += 2) {
                    if (c + 1 < nch) load_fr(c + 1, fb);
                    chunk(fa);
                    if (c + 1 < nch) {
                        if (c + 2 < nch) load_fr(c + 2, fa);
                        chunk(fb);
                    }
                }
                // this warp's partials: D[n][token] of the two logit tiles, the square-sum diagonal
                float *pw = sPart + ((size_t)(k & 1) * kCons + warp) * kTT * kPart;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * tig + e;
                    pw[t * kPart + gid] = acc0[e];
                    pw[t * kPart + gid + 8] = acc0[2 + e];
                    pw[t * kPart + 16 + gid] = acc1[e];
                }
                if (gdiag) pw[gid * kPart + 24] = gsel ? gq[1] : gq[0];
            }
            // partials of tile k are in; the heads of tile k - 1 are too (warp 0 wrote them before
            // it got here)
            named_sync(1, kCons * 32);
            if (k < my_tiles && warp == 0 && lane < kTT) {
                // ---- heads of tile k, one thread per token
                const int t = lane;
                const int64_t tok = tile_t0(k) + t;
                const float *pk = sPart + (size_t)(k & 1) * kCons * kTT * kPart;
                float *hk = sHead + (size_t)(k & 1) * kTT * 8;
                float z[kNumMix], sx2 = 0.f;
#pragma unroll
                for (int n = 0; n < kNumMix; ++n) z[n] = 0.f;
#pragma unroll
                for (int w = 0; w < kCons; ++w) {
                    const float *pp = pk + ((size_t)w * kTT + t) * kPart;
#pragma unroll
                    for (int n = 0; n < kNumMix; ++n) z[n] += pp[n];
                    sx2 += pp[24];
                }
                const float r = __frsqrt_rn((4.f * sx2) * inv_kh + sc.hc_norm_eps);
                float pre[kHC];
#pragma unroll
                for (int i = 0; i < kHC; ++i) pre[i] = __frcp_rn(1.f + expf(-(a_pre * (r * z[i]) + bias[i])));
                // sum_h X^2 = pre^T G pre with every Gram entry equal to sum_h x^2
                float sx = pre[0] * pre[0] * sx2 + pre[1] * pre[1] * sx2 + pre[2] * pre[2] * sx2 +
                           pre[3] * pre[3] * sx2;
                sx += 2.f * (pre[0] * pre[1] * sx2 + pre[0] * pre[2] * sx2 + pre[0] * pre[3] * sx2 +
                             pre[1] * pre[2] * sx2 + pre[1] * pre[3] * sx2 + pre[2] * pre[3] * sx2);
                const float rstd = __frsqrt_rn(fmaxf(sx, 0.f) * inv_h + sc.rmsnorm_eps);
#pragma unroll
                for (int i = 0; i < kHC; ++i) hk[t * 8 + i] = pre[i];
                hk[t * 8 + 4] = rstd;
                if (tok < T) {
#pragma unroll
                    for (int i = 0; i < kHC; ++i) {
                        pre_out[tok * 4 + i] = pre[i];
                        post_out[tok * 4 + i] =
                            sc.hc_post_scale / (1.f + expf(-(a_post * (r * z[4 + i]) + bias[4 + i])));
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) zstash[tok * 16 + e] = r * z[8 + e];  // normalised at the end
                }
            }
            if (k >= 1) {
                // ---- pass 2 of tile k - 1: items (token, 8-value vector) tid and tid + 256 of each chunk
                const int64_t t0 = tile_t0(k - 1);
                const float *hk = sHead + (size_t)((k - 1) & 1) * kTT * 8;
                const int ct = tid;  // < kCons * 32
                float pu[2][kHC], ru[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = (ct + kCons * 32 * u) >> 6;
#pragma unroll
                    for (int i = 0; i < kHC; ++i) pu[u][i] = hk[t * 8 + i];
                    ru[u] = hk[t * 8 + 4];
                }
                for (int c = 0; c < nch; ++c, ++seq) {
                    const int buf = (int)(seq % kNCh);
                    bwait(&full[buf], (uint32_t)((seq / kNCh) & 1), dead);
                    const unsigned char *cb = ring + (size_t)buf * kChunkBytes;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int v = ct + kCons * 32 * u;
                        const int t = v >> 6, j = v & 63, hb = j >> 3, g16 = j & 7;
                        const int h = c * kCW + hb * 64 + g16 * kVec;
                        if (t0 + t < T && h < H) {
                            float xf[8];
                            unpack8(*reinterpret_cast<const uint4 *>(cb + hb * 1024 + t * 128 + ((g16 ^ t) << 4)), xf);
                            const float rf[kHC][8] = {{xf[0], xf[1], xf[2], xf[3], xf[4], xf[5], xf[6], xf[7]},
                                                      {xf[0], xf[1], xf[2], xf[3], xf[4], xf[5], xf[6], xf[7]},
                                                      {xf[0], xf[1], xf[2], xf[3], xf[4], xf[5], xf[6], xf[7]},
                                                      {xf[0], xf[1], xf[2], xf[3], xf[4], xf[5], xf[6], xf[7]}};
                            float X[8];
                            combine_vec8_x2(rf, pu[u], X);
                            st_stream(X_out + (t0 + t) * (int64_t)H + h, norm_vec8(X, ru[u], ld_ro(gamma + h)));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[buf]);
                }
            }
        }
    }

    __syncthreads();  // every role is done; the tile heads' residual-mix logits are in zstash
    // ---- Sinkhorn of this CTA's tokens, one token per thread
    const float a_res = mix_scales[2];
    for (int i = tid; i < my_tiles * kTT; i += kNT) {
        const int64_t t = tile_t0(i / kTT) + (i % kTT);
        if (t >= T) continue;
        float M[16];
        const float4 *zs = reinterpret_cast<const float4 *>(zstash + t * 16);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float4 f = zs[x];
            M[4 * x] = f.x; M[4 * x + 1] = f.y; M[4 * x + 2] = f.z; M[4 * x + 3] = f.w;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) M[e] = expf(a_res * M[e] + bias[8 + e]);
        sinkhorn16(M, sc);
        float4 *ro = reinterpret_cast<float4 *>(res_out + t * 16);
#pragma unroll
        for (int x = 0; x < 4; ++x) ro[x] = make_float4(M[4 * x], M[4 * x + 1], M[4 * x + 2], M[4 * x + 3]);
    }
    if (__any_sync(0xffffffffu, dead) && lane == 0) atomicOr(status, 1u);
}

}  // namespace

bool bcast_supported(int64_t T, int64_t H) {
    // the (h % 64, t, h / 64) views need whole 64-wide blocks; token coordinates are 32-bit
    return H >= 64 && H % 64 == 0 && H <= (int64_t)1 << 20 && T >= 1 && T < ((int64_t)1 << 31) - kTT;
}

size_t bcast_pack_bytes(int64_t H) { return (size_t)((H + 15) / 16) * 3 * 32 * 16; }

size_t bcast_workspace_bytes(int64_t T, int64_t H) {
    return ((bcast_pack_bytes(H) + 255) & ~size_t(255)) + (size_t)T * 16 * 4;
}

cudaError_t launch_bcast_pre(const BcastArgs &a, unsigned int *status, void *scratch, int num_sms,
                             cudaStream_t stream) {
    if (!bcast_supported(a.T, a.H)) return cudaErrorInvalidValue;
    tma::EncodeTiledFn fn;
    cudaError_t e = tma::encoder(fn);
    if (e != cudaSuccess) return e;
    const cuuint64_t H = (cuuint64_t)a.H, T = (cuuint64_t)a.T;
    BcastMaps maps;
    std::memset(&maps, 0, sizeof maps);
    {
        const cuuint64_t dims[3] = {64, T, H / 64}, strides[2] = {H * 2, 128};
        const cuuint32_t box[3] = {64, (cuuint32_t)kTT, (cuuint32_t)kCHB};
        if ((e = tma::encode_bf16(fn, &maps.x, 3, a.x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    {
        const cuuint64_t dims[4] = {64, T, H / 64, 4}, strides[3] = {H * 8, 128, H * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)kTT, (cuuint32_t)kCHB, 1};
        if ((e = tma::encode_bf16(fn, &maps.R, 4, a.R_out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            cudaSuccess)
            return e;
    }
    uint4 *pack = static_cast<uint4 *>(scratch);
    float *zstash =
        reinterpret_cast<float *>(static_cast<char *>(scratch) + ((bcast_pack_bytes(a.H) + 255) & ~size_t(255)));
    const int nks = (a.H + 15) / 16;
    pack_phisum_kernel<<<(unsigned)((nks * 96 + 255) / 256), 256, 0, stream>>>(a.phi, a.H, nks, pack);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const size_t smem = BLayout::bytes() + 1024;  // + alignment slack
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        static std::mutex mu;
        static bool attr_set[64];
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if ((e = cudaFuncSetAttribute(bcast_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
                cudaSuccess)
                return e;
            attr_set[dev] = true;
        }
    }
    const int64_t ntiles = (a.T + kTT - 1) / kTT;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    // overlap the start (barriers, the first chunk loads and residual stores) with the packing
    // launch; the consumer warps wait for the packed phi_sum (griddepcontrol.wait)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(ntiles, std::max(num_sms, 1)));
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    mark_main_kernel(stream, true);
    e = cudaLaunchKernelEx(&cfg, bcast_pre_kernel, maps, (const uint4 *)pack, a.bias, a.mix_scales, a.gamma, a.s,
                           a.T, a.H, a.X_out, a.pre_out, a.post_out, a.res_out, zstash, status);
    mark_main_kernel(stream, false);
    return e;
}

}  // namespace mhc
