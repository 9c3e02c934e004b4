// Warp-specialised pipelined cluster schedule (schedule "ws"): the whole mHC
// post+pre step in one pass over HBM.
//
// A cluster of 16 CTAs (one per SM) owns groups of G = 8 tokens; CTA c owns
// the hidden slice [c*Hs, (c+1)*Hs) of each token (Hs a multiple of 64, at
// most 512).  Each role is its own set of warps, and the roles hand groups to
// one another through mbarriers only, so no role waits for another role's
// slowest warp and their latencies overlap:
//
//   producer (1 warp) : TMA tensor copies of group q (R as 64 x 8 x 4 boxes of
//                       4 KB, Y as 64 x 8 boxes, the previous mixes) into a
//                       5-deep ring once the combine has released the slot.
//   post (8 warps)    : warp t: token t of the group; R' = comb^T R + post Y in
//                       shared memory (R' overwrites R), R' to HBM.
//   projection (4)    : warp p: hidden blocks [p*Hs/4, (p+1)*Hs/4) of the
//                       slice, all four streams.  Per 16 hidden values two
//                       ldmatrix.x4 load the 8 tokens' R' of streams (0,1) and
//                       (2,3); the same fragments are the B operand of the
//                       projection (A = phi^T hi/lo fragments resident in
//                       tensor memory, mma.sync bf16, fp32 accumulate) and both
//                       operands of five Gram-matrix MMAs (R'_x . R'_j over the
//                       hidden values for the stream pairs, of which each token
//                       keeps its own diagonal entries).  The four warps' partials are summed
//                       into one 144-byte record per token (24 logits + 10 Gram
//                       entries) and sent to the token's owner CTA (st.async).
//   owner (1 warp)    : for the token this CTA owns in the group: sum the 16
//                       records, r, the pre and post heads, rstd of the combined
//                       row from the Gram matrix (sum_h X^2 = pre^T G pre),
//                       (pre, rstd) to all 16 CTAs; residual-mix logits kept.
//   combine (4 warps) : X = sum_i pre_i R'_i, RMSNorm * gamma, bf16 to HBM;
//                       then releases the ring slot to the producer.
// At the end all warps run the Sinkhorn normalisations of the owned tokens,
// one token per thread.
//
// Flow control: a ring slot is refilled only after the combine of the group
// that used it (which comes after that group's post and projection).  The
// owner's record buffer has two slots (its owned groups alternate); records
// of group q are sent only after (pre, rstd) of group q-4 arrived, which the
// owner sends after reading the slot.  The (pre, rstd) slots are 5 deep, and a
// group can only reach them after the combine of the group 5 earlier.
//
// Every mbarrier wait is bounded: on a timeout the CTA sets bit 0 of the
// status word and stops waiting (later waits give up at once), waits (again
// bounded) for its own tensor copies in flight, meets the cluster barrier at
// the end, frees its tensor memory and exits.
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

constexpr int kC = 16;                    // CTAs per cluster
constexpr int kG = 8;                     // tokens per group
constexpr int kP1 = kG;                   // post warps
constexpr int kP2 = 4;                    // projection warps (one tensor-memory lane quadrant each)
constexpr int kCB = 4;                    // combine warps
constexpr int kWP2 = kP1;                 // first projection warp
constexpr int kWCB = kP1 + kP2;           // first combine warp
constexpr int kWOwner = kP1 + kP2 + kCB;  // owner warp
constexpr int kWProd = kWOwner + 1;       // producer warp
constexpr int kNT = (kWProd + 1) * 32;
constexpr int kNBuf = 5;                  // ring of R / Y / mix tiles
constexpr int kNPre = 5;                  // (pre, rstd) slots; must be >= kNBuf
constexpr int kRec = 36;                  // floats per record: 24 logits, 10 Gram entries, 2 pad
constexpr int kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 25;
static_assert(kNPre >= kNBuf, "a (pre, rstd) slot is reused only after the combine of its last group");
static_assert(kWP2 % 4 == 0, "projection warp p must own tensor-memory lane quadrant p");

__device__ __forceinline__ void bwait(uint64_t *bar, uint32_t parity, bool &dead) {
    mbar_wait(bar, parity, dead, kWaitLimit);
}

// One k16 step's phi^T fragments (3 m-tiles x 4 registers) from tensor memory columns
// [col, col + 12) of this warp's lane quadrant.
__device__ __forceinline__ void tmem_ld12(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11])
                 : "r"(taddr + 8u)
                 : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- shared memory layout ---------------------------------------------------------
// Ring slot b: R' tile of nHB boxes of [stream 4][token 8][64 hidden] bf16 (4 KB each,
// TMA 128-byte swizzle), Y tile of nHB boxes [token 8][64 hidden], comb [8][16] and
// post [8][4] fp32.
struct Layout {
    int nHB;  // 64-wide hidden blocks per slice
    __host__ __device__ size_t rbuf() const { return (size_t)nHB * 4096; }
    __host__ __device__ size_t ybuf() const { return (size_t)nHB * 1024; }
    __host__ __device__ size_t r_off(int b) const { return (size_t)b * rbuf(); }
    __host__ __device__ size_t y_off(int b) const { return kNBuf * rbuf() + (size_t)b * ybuf(); }
    __host__ __device__ size_t comb_off(int b) const { return y_off(kNBuf) + (size_t)b * 512; }
    __host__ __device__ size_t post_off(int b) const { return comb_off(kNBuf) + (size_t)b * 128; }
    __host__ __device__ size_t part_off() const { return post_off(kNBuf); }                         // [2][kP2][8][36]
    __host__ __device__ size_t recv_off() const { return part_off() + (size_t)2 * kP2 * kG * kRec * 4; }  // [2][16][36]
    __host__ __device__ size_t prein_off() const { return recv_off() + (size_t)2 * kC * kRec * 4; }     // [kNPre][8][8]
    __host__ __device__ size_t gam_off() const { return prein_off() + (size_t)kNPre * kG * 8 * 4; }     // [Hs] bf16
    __host__ __device__ size_t bar_off() const { return gam_off() + (size_t)nHB * 64 * 2; }
    // full[kNBuf], postd[kNBuf], freeb[kNBuf], part_full[2], pre_full[kNPre]
    static constexpr int kBars = 3 * kNBuf + 2 + kNPre;
    __host__ __device__ size_t tmem_off() const { return bar_off() + (size_t)kBars * 8; }
    __host__ __device__ size_t bytes() const { return tmem_off() + 8; }
};

// Byte offset of 16-byte chunk c16 (8 hidden values) of (token t, stream j) in box hb.
// Box rows are stream-major (row = j*8 + t: the 8 tokens of one stream are consecutive
// rows, so an 8-token ldmatrix is conflict-free) when the tensor map could be encoded
// with the streams as the outer dimension, otherwise token-major (row = t*4 + j).
__device__ __forceinline__ uint32_t r_swz(int hb, int t, int j, int c16, bool jmajor) {
    const int row = jmajor ? j * 8 + t : t * 4 + j;
    return (uint32_t)(hb * 4096 + row * 128 + ((c16 ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t y_swz(int hb, int t, int c16) {
    return (uint32_t)(hb * 1024 + t * 128 + ((c16 ^ (t & 7)) << 4));
}

struct WsMaps {
    CUtensorMap R, Y, comb, post;
};

template <bool kPost>
__global__ void __launch_bounds__(kNT, 1)
ws_kernel(const __grid_constant__ WsMaps maps, const uint4 *__restrict__ phi_pack, const float *__restrict__ bias,
          const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma, Scalars sc, int64_t T, int H,
          int Hs, bool jmajor, uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out,
          float *__restrict__ pre_out, float *__restrict__ post_out, float *__restrict__ res_out,
          float *__restrict__ zstash, unsigned int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzled TMA boxes need a 1024-byte aligned base (1 KB of slack is allocated)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nHB = Hs / 64;
    const Layout L{nHB};
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float *sPart = reinterpret_cast<float *>(smem + L.part_off());
    float *sRecv = reinterpret_cast<float *>(smem + L.recv_off());
    float *sPreIn = reinterpret_cast<float *>(smem + L.prein_off());
    unsigned char *sGam = smem + L.gam_off();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off());
    uint64_t *full = bars, *postd = bars + kNBuf, *freeb = bars + 2 * kNBuf, *part_full = bars + 3 * kNBuf,
             *pre_full = bars + 3 * kNBuf + 2;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.tmem_off());
    // the projection and the combine wait for R' (post mode) or for the tile itself (pre only)
    uint64_t *rdy = kPost ? postd : full;

    const int h0 = c * Hs;
    const int nvec = Hs / kVec;  // <= 64
    const int64_t ngroups = (T + kG - 1) / kG;
    const int nclusters = gridDim.x / kC;
    const int cid = blockIdx.x / kC;
    const int n_it = cid < ngroups ? (int)((ngroups - cid + nclusters - 1) / nclusters) : 0;
    // token t of group q is owned by CTA (t + 8*(q&1)) % 16: CTAs 0-7 own in even groups, 8-15 in odd ones
    const int first_owned = c >= kG ? 1 : 0;
    const int nown = n_it > first_owned ? (n_it - first_owned + 1) / 2 : 0;
    auto group_t0 = [&](int q) { return (int64_t)(cid + (int64_t)q * nclusters) * kG; };
    bool dead = false;

    // ---- set-up
    if (warp == kWProd) {
        if (lane == 0) {
            for (int i = 0; i < kNBuf; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&postd[i], kP1);
                mbar_init(&freeb[i], kCB);
            }
            for (int i = 0; i < 2; ++i) mbar_init(&part_full[i], 1);
            for (int i = 0; i < kNPre; ++i) mbar_init(&pre_full[i], 1);
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
    if (warp >= kWP2 && warp < kWCB) {
        // phi^T fragments of this warp's hidden blocks: column (lb*4 + j)*16 holds the
        // 3 x 4 registers of k16 step s = j*(Hs/16) + p*nHB + lb
        const int p = warp - kWP2;
        const uint32_t tq = tbase + ((uint32_t)(32 * p) << 16);
        const uint4 *pack = phi_pack + (size_t)c * (kHC * Hs / 16) * 96;
        for (int lb = 0; lb < nHB; ++lb) {
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                const int s = j * (Hs / 16) + p * nHB + lb;
                uint32_t r[16];
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) {
                    const uint4 a = __ldg(pack + ((size_t)s * 3 + mt) * 32 + lane);
                    r[4 * mt] = a.x; r[4 * mt + 1] = a.y; r[4 * mt + 2] = a.z; r[4 * mt + 3] = a.w;
                }
                r[12] = r[13] = r[14] = r[15] = 0u;
                tmem_st16(tq + (uint32_t)((lb * 4 + j) * 16), r);
            }
        }
        tmem_wait_st();
    }
    if (warp >= kWCB && warp < kWOwner) {
        // this CTA's slice of the RMSNorm weight (zero beyond H)
        for (int v = tid - kWCB * 32; v < nvec; v += kCB * 32) {
            const int h = h0 + v * kVec;
            *reinterpret_cast<uint4 *>(sGam + v * 16) = h < H ? ld_ro(gamma + h) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (warp == kWProd && lane == 0) {
        // arm the message barriers for their first phases
        for (int i = 0; i < 2 && i < nown; ++i) mbar_arrive_expect_tx(&part_full[i], kC * kRec * 4);
        for (int i = 0; i < kNPre && i < n_it; ++i) mbar_arrive_expect_tx(&pre_full[i], kG * 32);
    }
    cluster.sync();  // every CTA's barriers exist before any message is sent

    if (warp == kWProd) {
        // ================================ producer
        if (lane == 0) {
            const uint32_t expect_bytes = (uint32_t)nHB * (4096 + (kPost ? 1024 : 0)) + (kPost ? 512 + 128 : 0);
            int issued = 0;
            for (int q = 0; q < n_it && !dead; ++q) {
                const int b = q % kNBuf;
                if (q >= kNBuf) bwait(&freeb[b], (uint32_t)((q / kNBuf - 1) & 1), dead);
                if (dead) break;
                const int t0 = (int)group_t0(q);
                mbar_arrive_expect_tx(&full[b], expect_bytes);
                for (int hb = 0; hb < nHB; ++hb) {
                    if (jmajor)
                        tma_load_3d(smem + L.r_off(b) + hb * 4096, &maps.R, h0 + hb * 64, t0, 0, &full[b]);
                    else
                        tma_load_3d(smem + L.r_off(b) + hb * 4096, &maps.R, h0 + hb * 64, 0, t0, &full[b]);
                    if (kPost) tma_load_2d(smem + L.y_off(b) + hb * 1024, &maps.Y, h0 + hb * 64, t0, &full[b]);
                }
                if (kPost) {
                    tma_load_2d(smem + L.comb_off(b), &maps.comb, 0, t0, &full[b]);
                    tma_load_2d(smem + L.post_off(b), &maps.post, 0, t0, &full[b]);
                }
                ++issued;
            }
            // the copies of the last kNBuf groups have landed (already true unless a wait timed out)
            bool drained = false;
            for (int q = issued > kNBuf ? issued - kNBuf : 0; q < issued; ++q)
                mbar_wait(&full[q % kNBuf], (uint32_t)((q / kNBuf) & 1), drained, kWaitLimit);
            dead = dead || drained;
        }
        __syncwarp();
    } else if (warp < kP1) {
        // ================================ post: token t = warp
        if (kPost) {
            const int t = warp;
            for (int q = 0; q < n_it; ++q) {
                const int b = q % kNBuf;
                bwait(&full[b], (uint32_t)((q / kNBuf) & 1), dead);
                const int64_t t0 = group_t0(q);
                unsigned char *rb = smem + L.r_off(b);
                float cm[kHC * kHC], pm[kHC];
                {
                    const float4 *cb = reinterpret_cast<const float4 *>(smem + L.comb_off(b)) + t * 4;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float4 f = cb[x];
                        cm[4 * x] = f.x; cm[4 * x + 1] = f.y; cm[4 * x + 2] = f.z; cm[4 * x + 3] = f.w;
                    }
                    const float4 f = *(reinterpret_cast<const float4 *>(smem + L.post_off(b)) + t);
                    pm[0] = f.x; pm[1] = f.y; pm[2] = f.z; pm[3] = f.w;
                }
                const bool valid_t = t0 + t < T;
                for (int v = lane; v < nvec; v += 32) {
                    const int hb = v >> 3, ch = v & 7;
                    uint4 r4[kHC], o[kHC];
                    float rf[kHC][8];
#pragma unroll
                    for (int j = 0; j < kHC; ++j) r4[j] = *reinterpret_cast<const uint4 *>(rb + r_swz(hb, t, j, ch, jmajor));
                    const uint4 y = *reinterpret_cast<const uint4 *>(smem + L.y_off(b) + y_swz(hb, t, ch));
                    post_vec8_x2(r4, y, cm, pm, o, rf);
#pragma unroll
                    for (int j = 0; j < kHC; ++j) *reinterpret_cast<uint4 *>(rb + r_swz(hb, t, j, ch, jmajor)) = o[j];
                    const int h = h0 + v * kVec;
                    if (valid_t && h < H) {
                        const int64_t base = (t0 + t) * kHC * (int64_t)H + h;
#pragma unroll
                        for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&postd[b]);
            }
        }
    } else if (warp < kWCB) {
        // ================================ projection + Gram partials, records
        const int p = warp - kWP2, pt = tid - kWP2 * 32;
        const int gid = lane >> 2, tig = lane & 3;
        const uint32_t tq = tbase + ((uint32_t)(32 * p) << 16);
        // ldmatrix.x4 lane address: matrices (stream i0, k 0-7), (i0+1, k 0-7), (i0, k 8-15), (i0+1, k 8-15),
        // row = token lane & 7
        const int lj = (lane >> 3) & 1, lt = lane & 7, lk = 8 * (lane >> 4);
        // the lanes holding a diagonal (token == token) entry of the Gram tiles: token gid, when gid/2 == tig
        const bool gdiag = (gid >> 1) == tig;
        const int gsel = gid & 1;
        for (int q = 0; q < n_it; ++q) {
            const int b = q % kNBuf;
            bwait(&rdy[b], (uint32_t)((q / kNBuf) & 1), dead);
            const uint32_t rb32 = smem_u32(smem + L.r_off(b));
            float acc[3][4], gd[5][4];
#pragma unroll
            for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
#pragma unroll
            for (int g = 0; g < 5; ++g)
#pragma unroll
                for (int e = 0; e < 4; ++e) gd[g][e] = 0.f;
            int hh = 16 * p * nHB + lk;  // this lane's hidden offset within the slice
            for (int lb = 0; lb < nHB; ++lb, hh += 16) {
                const int hb = hh >> 6, ch = (hh & 63) >> 3;
                uint32_t f[4], g[4];
                ldmatrix_x4(rb32 + r_swz(hb, lt, lj, ch, jmajor), f);      // streams 0, 1
                ldmatrix_x4(rb32 + r_swz(hb, lt, 2 + lj, ch, jmajor), g);  // streams 2, 3
                // Gram tiles: A rows are (stream x, token) for m < 8 and (stream y, token) for
                // m >= 8, B columns (stream j, token); 5 MMAs cover the 10 distinct pairs:
                // (0,2|0) (1,3|1) (2,1|2) (3,2|3) (1,3|0)
                mma_bf16(gd[0], f[0], g[0], f[2], g[2], f[0], f[2]);
                mma_bf16(gd[1], f[1], g[1], f[3], g[3], f[1], f[3]);
                mma_bf16(gd[2], g[0], f[1], g[2], f[3], g[0], g[2]);
                mma_bf16(gd[3], g[1], g[0], g[3], g[2], g[1], g[3]);
                mma_bf16(gd[4], f[1], g[1], f[3], g[3], f[0], f[2]);
                // projection: k16 steps of streams 0-3 at these 16 hidden values
#pragma unroll
                for (int jp = 0; jp < kHC; jp += 2) {
                    uint32_t a[24];
                    tmem_ld12(tq + (uint32_t)((lb * 4 + jp) * 16), a);
                    tmem_ld12(tq + (uint32_t)((lb * 4 + jp + 1) * 16), a + 12);
                    tmem_wait_ld();
                    const uint32_t b00 = jp ? g[0] : f[0], b01 = jp ? g[2] : f[2];
                    const uint32_t b10 = jp ? g[1] : f[1], b11 = jp ? g[3] : f[3];
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt)
                        mma_bf16(acc[mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], b00, b01);
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt)
                        mma_bf16(acc[mt], a[12 + 4 * mt], a[13 + 4 * mt], a[14 + 4 * mt], a[15 + 4 * mt], b10, b11);
                }
            }
            // partials of this warp: [token][24 logits (hi + lo rows), 10 Gram entries, 2 pad]
            float *pw = sPart + ((size_t)((q & 1) * kP2 + p) * kG) * kRec;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 2 * tig + e;
                pw[t * kRec + gid] = acc[0][e] + acc[1][2 + e];
                pw[t * kRec + gid + 8] = acc[0][2 + e] + acc[2][e];
                pw[t * kRec + gid + 16] = acc[1][e] + acc[2][2 + e];
            }
            if (gdiag) {
                // D[m][n]: rows m < 8 are stream x of token m, rows m >= 8 stream y; this lane
                // holds rows gid and gid + 8 at column gid
                float u[5], w[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    u[k] = gsel ? gd[k][1] : gd[k][0];
                    w[k] = gsel ? gd[k][3] : gd[k][2];
                }
                float *gq = pw + gid * kRec + kNumMix;
                // order (0,0) (1,1) (2,2) (3,3) (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
                gq[0] = u[0]; gq[1] = u[1]; gq[2] = u[2]; gq[3] = u[3];
                gq[4] = u[4]; gq[5] = w[0]; gq[6] = w[4]; gq[7] = w[2]; gq[8] = w[1]; gq[9] = w[3];
                gq[10] = 0.f; gq[11] = 0.f;
            }
            named_sync(2, kP2 * 32);
            if (pt < kG * (kRec / 4)) {
                // chunk qq of token t: sum of the warps' partials, sent to the owner's record slot
                const int t = pt / (kRec / 4), qq = pt % (kRec / 4);
                float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w2 = 0; w2 < kP2; ++w2) {
                    const float4 x = *reinterpret_cast<const float4 *>(
                        sPart + ((size_t)((q & 1) * kP2 + w2) * kG + t) * kRec + 4 * qq);
                    s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
                }
                // the owner has read its slot for group q-4 once (pre, rstd) of q-4 arrived
                if (q >= 4) bwait(&pre_full[(q - 4) % kNPre], (uint32_t)(((q - 4) / kNPre) & 1), dead);
                const uint32_t owner = (uint32_t)((t + 8 * (q & 1)) % kC);
                const int slot = (q >> 1) & 1;
                const uint32_t raddr = mapa(smem_u32(sRecv + ((size_t)slot * kC + c) * kRec + 4 * qq), owner);
                const uint32_t rbar = mapa(smem_u32(&part_full[slot]), owner);
                st_async16(raddr, rbar, make_uint4(__float_as_uint(s.x), __float_as_uint(s.y),
                                                   __float_as_uint(s.z), __float_as_uint(s.w)));
            }
        }
    } else if (warp < kWOwner) {
        // ================================ combine + RMSNorm
        const int ct = tid - kWCB * 32;
        constexpr int kStride = kCB * 32;
        // this thread's first item (token, vector) and the per-step advance, without divisions in the loop
        const int t_first = ct / nvec, v_first = ct % nvec, dt = kStride / nvec, dv = kStride % nvec;
        for (int q = 0; q < n_it; ++q) {
            const int b = q % kNBuf, s = q % kNPre;
            bwait(&rdy[b], (uint32_t)((q / kNBuf) & 1), dead);
            bwait(&pre_full[s], (uint32_t)((q / kNPre) & 1), dead);
            if (ct == 0 && q + kNPre < n_it) mbar_arrive_expect_tx(&pre_full[s], kG * 32);
            const int64_t t0 = group_t0(q);
            const unsigned char *rb = smem + L.r_off(b);
            int t = t_first, v = v_first;
            while (t < kG) {
                const int h = h0 + v * kVec;
                if (t0 + t < T && h < H) {
                    const float4 pr = *reinterpret_cast<const float4 *>(sPreIn + ((size_t)s * kG + t) * 8);
                    const float rstd = sPreIn[((size_t)s * kG + t) * 8 + 4];
                    const float pre[kHC] = {pr.x, pr.y, pr.z, pr.w};
                    float rf[kHC][8], x[8];
#pragma unroll
                    for (int j = 0; j < kHC; ++j)
                        unpack8(*reinterpret_cast<const uint4 *>(rb + r_swz(v >> 3, t, j, v & 7, jmajor)), rf[j]);
                    combine_vec8_x2(rf, pre, x);
                    st_stream(X_out + (t0 + t) * (int64_t)H + h,
                              norm_vec8(x, rstd, *reinterpret_cast<const uint4 *>(sGam + v * 16)));
                }
                t += dt;
                v += dv;
                if (v >= nvec) { v -= nvec; ++t; }
            }
            fence_proxy_async_smem();  // the slot is refilled by TMA after this
            __syncwarp();
            if (lane == 0) mbar_arrive(&freeb[b]);
        }
    } else {
        // ================================ owner
        for (int k = 0; k < nown; ++k) {
            const int q = first_owned + 2 * k, slot = k & 1;
            const int g = c - 8 * (q & 1);
            const int64_t t0 = group_t0(q);
            const bool valid = t0 + g < T;
            bwait(&part_full[slot], (uint32_t)((k >> 1) & 1), dead);
            // fixed-order sum over the 16 source CTAs: lane l takes float l, lanes 0-1 also
            // floats 32-33 (Gram entries 8 and 9)
            const float *rv = sRecv + (size_t)slot * kC * kRec;
            float a = 0.f, a2 = 0.f;
            for (int src = 0; src < kC; ++src) {
                a += rv[src * kRec + lane];
                if (lane < 2) a2 += rv[src * kRec + 32 + lane];
            }
            __syncwarp();
            if (lane == 0 && k + 2 < nown) mbar_arrive_expect_tx(&part_full[slot], kC * kRec * 4);
            float G[10];
#pragma unroll
            for (int e = 0; e < 8; ++e) G[e] = __shfl_sync(0xffffffffu, a, kNumMix + e);
            G[8] = __shfl_sync(0xffffffffu, a2, 0);
            G[9] = __shfl_sync(0xffffffffu, a2, 1);
            const float ss = (G[0] + G[1]) + (G[2] + G[3]);
            const float r = 1.f / sqrtf(ss / (float)(kHC * H) + sc.hc_norm_eps);
            const float z = r * a;
            const float pv = pre_head(z, bias, mix_scales);
            float pre[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pre[i] = __shfl_sync(0xffffffffu, pv, i);
            // sum_h X^2 = pre^T G pre
            float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] +
                       pre[3] * pre[3] * G[3];
            sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                         pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
            const float rstd = 1.f / sqrtf(fmaxf(sx, 0.f) / (float)H + sc.rmsnorm_eps);
            // (pre, rstd) to every CTA of the cluster: lane d < 16 sends to CTA d
            if (lane < kC) {
                const int s = q % kNPre;
                const uint32_t raddr = mapa(smem_u32(sPreIn + ((size_t)s * kG + g) * 8), (uint32_t)lane);
                const uint32_t rbar = mapa(smem_u32(&pre_full[s]), (uint32_t)lane);
                st_async16(raddr, rbar, make_uint4(__float_as_uint(pre[0]), __float_as_uint(pre[1]),
                                                   __float_as_uint(pre[2]), __float_as_uint(pre[3])));
                st_async16(raddr + 16, rbar, make_uint4(__float_as_uint(rstd), 0u, 0u, 0u));
            }
            if (valid) {
                const int64_t t = t0 + g;
                if (lane < 4) pre_out[t * 4 + lane] = pv;
                else if (lane < 8)
                    post_out[t * 4 + lane - 4] = sc.hc_post_scale / (1.f + expf(-(mix_scales[1] * z + bias[lane])));
                else if (lane < kNumMix) zstash[t * 16 + lane - 8] = z;  // residual-mix logits, normalised at the end
            }
        }
    }

    cluster.sync();  // all messages delivered; no CTA leaves while others may still write to it

    // ---- Sinkhorn of the tokens this CTA owned, one token per thread
    for (int k = tid; k < nown; k += kNT) {
        const int q = first_owned + 2 * k;
        const int64_t t = group_t0(q) + (c - 8 * (q & 1));
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
    const bool any_dead = __any_sync(0xffffffffu, dead);
    if (any_dead && lane == 0) atomicOr(status, 1u);
    tmem_fence_before();
    __syncthreads();
    if (warp == kWProd) tmem_dealloc(tbase, kTmemCols);
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
                   const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                   CUtensorMapSwizzle swz) {
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int ws_slice(int H) { return ((H + 64 * kC - 1) / (64 * kC)) * 64; }

bool ws_supported(int H) {
    const int Hs = ws_slice(H);
    // tensor memory: Hs/64 hidden blocks x 4 streams x 16 columns per projection warp
    return Hs <= kTmemCols && Hs / kVec <= 64 && Layout{Hs / 64}.bytes() + 1024 <= 227 * 1024;
}

size_t ws_pack_bytes(int H) {
    const int Hs = ws_slice(H);
    return (size_t)kC * (kHC * Hs / 16) * 96 * 16;
}

size_t ws_stash_bytes(int64_t T) { return (size_t)T * 16 * 4; }

cudaError_t launch_ws(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream) {
    if (!ws_supported(a.H)) return cudaErrorInvalidValue;
    const int Hs = ws_slice(a.H);
    const bool post = a.R_out != nullptr;
    EncodeTiledFn fn;
    cudaError_t e = get_encode(fn);
    if (e != cudaSuccess) return e;
    WsMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const cuuint64_t H = (cuuint64_t)a.H, T = (cuuint64_t)a.T;
    bool jmajor = true;
    {   // R [T][4][H] bf16 as (h, t, j) (box 64 x 8 x 4, stream-major rows in shared memory);
        // if the encoder refuses the non-monotonic strides, as (h, j, t) (box 64 x 4 x 8)
        const cuuint64_t dims[3] = {H, T, 4}, strides[2] = {H * 8, H * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kG, 4};
        if (encode(fn, &maps.R, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess) {
            jmajor = false;
            const cuuint64_t dims2[3] = {H, 4, T}, strides2[2] = {H * 2, H * 8};
            const cuuint32_t box2[3] = {64, 4, (cuuint32_t)kG};
            if ((e = encode(fn, &maps.R, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, dims2, strides2, box2,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
                return e;
        }
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

    const int64_t total = (int64_t)kC * (kHC * Hs / 16) * 96;
    launch_pack_phi(a.phi, a.H, kC, Hs, a.phi_pack, total, stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    auto kern = post ? ws_kernel<true> : ws_kernel<false>;
    const size_t smem = Layout{Hs / 64}.bytes() + 1024;  // + alignment slack
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
    // one CTA per SM (the kernel takes all 512 tensor-memory columns): always ask for
    // more than half of the SM's shared memory
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
                              a.H, Hs, jmajor, a.R_out, a.X_out, a.pre_out, a.post_out, a.res_out, zstash, status);
}

}  // namespace mhc
