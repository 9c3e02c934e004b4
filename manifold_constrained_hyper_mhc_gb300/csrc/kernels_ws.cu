// Warp-specialised pipelined cluster schedule (schedule "ws"): the whole mHC
// post+pre step in one pass over HBM.
//
// A cluster of 16 CTAs (one per SM) owns groups of G = 8 tokens; CTA c owns
// the hidden slice [c*Hs, (c+1)*Hs) of each token (Hs a multiple of 64, at
// most 512).  Each role is its own set of warps, and the roles hand groups to
// one another through mbarriers, so no role waits for another role's slowest
// warp and their latencies overlap:
//
//   post (7 warps)    : the group's (token, 8-value vector) items, two per
//                       thread; R' = comb^T R + post Y in shared memory (R'
//                       overwrites R), R' to HBM.
//   projection (7)    : warp p: tensor-memory lane quadrant (p + 7) % 4, a
//                       share of the slice's 16-wide blocks (at most four), all
//                       four streams.
//                       Per 16 hidden values two ldmatrix.x4 load the 8 tokens'
//                       R' of streams (0,1) and (2,3); the same fragments are the
//                       B operand of the projection (A = phi^T hi/lo fragments
//                       resident in tensor memory, mma.sync bf16, fp32
//                       accumulate) and both operands of six Gram-matrix MMAs
//                       (R'_i . R'_j over the hidden values for the stream
//                       pairs, of which each token keeps its own diagonal
//                       entries).  Each warp writes its partials to shared
//                       memory.
//   sender (1 warp)   : sums the seven warps' partials into one 144-byte record
//                       per token (24 logits + 10 Gram entries), sends it to the
//                       token's owner CTA (st.async), and refills the Y ring.
//   owner (1 warp)    : for the token this CTA owns in the group: sum the 16
//                       records, r, the pre and post heads, rstd of the combined
//                       row from the Gram matrix (sum_h X^2 = pre^T G pre),
//                       (pre, rstd) to all 16 CTAs; residual-mix logits kept.
//   combine (4 warps) : X = sum_i pre_i R'_i, RMSNorm * gamma, bf16 to HBM;
//                       then, the slot's last use being over, the four warps
//                       issue the TMA tensor copies of group q + 6 into it (R
//                       as 64 x 8 x 4 boxes of 4 KB; the sender copies Y as
//                       64 x 8 boxes and the previous mixes into the Y ring).
// At the end all warps run the Sinkhorn normalisations of the owned tokens,
// one token per thread.
//
// Flow control: a ring slot is refilled only after the combine of the group
// that used it (which comes after that group's post and projection).  The
// owner's record buffer has two slots (its owned groups alternate); records
// of group q are sent only after (pre, rstd) of group q-4 arrived, which the
// owner sends after reading the slot.  The (pre, rstd) slots are 6 deep, and a
// group can only reach them after the combine of the group 6 earlier.
//
// Every mbarrier wait is bounded: on a timeout the CTA sets bit 0 of the
// status word and stops waiting (later waits give up at once), issues no more
// copies, waits (again bounded) for its copies in flight, meets the cluster
// barrier at the end, frees its tensor memory and exits.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "mhc_device.cuh"
#include "mhc_kernels.h"
#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace mhc {

namespace {

using namespace ptx;

constexpr int kC = 16;                    // CTAs per cluster
constexpr int kG = 8;                     // tokens per group
constexpr int kP1 = 7;                    // post warps 0-6
constexpr int kWP2 = kP1;                 // projection warps 7-13
constexpr int kP2 = 7;
constexpr int kWOwner = kWP2 + kP2;       // owner warp (14)
constexpr int kWCB = kWOwner + 1;         // combine warps 15-18
constexpr int kCB = 4;
constexpr int kWSend = kWCB + kCB;        // sender warp (19): sums the projection partials, sends records
constexpr int kNT = (kWSend + 1) * 32;
constexpr int kMaxB16 = 4 * kP2;          // 16-wide hidden blocks per slice: at most four per projection warp
constexpr int kP1Items = (kG * kMaxB16 * 2 + kP1 * 32 - 1) / (kP1 * 32);  // post items per thread
constexpr int kCItems = (kG * kMaxB16 * 2 + kCB * 32 - 1) / (kCB * 32);   // combine items per thread
constexpr int kNBuf = 6;                  // ring of R tiles (R' in place), refilled after the combine
constexpr int kNY = 3;                    // ring of Y + previous-mix tiles, refilled after the projection
constexpr int kNPre = 6;                  // (pre, rstd) slots; must be >= kNBuf
constexpr int kRec = 36;                  // floats per record: 24 logits, 10 Gram entries, 2 pad
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait
static_assert(kNPre >= kNBuf, "a (pre, rstd) slot is reused only after the combine of its last group");

// phi [4H][24] fp32 -> per CTA rank c, k16-step s, m-tile mt, lane: the A
// fragment (4 x 32 bits, 8 bf16) of mma.m16n8k16 for the matrix
//   A[r][k] = hi(phi[k][r]) for r < 24, lo(phi[k][r-24]) for 24 <= r < 48,
// where hi = bf16(x), lo = bf16(x - hi), and the CTA-local k runs over
// (stream i, hidden h) as k_local = i*Hs + (h - c*Hs); zero where h >= H.
__global__ void __launch_bounds__(256)
pack_phi_kernel(const float *__restrict__ phi, int H, int C, int Hs, uint4 *__restrict__ out) {
    // a kernel launched after this one with programmatic stream serialization may start now;
    // it waits for this grid's results before reading them
    asm volatile("griddepcontrol.launch_dependents;");
    const int S = kHC * Hs / 16;
    const int64_t total = (int64_t)C * S * 3 * 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int lane = (int)(idx & 31);
    const int mt = (int)((idx >> 5) % 3);
    const int s = (int)((idx / 96) % S);
    const int c = (int)(idx / (96 * (int64_t)S));
    const int gid = lane >> 2, tig = lane & 3;
    auto val = [&](int r, int kl) -> float {
        const int i = kl / Hs, h = c * Hs + kl % Hs;
        if (h >= H) return 0.f;
        const float x = phi[((int64_t)i * H + h) * kNumMix + (r % kNumMix)];
        const float hi = __bfloat162float(__float2bfloat16_rn(x));
        return r < kNumMix ? hi : x - hi;
    };
    const int r0 = mt * 16 + gid, r1 = r0 + 8, k0 = 16 * s + 2 * tig;
    uint4 v;
    v.x = pack2_rn(val(r0, k0), val(r0, k0 + 1));
    v.y = pack2_rn(val(r1, k0), val(r1, k0 + 1));
    v.z = pack2_rn(val(r0, k0 + 8), val(r0, k0 + 9));
    v.w = pack2_rn(val(r1, k0 + 8), val(r1, k0 + 9));
    out[idx] = v;
}

__device__ __forceinline__ void bwait(uint64_t *bar, uint32_t parity, bool &dead) {
    mbar_wait_timed(bar, parity, dead, kWaitLimitNs);
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
// D = A x B (no accumulator input)
__device__ __forceinline__ void mma_bf16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
template <bool kFirst>
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    if constexpr (kFirst)
        mma_bf16_z(d, a0, a1, a2, a3, b0, b1);
    else
        mma_bf16(d, a0, a1, a2, a3, b0, b1);
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
    __host__ __device__ size_t comb_off(int b) const { return y_off(kNY) + (size_t)b * 512; }
    __host__ __device__ size_t post_off(int b) const { return comb_off(kNY) + (size_t)b * 128; }
    __host__ __device__ size_t part_off() const { return post_off(kNY); }                           // [2][kP2][8][36]
    __host__ __device__ size_t recv_off() const { return part_off() + (size_t)2 * kP2 * kG * kRec * 4; }  // [2][16][36]
    __host__ __device__ size_t prein_off() const { return recv_off() + (size_t)2 * kC * kRec * 4; }     // [kNPre][8][8]
    __host__ __device__ size_t gam_off() const { return prein_off() + (size_t)kNPre * kG * 8 * 4; }     // [Hs] bf16
    __host__ __device__ size_t bar_off() const { return gam_off() + (size_t)nHB * 64 * 2; }
    // full[kNBuf], postd[kNBuf], yfull[kNY], part_full[2], pre_full[kNPre], parts_ready[2], parts_free[2]
    static constexpr int kBars = 2 * kNBuf + kNY + 2 + kNPre + 4;
    __host__ __device__ size_t tmem_off() const { return bar_off() + (size_t)kBars * 8; }
    __host__ __device__ size_t bytes() const { return tmem_off() + 8; }
};

// R tile layout in shared memory.  Rows of 128 bytes (64 hidden values) hold one
// (stream j, 64-wide hidden block hb, token t); the TMA 128-byte swizzle puts 16-byte
// chunk c16 of a row at chunk c16 ^ (row % 8), and row % 8 = t in both layouts below,
// so the 8 tokens of one (j, hb) are 8 consecutive rows and an 8-token ldmatrix is
// conflict-free.
//   one box : a single 4-D copy [j 4][hb nHB][t 8][64]  (s_hb = 1024, s_j = nHB*1024)
//   per hb  : nHB 3-D copies   [hb nHB][j 4][t 8][64]  (s_hb = 4096, s_j = 1024)
struct RLayout {
    int s_hb, s_j;
    bool one_box;
};
__device__ __forceinline__ uint32_t r_swz(int hb, int t, int j, int c16, const RLayout &lay) {
    return (uint32_t)(hb * lay.s_hb + j * lay.s_j + t * 128 + ((c16 ^ t) << 4));
}
// Y tile: rows (hb, t), in both layouts.
__device__ __forceinline__ uint32_t y_swz(int hb, int t, int c16) {
    return (uint32_t)(hb * 1024 + t * 128 + ((c16 ^ (t & 7)) << 4));
}

struct WsMaps {
    CUtensorMap R, Y, comb, post;
};

template <bool kPost, bool kMx>
__global__ void __launch_bounds__(kNT, 1)
ws_kernel(const __grid_constant__ WsMaps maps, const uint4 *__restrict__ phi_pack, const float *__restrict__ bias,
          const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma, Scalars sc, int64_t T, int H,
          int Hs, RLayout lay, uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out,
          float *__restrict__ pre_out, float *__restrict__ post_out, float *__restrict__ res_out,
          float *__restrict__ zstash, unsigned int *__restrict__ redo_list, int64_t list_len,
          unsigned int *__restrict__ status, MxOut mx) {
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
    uint64_t *full = bars, *postd = bars + kNBuf, *yfull = postd + kNBuf, *part_full = yfull + kNY,
             *pre_full = part_full + 2,
             *parts_ready = pre_full + kNPre, *parts_free = parts_ready + 2;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.tmem_off());

    const int h0 = c * Hs;
    const int nvec = Hs / kVec;  // <= 56
    const int nB16 = Hs / 16;    // 16-wide hidden blocks of the slice, <= 28
    const int64_t ngroups = (T + kG - 1) / kG;
    const int nclusters = gridDim.x / kC;
    const int cid = blockIdx.x / kC;
    const int n_it = cid < ngroups ? (int)((ngroups - cid + nclusters - 1) / nclusters) : 0;
    // token t of group q is owned by CTA (t + 8*(q&1)) % 16: CTAs 0-7 own in even groups, 8-15 in odd ones
    const int first_owned = c >= kG ? 1 : 0;
    const int nown = n_it > first_owned ? (n_it - first_owned + 1) / 2 : 0;
    auto group_t0 = [&](int q) { return (int64_t)(cid + (int64_t)q * nclusters) * kG; };
    // the 16-wide blocks of projection warp p: [blk0(p), blk0(p) + nblk(p)), at most 4
    auto nblk = [&](int p) { return nB16 / kP2 + (p < nB16 % kP2 ? 1 : 0); };
    auto blk0 = [&](int p) { return p * (nB16 / kP2) + min(p, nB16 % kP2); };
    bool dead = false;

    // ---- set-up
    if (warp == kWOwner) {
        if (lane == 0) {
            for (int i = 0; i < kNY; ++i) mbar_init(&yfull[i], 1);
            for (int i = 0; i < kNBuf; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&postd[i], kP1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&part_full[i], 1);
                mbar_init(&parts_ready[i], kP2);
                mbar_init(&parts_free[i], 1);
            }
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
    // Up to here the kernel has touched only its own shared and tensor memory.  It is launched with
    // programmatic dependent launch, so this set-up may overlap the end of the launch before it on
    // the stream; from here on it reads and writes global memory, which that launch (the previous
    // call's kernels, the packing launch, or whatever else came before) may still be using: wait for
    // its completion.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the launches after this one (the token-tile kernel on the SMs the clusters leave idle, the
    // redo pass) may start now: they read the packed phi, complete by now, and neither waits for
    // this kernel before its end
    asm volatile("griddepcontrol.launch_dependents;");
    // the first groups' copies go out now, ahead of the phi fill and the cluster barrier: they
    // need only this CTA's barriers
    if (warp >= kWCB && warp < kWCB + kCB && lane == 0) {
        const int cw = warp - kWCB;
        for (int q = 0; q < kNBuf && q < n_it; ++q) {
            const int b = q % kNBuf;
            const int t0 = (int)group_t0(q);
            if (cw == 0) mbar_arrive_expect_tx(&full[b], (uint32_t)nHB * 4096);
            unsigned char *rs = smem + L.r_off(b);
            if (lay.one_box) {
                tma_load_4d(rs + cw * lay.s_j, &maps.R, 0, t0, h0 / 64, cw, &full[b]);
            } else {
                for (int hb = cw; hb < nHB; hb += kCB) tma_load_3d(rs + hb * 4096, &maps.R, h0 + hb * 64, t0, 0, &full[b]);
            }
        }
    }
    if (kPost && warp == kWSend && lane == 0) {
        const uint32_t ybytes = (uint32_t)nHB * 1024 + 512 + 128;
        for (int q = 0; q < kNY && q < n_it; ++q) {
            const int ys = q % kNY;
            const int t0 = (int)group_t0(q);
            mbar_arrive_expect_tx(&yfull[ys], ybytes);
            if (lay.one_box)
                tma_load_3d(smem + L.y_off(ys), &maps.Y, 0, t0, h0 / 64, &yfull[ys]);
            else
                for (int hb = 0; hb < nHB; ++hb)
                    tma_load_2d(smem + L.y_off(ys) + hb * 1024, &maps.Y, h0 + hb * 64, t0, &yfull[ys]);
            tma_load_2d(smem + L.comb_off(ys), &maps.comb, 0, t0, &yfull[ys]);
            tma_load_2d(smem + L.post_off(ys), &maps.post, 0, t0, &yfull[ys]);
        }
    }
    // projection warp p = warp - kWP2 keeps the phi^T fragments of its blocks in tensor-memory
    // lane quadrant warp % 4, after those of the lower projection warps of the same quadrant:
    // block i, stream j at column col0 + (i*4 + j)*16 (3 x 4 registers of k16 step
    // s = j*(Hs/16) + blk0(p) + i)
    uint32_t tq = 0;
    if (warp >= kWP2 && warp < kWP2 + kP2) {
        const int p = warp - kWP2;
        int col0 = 0;
        for (int p2 = 0; p2 < p; ++p2)
            if (((p2 + kWP2) & 3) == (warp & 3)) col0 += 64 * nblk(p2);
        tq = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col0;
        const uint4 *pack = phi_pack + (size_t)c * (kHC * Hs / 16) * 96;
        for (int i = 0; i < nblk(p); ++i) {
            // the block's 12 fragment loads in flight together (a tensor-memory store orders memory,
            // so loads issued after one wait for it)
            uint4 fa[kHC][3];
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                const int s = j * nB16 + blk0(p) + i;
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) fa[j][mt] = __ldg(pack + ((size_t)s * 3 + mt) * 32 + lane);
            }
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                uint32_t r[16];
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) {
                    r[4 * mt] = fa[j][mt].x; r[4 * mt + 1] = fa[j][mt].y; r[4 * mt + 2] = fa[j][mt].z; r[4 * mt + 3] = fa[j][mt].w;
                }
                r[12] = r[13] = r[14] = r[15] = 0u;
                tmem_st16(tq + (uint32_t)((i * 4 + j) * 16), r);
            }
        }
        tmem_wait_st();
    }
    if (warp >= kWCB && warp < kWCB + kCB) {
        // this CTA's slice of the RMSNorm weight (zero beyond H)
        for (int v = tid - kWCB * 32; v < nvec; v += kCB * 32) {
            const int h = h0 + v * kVec;
            *reinterpret_cast<uint4 *>(sGam + v * 16) = h < H ? ld_ro(gamma + h) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (warp == kWOwner && lane == 0) {
        // arm the message barriers for their first phases
        for (int i = 0; i < 2 && i < nown; ++i) mbar_arrive_expect_tx(&part_full[i], kC * kRec * 4);
        for (int i = 0; i < kNPre && i < n_it; ++i) mbar_arrive_expect_tx(&pre_full[i], kG * 32);
    }
    cluster.sync();  // every CTA's barriers exist before any message is sent

    if (warp < kP1) {
        // ================================ post: items (token, vector) pt + k * 224 of the group
        if (kPost) {
            // token-major items: thread tid works on token tid / kTPT, vectors tid % kTPT + kTPT * k, so
            // the token's mixes are loaded once per group; 8 consecutive lanes read and write 8
            // consecutive chunks of a 128-byte row.  The items are the same in every group: their offsets
            // are computed once.
            constexpr int kTPT = kP1 * 32 / kG;  // threads per token (28)
            const int p_tok = tid / kTPT;
            uint32_t p_roff[kP1Items], p_yoff[kP1Items];
            int p_goff[kP1Items];
            bool p_on[kP1Items];
#pragma unroll
            for (int k = 0; k < kP1Items; ++k) {
                const int v = tid % kTPT + kTPT * k;
                p_on[k] = v < nvec && h0 + v * kVec < H;
                p_roff[k] = r_swz(v >> 3, p_tok, 0, v & 7, lay);
                p_yoff[k] = y_swz(v >> 3, p_tok, v & 7);
                p_goff[k] = p_tok * kHC * H + h0 + v * kVec;
            }
            for (int q = 0; q < n_it; ++q) {
                const int b = q % kNBuf, ys = q % kNY;
                bwait(&full[b], (uint32_t)((q / kNBuf) & 1), dead);
                bwait(&yfull[ys], (uint32_t)((q / kNY) & 1), dead);
                unsigned char *rb = smem + L.r_off(b);
                const int64_t t0 = group_t0(q);
                uint16_t *rrow = R_out + t0 * kHC * (int64_t)H;
                float cm[kHC * kHC], pm[kHC];
                {
                    const float4 *cb = reinterpret_cast<const float4 *>(smem + L.comb_off(ys)) + p_tok * 4;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float4 f = cb[x];
                        cm[4 * x] = f.x; cm[4 * x + 1] = f.y; cm[4 * x + 2] = f.z; cm[4 * x + 3] = f.w;
                    }
                    const float4 f = *(reinterpret_cast<const float4 *>(smem + L.post_off(ys)) + p_tok);
                    pm[0] = f.x; pm[1] = f.y; pm[2] = f.z; pm[3] = f.w;
                }
                const int t = p_tok;
#pragma unroll
                for (int k = 0; k < kP1Items; ++k) {
                    if (p_on[k]) {
                        const float *cb = cm;
                        const float *pb = pm;
                        unsigned char *rp = rb + p_roff[k];
                        uint4 r4[kHC], o[kHC];
                        float rf[kHC][8];
#pragma unroll
                        for (int j = 0; j < kHC; ++j) r4[j] = *reinterpret_cast<const uint4 *>(rp + j * lay.s_j);
                        const uint4 y = *reinterpret_cast<const uint4 *>(smem + L.y_off(ys) + p_yoff[k]);
                        post_vec8_x2(r4, y, cb, pb, o, rf);
#pragma unroll
                        for (int j = 0; j < kHC; ++j) *reinterpret_cast<uint4 *>(rp + j * lay.s_j) = o[j];
                        if (t0 + t < T) {
                            uint16_t *dst = rrow + p_goff[k];
#pragma unroll
                            for (int i = 0; i < kHC; ++i) st_stream(dst + (int64_t)i * H, o[i]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&postd[b]);
            }
        }
    } else if (warp < kWP2 + kP2) {
        // ================================ projection + Gram partials of this warp's blocks, records
        const int p = warp - kWP2;
        const int nb = nblk(p), bstart = blk0(p);
        const int gid = lane >> 2, tig = lane & 3;
        // ldmatrix.x4 over the 8 tokens (row = token lane & 7) of streams (i0, i0+1) in the order
        // (i0, k 0-7) (i0, k 8-15) (i0+1, k 0-7) (i0+1, k 8-15): registers {0,1} and {2,3} are the B
        // fragments of streams i0 and i0+1, and {0,2,1,3} the A fragment of the 16 rows (stream i0
        // tokens, stream i0+1 tokens).  Streams (2, 3) are 2 * s_j bytes further.
        const int lt = lane & 7;
        const int bj = lane >> 4, bk = 8 * ((lane >> 3) & 1);  // stream offset, k offset
        auto lds_off = [&](int i, int j, int k) {
            const int h = 16 * (bstart + i) + k;
            return r_swz(h >> 6, lt, j, (h & 63) >> 3, lay);
        };
        const uint32_t s2j = 2u * (uint32_t)lay.s_j;
        // the lanes holding a diagonal (token == token) entry of the Gram tiles: token gid, when gid/2 == tig
        const bool gdiag = (gid >> 1) == tig;
        const int gsel = gid & 1;
        uint64_t *rdy = kPost ? postd : full;
        for (int q = 0; q < n_it; ++q) {
            const int b = q % kNBuf;
            bwait(&rdy[b], (uint32_t)((q / kNBuf) & 1), dead);
            const uint32_t rb32 = smem_u32(smem + L.r_off(b));
            float *pw = sPart + ((size_t)((q & 1) * kP2 + p) * kG) * kRec;
            // the sender has read this partial slot's previous group (q - 2)
            if (q >= 2) bwait(&parts_free[q & 1], (uint32_t)(((q - 2) >> 1) & 1), dead);
            // per block: one ldmatrix.x4 per stream pair feeds the Gram tiles D = A x B (A rows
            // (stream i0 | i0+1, token), B columns (stream j, token); tiles (0,1|0) (0,1|1) (0,1|2)
            // (0,1|3) (2,3|2) (2,3|3) cover the 10 distinct pairs) and the projection's k16 steps of
            // streams 0-3 (phi^T fragments from tensor memory, B = R')
            float gd[6][4], acc[3][4];
            auto block = [&](auto first_tag, int i) {
                constexpr bool kF = decltype(first_tag)::value;
                const uint32_t oB = lds_off(i, bj, bk);
                uint32_t f[4], g[4];
                ldmatrix_x4(rb32 + oB, f);
                ldmatrix_x4(rb32 + oB + s2j, g);
                uint32_t a[24];
                tmem_ld12(tq + (uint32_t)((i * 4) * 16), a);
                tmem_ld12(tq + (uint32_t)((i * 4 + 1) * 16), a + 12);
                // the A-order fragment of streams (i0, i0+1) is the B-order load permuted:
                // (i0 k0-7, i0+1 k0-7, i0 k8-15, i0+1 k8-15) = (f0, f2, f1, f3)
                mma_acc<kF>(gd[0], f[0], f[2], f[1], f[3], f[0], f[1]);
                mma_acc<kF>(gd[1], f[0], f[2], f[1], f[3], f[2], f[3]);
                mma_acc<kF>(gd[2], f[0], f[2], f[1], f[3], g[0], g[1]);
                tmem_wait_ld();
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
                    mma_acc<kF>(acc[mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], f[0], f[1]);
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
                    mma_bf16(acc[mt], a[12 + 4 * mt], a[13 + 4 * mt], a[14 + 4 * mt], a[15 + 4 * mt], f[2], f[3]);
                tmem_ld12(tq + (uint32_t)((i * 4 + 2) * 16), a);
                tmem_ld12(tq + (uint32_t)((i * 4 + 3) * 16), a + 12);
                // the rest of the Gram tiles cover the second tensor-memory load
                mma_acc<kF>(gd[3], f[0], f[2], f[1], f[3], g[2], g[3]);
                mma_acc<kF>(gd[4], g[0], g[2], g[1], g[3], g[0], g[1]);
                mma_acc<kF>(gd[5], g[0], g[2], g[1], g[3], g[2], g[3]);
                tmem_wait_ld();
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
                    mma_bf16(acc[mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], g[0], g[1]);
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
                    mma_bf16(acc[mt], a[12 + 4 * mt], a[13 + 4 * mt], a[14 + 4 * mt], a[15 + 4 * mt], g[2], g[3]);
            };
            if (nb > 0) {
                block(std::true_type{}, 0);
                for (int i = 1; i < nb; ++i) block(std::false_type{}, i);
            } else {
#pragma unroll
                for (int k = 0; k < 6; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) gd[k][e] = 0.f;
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
            }
            if (gdiag) {
                // D[m][n]: rows m < 8 are stream i0 of token m, rows m >= 8 stream i0+1; this lane
                // holds rows gid and gid + 8 at column gid
                float u[6], w[6];
#pragma unroll
                for (int k = 0; k < 6; ++k) {
                    u[k] = gsel ? gd[k][1] : gd[k][0];
                    w[k] = gsel ? gd[k][3] : gd[k][2];
                }
                float *gq = pw + gid * kRec + kNumMix;
                // order (0,0) (1,1) (2,2) (3,3) (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
                gq[0] = u[0]; gq[1] = w[1]; gq[2] = u[4]; gq[3] = w[5];
                gq[4] = u[1]; gq[5] = u[2]; gq[6] = u[3]; gq[7] = w[2]; gq[8] = w[3]; gq[9] = u[5];
                gq[10] = 0.f; gq[11] = 0.f;
            }
            // partial logits of this warp: [token][24 (hi + lo rows)]
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 2 * tig + e;
                pw[t * kRec + gid] = acc[0][e] + acc[1][2 + e];
                pw[t * kRec + gid + 8] = acc[0][2 + e] + acc[2][e];
                pw[t * kRec + gid + 16] = acc[1][e] + acc[2][2 + e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&parts_ready[q & 1]);
        }
    } else if (warp >= kWCB && warp < kWCB + kCB) {
        // ================================ combine + RMSNorm
        const int ct = tid - kWCB * 32, cw = warp - kWCB;
        constexpr int kStride = kCB * 32;
        uint64_t *rdy = kPost ? postd : full;
        // Tensor copies of group q's R tile into ring slot q % kNBuf, shared by the four combine warps
        // (one per SM sub-partition): warp cw copies stream cw (one box) or the 64-wide blocks
        // hb = cw mod 4 of the per-block layout.  Warp 0 sets the expected byte count.
        const uint32_t expect_bytes = (uint32_t)nHB * 4096;
        auto issue = [&](int q) {
            const int b = q % kNBuf;
            const int t0 = (int)group_t0(q);
            if (cw == 0) mbar_arrive_expect_tx(&full[b], expect_bytes);
            unsigned char *rs = smem + L.r_off(b);
            if (lay.one_box) {
                tma_load_4d(rs + cw * lay.s_j, &maps.R, 0, t0, h0 / 64, cw, &full[b]);
            } else {
                for (int hb = cw; hb < nHB; hb += kCB) tma_load_3d(rs + hb * 4096, &maps.R, h0 + hb * 64, t0, 0, &full[b]);
            }
        };

        // token-major items: thread ct works on token ct / kCPT, vectors ct % kCPT + kCPT * k, so the
        // token's (pre, rstd) is read once per group; offsets computed once.  With the MXFP8 output
        // the thread instead takes the four vectors of block b = ct % kCPT (at most 14 blocks of
        // 32 in a slice), vector j = (k + b / 2) % 4 of it at step k: the 16-byte chunks read by
        // lanes 0-7 (and 8-15) of one token then all differ, so the loads stay conflict-free, and
        // the block's scale needs no data from other lanes.
        constexpr int kCPT = kStride / kG;  // threads per token (16)
        static_assert(!kMx || kCItems == 4, "one block of four vectors per thread");
        const int c_tok = ct / kCPT;
        uint32_t c_roff[kCItems];
        int c_xoff[kCItems], c_v[kCItems], c_j[kCItems];
        bool c_on[kCItems];
#pragma unroll
        for (int k = 0; k < kCItems; ++k) {
            const int b = ct % kCPT;
            c_j[k] = (k + (b >> 1)) & 3;
            const int v = kMx ? 4 * b + c_j[k] : ct % kCPT + kCPT * k;
            c_on[k] = v < nvec && h0 + v * kVec < H;
            c_v[k] = v;
            c_roff[k] = r_swz(v >> 3, c_tok, 0, v & 7, lay);
            c_xoff[k] = c_tok * H + h0 + v * kVec;
        }
        const int c_scol = kMx ? mx_scale_col((h0 + (ct % kCPT) * 32) / 32) : 0;
        for (int q = 0; q < n_it; ++q) {
            const int b = q % kNBuf, s = q % kNPre;
            bwait(&rdy[b], (uint32_t)((q / kNBuf) & 1), dead);
            bwait(&pre_full[s], (uint32_t)((q / kNPre) & 1), dead);
            if (ct == 0 && q + kNPre < n_it) mbar_arrive_expect_tx(&pre_full[s], kG * 32);
            const int64_t t0 = group_t0(q);
            const unsigned char *rb = smem + L.r_off(b);
            const float *pin = sPreIn + (size_t)s * kG * 8;
            uint16_t *xrow = X_out + t0 * (int64_t)H;
            const float4 pr = *reinterpret_cast<const float4 *>(pin + c_tok * 8);
            const float rstd = pin[c_tok * 8 + 4];
            const float pre[kHC] = {pr.x, pr.y, pr.z, pr.w};
            const bool tok_ok = t0 + c_tok < T;
            uint8_t *const srow = kMx ? mx.scale + mx_scale_row(t0 + c_tok, H) : nullptr;
            uint8_t *const qrow = kMx ? mx.q + t0 * (int64_t)H : nullptr;
            uint4 ob[kCItems];
#pragma unroll
            for (int k = 0; k < kCItems; ++k) {
                ob[k] = make_uint4(0u, 0u, 0u, 0u);
                if (c_on[k] && tok_ok) {
                    const unsigned char *rp = rb + c_roff[k];
                    float rf[kHC][8], x[8];
#pragma unroll
                    for (int j = 0; j < kHC; ++j) unpack8(*reinterpret_cast<const uint4 *>(rp + j * lay.s_j), rf[j]);
                    combine_vec8_x2(rf, pre, x);
                    ob[k] = norm_vec8(x, rstd, *reinterpret_cast<const uint4 *>(sGam + c_v[k] * 16));
                    if (!kMx || X_out != nullptr) st_stream(xrow + c_xoff[k], ob[k]);
                }
            }
            // every use of the slot (post, projection, combine) is over: refill it with group q + kNBuf
            fence_proxy_async_smem();
            named_sync(3, kCB * 32);
            if (lane == 0 && q + kNBuf < n_it && !dead) issue(q + kNBuf);
            if (kMx && c_on[0] && tok_ok)  // from registers, after the refill; the block is in range or not as a whole
                mx_quantize_block(ob, c_j, mx.mode, qrow + c_xoff[0] - 8 * c_j[0], srow + c_scol);
        }
        if (lane == 0 && cw == 0) {
            // the copies of the last groups issued have landed (already true unless a wait timed out)
            bool drained = false;
            for (int q = n_it > kNBuf ? n_it - kNBuf : 0; q < n_it; ++q)
                mbar_wait_timed(&full[q % kNBuf], (uint32_t)((q / kNBuf) & 1), drained, kWaitLimitNs);
            dead = dead || drained;
        }
    } else if (warp == kWSend) {
        // ================================ sender: records of the group from the projection partials;
        // also refills the Y ring: once group q's partials are in, the post is done with Y slot
        // q % kNY, and lane 0 copies Y and the previous mixes of group q + kNY into it
        const uint32_t ybytes = (uint32_t)nHB * 1024 + 512 + 128;
        auto issue_y = [&](int q) {
            const int ys = q % kNY;
            const int t0 = (int)group_t0(q);
            mbar_arrive_expect_tx(&yfull[ys], ybytes);
            if (lay.one_box)
                tma_load_3d(smem + L.y_off(ys), &maps.Y, 0, t0, h0 / 64, &yfull[ys]);
            else
                for (int hb = 0; hb < nHB; ++hb)
                    tma_load_2d(smem + L.y_off(ys) + hb * 1024, &maps.Y, h0 + hb * 64, t0, &yfull[ys]);
            tma_load_2d(smem + L.comb_off(ys), &maps.comb, 0, t0, &yfull[ys]);
            tma_load_2d(smem + L.post_off(ys), &maps.post, 0, t0, &yfull[ys]);
        };

        for (int q = 0; q < n_it; ++q) {
            bwait(&parts_ready[q & 1], (uint32_t)((q >> 1) & 1), dead);
            // chunk (token t, 16-byte piece qq) = lane + 32 k: sum of the warps' partials, fixed order
            float4 sum[3];
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int ch = lane + 32 * k;
                sum[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ch < kG * (kRec / 4)) {
                    const int t = ch / (kRec / 4), qq = ch % (kRec / 4);
#pragma unroll
                    for (int w2 = 0; w2 < kP2; ++w2) {
                        const float4 x = *reinterpret_cast<const float4 *>(
                            sPart + ((size_t)((q & 1) * kP2 + w2) * kG + t) * kRec + 4 * qq);
                        sum[k].x += x.x; sum[k].y += x.y; sum[k].z += x.z; sum[k].w += x.w;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&parts_free[q & 1]);
            // the owner has read its record slot for group q-4 once (pre, rstd) of q-4 arrived
            if (q >= 4) bwait(&pre_full[(q - 4) % kNPre], (uint32_t)(((q - 4) / kNPre) & 1), dead);
            const int slot = (q >> 1) & 1;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int ch = lane + 32 * k;
                if (ch < kG * (kRec / 4)) {
                    const int t = ch / (kRec / 4), qq = ch % (kRec / 4);
                    const uint32_t owner = (uint32_t)((t + 8 * (q & 1)) % kC);
                    const uint32_t raddr = mapa(smem_u32(sRecv + ((size_t)slot * kC + c) * kRec + 4 * qq), owner);
                    const uint32_t rbar = mapa(smem_u32(&part_full[slot]), owner);
                    st_async16(raddr, rbar, make_uint4(__float_as_uint(sum[k].x), __float_as_uint(sum[k].y),
                                                       __float_as_uint(sum[k].z), __float_as_uint(sum[k].w)));
                }
            }
            if (kPost && lane == 0 && q + kNY < n_it && !dead) {
                fence_proxy_async_smem();
                issue_y(q + kNY);
            }
        }
        if (kPost && lane == 0) {
            // the last Y copies issued have landed (already true unless a wait timed out)
            bool drained = false;
            for (int q = n_it > kNY ? n_it - kNY : 0; q < n_it; ++q)
                mbar_wait_timed(&yfull[q % kNY], (uint32_t)((q / kNY) & 1), drained, kWaitLimitNs);
            dead = dead || drained;
        }
    } else {
        // ================================ owner
        const float a_pre = mix_scales[0], a_post = mix_scales[1];
        const float bl = lane < kNumMix ? bias[lane] : 0.f;
        // the reductions' mean and the reciprocal square roots use a reciprocal multiply and the
        // correctly rounded rsqrt / rcp: within 1 ulp of the divide-based forms, and a shorter
        // dependent chain on the path every CTA's combine waits for
        const float inv_kh = 1.f / (float)(kHC * H), inv_h = 1.f / (float)H;
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
#pragma unroll
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
            const float r = __frsqrt_rn(ss * inv_kh + sc.hc_norm_eps);
            const float z = r * a;
            // pre head (lanes 0-3)
            const float pv = lane < 4 ? __frcp_rn(1.f + expf(-(a_pre * z + bl))) : 0.f;
            float pre[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pre[i] = __shfl_sync(0xffffffffu, pv, i);
            // sum_h X^2 = pre^T G pre
            float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] +
                       pre[3] * pre[3] * G[3];
            sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                         pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
            const float rstd = __frsqrt_rn(fmaxf(sx, 0.f) * inv_h + sc.rmsnorm_eps);
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
                // streams that cancel in X: the combine ran with this rstd; the token goes on the
                // list whose layer inputs redo_kernel recomputes with a direct sum after this
                // kernel (checked after the sends, off the path every CTA's combine waits for)
                if (lane == 0 && gram_cancels(sx, pre, G)) {
                    const unsigned int idx = atomicAdd(status + kRedoCountWord, 1u);
                    if (idx < (unsigned int)list_len) redo_list[idx] = (unsigned int)t;
                }
                if (lane < 4) pre_out[t * 4 + lane] = pv;
                else if (lane < 8)
                    post_out[t * 4 + lane - 4] = sc.hc_post_scale / (1.f + expf(-(a_post * z + bl)));
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
    if (warp == kWOwner) tmem_dealloc(tbase, kTmemCols);
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
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};  // one per dimension, up to rank 5
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int ws_slice(int H) { return ((H + 64 * kC - 1) / (64 * kC)) * 64; }

bool ws_supported(int H) {
    const int Hs = ws_slice(H);
    // at most four 16-wide blocks per projection warp (so at most 8 blocks, 512 tensor-memory
    // columns, per lane quadrant)
    return Hs / 16 <= kMaxB16 && Layout{Hs / 64}.bytes() + 1024 <= 227 * 1024;
}

size_t ws_pack_bytes(int H) {
    const int Hs = ws_slice(H);
    return (size_t)kC * (kHC * Hs / 16) * 96 * 16;
}

cudaError_t launch_ws_pack(const float *phi, int H, uint4 *out, cudaStream_t stream) {
    const int Hs = ws_slice(H);
    const int64_t total = (int64_t)kC * (kHC * Hs / 16) * 96;
    pack_phi_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(phi, H, kC, Hs, out);
    return cudaGetLastError();
}

// residual-mix logits [T][16] fp32, then the list of tokens for redo_kernel [T] u32
size_t ws_stash_bytes(int64_t T) { return (size_t)T * 16 * 4 + (size_t)T * 4; }

cudaError_t ws_resident_ctas(int H, bool post, int &ctas) {
    const Layout L{ws_slice(H) / 64};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static int cache[64][2];
    std::lock_guard<std::mutex> lock(g_mu);
    int &mc = cache[dev][post ? 1 : 0];
    if (mc == 0) {
        auto kern = post ? ws_kernel<true, false> : ws_kernel<false, false>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kC;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        q.gridDim = dim3(kC);
        q.blockDim = dim3(kNT);
        q.dynamicSmemBytes = std::max<size_t>(L.bytes() + 1024, 227 * 1024 / 2 + 1024);
        q.attrs = attr;
        q.numAttrs = 1;
        int n = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &q)) != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        mc = n;
    }
    ctas = mc * kC;
    return cudaSuccess;
}

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
    const int nHB = Hs / 64;
    RLayout lay{1024, nHB * 1024, true};
    // R [T][4][H] bf16 as (h % 64, t, h / 64, j), one box {64, 8, nHB, 1} per stream and group, and
    // Y [T][H] as (h % 64, t, h / 64), one box {64, 8, nHB} per group: needs H % 64 == 0
    // (otherwise a block would run into the next row instead of the zero fill)
    if (a.H % 64 != 0) lay.one_box = false;
    if (lay.one_box) {
        const cuuint64_t dims[4] = {64, T, H / 64, 4}, strides[3] = {H * 8, 128, H * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)kG, (cuuint32_t)nHB, 1};
        lay.one_box = encode(fn, &maps.R, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.R, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B) == cudaSuccess;
    }
    if (lay.one_box && post) {
        const cuuint64_t dims[3] = {64, T, H / 64}, strides[2] = {H * 2, 128};
        const cuuint32_t box[3] = {64, (cuuint32_t)kG, (cuuint32_t)nHB};
        lay.one_box = encode(fn, &maps.Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Y, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B) == cudaSuccess;
    }
    if (!lay.one_box) {
        // per 64-wide block: R as (h, t, j), box {64, 8, 4}; Y as (h, t), box {64, 8}
        lay = RLayout{4096, 1024, false};
        const cuuint64_t dims[3] = {H, T, 4}, strides[2] = {H * 8, H * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kG, 4};
        if ((e = encode(fn, &maps.R, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        if (post) {
            const cuuint64_t dy[2] = {H, T}, sy[1] = {H * 2};
            const cuuint32_t by[2] = {64, (cuuint32_t)kG};
            if ((e = encode(fn, &maps.Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Y, dy, sy, by,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
                return e;
        }
    }
    if (post) {
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

    if (!a.prepacked && (e = launch_ws_pack(a.phi, a.H, a.phi_pack, stream)) != cudaSuccess) return e;

    const bool mxo = a.mx.q != nullptr;
    auto kern = post ? (mxo ? ws_kernel<true, true> : ws_kernel<true, false>)
                     : (mxo ? ws_kernel<false, true> : ws_kernel<false, false>);
    const size_t smem = Layout{Hs / 64}.bytes() + 1024;  // + alignment slack
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static int max_clusters[64][4];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the set-up (barriers, tensor memory) overlaps the end of the
    // launch before this one (the packing launch, or the previous call's last kernel); the kernel
    // waits for that launch's completion (griddepcontrol.wait) before it touches global memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kNT);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.stream = stream;
    // one CTA per SM (the kernel takes all 512 tensor-memory columns): always ask for
    // more than half of the SM's shared memory
    cfg.dynamicSmemBytes = std::max<size_t>(smem, 227 * 1024 / 2 + 1024);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int &mc = max_clusters[dev][(post ? 1 : 0) + (mxo ? 2 : 0)];
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
    mark_main_kernel(stream, true);
    e = cudaLaunchKernelEx(&cfg, kern, maps, (const uint4 *)a.phi_pack, a.bias, a.mix_scales, a.gamma, a.s, a.T,
                           a.H, Hs, lay, a.R_out, a.X_out, a.pre_out, a.post_out, a.res_out, zstash, a.redo_list,
                           a.redo_len, status, a.mx);
    if (!a.side_follows) mark_main_kernel(stream, false);  // else after the side kernel
    return e;
}

}  // namespace mhc
