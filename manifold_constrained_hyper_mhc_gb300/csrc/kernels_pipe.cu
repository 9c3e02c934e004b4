// Pipelined cluster schedule: the whole mHC post+pre step in one pass over
// HBM, with no cluster-wide barrier in the steady state.
//
// A cluster of 16 CTAs (one per SM) owns groups of G = 8 tokens; CTA c owns
// the hidden slice [c*Hs, (c+1)*Hs) of each token (Hs a multiple of 64).
// Warps 0-15 are workers, warp 16 is the control warp.
//
//   control: issues the TMA tensor copies of group k+2 (R as 64x4x8 boxes of
//            4 KB, Y as 64x8 boxes, the previous mixes) into a triple buffer
//            once the workers released it; and, for the tokens this CTA owns
//            in group k, reduces the 16 partial records the CTAs sent it,
//            computes r, the pre head, rstd of the combined row, sends
//            (pre, rstd) to all 16 CTAs, then the post head and the Sinkhorn
//            residual mix, and writes the three mixes.
//   workers: group k: P1 post in shared memory (R' overwrites R in place),
//            R' to HBM, the 4x4 Gram matrix of the slice's streams; P2 the
//            projection partials on the tensor cores (mma.sync bf16, A =
//            phi^T hi/lo fragments resident in tensor memory, B = R' via
//            ldmatrix); one 144-byte record per token (24 logits + 10 Gram
//            entries) sent to the token's owner CTA with st.async; then the
//            combine + RMSNorm of group k-1, whose (pre, rstd) arrived while
//            group k was being computed.
//
// Messages between CTAs are st.async writes into the receiver's shared
// memory that complete bytes on the receiver's mbarrier, so a CTA waits only
// for the data it needs.  The square sum of X = sum_i pre_i R'_i over the row
// comes from the Gram matrix G of the bf16 streams (sum_h X^2 = pre^T G pre,
// an identity), so the combine needs no second reduction.
//
// Every mbarrier wait is bounded: on a timeout the CTA sets bit 0 of the
// status word and stops waiting (later waits give up at once), keeps to the
// cluster barrier at the end, frees its tensor memory and exits.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace cg = cooperative_groups;

namespace mhc {

namespace {

constexpr int kC = 16;                 // CTAs per cluster
constexpr int kG = 8;                  // tokens per group
constexpr int kWorkers = 16;           // worker warps
constexpr int kNT = (kWorkers + 1) * 32;
constexpr int kNBuf = 3;               // R' buffers (group k loading, k in P1/P2, k-1 in combine)
constexpr int kTmemCols = 512;
constexpr int kColsPerStep = 16;
constexpr int kRec = 36;               // floats per record: 24 logits, 10 Gram entries, 2 pad
constexpr uint32_t kWaitLimit = 1u << 25;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarriers ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
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
// Bounded wait.  After one timeout (`dead`), further waits give up at once.
__device__ __forceinline__ void mbar_wait(uint64_t *bar, uint32_t parity, bool &dead) {
    const uint32_t limit = dead ? 1u : kWaitLimit;
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return;
    dead = true;
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---- TMA tensor copies ---------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// ---- distributed shared memory messages ------------------------------------------
__device__ __forceinline__ uint32_t mapa(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// 16 bytes into another CTA's shared memory, completing 16 bytes on its mbarrier.
__device__ __forceinline__ void st_async16(uint32_t raddr, uint32_t rbar, uint4 v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(
                     raddr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
                 : "memory");
}

// ---- tensor memory -----------------------------------------------------------------
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
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kWorkers * 32) : "memory"); }

// ---- shared memory layout ---------------------------------------------------------
// R' buffer of one group: nHB boxes of [token 8][stream 4][64 hidden] bf16, each
// box 4 KB with the TMA 128-byte swizzle (16-byte chunk index XOR row % 8).
struct Layout {
    int nHB;  // 64-wide hidden blocks per slice
    __host__ __device__ size_t rbuf() const { return (size_t)nHB * 4096; }
    __host__ __device__ size_t ybuf() const { return (size_t)nHB * 1024; }
    __host__ __device__ size_t r_off(int b) const { return (size_t)b * rbuf(); }
    __host__ __device__ size_t y_off(int b) const { return kNBuf * rbuf() + (size_t)b * ybuf(); }
    __host__ __device__ size_t comb_off(int b) const { return y_off(kNBuf) + (size_t)b * 512; }
    __host__ __device__ size_t post_off(int b) const { return comb_off(kNBuf) + (size_t)b * 128; }
    __host__ __device__ size_t z_off() const { return post_off(kNBuf); }                               // [16][8][24]
    __host__ __device__ size_t gram_off() const { return z_off() + (size_t)kWorkers * kG * kNumMix * 4; }  // [16][12]
    __host__ __device__ size_t rec_off() const { return gram_off() + (size_t)kWorkers * 12 * 4; }     // [8][36]
    __host__ __device__ size_t recv_off() const { return rec_off() + (size_t)kG * kRec * 4; }         // [16][36]
    __host__ __device__ size_t prein_off() const { return recv_off() + (size_t)kC * kRec * 4; }       // [2][8][8]
    __host__ __device__ size_t gam_off() const { return prein_off() + 2 * kG * 8 * 4; }       // [Hs] bf16
    __host__ __device__ size_t bar_off() const { return gam_off() + (size_t)nHB * 64 * 2; }
    // full[3], free[3], part_full, pre_full[2]
    __host__ __device__ size_t tmem_off() const { return bar_off() + 9 * 8; }
    __host__ __device__ size_t bytes() const { return tmem_off() + 8; }
};

// R box rows: stream-major (row = j*8 + t, the eight tokens of one stream are
// consecutive rows, so an ldmatrix over 8 tokens is conflict-free) when the
// tensor map could be encoded with the streams as the outer dimension,
// otherwise token-major (row = t*4 + j).
__device__ __forceinline__ uint32_t r_swz(int hb, int t, int j, int c16, bool jmajor) {
    const int row = jmajor ? j * 8 + t : t * 4 + j;
    return (uint32_t)(hb * 4096 + row * 128 + ((c16 ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t y_swz(int hb, int t, int c16) {
    return (uint32_t)(hb * 1024 + t * 128 + ((c16 ^ (t & 7)) << 4));
}

// Gram index order: (0,0) (1,1) (2,2) (3,3) (0,1) (0,2) (0,3) (1,2) (1,3) (2,3).
// Even and odd elements accumulate in the two halves of packed fp32 pairs.
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

// Warp sum of 10 per-lane values, as a butterfly reduce-scatter (12 shuffles
// instead of 50): each level hands half of the values still held to the
// partner lane and adds the half it keeps.  Afterwards lane l holds the total
// of value idx(l) (see gram_lane_index), or padding; fixed order.
__device__ __forceinline__ float gram_reduce_scatter(const float (&v)[10]) {
    const int lane = threadIdx.x & 31;
    // level 1 (xor 16): 10 -> 5
    float a[6];
    {
        const bool hi = lane & 16;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const float keep = hi ? v[5 + i] : v[i], give = hi ? v[i] : v[5 + i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
        }
        a[5] = 0.f;
    }
    // level 2 (xor 8): 6 -> 3
    float b[4];
    {
        const bool hi = lane & 8;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const float keep = hi ? a[3 + i] : a[i], give = hi ? a[i] : a[3 + i];
            b[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
        b[3] = 0.f;
    }
    // level 3 (xor 4): 4 -> 2
    float c2[2];
    {
        const bool hi = lane & 4;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float keep = hi ? b[2 + i] : b[i], give = hi ? b[i] : b[2 + i];
            c2[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
        }
    }
    // level 4 (xor 2): 2 -> 1
    float d;
    {
        const bool hi = lane & 2;
        const float keep = hi ? c2[1] : c2[0], give = hi ? c2[0] : c2[1];
        d = keep + __shfl_xor_sync(0xffffffffu, give, 2);
    }
    // level 5 (xor 1): both lanes end with the full sum
    return d + __shfl_xor_sync(0xffffffffu, d, 1);
}
// Which of the 10 values lane l holds after gram_reduce_scatter (-1: padding).
__device__ __forceinline__ int gram_lane_index(int lane) {
    // level 2 leaves values {0,1,2} (bit 3 clear) or {3,4} (bit 3 set) of each half,
    // levels 3-4 pick one of them (or padding) by bits 2 and 1
    const int base = (lane & 16) ? 5 : 0;
    const bool upper = lane & 8;
    const int bi = ((lane & 4) ? 2 : 0) + ((lane & 2) ? 1 : 0);
    if (bi >= (upper ? 2 : 3)) return -1;
    return base + (upper ? 3 : 0) + bi;
}

struct PipeMaps {
    CUtensorMap R, Y, comb, post;
};

template <bool kPost>
__global__ void __launch_bounds__(kNT, 1)
pipe_kernel(const __grid_constant__ PipeMaps maps, const uint4 *__restrict__ phi_pack,
            const float *__restrict__ bias, const float *__restrict__ mix_scales,
            const uint16_t *__restrict__ gamma, Scalars sc, int64_t T, int H, int Hs, bool jmajor,
            uint16_t *__restrict__ R_out, uint16_t *__restrict__ X_out, float *__restrict__ pre_out,
            float *__restrict__ post_out, float *__restrict__ res_out, float *__restrict__ zstash,
            unsigned int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzled TMA boxes need a 1024-byte aligned base (1 KB of slack is allocated)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nHB = Hs / 64;
    const Layout L{nHB};
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool control = warp == kWorkers;

    float *sZ = reinterpret_cast<float *>(smem + L.z_off());
    float *sGram = reinterpret_cast<float *>(smem + L.gram_off());
    float *sRec = reinterpret_cast<float *>(smem + L.rec_off());
    float *sRecv = reinterpret_cast<float *>(smem + L.recv_off());
    float *sPreIn = reinterpret_cast<float *>(smem + L.prein_off());
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off());
    uint64_t *full = bars, *freeb = bars + 3, *part_full = bars + 6, *pre_full = bars + 7;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.tmem_off());
    unsigned char *sGam = smem + L.gam_off();

    const int h0 = c * Hs;
    const int nvec = Hs / kVec;                          // <= 64
    const int S = kHC * Hs / 16;                         // k16 steps of the slice
    const int spw = (S + kWorkers - 1) / kWorkers;       // <= 8 (checked on the host)
    const int64_t ngroups = (T + kG - 1) / kG;
    const int nclusters = gridDim.x / kC;
    const int cid = blockIdx.x / kC;
    const int n_it = cid < ngroups ? (int)((ngroups - cid + nclusters - 1) / nclusters) : 0;
    // token t of the group in iteration `it` is owned by CTA (t + 8*(it&1)) % 16
    auto owned_token = [&](int it) { return c - 8 * (it & 1); };  // valid if in [0, 8)
    bool dead = false;

    // ---- set-up
    if (control) {
        if (lane == 0) {
            for (int i = 0; i < 3; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&freeb[i], kWorkers);
            }
            mbar_init(part_full, 1);
            mbar_init(&pre_full[0], 1);
            mbar_init(&pre_full[1], 1);
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
    const uint32_t tw = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * spw * kColsPerStep);
    const int s_begin = min(S, spw * warp), s_end = min(S, spw * (warp + 1));
    if (!control) {
        // this CTA's slice of the RMSNorm weight (zero beyond H)
        for (int v = tid; v < nvec; v += kWorkers * 32) {
            const int h = h0 + v * kVec;
            *reinterpret_cast<uint4 *>(sGam + v * 16) = h < H ? ld_ro(gamma + h) : make_uint4(0u, 0u, 0u, 0u);
        }
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
    if (control && lane == 0) {
        // arm the message barriers for their first phases
        int first_owned = -1;
        for (int it = 0; it < n_it && first_owned < 0; ++it)
            if (owned_token(it) >= 0 && owned_token(it) < kG) first_owned = it;
        if (first_owned >= 0) mbar_arrive_expect_tx(part_full, kC * kRec * 4);
        if (n_it > 0) mbar_arrive_expect_tx(&pre_full[0], kG * 32);
        if (n_it > 1) mbar_arrive_expect_tx(&pre_full[1], kG * 32);
    }
    cluster.sync();  // every CTA's barriers exist before any message is sent

    const uint32_t expect_bytes = (uint32_t)nHB * (4096 + (kPost ? 1024 : 0)) + (kPost ? 512 + 128 : 0);
    auto issue = [&](int it) {  // control lane 0: tensor copies of iteration `it` into buffer it % 3
        const int b = it % kNBuf, yb = b;
        const int64_t t0 = (int64_t)(cid + (int64_t)it * nclusters) * kG;
        mbar_arrive_expect_tx(&full[b], expect_bytes);
        for (int hb = 0; hb < nHB; ++hb) {
            if (jmajor)
                tma_load_3d(smem + L.r_off(b) + hb * 4096, &maps.R, h0 + hb * 64, (int)t0, 0, &full[b]);
            else
                tma_load_3d(smem + L.r_off(b) + hb * 4096, &maps.R, h0 + hb * 64, 0, (int)t0, &full[b]);
            if (kPost) tma_load_2d(smem + L.y_off(yb) + hb * 1024, &maps.Y, h0 + hb * 64, (int)t0, &full[b]);
        }
        if (kPost) {
            tma_load_2d(smem + L.comb_off(yb), &maps.comb, 0, (int)t0, &full[b]);
            tma_load_2d(smem + L.post_off(yb), &maps.post, 0, (int)t0, &full[b]);
        }
    };

    if (control) {
        // ================================ control warp
        if (lane == 0) {
            for (int it = 0; it < kNBuf - 1 && it < n_it; ++it) issue(it);
        }
        int owned_done = 0;
        for (int it = 0; it < n_it; ++it) {
            const int nxt = it + kNBuf - 1;
            if (nxt < n_it) {
                // buffer nxt % 3 was last used by iteration it - 1
                if (it >= 1) mbar_wait(&freeb[(it - 1) % kNBuf], (uint32_t)(((it - 1) / kNBuf) & 1), dead);
                if (lane == 0) issue(nxt);
                __syncwarp();
            }
            const int g = owned_token(it);
            if (g < 0 || g >= kG) continue;
            const int64_t t0 = (int64_t)(cid + (int64_t)it * nclusters) * kG;
            const bool valid = t0 + g < T;
            mbar_wait(part_full, (uint32_t)(owned_done & 1), dead);
            ++owned_done;
            // fixed-order sum over the 16 source CTAs: lane l < 32 takes float l,
            // lanes 0-1 also take floats 32-33 (Gram entries 8 and 9)
            float a = 0.f, a2 = 0.f;
            for (int q = 0; q < kC; ++q) {
                a += sRecv[q * kRec + lane];
                if (lane < 2) a2 += sRecv[q * kRec + 32 + lane];
            }
            __syncwarp();
            if (lane == 0) {
                // re-arm for this CTA's next owned iteration (it + 2), if any
                if (it + 2 < n_it) mbar_arrive_expect_tx(part_full, kC * kRec * 4);
            }
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
            // sum_h X^2 = pre^T G pre
            float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] +
                       pre[3] * pre[3] * G[3];
            sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                         pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
            const float rstd = 1.f / sqrtf(fmaxf(sx, 0.f) / (float)H + sc.rmsnorm_eps);
            // (pre, rstd) to every CTA of the cluster: lane q < 16 sends to CTA q
            if (lane < kC) {
                const int s = it & 1;
                const uint32_t laddr = smem_u32(sPreIn + ((size_t)s * kG + g) * 8);
                const uint32_t raddr = mapa(laddr, (uint32_t)lane);
                const uint32_t rbar = mapa(smem_u32(&pre_full[s]), (uint32_t)lane);
                st_async16(raddr, rbar, make_uint4(__float_as_uint(pre[0]), __float_as_uint(pre[1]),
                                                   __float_as_uint(pre[2]), __float_as_uint(pre[3])));
                st_async16(raddr + 16, rbar, make_uint4(__float_as_uint(rstd), 0u, 0u, 0u));
            }
            if (valid) {
                const int64_t t = t0 + g;
                if (lane < 4) pre_out[t * 4 + lane] = p;
                else if (lane < 8)
                    post_out[t * 4 + lane - 4] = sc.hc_post_scale / (1.f + expf(-(mix_scales[1] * z + bias[lane])));
                else if (lane < 24) zstash[t * 16 + lane - 8] = z;  // residual-mix logits, normalised at the end
            }
        }
    } else {
        // ================================ workers
        const int gid = lane >> 2, tig = lane & 3;
        auto combine = [&](int it) {
            const int b = it % kNBuf, s = it & 1;
            mbar_wait(&pre_full[s], (uint32_t)((it >> 1) & 1), dead);
            if (tid == 0 && it + 2 < n_it) mbar_arrive_expect_tx(&pre_full[s], kG * 32);
            const int64_t t0 = (int64_t)(cid + (int64_t)it * nclusters) * kG;
            const unsigned char *rb = smem + L.r_off(b);
            for (int item = tid; item < kG * nvec; item += kWorkers * 32) {
                const int t = item / nvec, v = item % nvec;
                const int h = h0 + v * kVec;
                if (t0 + t >= T || h >= H) continue;
                const float *pi = sPreIn + ((size_t)s * kG + t) * 8;
                const float pre[kHC] = {pi[0], pi[1], pi[2], pi[3]};
                const float rstd = pi[4];
                float rf[kHC][8], x[8];
#pragma unroll
                for (int j = 0; j < kHC; ++j)
                    unpack8(*reinterpret_cast<const uint4 *>(rb + r_swz(v >> 3, t, j, v & 7, jmajor)), rf[j]);
                combine_vec8_x2(rf, pre, x);
                st_stream(X_out + (t0 + t) * (int64_t)H + h,
                          norm_vec8(x, rstd, *reinterpret_cast<const uint4 *>(sGam + v * 16)));
            }
            fence_proxy_async_smem();  // the buffer is refilled by TMA after this
            __syncwarp();
            if (lane == 0) mbar_arrive(&freeb[b]);
        };

        for (int it = 0; it < n_it; ++it) {
            const int b = it % kNBuf, yb = b;
            const int64_t t0 = (int64_t)(cid + (int64_t)it * nclusters) * kG;
            mbar_wait(&full[b], (uint32_t)((it / kNBuf) & 1), dead);
            unsigned char *rb = smem + L.r_off(b);

            // ---- P1: post in place, R' to HBM, Gram partials.  Warp w: token w/2,
            // half w%2 of the slice's vectors (one vector per lane).
            {
                const int t = warp >> 1, half = warp & 1;
                const int nh = (nvec + 1) >> 1;
                const int v = half * nh + lane;
                float2 gm2[10];
#pragma unroll
                for (int q = 0; q < 10; ++q) gm2[q] = make_float2(0.f, 0.f);
                if (lane < nh && v < nvec) {
                    const int hb = v >> 3, ch = v & 7;
                    float rf[kHC][8];
                    if (kPost) {
                        uint4 r4[kHC], o[kHC];
#pragma unroll
                        for (int j = 0; j < kHC; ++j) r4[j] = *reinterpret_cast<const uint4 *>(rb + r_swz(hb, t, j, ch, jmajor));
                        const uint4 y = *reinterpret_cast<const uint4 *>(smem + L.y_off(yb) + y_swz(hb, t, ch));
                        const float *cb = reinterpret_cast<const float *>(smem + L.comb_off(yb)) + t * 16;
                        const float *pb = reinterpret_cast<const float *>(smem + L.post_off(yb)) + t * 4;
                        post_vec8_x2(r4, y, cb, pb, o, rf);
#pragma unroll
                        for (int j = 0; j < kHC; ++j) *reinterpret_cast<uint4 *>(rb + r_swz(hb, t, j, ch, jmajor)) = o[j];
                        const int h = h0 + v * kVec;
                        if (t0 + t < T && h < H) {
                            const int64_t base = (t0 + t) * kHC * (int64_t)H + h;
#pragma unroll
                            for (int i = 0; i < kHC; ++i) st_stream(R_out + base + (int64_t)i * H, o[i]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kHC; ++j)
                            unpack8(*reinterpret_cast<const uint4 *>(rb + r_swz(hb, t, j, ch, jmajor)), rf[j]);
                    }
                    gram_acc(rf, gm2);
                }
                float gm[10];
#pragma unroll
                for (int e = 0; e < 10; ++e) gm[e] = gm2[e].x + gm2[e].y;
                const float tot = gram_reduce_scatter(gm);
                const int gi = gram_lane_index(lane);
                if (gi >= 0 && (lane & 1) == 0) sGram[warp * 12 + gi] = tot;
            }
            workers_sync();

            // ---- P2: projection partials of this warp's k16 steps for the 8 tokens
            {
                float acc[3][4];
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[mt][q] = 0.f;
                const uint32_t rb32 = smem_u32(rb);
                const int lt = lane & 7, lk = 8 * ((lane >> 3) & 1);
                // k = 16 s + lk = j*Hs + h, advanced incrementally (Hs is a multiple of 64, steps of 16
                // never cross a stream)
                int sj = (16 * s_begin) / Hs, sh = (16 * s_begin) % Hs;
                auto bfrag = [&](int j, int h, uint32_t &b0, uint32_t &b1) {
                    const int hh = h + lk;
                    ldmatrix_x2(rb32 + r_swz(hh >> 6, lt, j, (hh & 63) >> 3, jmajor), b0, b1);
                };
                auto advance = [&]() {
                    sh += 16;
                    if (sh >= Hs) { sh -= Hs; ++sj; }
                };
                int s = s_begin;
                for (; s + 1 < s_end; s += 2) {  // two k16 steps per tensor-memory load
                    uint32_t a[32];
                    tmem_ld32(tw + (uint32_t)((s - s_begin) * kColsPerStep), a);
                    uint32_t b0, b1, b2, b3;
                    bfrag(sj, sh, b0, b1);
                    advance();
                    bfrag(sj, sh, b2, b3);
                    advance();
                    tmem_wait_ld();
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt) mma_bf16(acc[mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], b0, b1);
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt)
                        mma_bf16(acc[mt], a[16 + 4 * mt], a[17 + 4 * mt], a[18 + 4 * mt], a[19 + 4 * mt], b2, b3);
                }
                if (s < s_end) {
                    uint32_t a[16];
                    tmem_ld16(tw + (uint32_t)((s - s_begin) * kColsPerStep), a);
                    uint32_t b0, b1;
                    bfrag(sj, sh, b0, b1);
                    tmem_wait_ld();
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt) mma_bf16(acc[mt], a[4 * mt], a[4 * mt + 1], a[4 * mt + 2], a[4 * mt + 3], b0, b1);
                }
                float *zw = sZ + (size_t)warp * kG * kNumMix;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * tig + e;
                    zw[t * kNumMix + gid] = acc[0][e] + acc[1][2 + e];
                    zw[t * kNumMix + gid + 8] = acc[0][2 + e] + acc[2][e];
                    zw[t * kNumMix + gid + 16] = acc[1][e] + acc[2][2 + e];
                }
            }
            // ---- combine + RMSNorm of the previous group (overlaps other warps' MMA chains)
            if (it >= 1) combine(it - 1);
            workers_sync();

            // ---- records: 24 logits (sum over the 16 warps, fixed order) + 10 Gram entries
            for (int idx = tid; idx < kG * kRec; idx += kWorkers * 32) {
                const int t = idx / kRec, n = idx % kRec;
                float v = 0.f;
                if (n < kNumMix) {
                    for (int w = 0; w < kWorkers; ++w) v += sZ[((size_t)w * kG + t) * kNumMix + n];
                } else if (n < kNumMix + 10) {
                    v = sGram[(2 * t) * 12 + (n - kNumMix)] + sGram[(2 * t + 1) * 12 + (n - kNumMix)];
                }
                sRec[idx] = v;
            }
            workers_sync();
            if (tid < kG * (kRec / 4)) {
                const int t = tid / (kRec / 4), q = tid % (kRec / 4);
                const uint32_t owner = (uint32_t)((t + 8 * (it & 1)) % kC);
                const uint4 val = *reinterpret_cast<const uint4 *>(sRec + t * kRec + 4 * q);
                const uint32_t raddr = mapa(smem_u32(sRecv + c * kRec + 4 * q), owner);
                const uint32_t rbar = mapa(smem_u32(part_full), owner);
                st_async16(raddr, rbar, val);
            }

        }
        if (n_it >= 1) combine(n_it - 1);
    }

    cluster.sync();  // all messages delivered; no CTA leaves while others may still write to it

    // ---- Sinkhorn of the tokens this CTA owned, one token per thread
    {
        const int first = c >= 8 ? 1 : 0;
        const int nown = n_it > first ? (n_it - first + 1) / 2 : 0;
        for (int k = tid; k < nown; k += kNT) {
            const int it = first + 2 * k;
            const int64_t t = (int64_t)(cid + (int64_t)it * nclusters) * kG + (c - 8 * (it & 1));
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
    if (control) tmem_dealloc(tbase, kTmemCols);
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

int pipe_slice(int H) { return ((H + 64 * kC - 1) / (64 * kC)) * 64; }

bool pipe_supported(int H) {
    const int Hs = pipe_slice(H);
    const int S = kHC * Hs / 16;
    const int spw = (S + kWorkers - 1) / kWorkers;
    return 4 * spw * kColsPerStep <= kTmemCols && Hs / kVec <= 64 && Layout{Hs / 64}.bytes() <= 227 * 1024;
}

size_t pipe_pack_bytes(int H) {
    const int Hs = pipe_slice(H);
    return (size_t)kC * (kHC * Hs / 16) * 96 * 16;
}

size_t pipe_stash_bytes(int64_t T) { return (size_t)T * 16 * 4; }

cudaError_t launch_pipe(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream) {
    if (!pipe_supported(a.H)) return cudaErrorInvalidValue;
    const int Hs = pipe_slice(a.H);
    const bool post = a.R_out != nullptr;
    EncodeTiledFn fn;
    cudaError_t e = get_encode(fn);
    if (e != cudaSuccess) return e;
    PipeMaps maps;
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

    auto kern = post ? pipe_kernel<true> : pipe_kernel<false>;
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
    // one CTA per SM (the kernel takes all 512 TMEM columns): always ask for more
    // than half of the SM's shared memory
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
