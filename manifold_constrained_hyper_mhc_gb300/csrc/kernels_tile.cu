// Token-tile schedule (schedule "tile"): the whole fused mHC post+pre step for tiles of 18
// tokens, one CTA per SM, no clusters.  It runs on its own (every SM, H % 64 == 0, H > 256), or
// beside the ws schedule on the SMs that ws's 16-CTA clusters cannot use, on a share of the
// tokens (ws takes the leading tokens, this kernel the rest).
//
// A tile's row (4 streams x H) does not fit in shared memory, so it is walked twice in chunks of
// 18 tokens x 256 hidden values:
//   pass 1: the post (R' = comb^T R + post Y, fp32, rounded to bf16) in shared memory, R' to HBM
//           by a TMA store with the L2 evict-last policy; the 10 Gram entries per token
//           (sum_h R'_i R'_j) in fp32 from the post's registers; the projection onto the 24
//           logits on the tensor cores (mma.sync m16n8k16 bf16: A = phi^T as bf16 high part and
//           remainder, the packed form of the ws schedule read from L2; B = R', the 18 tokens as
//           three n8 tiles, the last part-filled; fp32 accumulate);
//   heads:  r, the pre and post mixes, rstd from the Gram matrix, the residual-mix logits kept
//           for the Sinkhorn at the end of the kernel;
//   pass 2: R' read back from L2, X = sum_i pre_i R'_i, RMSNorm * gamma, bf16 to HBM (and, when
//           asked for, its MXFP8 form: E4M3 codes and a UE8M0 scale per block of 32).
// Pass-2 chunks of tile k-1 are interleaved with pass-1 chunks of tile k (two chunks behind),
// so the HBM reads of pass 1, the L2 reads of both passes and the heads overlap.  HBM moves
// 20H + 176 bytes per token, as in the single-pass schedules; L2 additionally serves phi
// (24 * 4H * 4 bytes per tile) and the R' re-read.  18 tokens (not 16) per tile: the busiest
// elementwise warp still takes three tokens, only the projection's third n8 tile is extra, and
// the larger share per SM lets this kernel take more of a call's tokens beside ws.
//
// Roles (16 warps, so 128 registers a thread): 7 elementwise warps (the post in pass 1, the
// combine in pass 2; warp w takes tokens w, w + 7, w + 14 of each chunk, lane v the chunk's
// 8-value vector v), 8 projection warps (warp p the 16-wide blocks 2p and 2p + 1 of each chunk,
// all four streams; warp 0 also computes the heads) and one thread that issues the TMA loads
// into a 4-slot ring and the TMA stores of R'.  Every mbarrier wait is bounded (1 s): on a
// timeout the thread sets bit 0 of the status word and stops waiting, and the load/store
// thread waits (again bounded) for its copies in flight before the CTA exits.
//
// Launched beside ws (programmatic dependent launch after it, so that ws's clusters are placed
// first), it never waits for ws while it works; at its very end it waits for ws's completion
// (griddepcontrol.wait), so whatever follows it on the stream sees both kernels' outputs.  The
// last CTA to finish then redoes the layer input of the tokens whose streams cancel in X (listed
// by both kernels; see redo_token), so no separate redo launch follows.
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

constexpr int kTT = 18;                         // tokens per tile: three n8 tiles of the MMAs, the last part-filled
constexpr int kNT8 = (kTT + 7) / 8;             // n8 tiles
constexpr int kCW = 256;                        // hidden values per chunk
constexpr int kCHB = kCW / 64;                  // 64-wide blocks per chunk (TMA box depth)
constexpr int kRB = kHC * kCHB * kTT * 128;     // R or R' of a chunk: 32 KB
constexpr int kYB = kCHB * kTT * 128;           // Y of a chunk: 8 KB
constexpr int kSlot = kRB + kYB;                // one ring slot
constexpr int kNSlot = 4;
constexpr int kEW = 7, kPW = 8;                 // elementwise warps 0-6, projection warps 7-14
constexpr int kWProd = kEW + kPW;               // warp 15: loads and stores (one thread)
constexpr int kNT = (kWProd + 1) * 32;          // 16 warps: 4 per SM sub-partition, 128 registers
constexpr int kItems = kTT * (kCW / kVec);      // (token, vector) items of a chunk: 32 per token
constexpr int kMixB = (kTT * 80 + 127) / 128 * 128;  // comb [kTT][16] + post [kTT][4] fp32, 128-byte aligned
constexpr int kLag = 2;                         // pass-2 chunks trail pass-1 chunks by this many
constexpr int kEmptyCount = kEW + kPW + 1;      // every role releases every slot (the producer too)
constexpr uint64_t kWaitNs = 1000000000ull;
static_assert(kSlot % 1024 == 0 && kRB % 1024 == 0, "ring slots and their Y part start on the swizzle period");
static_assert(kTT <= 24 && kTT <= 32, "three n8 tiles at most; one head lane per token");

__device__ __forceinline__ void bwait(uint64_t *bar, uint32_t parity, bool &dead) {
    mbar_wait_timed(bar, parity, dead, kWaitNs);
}
// (the "memory" clobber keeps the read after the mbarrier wait that makes the data visible)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// 16 bytes of the packed phi: read-only path, not kept in L1 (a chunk's fragments outsize it),
// kept in L2 with the given (evict-last) policy, since every tile reads phi again while the rest of
// the traffic streams through L2
__device__ __forceinline__ uint4 ldg_keep(const uint4 *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}
// Byte offset of 16-byte chunk c16 of row `row` of a ring slot: TMA's 128-byte swizzle XORs the
// chunk index with the row's position in its 1024-byte period (rows of 128 bytes, counted from the
// slot's 1024-aligned start across the box's (stream, block) planes of kTT rows each)
__device__ __forceinline__ uint32_t swz(int row, int c16) { return (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4)); }
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Shared memory (after the 1 KB-aligned ring).
struct TLayout {
    __host__ __device__ static constexpr size_t ring() { return 0; }
    __host__ __device__ static constexpr size_t mix() { return ring() + (size_t)kNSlot * kSlot; }          // [2][kMixB]
    __host__ __device__ static constexpr size_t part() { return mix() + 2 * (size_t)kMixB; }             // [2][kPW][kTT][24]
    __host__ __device__ static constexpr size_t gram() { return part() + (size_t)2 * kPW * kTT * 24 * 4; } // [2][kTT][12]
    __host__ __device__ static constexpr size_t head() { return gram() + (size_t)2 * kTT * 12 * 4; }       // [2][kTT][8]
    // full, postd, empty [kNSlot]; mixfull, mixempty, gfull, hfull [2]
    __host__ __device__ static constexpr size_t bars() { return head() + (size_t)2 * kTT * 8 * 4; }
    __host__ __device__ static constexpr size_t flag() { return bars() + (size_t)(3 * kNSlot + 8) * 8; }  // u32
    __host__ __device__ static constexpr size_t bytes() { return flag() + 16; }
};

struct TileMaps {
    CUtensorMap R;     // residual (or R' for the pre alone) [T][4][H] as (h % 64, t, h / 64, stream)
    CUtensorMap Y;     // layer output [T][H] as (h % 64, t, h / 64)
    CUtensorMap Rout;  // R' [T][4][H], stored in pass 1 and read back in pass 2
    CUtensorMap comb, post;
};

// One job of the chunk walk: pass (0 or 1) of chunk c of the CTA's tile k.
// Pass-1 chunk c of tile k at time k * nch + c, pass-2 chunk c of tile k at time
// (k + 1) * nch + c + lag (lag < nch); at equal times pass 1 goes first.
template <typename F>
__device__ __forceinline__ void walk(int my_tiles, int nch, int lag, F &&f) {
    int seq = 0;
    const int tend = my_tiles * nch + lag;  // last pass-2 time + 1 - nch
    for (int tau = 0; tau < tend + nch; ++tau) {
        if (tau < my_tiles * nch) f(tau / nch, 0, tau % nch, seq++);
        const int u = tau - nch - lag;
        if (u >= 0 && u < my_tiles * nch) f(u / nch, 1, u % nch, seq++);
    }
}

// The same order as walk(), one job at a time.
struct JobGen {
    int tau = 0, sub = 0, my_tiles, nch, lag;
    __device__ JobGen(int m, int n, int l) : my_tiles(m), nch(n), lag(l) {}
    __device__ bool next(int &k, int &pass, int &c) {
        while (tau < my_tiles * nch + lag + nch) {
            if (sub == 0) {
                sub = 1;
                if (tau < my_tiles * nch) {
                    k = tau / nch, pass = 0, c = tau % nch;
                    return true;
                }
            }
            sub = 0;
            const int u = tau - nch - lag;
            ++tau;
            if (u >= 0 && u < my_tiles * nch) {
                k = u / nch, pass = 1, c = u % nch;
                return true;
            }
        }
        return false;
    }
};

template <bool kPost>
__global__ void __launch_bounds__(kNT, 1)
tile_kernel(const __grid_constant__ TileMaps maps, const uint4 *__restrict__ pack, const float *__restrict__ bias,
            const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma, Scalars sc, int64_t t_begin,
            int64_t T, int H, int Hs_pack, uint16_t *__restrict__ X_out, float *__restrict__ pre_out,
            float *__restrict__ post_out, float *__restrict__ res_out, float *__restrict__ zstash,
            unsigned int *__restrict__ redo_list, unsigned int *__restrict__ status, int wait_pack, MxOut mx,
            const uint16_t *__restrict__ Rp) {
    // a kernel after this one (the redo pass) may be scheduled now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *ring = smem + TLayout::ring();
    unsigned char *mixb = smem + TLayout::mix();
    float *sPart = reinterpret_cast<float *>(smem + TLayout::part());
    float *sGram = reinterpret_cast<float *>(smem + TLayout::gram());
    float *sHead = reinterpret_cast<float *>(smem + TLayout::head());
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TLayout::bars());
    uint64_t *postd = full + kNSlot, *empty = postd + kNSlot;
    uint64_t *mixfull = empty + kNSlot, *mixempty = mixfull + 2, *gfull = mixempty + 2, *hfull = gfull + 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_tok = T - t_begin;
    const int ntiles = (int)((n_tok + kTT - 1) / kTT);
    const int nch = (H + kCW - 1) / kCW;
    const int lag = kLag < nch ? kLag : nch - 1;
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_t0 = [&](int k) { return t_begin + ((int64_t)blockIdx.x + (int64_t)k * gridDim.x) * kTT; };
    bool dead = false;

    if (tid == 0) {
        for (int i = 0; i < kNSlot; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&postd[i], kEW);
            mbar_init(&empty[i], kEmptyCount);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mixfull[i], 1);
            mbar_init(&mixempty[i], kEW);
            mbar_init(&gfull[i], kEW);
            mbar_init(&hfull[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWProd) {
        // ================================ producer: TMA loads into the ring, and the R' stores.
        // One thread, two cursors over the job sequence: the next job to load and the next loaded
        // job to finish (store its R' once the post is done, release the slot).  Each turn it
        // does whichever is ready, so neither waits behind the other; a turn that finds nothing
        // ready for 1 s gives up (status word).
        if (lane == 0) {
            const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
            JobGen gl(my_tiles, nch, lag), gs(my_tiles, nch, lag);
            int lk = 0, lp = 0, lc = 0, sk = 0, sp = 0, sc2 = 0;
            bool lmore = gl.next(lk, lp, lc), smore = false;
            int nload = 0, nstore = 0, stored_tiles = 0;  // tiles whose R' stores are complete
            uint64_t idle_since = globaltimer_ns();
            while (!dead && (lmore || nstore < nload)) {
                bool progress = false;
                // ---- finish the oldest loaded job
                if (nstore < nload) {
                    if (!smore) smore = gs.next(sk, sp, sc2);
                    const int slot = nstore % kNSlot;
                    const uint32_t ph = (uint32_t)((nstore / kNSlot) & 1);
                    const bool store = kPost && sp == 0;
                    if (!store || mbar_try_wait(&postd[slot], ph)) {
                        if (store) {
                            tma_store_4d_hint(&maps.Rout, ring + (size_t)slot * kSlot, 0, (int)tile_t0(sk), sc2 * kCHB,
                                              0, keep);
                            bulk_commit();
                            bulk_wait_read<0>();  // the store has read the slot
                            if (sc2 == nch - 1) {
                                bulk_wait<0>();  // every R' store of tile sk is complete
                                fence_proxy_async_global();
                                stored_tiles = sk + 1;
                            }
                        }
                        mbar_arrive(&empty[slot]);
                        ++nstore;
                        smore = false;
                        progress = true;
                    }
                }
                // ---- load the next job into its slot
                if (lmore) {
                    const int slot = nload % kNSlot;
                    bool ready = nload < kNSlot || mbar_try_wait(&empty[slot], (uint32_t)(((nload / kNSlot) - 1) & 1));
                    if (ready && kPost && lp == 0 && lc == 0 && lk >= 2)  // the mix buffer of tile lk - 2 is free
                        ready = mbar_try_wait(&mixempty[lk & 1], (uint32_t)(((lk >> 1) - 1) & 1));
                    if (ready && kPost && lp == 1 && lc == 0) ready = stored_tiles > lk;  // R' of tile lk is out
                    if (ready) {
                        unsigned char *dst = ring + (size_t)slot * kSlot;
                        const int t0 = (int)tile_t0(lk);
                        if (lp == 0) {
                            if (kPost && lc == 0) {  // the tile's previous mixes, with its first chunk
                                unsigned char *m = mixb + (size_t)(lk & 1) * kMixB;
                                mbar_arrive_expect_tx(&mixfull[lk & 1], kTT * 80);  // the two copies' bytes (the buffer is padded)
                                tma_load_2d(m, &maps.comb, 0, t0, &mixfull[lk & 1]);
                                tma_load_2d(m + kTT * 64, &maps.post, 0, t0, &mixfull[lk & 1]);
                            }
                            mbar_arrive_expect_tx(&full[slot], kPost ? kSlot : kRB);
                            tma_load_4d_hint(dst, &maps.R, 0, t0, lc * kCHB, 0, &full[slot], drop);
                            if (kPost) tma_load_3d_hint(dst + kRB, &maps.Y, 0, t0, lc * kCHB, &full[slot], drop);
                        } else {
                            mbar_arrive_expect_tx(&full[slot], kRB);
                            tma_load_4d_hint(dst, kPost ? &maps.Rout : &maps.R, 0, t0, lc * kCHB, 0, &full[slot], drop);
                        }
                        ++nload;
                        lmore = gl.next(lk, lp, lc);
                        progress = true;
                    }
                }
                if (progress) {
                    idle_since = globaltimer_ns();
                } else {
                    __nanosleep(64);
                    if (globaltimer_ns() - idle_since > kWaitNs) dead = true;
                }
            }
            // the copies issued last have landed and the stores are complete (already true unless a
            // wait timed out)
            bool drained = false;
            for (int q = nload > kNSlot ? nload - kNSlot : 0; q < nload; ++q)
                mbar_wait_timed(&full[q % kNSlot], (uint32_t)((q / kNSlot) & 1), drained, kWaitNs);
            bulk_wait<0>();
            dead = dead || drained;
        }
    } else if (warp < kEW) {
        // ================================ elementwise: the post (pass 1), the combine (pass 2).
        // Item i = tid + 224 u (u = 0, 1, 2; i < 32 kTT) of a chunk: token i / 32, vector i % 32, so
        // warp w takes tokens w, w + 7 and (w < kTT - 14) w + 14, lane v the chunk's vector v.
        constexpr int kU = (kItems + kEW * 32 - 1) / (kEW * 32);  // 3
        float g[kU][10];  // Gram partials of the warp's tokens over the tile
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
            for (int e = 0; e < 10; ++e) g[u][e] = 0.f;
        float hp[kU][kHC], hr[kU];  // (pre, rstd) of the warp's tokens in pass 2
        const int v = lane, hb = v >> 3, c16 = v & 7;
        walk(my_tiles, nch, lag, [&](int k, int pass, int c, int seq) {
            const int slot = seq % kNSlot;
            const uint32_t ph = (uint32_t)((seq / kNSlot) & 1);
            const int h = c * kCW + v * kVec;
            // pass 2: this lane's 8 values of gamma, loaded before the wait for the slot
            const uint4 gv = pass == 1 && h < H ? ld_ro(gamma + h) : make_uint4(0u, 0u, 0u, 0u);
            bwait(&full[slot], ph, dead);
            unsigned char *sl = ring + (size_t)slot * kSlot;
            const int64_t t0 = tile_t0(k);
            if (pass == 0) {
                if (kPost && c == 0) bwait(&mixfull[k & 1], (uint32_t)((k >> 1) & 1), dead);
                const float *mx = reinterpret_cast<const float *>(mixb + (size_t)(k & 1) * kMixB);
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int t = warp + kEW * u;
                    if (t >= kTT || t0 + t >= T || h >= H) continue;
                    float rf[kHC][8];
                    uint4 r4[kHC];
#pragma unroll
                    for (int j = 0; j < kHC; ++j)
                        r4[j] = *reinterpret_cast<const uint4 *>(sl + swz((j * kCHB + hb) * kTT + t, c16));
                    if (kPost) {
                        const uint4 y = *reinterpret_cast<const uint4 *>(sl + kRB + swz(hb * kTT + t, c16));
                        uint4 o[kHC];
                        post_vec8_x2(r4, y, mx + t * 16, mx + kTT * 16 + t * 4, o, rf);
#pragma unroll
                        for (int j = 0; j < kHC; ++j)
                            *reinterpret_cast<uint4 *>(sl + swz((j * kCHB + hb) * kTT + t, c16)) = o[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < kHC; ++j) unpack8(r4[j], rf[j]);
                    }
                    // Gram entries (0,0) (1,1) (2,2) (3,3) (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        auto dot = [&](int i0, int j0, float &acc) {
                            acc = fmaf(rf[i0][e + 1], rf[j0][e + 1], fmaf(rf[i0][e], rf[j0][e], acc));
                        };
                        dot(0, 0, g[u][0]); dot(1, 1, g[u][1]); dot(2, 2, g[u][2]); dot(3, 3, g[u][3]);
                        dot(0, 1, g[u][4]); dot(0, 2, g[u][5]); dot(0, 3, g[u][6]);
                        dot(1, 2, g[u][7]); dot(1, 3, g[u][8]); dot(2, 3, g[u][9]);
                    }
                }
                if (kPost) fence_proxy_async_smem();  // R' written here, read by the TMA store
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&postd[slot]);
                    mbar_arrive(&empty[slot]);
                }
                if (c == nch - 1) {
                    // the tile's Gram entries: xor tree over the lanes, then to the heads
#pragma unroll
                    for (int u = 0; u < kU; ++u)
#pragma unroll
                        for (int e = 0; e < 10; ++e) {
                            float a = g[u][e];
#pragma unroll
                            for (int m = 16; m > 0; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
                            g[u][e] = a;
                        }
                    if (lane == 0)
#pragma unroll
                        for (int u = 0; u < kU; ++u)
                            if (warp + kEW * u < kTT)
#pragma unroll
                                for (int e = 0; e < 10; ++e) sGram[((k & 1) * kTT + warp + kEW * u) * 12 + e] = g[u][e];
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&gfull[k & 1]);
                        if (kPost) mbar_arrive(&mixempty[k & 1]);
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u)
#pragma unroll
                        for (int e = 0; e < 10; ++e) g[u][e] = 0.f;
                }
            } else {
                if (c == 0) {
                    bwait(&hfull[k & 1], (uint32_t)((k >> 1) & 1), dead);
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int t = warp + kEW * u < kTT ? warp + kEW * u : 0;
                        const float *hd = sHead + ((k & 1) * kTT + t) * 8;
#pragma unroll
                        for (int i0 = 0; i0 < kHC; ++i0) hp[u][i0] = hd[i0];
                        hr[u] = hd[4];
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int t = warp + kEW * u;
                    if (t >= kTT || t0 + t >= T) continue;  // warp-uniform
                    const bool act = h < H;
                    uint4 ob = make_uint4(0u, 0u, 0u, 0u);
                    if (act) {
                        float rf[kHC][8], x[8];
#pragma unroll
                        for (int j = 0; j < kHC; ++j)
                            unpack8(*reinterpret_cast<const uint4 *>(sl + swz((j * kCHB + hb) * kTT + t, c16)), rf[j]);
                        combine_vec8_x2(rf, hp[u], x);
                        ob = norm_vec8(x, hr[u], gv);
                        if (X_out != nullptr) st_stream(X_out + (t0 + t) * (int64_t)H + h, ob);
                    }
                    // MXFP8 layer input: lanes 4a .. 4a+3 hold the block of 32 values a of the chunk
                    // (H % 32 == 0, so a block is in range or not as a whole)
                    if (mx.q != nullptr)
                        mx_quantize8(ob, act, mx.mode, mx.q + (t0 + t) * (int64_t)H + h,
                                     mx.scale + mx_scale_offset(t0 + t, h / 32, H));
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&postd[slot]);
                    mbar_arrive(&empty[slot]);
                }
            }
        });
    } else {
        // ================================ projection (+ the heads in warp 0 of the role)
        const int p = warp - kEW;
        const int gid = lane >> 2, tig = lane & 3;
        // ldmatrix.x4 rows: lanes 0-15 tokens 0-7 (k 0-7, then k 8-15), lanes 16-31 tokens 8-15
        const int lt = (lane & 7) + 8 * (lane >> 4), lk = ((lane >> 3) & 1) * 8;
        const int nsteps_pack = kHC * Hs_pack / 16;  // k16 steps per CTA slice of the packed phi
        float acc[3][kNT8][4];
#pragma unroll
        for (int mt = 0; mt < 3; ++mt)
#pragma unroll
            for (int nt = 0; nt < kNT8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        // phi^T fragments: the packed form (ws's) holds, per CTA slice cr of Hs_pack hidden values and
        // k16 step sl = stream * (Hs_pack / 16) + block within the slice, 3 m-tiles x 32 lanes of uint4.
        // base(c, b): this lane's first uint4 for block 2p + b of chunk c, stream 0 (nullptr beyond H);
        // stream j is j * (Hs_pack / 16) * 96 uint4 further.
        const size_t jstride = (size_t)(Hs_pack / 16) * 96;
        const uint64_t keep_phi = l2_policy_evict_last();
        auto base = [&](int c, int b) -> const uint4 * {
            const int h = (c * (kCW / 16) + 2 * p + b) * 16;
            if (h >= H) return nullptr;
            const int cr = h / Hs_pack;
            return pack + ((size_t)cr * nsteps_pack + (h - cr * Hs_pack) / 16) * 96 + lane;
        };
        auto frag = [&](const uint4 *src, int j, uint4 (&f)[3]) {
            if (src == nullptr) {
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) f[mt] = make_uint4(0u, 0u, 0u, 0u);
                return;
            }
#pragma unroll
            for (int mt = 0; mt < 3; ++mt) f[mt] = ldg_keep(src + j * jstride + mt * 32, keep_phi);
        };
        // alone after the packing launch (programmatic dependent launch): wait for the packed phi.
        // Beside ws the launch before this one is ws, which lets this kernel start only once the
        // packed phi is complete, so there is nothing to wait for here (waiting would wait for ws).
        if (wait_pack) asm volatile("griddepcontrol.wait;" ::: "memory");
        uint4 fr[4][3];  // steps s .. s + 3 in flight
        if (my_tiles > 0) {
            const uint4 *b0 = base(0, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s) frag(b0, s, fr[s]);
        }
        walk(my_tiles, nch, lag, [&](int k, int pass, int c, int seq) {
            const int slot = seq % kNSlot;
            const uint32_t ph = (uint32_t)((seq / kNSlot) & 1);
            // every job's postd phase is waited for, pass 2 included: a parity wait only tells the
            // phase it names from the one before it, so a warp must never skip a phase of a barrier
            // it waits on (a pass-2 job still being combined would otherwise let this warp read the
            // next job's slot before it is loaded)
            bwait(&postd[slot], ph, dead);
            if (pass == 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                return;
            }
            const uint32_t sl = smem_u32(ring + (size_t)slot * kSlot);
            const int cn = c + 1 < nch ? c + 1 : 0;  // the next pass-1 chunk (phi is the same in every tile)
            const uint4 *b1 = base(c, 1), *bn = base(cn, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int b = 2 * p + (s >> 2), j = s & 3;
                const int hh = b * 16 + lk;  // hidden offset within the chunk of this lane's row
                const int row0 = (j * kCHB + (hh >> 6)) * kTT, c16 = (hh & 63) >> 3;
                uint32_t r[4];
                ldsm_x4(sl + swz(row0 + lt, c16), r);
                uint32_t r2[2];
                // tokens 16-23 (lanes 0-15 give the rows; rows past the tile read the next plane's rows,
                // inside the slot, and only feed columns that are dropped)
                if (kNT8 > 2) ldsm_x2(sl + swz(row0 + 16 + (lane & 7), c16), r2);
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) {
                    mma16816(acc[mt][0], fr[s & 3][mt], r[0], r[1]);
                    mma16816(acc[mt][1], fr[s & 3][mt], r[2], r[3]);
                    if (kNT8 > 2) mma16816(acc[mt][2], fr[s & 3][mt], r2[0], r2[1]);
                }
                // refill this ring entry with the step four ahead
                if (s < 4) frag(b1, s, fr[s & 3]);
                else frag(bn, s - 4, fr[s & 3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (c < nch - 1) return;
            // ---- the tile's logit partials of this warp: token nt * 8 + 2 tig + e, logits gid, gid + 8,
            // gid + 16 (rows 0-23 hold phi's high part, rows 24-47 the remainder of the same logit)
            // (two buffers, by tile parity)
            float *pw = sPart + (size_t)((k & 1) * kPW + p) * kTT * 24;
#pragma unroll
            for (int nt = 0; nt < kNT8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = nt * 8 + 2 * tig + e;
                    if (t >= kTT) continue;
                    pw[t * 24 + gid] = acc[0][nt][e] + acc[1][nt][2 + e];
                    pw[t * 24 + gid + 8] = acc[0][nt][2 + e] + acc[2][nt][e];
                    pw[t * 24 + gid + 16] = acc[1][nt][e] + acc[2][nt][2 + e];
                }
#pragma unroll
            for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                for (int nt = 0; nt < kNT8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
            named_sync(1, kPW * 32);
            if (p != 0) return;
            // ---- heads of tile k: one lane per token
            bwait(&gfull[k & 1], (uint32_t)((k >> 1) & 1), dead);
            if (lane < kTT) {
                const int t = lane;
                const int64_t tok = tile_t0(k) + t;
                float z[kNumMix];
#pragma unroll
                for (int n = 0; n < kNumMix; ++n) z[n] = 0.f;
#pragma unroll
                for (int w = 0; w < kPW; ++w) {
                    const float4 *pp = reinterpret_cast<const float4 *>(sPart + ((size_t)((k & 1) * kPW + w) * kTT + t) * 24);
#pragma unroll
                    for (int q = 0; q < 6; ++q) {
                        const float4 f = pp[q];
                        z[4 * q] += f.x; z[4 * q + 1] += f.y; z[4 * q + 2] += f.z; z[4 * q + 3] += f.w;
                    }
                }
                float G[10];
#pragma unroll
                for (int e = 0; e < 10; ++e) G[e] = sGram[((k & 1) * kTT + t) * 12 + e];
                const float inv_kh = 1.f / (float)(kHC * H), inv_h = 1.f / (float)H;
                const float ss = (G[0] + G[1]) + (G[2] + G[3]);
                const float r = __frsqrt_rn(ss * inv_kh + sc.hc_norm_eps);
                const float a_pre = mix_scales[0], a_post = mix_scales[1];
                float pre[kHC];
#pragma unroll
                for (int i = 0; i < kHC; ++i) pre[i] = __frcp_rn(1.f + expf(-(a_pre * (r * z[i]) + bias[i])));
                float sx = pre[0] * pre[0] * G[0] + pre[1] * pre[1] * G[1] + pre[2] * pre[2] * G[2] +
                           pre[3] * pre[3] * G[3];
                sx += 2.f * (pre[0] * pre[1] * G[4] + pre[0] * pre[2] * G[5] + pre[0] * pre[3] * G[6] +
                             pre[1] * pre[2] * G[7] + pre[1] * pre[3] * G[8] + pre[2] * pre[3] * G[9]);
                const float rstd = __frsqrt_rn(fmaxf(sx, 0.f) * inv_h + sc.rmsnorm_eps);
                float *hd = sHead + ((k & 1) * kTT + t) * 8;
#pragma unroll
                for (int i = 0; i < kHC; ++i) hd[i] = pre[i];
                hd[4] = rstd;
                if (tok < T) {
#pragma unroll
                    for (int i = 0; i < kHC; ++i) {
                        pre_out[tok * 4 + i] = pre[i];
                        post_out[tok * 4 + i] = sc.hc_post_scale / (1.f + expf(-(a_post * (r * z[4 + i]) + bias[4 + i])));
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) zstash[tok * 16 + e] = r * z[8 + e];  // normalised at the end
                    // streams that cancel in X: the layer input is redone with a direct sum after
                    // this kernel (the redo pass)
                    if (gram_cancels(sx, pre, G)) {
                        const unsigned int idx = atomicAdd(status + kRedoCountWord, 1u);
                        if (idx < (unsigned int)T) redo_list[idx] = (unsigned int)tok;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hfull[k & 1]);
        });
    }

    __syncthreads();  // every role is done; the residual-mix logits are in zstash
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
    // ---- the redo pass: the layer input of the tokens whose streams cancel in X (listed by this
    // kernel's heads and by ws's owners), redone by the last CTA of the grid to get here once ws
    // is complete.  Each CTA counts itself done after its own tokens are listed.
    unsigned int &sLast = *reinterpret_cast<unsigned int *>(smem + TLayout::flag());
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        sLast = atomicAdd(status + kRedoDoneWord, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    // beside ws: this grid completes only after ws has (what follows on the stream sees both), and
    // ws's list entries and outputs are visible from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!sLast) return;
    __threadfence();
    // (a list longer than the call's tokens can only be left over from an aborted call)
    const unsigned int n0 = *reinterpret_cast<volatile unsigned int *>(status + kRedoCountWord);
    const unsigned int n = n0 < (unsigned int)T ? n0 : (unsigned int)T;
    for (unsigned int i = (unsigned int)warp; i < n; i += kNT / 32)
        redo_token(Rp, gamma, sc.rmsnorm_eps, H, pre_out, X_out, mx, (int64_t)__ldcg(redo_list + i));
    __syncthreads();
    if (tid == 0) {
        status[kRedoCountWord] = 0u;
        status[kRedoDoneWord] = 0u;
    }
}

}  // namespace

bool tile_supported(int64_t T, int64_t H) {
    // the (h % 64, t, h / 64) tensor views need whole 64-wide blocks; at least two chunks per row;
    // token coordinates are 32-bit
    return H > kCW && H % 64 == 0 && H <= ((int64_t)1 << 20) && T >= 1 && T < ((int64_t)1 << 31) - kTT;
}

size_t tile_smem_bytes() { return TLayout::bytes() + 1024; }

int tile_tokens() { return kTT; }

cudaError_t launch_tile(const FusedArgs &a, int64_t t_begin, unsigned int *status, float *zstash, int grid,
                        bool beside, cudaStream_t stream) {
    if (!tile_supported(a.T, a.H) || t_begin < 0 || t_begin >= a.T || grid < 1) return cudaErrorInvalidValue;
    const bool post = a.R_out != nullptr;
    tma::EncodeTiledFn fn;
    cudaError_t e = tma::encoder(fn);
    if (e != cudaSuccess) return e;
    const cuuint64_t H = (cuuint64_t)a.H, T = (cuuint64_t)a.T;
    TileMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const cuuint64_t dR[4] = {64, T, H / 64, 4}, sR[3] = {H * 8, 128, H * 2};
    const cuuint32_t bR[4] = {64, (cuuint32_t)kTT, (cuuint32_t)kCHB, (cuuint32_t)kHC};
    if ((e = tma::encode_bf16(fn, &maps.R, 4, a.R, dR, sR, bR, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    if (post) {
        if ((e = tma::encode_bf16(fn, &maps.Rout, 4, a.R_out, dR, sR, bR, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        const cuuint64_t dY[3] = {64, T, H / 64}, sY[2] = {H * 2, 128};
        const cuuint32_t bY[3] = {64, (cuuint32_t)kTT, (cuuint32_t)kCHB};
        if ((e = tma::encode_bf16(fn, &maps.Y, 3, a.Y, dY, sY, bY, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        const cuuint32_t es[2] = {1, 1};
        const cuuint64_t dc[2] = {16, T}, scm[1] = {64};
        const cuuint32_t bc[2] = {16, (cuuint32_t)kTT};
        const cuuint64_t dp[2] = {4, T}, sp[1] = {16};
        const cuuint32_t bp[2] = {4, (cuuint32_t)kTT};
        if (fn(&maps.comb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.prev_comb), dc, scm, bc, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            fn(&maps.post, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.prev_post), dp, sp, bp, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t smem = tile_smem_bytes();
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        static std::mutex mu;
        static bool attr_set[64][2];
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev][post ? 1 : 0]) {
            auto kern = post ? tile_kernel<true> : tile_kernel<false>;
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
                return e;
            attr_set[dev][post ? 1 : 0] = true;
        }
    }
    const int64_t ntiles = (a.T - t_begin + kTT - 1) / kTT;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    // beside ws: may start once ws's CTAs are all resident (ws signals at its start); alone after
    // the packing launch: may start with it (the projection warps wait for the packed phi)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(ntiles, grid));
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (beside || !a.prepacked) ? 1 : 0;
    const int Hs_pack = ws_slice(a.H);
    unsigned int *list = a.redo_list;
    const uint16_t *Rp = post ? a.R_out : a.R;  // R' for the redo pass in the kernel's tail
    if (!beside) mark_main_kernel(stream, true);
    e = post ? cudaLaunchKernelEx(&cfg, tile_kernel<true>, maps, (const uint4 *)a.phi_pack, a.bias, a.mix_scales,
                                  a.gamma, a.s, t_begin, a.T, a.H, Hs_pack, a.X_out, a.pre_out, a.post_out, a.res_out,
                                  zstash, list, status, (!beside && !a.prepacked) ? 1 : 0, a.mx, Rp)
             : cudaLaunchKernelEx(&cfg, tile_kernel<false>, maps, (const uint4 *)a.phi_pack, a.bias, a.mix_scales,
                                  a.gamma, a.s, t_begin, a.T, a.H, Hs_pack, a.X_out, a.pre_out, a.post_out, a.res_out,
                                  zstash, list, status, (!beside && !a.prepacked) ? 1 : 0, a.mx, Rp);
    if (!beside) mark_main_kernel(stream, false);
    return e;
}

}  // namespace mhc
