// Cluster schedule: the whole mHC post+pre step in one pass over HBM.
//
// A thread-block cluster of C CTAs owns a group of G tokens at a time; CTA c
// of the cluster owns the hidden slice [c*Hs, (c+1)*Hs) of every token in the
// group (Hs = H / C rounded up to 16).  Per group:
//
//   P1  post: stream R and Y of its slice (16-byte vectors), form R' in fp32,
//       round to bf16, write R' to HBM and keep it in shared memory; square
//       sums per token.
//   P2  projection of the slice onto the 24 logits on the tensor cores:
//       mma.sync m16n8k16 bf16 with A = phi^T split into bf16 hi and lo parts
//       (48 rows = three m16 tiles; pre-packed in fragment order by
//       pack_phi_kernel) and B = R' straight from shared memory (ldmatrix).
//   P3  cluster reduce: every CTA publishes its 25 partial sums per token in
//       shared memory; after a cluster barrier the owner CTA of each token sums
//       the C partials through distributed shared memory in a fixed order,
//       computes r, the sigmoid heads and the Sinkhorn mix (one warp per
//       token), writes the mixes and pushes pre to every CTA of the cluster.
//   P4  combine: X = sum_i pre_i R'_i from shared memory, square sum of X per
//       token exchanged the same way, then RMSNorm * gamma and the bf16 write.
//
// So each token's R and Y are read once and R' and the layer input written
// once: 20H + 176 bytes per token.  Cluster barriers are hardware barriers
// (no spinning), every reduction has a fixed order (results do not depend on
// timing), and R' never leaves the chip between the post and the combine.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>

#include "mhc_device.cuh"
#include "mhc_kernels.h"

namespace cg = cooperative_groups;

namespace mhc {

namespace {


// Split cluster barrier: arrive (release) now, wait (acquire) later.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Shared memory of one CTA (dynamic).  R' rows are padded by 16 bytes so the
// eight rows an ldmatrix reads fall into distinct bank groups.
template <int G, int kWarps>
struct FusedSmem {
    static constexpr int kPartStride = 32;
    // offsets in bytes
    __host__ __device__ static size_t rows_bytes(int Hs) { return (size_t)G * row_bytes(Hs); }
    __host__ __device__ static size_t row_bytes(int Hs) { return (size_t)kHC * Hs * 2 + 16; }
    __host__ __device__ static size_t zpart_off(int Hs) { return rows_bytes(Hs); }                                  // [kWarps][G][24] f32
    __host__ __device__ static size_t part_off(int Hs) { return zpart_off(Hs) + (size_t)kWarps * G * kNumMix * 4; }  // [G][32] f32
    __host__ __device__ static size_t ss_off(int Hs) { return part_off(Hs) + (size_t)G * kPartStride * 4; }          // [G] f32
    __host__ __device__ static size_t pre_off(int Hs) { return ss_off(Hs) + (size_t)G * 4; }                         // [G][4] f32
    __host__ __device__ static size_t xsq_off(int Hs) { return pre_off(Hs) + (size_t)G * 16; }                       // [G] f32
    __host__ __device__ static size_t mix_off(int Hs) { return xsq_off(Hs) + (size_t)G * 4; }                        // [G][20] f32
    __host__ __device__ static size_t bytes(int Hs) { return mix_off(Hs) + (size_t)G * 20 * 4; }
};

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

template <int C, int G, int kWarps, int kMinBlocks, bool kPost>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks)
fused_cluster_kernel(const uint16_t *__restrict__ R, const uint16_t *__restrict__ Y,
                     const float *__restrict__ prev_post, const float *__restrict__ prev_comb,
                     const uint4 *__restrict__ phi_pack, const float *__restrict__ bias,
                     const float *__restrict__ mix_scales, const uint16_t *__restrict__ gamma,
                     Scalars sc, int64_t T, int H, int Hs, uint16_t *__restrict__ R_out,
                     uint16_t *__restrict__ X_out, float *__restrict__ pre_out,
                     float *__restrict__ post_out, float *__restrict__ res_out) {
    using SM = FusedSmem<G, kWarps>;
    constexpr int kThreads = kWarps * 32;
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;

    const size_t rowb = SM::row_bytes(Hs);
    unsigned char *sR = smem;
    float *sZ = reinterpret_cast<float *>(smem + SM::zpart_off(Hs));
    float *sPart = reinterpret_cast<float *>(smem + SM::part_off(Hs));
    float *sSS = reinterpret_cast<float *>(smem + SM::ss_off(Hs));
    float *sPre = reinterpret_cast<float *>(smem + SM::pre_off(Hs));
    float *sXsq = reinterpret_cast<float *>(smem + SM::xsq_off(Hs));
    float *sMix = reinterpret_cast<float *>(smem + SM::mix_off(Hs));

    const int h0 = c * Hs;
    const int hv = max(0, min(Hs, H - h0));  // valid hidden elements of this slice
    const int nvec = Hs / kVec;              // vectors per stream row of the slice
    const int nvec_valid = hv / kVec;
    const int S = kHC * Hs / 16;             // k16-steps of the slice
    const uint4 *pack = phi_pack + (size_t)c * S * 96;

    const int64_t ngroups = (T + G - 1) / G;
    const int nclusters = gridDim.x / C;
    const int cid = blockIdx.x / C;

    for (int64_t grp = cid; grp < ngroups; grp += nclusters) {
        const int64_t t0 = grp * G;
        const int gv = (int)(T - t0 < G ? T - t0 : G);  // valid tokens in the group

        if (kPost) {
            for (int idx = tid; idx < G * 20; idx += kThreads) {
                const int g = idx / 20, m = idx % 20;
                float v = 0.f;
                if (g < gv) v = m < 16 ? prev_comb[(t0 + g) * 16 + m] : prev_post[(t0 + g) * 4 + (m - 16)];
                sMix[idx] = v;
            }
            __syncthreads();
        }

        // ---- P1: post for this slice, R' to HBM and shared memory, square sums
        for (int g = warp; g < G; g += kWarps) {
            float ss = 0.f;
            if (g < gv) {
                const int64_t t = t0 + g;
                const int64_t rbase = t * kHC * (int64_t)H + h0;
                unsigned char *row = sR + g * rowb;
                for (int v0 = lane; v0 < nvec; v0 += 64) {
                    // two vectors per lane in flight
                    uint4 in[2][kHC + 1];
                    bool ok[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int v = v0 + 32 * u;
                        ok[u] = v < nvec_valid;
                        if (ok[u]) {
#pragma unroll
                            for (int j = 0; j < kHC; ++j) in[u][j] = ld_stream(R + rbase + (int64_t)j * H + v * kVec);
                            if (kPost) in[u][kHC] = ld_stream(Y + t * (int64_t)H + h0 + v * kVec);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int v = v0 + 32 * u;
                        if (v >= nvec) continue;
                        uint4 o[kHC] = {};
                        if (ok[u]) {
                            float rf[kHC][8];
                            if (kPost) {
                                uint4 r4[kHC] = {in[u][0], in[u][1], in[u][2], in[u][3]};
                                post_vec8(r4, in[u][kHC], &sMix[g * 20], &sMix[g * 20 + 16], o, rf);
#pragma unroll
                                for (int i = 0; i < kHC; ++i)
                                    st_stream(R_out + rbase + (int64_t)i * H + v * kVec, o[i]);
                            } else {
#pragma unroll
                                for (int i = 0; i < kHC; ++i) {
                                    o[i] = in[u][i];
                                    unpack8(o[i], rf[i]);
                                }
                            }
#pragma unroll
                            for (int i = 0; i < kHC; ++i)
#pragma unroll
                                for (int e = 0; e < 8; ++e) ss = fmaf(rf[i][e], rf[i][e], ss);
                        }
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

        // ---- P2: projection partials on the tensor cores.  Warp w takes a
        // contiguous range of k16-steps for all G tokens.
        {
            float acc[G / 8][3][4];
#pragma unroll
            for (int nt = 0; nt < G / 8; ++nt)
#pragma unroll
                for (int mt = 0; mt < 3; ++mt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[nt][mt][q] = 0.f;
            const int s_begin = (int)((int64_t)S * warp / kWarps), s_end = (int)((int64_t)S * (warp + 1) / kWarps);
            // ldmatrix row addresses: lane l -> token 8*(l/16) + (l%8) (x4: two n-tiles),
            // k offset 8*((l/8)%2)
            const int ltok = 8 * ((lane >> 4) & 1) + (lane & 7);
            const int lk = 8 * ((lane >> 3) & 1);
            const uint32_t sR_u32 = smem_u32(sR);
            uint4 a_next[3];
            if (s_begin < s_end) {
#pragma unroll
                for (int mt = 0; mt < 3; ++mt) a_next[mt] = ld_ro(pack + ((size_t)s_begin * 3 + mt) * 32 + lane);
            }
            for (int s = s_begin; s < s_end; ++s) {
                uint4 a[3] = {a_next[0], a_next[1], a_next[2]};
                if (s + 1 < s_end) {
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt) a_next[mt] = ld_ro(pack + ((size_t)(s + 1) * 3 + mt) * 32 + lane);
                }
                const int kl = 16 * s + lk;  // CTA-local k of this lane's ldmatrix row
#pragma unroll
                for (int np = 0; np < G / 16; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(sR_u32 + (uint32_t)((16 * np + ltok) * rowb + (size_t)kl * 2), b0, b1, b2, b3);
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt) {
                        mma_bf16(acc[2 * np][mt], a[mt], b0, b1);
                        mma_bf16(acc[2 * np + 1][mt], a[mt], b2, b3);
                    }
                }
                if (G % 16 == 8) {
                    uint32_t b0, b1;
                    ldmatrix_x2(sR_u32 + (uint32_t)((16 * (G / 16) + (lane & 7)) * rowb + (size_t)kl * 2), b0, b1);
#pragma unroll
                    for (int mt = 0; mt < 3; ++mt) mma_bf16(acc[G / 8 - 1][mt], a[mt], b0, b1);
                }
            }
            // hi + lo rows -> 24 logits; thread holds logits gid, gid+8, gid+16 for
            // tokens 2*tig, 2*tig+1 of each n-tile.
            float *zw = sZ + (size_t)warp * G * kNumMix;
#pragma unroll
            for (int nt = 0; nt < G / 8; ++nt) {
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
        // sum the warp partials in a fixed order -> this CTA's partial record
        for (int idx = tid; idx < G * 32; idx += kThreads) {
            const int g = idx >> 5, n = idx & 31;
            float v = 0.f;
            if (n < kNumMix) {
                for (int w = 0; w < kWarps; ++w) v += sZ[((size_t)w * G + g) * kNumMix + n];
            } else if (n == kNumMix) {
                v = sSS[g];
            }
            sPart[idx] = v;
        }
        cluster.sync();  // #1: every CTA's partial records are complete

        // ---- P3: owner CTA of token g (g % C == c) reduces the C records and
        // pushes pre to every CTA; the post head and the Sinkhorn mix follow
        // after this warp has arrived at the cluster barrier, so they overlap
        // the other warps' combine instead of delaying it.
        float zkeep[(G + C * kWarps - 1) / (C * kWarps)];
        {
            int u = 0;
            for (int g = c + C * warp; g < gv; g += C * kWarps, ++u) {
                float acc = 0.f;
                if (lane <= kNumMix) {
                    for (int q = 0; q < C; ++q) acc += cluster.map_shared_rank(sPart, q)[g * 32 + lane];
                }
                const float ss = __shfl_sync(0xffffffffu, acc, kNumMix);
                const float r = 1.f / sqrtf(ss / (float)(kHC * H) + sc.hc_norm_eps);
                zkeep[u] = r * acc;
                const float p = pre_head(zkeep[u], bias, mix_scales);
                if (lane < 4) {
                    pre_out[(t0 + g) * 4 + lane] = p;
                    for (int q = 0; q < C; ++q) cluster.map_shared_rank(sPre, q)[g * 4 + lane] = p;
                }
            }
        }
        cluster_arrive();  // #2: pre of every token is in every CTA
        {
            int u = 0;
            for (int g = c + C * warp; g < gv; g += C * kWarps, ++u) {
                const float v = post_and_sinkhorn(zkeep[u], bias, mix_scales, sc);
                const int64_t t = t0 + g;
                if (lane >= 4 && lane < 8) post_out[t * 4 + lane - 4] = v;
                else if (lane >= 8 && lane < 24) res_out[t * 16 + lane - 8] = v;
            }
        }
        cluster_wait();

        // ---- P4: combine, square sum of X per token
        for (int g = warp; g < gv; g += kWarps) {
            const float pre[kHC] = {sPre[g * 4], sPre[g * 4 + 1], sPre[g * 4 + 2], sPre[g * 4 + 3]};
            const unsigned char *row = sR + g * rowb;
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
        cluster.sync();  // #3: every CTA's square sums of X are published

        for (int g = warp; g < gv; g += kWarps) {
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < C; ++q) tot += cluster.map_shared_rank(sXsq, q)[g];
            const float rstd = 1.f / sqrtf(tot / (float)H + sc.rmsnorm_eps);
            const float pre[kHC] = {sPre[g * 4], sPre[g * 4 + 1], sPre[g * 4 + 2], sPre[g * 4 + 3]};
            const unsigned char *row = sR + g * rowb;
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
        __syncthreads();  // shared rows and mixes are reused by the next group
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// Per-device, per-kernel launch set-up, done once: the shared-memory attribute
// (set to the largest size this kernel can need) and the number of clusters
// that fit on the device at that size.
struct LaunchSetup {
    bool ready = false;
    int max_clusters = 0;
};
constexpr int kMaxDevices = 64;

template <typename Kern>
cudaError_t launch_setup(Kern kern, int C, int threads, size_t smem_max, LaunchSetup &st) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_max;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(C);
    e = cudaOccupancyMaxActiveClusters(&st.max_clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (st.max_clusters < 1) return cudaErrorInvalidConfiguration;
    st.ready = true;
    return cudaSuccess;
}

std::mutex g_setup_mu;

template <int C, int G, int NW, int MB>
cudaError_t launch_fused_cg(const FusedArgs &a, int Hs, cudaStream_t stream) {
    using SM = FusedSmem<G, NW>;
    const size_t smem = SM::bytes(Hs);
    const bool post = a.R_out != nullptr;
    auto kern = post ? fused_cluster_kernel<C, G, NW, MB, true> : fused_cluster_kernel<C, G, NW, MB, false>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    static LaunchSetup setup[kMaxDevices][2];  // one per template instance and device
    int max_clusters;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        LaunchSetup &st = setup[dev][post ? 1 : 0];
        if (!st.ready) {
            // occupancy at the largest shared-memory size this instance may use
            e = launch_setup(kern, C, NW * 32, MB == 1 ? 227 * 1024 : 227 * 1024 / MB - 1024, st);
            if (e != cudaSuccess) return e;
        }
        max_clusters = st.max_clusters;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t ngroups = (a.T + G - 1) / G;
    const int nclusters = (int)std::min<int64_t>(ngroups, max_clusters);
    cfg.gridDim = dim3(nclusters * C);
    return cudaLaunchKernelEx(&cfg, kern, a.R, a.Y, a.prev_post, a.prev_comb, (const uint4 *)a.phi_pack, a.bias,
                              a.mix_scales, a.gamma, a.s, a.T, a.H, Hs, a.R_out, a.X_out, a.pre_out, a.post_out,
                              a.res_out);
}

}  // namespace

void launch_pack_phi(const float *phi, int H, int C, int Hs, uint4 *out, int64_t total, cudaStream_t stream) {
    pack_phi_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(phi, H, C, Hs, out);
}

int fused_slice(int H, int C) { return ((H + 16 * C - 1) / (16 * C)) * 16; }

size_t fused_pack_bytes(int H, int C) {
    const int Hs = fused_slice(H, C);
    return (size_t)C * (kHC * Hs / 16) * 96 * 16;
}

size_t fused_smem_bytes(int H, int C, int G) {
    const int Hs = fused_slice(H, C);
    if (C == 8 && G == 16) return FusedSmem<16, 16>::bytes(Hs);
    if (C == 8 && G == 8) return FusedSmem<8, 8>::bytes(Hs);
    return (size_t)-1;
}

cudaError_t launch_fused(const FusedArgs &a, cudaStream_t stream) {
    const int Hs = fused_slice(a.H, a.C);
    // 1. pack phi into mma fragment order (workspace)
    const int64_t total = (int64_t)a.C * (kHC * Hs / 16) * 96;
    pack_phi_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(a.phi, a.H, a.C, Hs, a.phi_pack);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. the fused pass
    if (a.C == 8 && a.G == 16) return launch_fused_cg<8, 16, 16, 1>(a, Hs, stream);
    if (a.C == 8 && a.G == 8) return launch_fused_cg<8, 8, 8, 2>(a, Hs, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mhc
