// C-ABI layer of libmhc.so: argument validation, schedule choice, launches.
// The contract of every entry point is stated in include/mhc.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <cstdint>
#include <string>

#include "mhc.h"
#include "mhc_kernels.h"

namespace {

thread_local std::string g_last_error;
thread_local int g_launches = 0;
std::atomic<int> g_forced_schedule{MHC_SCHEDULE_AUTO};

mhc_status fail(mhc_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
mhc_status fail(mhc_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

mhc_status cuda_fail(cudaError_t e, const char *what) {
    return fail(MHC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    const void *p;
    size_t bytes;
};

bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

mhc_status check_sizes(int64_t T, int64_t H) {
    if (T < 0 || T > MHC_MAX_TOKENS)
        return fail(MHC_ERR_INVALID_ARG, "T=%lld outside [0, %d]", (long long)T, MHC_MAX_TOKENS);
    if (H < 8 || H > MHC_MAX_HIDDEN || H % 8 != 0)
        return fail(MHC_ERR_INVALID_ARG, "H=%lld must be a multiple of 8 in [8, %d]", (long long)H,
                    MHC_MAX_HIDDEN);
    return MHC_OK;
}

mhc_status check_ptrs(std::initializer_list<std::pair<const void *, const char *>> ptrs) {
    for (auto &pn : ptrs) {
        if (pn.first == nullptr) return fail(MHC_ERR_INVALID_ARG, "%s is NULL", pn.second);
        if (!aligned16(pn.first)) return fail(MHC_ERR_INVALID_ARG, "%s is not 16-byte aligned", pn.second);
    }
    return MHC_OK;
}

mhc_status check_scalars(float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                         float sinkhorn_eps, int iters) {
    auto bad_eps = [](float e) { return !std::isfinite(e) || e < 0.f; };
    if (bad_eps(hc_norm_eps)) return fail(MHC_ERR_INVALID_ARG, "hc_norm_eps must be finite and >= 0");
    if (bad_eps(rmsnorm_eps)) return fail(MHC_ERR_INVALID_ARG, "rmsnorm_eps must be finite and >= 0");
    if (bad_eps(sinkhorn_eps)) return fail(MHC_ERR_INVALID_ARG, "sinkhorn_eps must be finite and >= 0");
    if (!std::isfinite(hc_post_scale)) return fail(MHC_ERR_INVALID_ARG, "hc_post_scale must be finite");
    if (iters < 0 || iters > MHC_MAX_SINKHORN_ITERS)
        return fail(MHC_ERR_INVALID_ARG, "sinkhorn_iters=%d outside [0, %d]", iters, MHC_MAX_SINKHORN_ITERS);
    return MHC_OK;
}

struct Device {
    int id, sms, major, minor;
};

mhc_status current_device(Device &d) {
    cudaError_t e = cudaGetDevice(&d.id);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, d.id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, d.id)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, d.id)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (d.major != 10 || d.minor != 3)
        return fail(MHC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    d.id, d.major, d.minor);
    return MHC_OK;
}

// Beyond ws's hidden size (H > 7168) the token-tile kernel alone beats the split schedule from
// about this many tokens: one round of its tiles costs about 100-110 us at H = 7232-8192, the
// split schedule about 0.23-0.25 us per token (graph-replayed: T = 512, H = 8192: 111.5 vs
// 152.8 us; T = 128: 110.1 vs 46.0 us; T = 8192: 410 vs 2,032 us).
constexpr int64_t kTileAloneMinT = 448;

// The split schedule's MXFP8-only call quantizes a bf16 layer input that it first writes here,
// after the split scratch.  Only reserved where AUTO can choose split (a forced split call with a
// larger T and no bf16 output is refused when the workspace has no room).
size_t split_mx_scratch_offset(int64_t T, int64_t H) {
    return mhc::kControlBytes + ((mhc::split_workspace_bytes(T, H) + 255) & ~size_t(255));
}
bool split_mx_scratch_reserved(int64_t T, int64_t H) {
    return H >= 8 && H <= MHC_MAX_HIDDEN && !mhc::ws_supported((int)H) && T < kTileAloneMinT;
}

size_t workspace_bytes_for(int64_t T, int64_t H) {
    size_t sched = mhc::split_workspace_bytes(T, H);
    if (split_mx_scratch_reserved(T, H))
        sched = ((sched + 255) & ~size_t(255)) + (size_t)T * (size_t)H * 2;
    if (H >= 8 && H <= MHC_MAX_HIDDEN)
    {
        sched = std::max(sched, ((mhc::ws_pack_bytes((int)H) + 255) & ~size_t(255)) + mhc::ws_stash_bytes(T));
        sched = std::max(sched, mhc::small_workspace_bytes(T, (int)H));
        sched = std::max(sched, mhc::bcast_workspace_bytes(T, H));
    }
    size_t b = mhc::kControlBytes + sched;
    return (b + 255) & ~size_t(255);
}

// Up to this many tokens the one-barrier small-T schedule has the lower latency.
constexpr int64_t kSmallAutoMaxT = 32;


int auto_schedule(int64_t T, int64_t H, int sms, bool mx = false) {
    if (T <= kSmallAutoMaxT && mhc::small_supported(T, (int)H, sms, mx)) return MHC_SCHEDULE_SMALL;
    if (mhc::ws_supported((int)H)) return MHC_SCHEDULE_WS;
    if (mhc::tile_supported(T, H) && T >= kTileAloneMinT) return MHC_SCHEDULE_TILE;
    return MHC_SCHEDULE_SPLIT;
}

int choose_schedule(int64_t T, int64_t H, int sms, bool mx) {
    const int forced = g_forced_schedule.load(std::memory_order_relaxed);
    // the broadcast schedule only concerns mhc_pre_broadcast; the other calls choose as AUTO
    if (forced != MHC_SCHEDULE_AUTO && forced != MHC_SCHEDULE_BCAST) return forced;
    return auto_schedule(T, H, sms, mx);
}

int forced_schedule() { return g_forced_schedule.load(std::memory_order_relaxed); }

// The token-tile kernel beside ws: below this many tokens (or with fewer idle SMs) ws runs alone.
constexpr int64_t kSideMinT = 2048;
constexpr int kSideMinSms = 8;
// Per-SM rate of the token-tile kernel relative to ws's while both run (long prefill, T = 65536,
// H = 7168: the split at which both kernels end together; rates 0.50-0.58 gave the tile kernel
// 15-16 rounds and 1,878-1,851 us, 0.62 gave it 17 rounds and made it the tail at 1,947 us).
constexpr double kSideRate = 0.58;

// The first token of the token-tile kernel's share (T: ws alone), and in `idle` the SMs ws leaves
// idle (the tile kernel's grid).  The share follows the two kernels' rates (ws on its resident
// CTAs, the tile kernel on the idle SMs) and is a whole number of tiles per idle SM, so
// the tile kernel's CTAs finish together; ws keeps whole groups of 8 tokens.
int64_t side_split(int64_t T, int64_t H, bool fused, int sms, int &idle) {
    idle = 0;
    if (T < kSideMinT || !mhc::tile_supported(T, H)) return T;
    int ws_ctas = 0;
    if (mhc::ws_resident_ctas((int)H, fused, ws_ctas) != cudaSuccess) return T;
    idle = sms - ws_ctas;
    if (idle < kSideMinSms) return T;
    const double f = idle * kSideRate / (ws_ctas + idle * kSideRate);
    const int64_t per_round = (int64_t)idle * mhc::tile_tokens();
    const int64_t rounds = (int64_t)(T * f / per_round + 0.5);
    if (rounds < 1) return T;
    return (T - rounds * per_round) / 8 * 8;
}

size_t mx_scale_bytes(int64_t T, int64_t H) {
    return (size_t)((T + 127) / 128 * 128) * (size_t)((H / 32 + 3) / 4 * 4);
}

// Common body of the fused call (post != nullptr) and the pre-only call.
mhc_status run_post_pre(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                        const float *prev_post_mix, const float *prev_comb_res_mix,
                        const float *phi, const float *bias, const float *mix_scales,
                        const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps,
                        float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps,
                        int sinkhorn_iters, mhc_bf16 *residual_out, mhc_bf16 *layer_in_out,
                        float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
                        void *workspace, size_t workspace_bytes, void *stream, bool fused,
                        uint8_t *mx_q = nullptr, uint8_t *mx_scale = nullptr, int mx_mode = 0,
                        const mhc::SideStream *side = nullptr, const void *packed_phi = nullptr) {
    mhc_status st;
    g_launches = 0;
    const bool mx = mx_q != nullptr || mx_scale != nullptr;
    if ((st = check_sizes(T, H)) != MHC_OK) return st;
    if ((st = check_scalars(hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters)) != MHC_OK)
        return st;
    if (T == 0) return MHC_OK;
    if ((st = check_ptrs({{residual, "residual"}, {phi, "phi"}, {bias, "bias"},
                          {mix_scales, "mix_scales"}, {rmsnorm_weight, "rmsnorm_weight"},
                          {pre_mix_out, "pre_mix_out"},
                          {post_mix_out, "post_mix_out"}, {comb_res_mix_out, "comb_res_mix_out"}})) != MHC_OK)
        return st;
    if ((!mx || layer_in_out != nullptr) && (st = check_ptrs({{layer_in_out, "layer_in_out"}})) != MHC_OK) return st;
    if (mx) {
        if (H % 32 != 0) return fail(MHC_ERR_INVALID_ARG, "the MXFP8 output needs H %% 32 == 0 (H=%lld)", (long long)H);
        if (mx_mode != MHC_MX_SCALE_FLOOR && mx_mode != MHC_MX_SCALE_CEIL)
            return fail(MHC_ERR_INVALID_ARG, "unknown MXFP8 scale mode %d", mx_mode);
        if ((st = check_ptrs({{mx_q, "layer_in_fp8"}})) != MHC_OK) return st;
        if (mx_scale == nullptr) return fail(MHC_ERR_INVALID_ARG, "layer_in_scales is NULL");
    }
    if (fused && (st = check_ptrs({{layer_out, "layer_out"}, {prev_post_mix, "prev_post_mix"},
                                   {prev_comb_res_mix, "prev_comb_res_mix"},
                                   {residual_out, "residual_out"}})) != MHC_OK)
        return st;
    if (packed_phi != nullptr && !aligned16(packed_phi))
        return fail(MHC_ERR_INVALID_ARG, "packed_phi is not 16-byte aligned");
    if (workspace == nullptr) return fail(MHC_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MHC_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    const size_t need = workspace_bytes_for(T, H);
    if (workspace_bytes < need)
        return fail(MHC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);

    const size_t tok = (size_t)T;
    const Span sR{residual, tok * 4 * H * 2}, sY{fused ? layer_out : nullptr, tok * H * 2},
        sPP{fused ? prev_post_mix : nullptr, tok * 16}, sPC{fused ? prev_comb_res_mix : nullptr, tok * 64},
        sPhi{phi, (size_t)H * 4 * 24 * 4}, sB{bias, 96}, sMS{mix_scales, 12}, sG{rmsnorm_weight, (size_t)H * 2},
        sW{workspace, need};
    const Span sPk{packed_phi, packed_phi != nullptr ? mhc::ws_pack_bytes((int)H) : 0};
    const Span ins[] = {sR, sY, sPP, sPC, sPhi, sB, sMS, sG, sPk};
    const Span oRo{fused ? residual_out : nullptr, tok * 4 * H * 2}, oX{layer_in_out, tok * H * 2},
        oPre{pre_mix_out, tok * 16}, oPost{post_mix_out, tok * 16}, oRes{comb_res_mix_out, tok * 64};
    const Span oQ{mx_q, mx ? tok * H : 0}, oS{mx_scale, mx ? mx_scale_bytes(T, H) : 0};
    const Span outs[] = {oRo, oX, oPre, oPost, oRes, sW, oQ, oS};
    const char *out_names[] = {"residual_out", "layer_in_out", "pre_mix_out", "post_mix_out",
                               "comb_res_mix_out", "workspace", "layer_in_fp8", "layer_in_scales"};
    for (int o = 0; o < 8; ++o) {
        for (int i = 0; i < 9; ++i) {
            if (o == 0 && i == 0 && residual_out == residual) continue;  // in-place residual update
            if (overlap(outs[o], ins[i]))
                return fail(MHC_ERR_INVALID_ARG, "%s overlaps an input", out_names[o]);
        }
        for (int p = o + 1; p < 8; ++p)
            if (overlap(outs[o], outs[p]))
                return fail(MHC_ERR_INVALID_ARG, "%s overlaps %s", out_names[o], out_names[p]);
    }

    Device dev;
    if ((st = current_device(dev)) != MHC_OK) return st;

    // mix_scales stays a device pointer: the kernels read the three alphas.
    mhc::Scalars s{hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters};
    const int sched = choose_schedule(T, H, dev.sms, mx);
    const mhc::MxOut mxo{mx_q, mx_scale, mx_mode};
    // the split schedule writes its bf16 layer input first (to the caller's buffer, or to the
    // workspace when only the MXFP8 form is wanted) and quantizes it in a second pass
    uint16_t *split_x = layer_in_out;
    if (mx && sched == MHC_SCHEDULE_SPLIT && layer_in_out == nullptr) {
        const size_t need = split_mx_scratch_offset(T, H) + (size_t)T * (size_t)H * 2;
        if (workspace_bytes < need)
            return fail(MHC_ERR_WORKSPACE, "the split schedule's MXFP8-only call needs %zu workspace bytes, got %zu",
                        need, workspace_bytes);
        split_x = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) + split_mx_scratch_offset(T, H));
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (sched) {
        case MHC_SCHEDULE_SPLIT: {
            mhc::SplitArgs a{};
            a.R = residual; a.Y = layer_out; a.prev_post = prev_post_mix; a.prev_comb = prev_comb_res_mix;
            a.phi = phi; a.bias = bias; a.mix_scales = mix_scales; a.gamma = rmsnorm_weight;
            a.T = T; a.H = (int)H; a.s = s;
            a.R_out = fused ? residual_out : nullptr;
            a.X_out = split_x; a.pre_out = pre_mix_out; a.post_out = post_mix_out;
            a.res_out = comb_res_mix_out;
            a.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + mhc::kControlBytes);
            e = mhc::launch_split(a, cs);
            g_launches = 3;
            if (e == cudaSuccess && mx) {
                e = mhc::launch_mx_quantize(split_x, T, (int)H, mxo, dev.sms, cs);
                g_launches += 1;
            }
            break;
        }
        case MHC_SCHEDULE_WS:
        case MHC_SCHEDULE_TILE: {
            const bool tile_alone = sched == MHC_SCHEDULE_TILE;
            if (!tile_alone && !mhc::ws_supported((int)H))
                return fail(MHC_ERR_UNSUPPORTED, "H=%lld does not fit the ws schedule", (long long)H);
            if (tile_alone && !mhc::tile_supported(T, H))
                return fail(MHC_ERR_UNSUPPORTED, "the tile schedule needs H %% 64 == 0 and H > 256 (H=%lld)",
                            (long long)H);
            mhc::FusedArgs a{};
            a.R = residual; a.Y = layer_out; a.prev_post = prev_post_mix; a.prev_comb = prev_comb_res_mix;
            a.phi = phi; a.bias = bias; a.mix_scales = mix_scales; a.gamma = rmsnorm_weight;
            a.T = T; a.H = (int)H; a.s = s;
            a.R_out = fused ? residual_out : nullptr;
            a.X_out = layer_in_out; a.pre_out = pre_mix_out; a.post_out = post_mix_out;
            a.res_out = comb_res_mix_out;
            char *ws = static_cast<char *>(workspace) + mhc::kControlBytes;
            a.phi_pack = packed_phi != nullptr ? static_cast<uint4 *>(const_cast<void *>(packed_phi))
                                               : reinterpret_cast<uint4 *>(ws);
            a.prepacked = packed_phi != nullptr;
            float *zstash = reinterpret_cast<float *>(ws + ((mhc::ws_pack_bytes((int)H) + 255) & ~size_t(255)));
            a.redo_list = reinterpret_cast<unsigned int *>(zstash + (size_t)T * 16);
            a.redo_len = T;
            unsigned int *ctrl = static_cast<unsigned int *>(workspace);
            // with the bf16 layer input wanted as well, a separate streaming quantize pass over it is
            // cheaper than ws's in-kernel epilogue (which lengthens the ring's critical chain); both
            // give the same bits
            const bool mx_pass = mx && layer_in_out != nullptr;
            a.mx = mx_pass ? mhc::MxOut{nullptr, nullptr, 0} : mxo;
            bool tile_ran = false;  // the token-tile kernel's tail does the redo pass
            if (tile_alone) {
                // the token-tile kernel alone on every SM (with the packing launch before it)
                if (!a.prepacked && (e = mhc::launch_ws_pack(phi, (int)H, a.phi_pack, cs)) != cudaSuccess) break;
                e = mhc::launch_tile(a, 0, ctrl, zstash, dev.sms, false, cs);
                g_launches = a.prepacked ? 1 : 2;
                tile_ran = true;
            } else {
                // AUTO on a large call: ws on the leading tokens, the token-tile kernel beside it on
                // the SMs its clusters leave idle (side_split decides the share)
                int side_ctas = 0;
                const int64_t t_ws =
                    forced_schedule() == MHC_SCHEDULE_WS ? T : side_split(T, H, fused, dev.sms, side_ctas);
                const bool side = t_ws < T;
                mhc::FusedArgs aw = a;
                aw.T = t_ws;
                aw.side_follows = side;
                e = mhc::launch_ws(aw, ctrl, zstash, cs);
                g_launches = a.prepacked ? 1 : 2;
                if (e == cudaSuccess && side) {
                    e = mhc::launch_tile(a, t_ws, ctrl, zstash, side_ctas, true, cs);
                    mhc::mark_main_kernel(cs, false);
                    g_launches += 1;
                    tile_ran = true;
                }
            }
            if (e == cudaSuccess && !tile_ran) {
                // tokens whose streams cancel in X, listed by ws: layer input redone
                e = mhc::launch_redo(fused ? residual_out : residual, rmsnorm_weight, rmsnorm_eps, T, (int)H,
                                     pre_mix_out, layer_in_out, a.mx, ctrl, a.redo_list, cs);
                g_launches += 1;
            }
            if (e == cudaSuccess && mx_pass) {
                e = mhc::launch_mx_quantize(layer_in_out, T, (int)H, mxo, dev.sms, cs);
                g_launches += 1;
            }
            break;
        }
        case MHC_SCHEDULE_SMALL: {
            if (!mhc::small_supported(T, (int)H, dev.sms, mx))
                return fail(MHC_ERR_UNSUPPORTED, "T=%lld, H=%lld does not fit the small schedule (T <= %d)",
                            (long long)T, (long long)H, mhc::kSmallMaxT);
            mhc::SplitArgs a{};
            a.R = residual; a.Y = layer_out; a.prev_post = prev_post_mix; a.prev_comb = prev_comb_res_mix;
            a.phi = phi; a.bias = bias; a.mix_scales = mix_scales; a.gamma = rmsnorm_weight;
            a.T = T; a.H = (int)H; a.s = s;
            a.R_out = fused ? residual_out : nullptr;
            a.X_out = layer_in_out; a.pre_out = pre_mix_out; a.post_out = post_mix_out;
            a.res_out = comb_res_mix_out;
            a.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + mhc::kControlBytes);
            a.mx = mxo;
            a.side = side;
            e = mhc::launch_small(a, static_cast<unsigned int *>(workspace), dev.sms, cs);
            g_launches = side != nullptr ? 2 : 1;
            side = nullptr;  // done: the tail kernel ran on the side stream
            break;
        }
        default:
            return fail(MHC_ERR_UNSUPPORTED, "schedule %d is not available", sched);
    }
    if (e == cudaSuccess && side != nullptr) {
        // a split call on a schedule without a side part: the mixes are complete on the main
        // stream; the side stream still gets the fork and the join, so the contract holds
        e = cudaEventRecord(side->fork, cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e == cudaSuccess) e = cudaEventRecord(side->join, side->stream);
    }
    if (e != cudaSuccess) {
        g_launches = 0;
        return cuda_fail(e, "kernel launch");
    }
    return MHC_OK;
}

}  // namespace

namespace mhc {
void set_last_error(const char *msg) { g_last_error = msg; }

namespace {
thread_local cudaEvent_t g_kev_start = nullptr, g_kev_stop = nullptr;
}
void mark_main_kernel(cudaStream_t stream, bool start) {
    cudaEvent_t ev = start ? g_kev_start : g_kev_stop;
    if (ev == nullptr) return;
    // inside a stream capture only an external record becomes a record node of the graph
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, stream);
}
}  // namespace mhc

extern "C" {

size_t mhc_workspace_size(int64_t T, int64_t H) {
    if (T < 0 || H < 0) return 0;
    return workspace_bytes_for(T, H);
}

mhc_status mhc_shifted_post_pre(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                                const float *prev_post_mix, const float *prev_comb_res_mix,
                                const float *phi, const float *bias, const float *mix_scales,
                                const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H,
                                float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                                float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
                                mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                                float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return run_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                        rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                        sinkhorn_iters, residual_out, layer_in_out, pre_mix_out, post_mix_out,
                        comb_res_mix_out, workspace, workspace_bytes, stream, true);
}

mhc_status mhc_shifted_post_pre_split(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                                      const float *prev_post_mix, const float *prev_comb_res_mix,
                                      const float *phi, const float *bias, const float *mix_scales,
                                      const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H,
                                      float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                                      float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
                                      mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                                      float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                      void *stream, void *side_stream, void *fork_event, void *join_event) {
    if (fork_event == nullptr || join_event == nullptr) {
        g_launches = 0;
        return fail(MHC_ERR_INVALID_ARG, "fork_event and join_event must be events");
    }
    if (side_stream == stream) {
        g_launches = 0;
        return fail(MHC_ERR_INVALID_ARG, "side_stream must differ from stream");
    }
    const mhc::SideStream side{static_cast<cudaStream_t>(side_stream), static_cast<cudaEvent_t>(fork_event),
                               static_cast<cudaEvent_t>(join_event)};
    const mhc_status st = run_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                                       rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                                       sinkhorn_iters, residual_out, layer_in_out, pre_mix_out, post_mix_out,
                                       comb_res_mix_out, workspace, workspace_bytes, stream, true, nullptr, nullptr,
                                       0, &side);
    if (st == MHC_OK && T == 0) {  // nothing to compute: the events still mark the (empty) work done
        cudaError_t e = cudaEventRecord(side.fork, static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side.stream, side.fork, 0);
        if (e == cudaSuccess) e = cudaEventRecord(side.join, side.stream);
        if (e != cudaSuccess) return cuda_fail(e, "event record");
    }
    return st;
}

size_t mhc_mxfp8_scale_bytes(int64_t T, int64_t H) {
    if (T < 0 || H < 0 || H % 32 != 0) return 0;
    return mx_scale_bytes(T, H);
}

mhc_status mhc_shifted_post_pre_mxfp8(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                                      const float *prev_post_mix, const float *prev_comb_res_mix,
                                      const float *phi, const float *bias, const float *mix_scales,
                                      const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H,
                                      float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                                      float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
                                      mhc_bf16 *layer_in_out, uint8_t *layer_in_fp8, uint8_t *layer_in_scales,
                                      int scale_mode, float *pre_mix_out, float *post_mix_out,
                                      float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                      void *stream) {
    if (layer_in_fp8 == nullptr && T > 0) return fail(MHC_ERR_INVALID_ARG, "layer_in_fp8 is NULL");
    return run_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                        rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                        sinkhorn_iters, residual_out, layer_in_out, pre_mix_out, post_mix_out,
                        comb_res_mix_out, workspace, workspace_bytes, stream, true, layer_in_fp8,
                        layer_in_scales, scale_mode);
}

mhc_status mhc_pre(const mhc_bf16 *residual, const float *phi, const float *bias,
                   const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H,
                   float hc_norm_eps, float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps,
                   int sinkhorn_iters, mhc_bf16 *layer_in_out, float *pre_mix_out,
                   float *post_mix_out, float *comb_res_mix_out, void *workspace,
                   size_t workspace_bytes, void *stream) {
    return run_post_pre(residual, nullptr, nullptr, nullptr, phi, bias, mix_scales, rmsnorm_weight, T,
                        H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters,
                        nullptr, layer_in_out, pre_mix_out, post_mix_out, comb_res_mix_out, workspace,
                        workspace_bytes, stream, false);
}

mhc_status mhc_pre_broadcast(const mhc_bf16 *x, const float *phi, const float *bias, const float *mix_scales,
                             const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps,
                             float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters,
                             mhc_bf16 *residual_out, mhc_bf16 *layer_in_out, float *pre_mix_out,
                             float *post_mix_out, float *comb_res_mix_out, void *workspace,
                             size_t workspace_bytes, void *stream) {
    mhc_status st;
    g_launches = 0;
    if ((st = check_sizes(T, H)) != MHC_OK) return st;
    if ((st = check_scalars(hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters)) != MHC_OK)
        return st;
    if (T == 0) return MHC_OK;
    if ((st = check_ptrs({{x, "x"}, {residual_out, "residual_out"}})) != MHC_OK) return st;
    const size_t tok = (size_t)T;
    const Span sx{x, tok * H * 2};
    const Span outs[] = {{residual_out, tok * 4 * H * 2}, {layer_in_out, tok * H * 2}, {pre_mix_out, tok * 16},
                         {post_mix_out, tok * 16}, {comb_res_mix_out, tok * 64},
                         {workspace, workspace_bytes < workspace_bytes_for(T, H) ? workspace_bytes
                                                                                : workspace_bytes_for(T, H)}};
    const Span ins[] = {sx, {phi, (size_t)H * 4 * 24 * 4}, {bias, 96}, {mix_scales, 12}, {rmsnorm_weight, (size_t)H * 2}};
    for (int a = 0; a < 6; ++a) {
        for (const Span &i : ins)
            if (overlap(outs[a], i)) return fail(MHC_ERR_INVALID_ARG, "an output overlaps an input");
        for (int b = a + 1; b < 6; ++b)
            if (overlap(outs[a], outs[b])) return fail(MHC_ERR_INVALID_ARG, "two outputs overlap");
    }
    // the pre's own checks (pointers, workspace) also run here, before anything is launched
    if (workspace == nullptr) return fail(MHC_ERR_WORKSPACE, "workspace is NULL");
    if (workspace_bytes < workspace_bytes_for(T, H))
        return fail(MHC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, workspace_bytes_for(T, H));
    if ((st = check_ptrs({{phi, "phi"}, {bias, "bias"}, {mix_scales, "mix_scales"}, {rmsnorm_weight, "rmsnorm_weight"},
                          {layer_in_out, "layer_in_out"}, {pre_mix_out, "pre_mix_out"}, {post_mix_out, "post_mix_out"},
                          {comb_res_mix_out, "comb_res_mix_out"}})) != MHC_OK)
        return st;
    const int forced = g_forced_schedule.load(std::memory_order_relaxed);
    const bool fusable = mhc::bcast_supported(T, H);
    if (forced == MHC_SCHEDULE_BCAST && !fusable)
        return fail(MHC_ERR_UNSUPPORTED, "the broadcast schedule needs H %% 64 == 0 (H=%lld)", (long long)H);
    Device dev;
    if ((st = current_device(dev)) != MHC_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the fused kernel from x alone, for all but the small-T calls (there the small schedule's
    // one launch over every SM is faster than one CTA per 8 tokens)
    if (forced == MHC_SCHEDULE_BCAST || (forced == MHC_SCHEDULE_AUTO && fusable && T > kSmallAutoMaxT)) {
        mhc::BcastArgs a{};
        a.x = x; a.phi = phi; a.bias = bias; a.mix_scales = mix_scales; a.gamma = rmsnorm_weight;
        a.T = T; a.H = (int)H;
        a.s = mhc::Scalars{hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters};
        a.R_out = residual_out; a.X_out = layer_in_out;
        a.pre_out = pre_mix_out; a.post_out = post_mix_out; a.res_out = comb_res_mix_out;
        cudaError_t e = mhc::launch_bcast_pre(a, static_cast<unsigned int *>(workspace),
                                              static_cast<char *>(workspace) + mhc::kControlBytes, dev.sms, cs);
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        g_launches = 2;
        return MHC_OK;
    }
    cudaError_t e = mhc::launch_broadcast4(x, T, (int)H, residual_out, dev.sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    st = run_post_pre(residual_out, nullptr, nullptr, nullptr, phi, bias, mix_scales, rmsnorm_weight, T, H,
                      hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters, nullptr, layer_in_out,
                      pre_mix_out, post_mix_out, comb_res_mix_out, workspace, workspace_bytes, stream, false);
    if (st == MHC_OK) g_launches += 1;
    return st;
}

mhc_status mhc_post(const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
                    const float *prev_comb_res_mix, int64_t T, int64_t H, mhc_bf16 *residual_out,
                    void *stream) {
    mhc_status st;
    g_launches = 0;
    if ((st = check_sizes(T, H)) != MHC_OK) return st;
    if (T == 0) return MHC_OK;
    if ((st = check_ptrs({{residual, "residual"}, {layer_out, "layer_out"}, {prev_post_mix, "prev_post_mix"},
                          {prev_comb_res_mix, "prev_comb_res_mix"}, {residual_out, "residual_out"}})) != MHC_OK)
        return st;
    const size_t tok = (size_t)T;
    const Span o{residual_out, tok * 4 * H * 2};
    if (residual_out != residual && overlap(o, {residual, tok * 4 * H * 2}))
        return fail(MHC_ERR_INVALID_ARG, "residual_out overlaps residual");
    if (overlap(o, {layer_out, tok * H * 2}) || overlap(o, {prev_post_mix, tok * 16}) ||
        overlap(o, {prev_comb_res_mix, tok * 64}))
        return fail(MHC_ERR_INVALID_ARG, "residual_out overlaps an input");
    Device dev;
    if ((st = current_device(dev)) != MHC_OK) return st;
    cudaError_t e = mhc::launch_post(residual, layer_out, prev_post_mix, prev_comb_res_mix, T, (int)H,
                                     residual_out, dev.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches = 1;
    return MHC_OK;
}

namespace {
// Common body of mhc_post_int8 and mhc_post_sqrsum.
mhc_status run_post_ex(const mhc_bf16 *residual, const mhc_bf16 *layer_out, const int8_t *layer_out_q,
                       const float *x_scales, const float *prev_post_mix, const float *prev_comb_res_mix,
                       int64_t T, int64_t H, mhc_bf16 *residual_out, float *sqrsum_out, void *stream) {
    mhc_status st;
    g_launches = 0;
    if ((st = check_sizes(T, H)) != MHC_OK) return st;
    if (T > INT32_MAX) return fail(MHC_ERR_INVALID_ARG, "T too large");
    if (T == 0) return MHC_OK;
    const bool i8 = layer_out_q != nullptr;
    if ((st = check_ptrs({{residual, "residual"}, {prev_post_mix, "prev_post_mix"},
                          {prev_comb_res_mix, "prev_comb_res_mix"}, {residual_out, "residual_out"}})) != MHC_OK)
        return st;
    if (i8) {
        if ((st = check_ptrs({{layer_out_q, "layer_out_q"}, {x_scales, "x_scales"}})) != MHC_OK) return st;
    } else if ((st = check_ptrs({{layer_out, "layer_out"}})) != MHC_OK) {
        return st;
    }
    if (sqrsum_out != nullptr && (st = check_ptrs({{sqrsum_out, "sqrsum_out"}})) != MHC_OK) return st;
    const size_t tok = (size_t)T;
    const Span o{residual_out, tok * 4 * H * 2}, oS{sqrsum_out, sqrsum_out ? tok * 4 : 0};
    const Span ins[] = {{residual, tok * 4 * H * 2}, {layer_out, i8 ? 0 : tok * H * 2},
                        {layer_out_q, i8 ? tok * H : 0}, {x_scales, i8 ? tok * 4 : 0},
                        {prev_post_mix, tok * 16}, {prev_comb_res_mix, tok * 64}};
    for (int i = 0; i < 6; ++i) {
        if (i == 0 && residual_out == residual) continue;  // in-place residual update
        if (overlap(o, ins[i])) return fail(MHC_ERR_INVALID_ARG, "residual_out overlaps an input");
        if (overlap(oS, ins[i])) return fail(MHC_ERR_INVALID_ARG, "sqrsum_out overlaps an input");
    }
    if (overlap(o, oS)) return fail(MHC_ERR_INVALID_ARG, "sqrsum_out overlaps residual_out");
    Device dev;
    if ((st = current_device(dev)) != MHC_OK) return st;
    cudaError_t e = mhc::launch_post_ex(residual, i8 ? nullptr : layer_out, layer_out_q, x_scales, prev_post_mix,
                                        prev_comb_res_mix, T, (int)H, residual_out, sqrsum_out,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches = 1;
    return MHC_OK;
}
}  // namespace

mhc_status mhc_post_int8(const mhc_bf16 *residual, const int8_t *layer_out_q, const float *x_scales,
                         const float *prev_post_mix, const float *prev_comb_res_mix, int64_t T, int64_t H,
                         mhc_bf16 *residual_out, float *sqrsum_out, void *stream) {
    if (layer_out_q == nullptr && T > 0) return fail(MHC_ERR_INVALID_ARG, "layer_out_q is NULL");
    return run_post_ex(residual, nullptr, layer_out_q, x_scales, prev_post_mix, prev_comb_res_mix, T, H,
                       residual_out, sqrsum_out, stream);
}

mhc_status mhc_post_sqrsum(const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
                           const float *prev_comb_res_mix, int64_t T, int64_t H, mhc_bf16 *residual_out,
                           float *sqrsum_out, void *stream) {
    if (sqrsum_out == nullptr && T > 0) return fail(MHC_ERR_INVALID_ARG, "sqrsum_out is NULL");
    return run_post_ex(residual, layer_out, nullptr, nullptr, prev_post_mix, prev_comb_res_mix, T, H,
                       residual_out, sqrsum_out, stream);
}

size_t mhc_packed_phi_bytes(int64_t H) {
    if (H < 8 || H > MHC_MAX_HIDDEN || H % 8 != 0) return 0;
    return mhc::ws_pack_bytes((int)H);
}

mhc_status mhc_pack_phi(const float *phi, int64_t H, void *packed_phi, size_t packed_bytes, void *stream) {
    mhc_status st;
    g_launches = 0;
    if ((st = check_sizes(1, H)) != MHC_OK) return st;
    if ((st = check_ptrs({{phi, "phi"}, {packed_phi, "packed_phi"}})) != MHC_OK) return st;
    const size_t need = mhc::ws_pack_bytes((int)H);
    if (packed_bytes < need) return fail(MHC_ERR_INVALID_ARG, "packed_phi has %zu bytes, needs %zu", packed_bytes, need);
    if (overlap({phi, (size_t)H * 4 * 24 * 4}, {packed_phi, need}))
        return fail(MHC_ERR_INVALID_ARG, "packed_phi overlaps phi");
    Device dev;
    if ((st = current_device(dev)) != MHC_OK) return st;
    cudaError_t e = mhc::launch_ws_pack(phi, (int)H, static_cast<uint4 *>(packed_phi), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches = 1;
    return MHC_OK;
}

mhc_status mhc_shifted_post_pre_prepacked(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                                          const float *prev_post_mix, const float *prev_comb_res_mix,
                                          const float *phi, const void *packed_phi, const float *bias,
                                          const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T,
                                          int64_t H, float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                                          float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
                                          mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                                          float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    if (packed_phi == nullptr && T > 0) {
        g_launches = 0;
        return fail(MHC_ERR_INVALID_ARG, "packed_phi is NULL");
    }
    return run_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                        rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                        sinkhorn_iters, residual_out, layer_in_out, pre_mix_out, post_mix_out,
                        comb_res_mix_out, workspace, workspace_bytes, stream, true, nullptr, nullptr, 0, nullptr,
                        packed_phi);
}

mhc_status mhc_shifted_post_pre_mxfp8_prepacked(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix, const float *prev_comb_res_mix,
    const float *phi, const void *packed_phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
    float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out, mhc_bf16 *layer_in_out, uint8_t *layer_in_fp8,
    uint8_t *layer_in_scales, int scale_mode, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *workspace, size_t workspace_bytes, void *stream) {
    g_launches = 0;
    if (packed_phi == nullptr && T > 0) return fail(MHC_ERR_INVALID_ARG, "packed_phi is NULL");
    if (layer_in_fp8 == nullptr && T > 0) return fail(MHC_ERR_INVALID_ARG, "layer_in_fp8 is NULL");
    return run_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                        rmsnorm_weight, T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                        sinkhorn_iters, residual_out, layer_in_out, pre_mix_out, post_mix_out,
                        comb_res_mix_out, workspace, workspace_bytes, stream, true, layer_in_fp8,
                        layer_in_scales, scale_mode, nullptr, packed_phi);
}

mhc_status mhc_pre_prepacked(const mhc_bf16 *residual, const float *phi, const void *packed_phi, const float *bias,
                             const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H,
                             float hc_norm_eps, float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps,
                             int sinkhorn_iters, mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                             float *comb_res_mix_out, void *workspace, size_t workspace_bytes, void *stream) {
    if (packed_phi == nullptr && T > 0) {
        g_launches = 0;
        return fail(MHC_ERR_INVALID_ARG, "packed_phi is NULL");
    }
    return run_post_pre(residual, nullptr, nullptr, nullptr, phi, bias, mix_scales, rmsnorm_weight, T, H,
                        hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters, nullptr, layer_in_out,
                        pre_mix_out, post_mix_out, comb_res_mix_out, workspace, workspace_bytes, stream, false,
                        nullptr, nullptr, 0, nullptr, packed_phi);
}

mhc_status mhc_set_schedule(int schedule) {
    if (schedule != MHC_SCHEDULE_AUTO && schedule != MHC_SCHEDULE_SPLIT && schedule != MHC_SCHEDULE_WS &&
        schedule != MHC_SCHEDULE_SMALL && schedule != MHC_SCHEDULE_BCAST && schedule != MHC_SCHEDULE_TILE)
        return fail(MHC_ERR_INVALID_ARG, "unknown schedule %d", schedule);
    g_forced_schedule.store(schedule, std::memory_order_relaxed);
    return MHC_OK;
}

int mhc_auto_schedule(int64_t T, int64_t H) {
    Device dev;
    if (current_device(dev) != MHC_OK) return MHC_SCHEDULE_AUTO;
    return auto_schedule(T, H, dev.sms);
}

int64_t mhc_auto_side_tokens(int64_t T, int64_t H, int fused) {
    if (T < 0 || H < 0) return -1;
    Device dev;
    if (current_device(dev) != MHC_OK) return -1;
    if (auto_schedule(T, H, dev.sms) != MHC_SCHEDULE_WS) return 0;
    int idle = 0;
    return T - side_split(T, H, fused != 0, dev.sms, idle);
}

mhc_status mhc_check_status(void *workspace, void *stream) {
    if (workspace == nullptr) return fail(MHC_ERR_WORKSPACE, "workspace is NULL");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    if (word != 0) {
        // a wait that gave up can leave barrier words mid-count: clear the whole control block
        e = cudaMemsetAsync(workspace, 0, mhc::kControlBytes, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(control block)");
        return fail(MHC_ERR_DEVICE_TIMEOUT, "device status word 0x%08x", word);
    }
    return MHC_OK;
}

const char *mhc_status_string(int status) {
    switch (status) {
        case MHC_OK: return "MHC_OK: success";
        case MHC_ERR_INVALID_ARG: return "MHC_ERR_INVALID_ARG: invalid argument";
        case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: unsupported device or schedule";
        case MHC_ERR_WORKSPACE: return "MHC_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: CUDA runtime error";
        case MHC_ERR_DEVICE_TIMEOUT: return "MHC_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
        default: return "unknown mhc_status";
    }
}

const char *mhc_last_error(void) { return g_last_error.c_str(); }

int mhc_last_launch_count(void) { return g_launches; }

void mhc_set_main_kernel_events(void *start, void *stop) {
    mhc::g_kev_start = static_cast<cudaEvent_t>(start);
    mhc::g_kev_stop = static_cast<cudaEvent_t>(stop);
}

}  // extern "C"
