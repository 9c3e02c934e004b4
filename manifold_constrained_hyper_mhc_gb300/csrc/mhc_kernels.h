// Internal launch interface between the C-ABI layer (mhc_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "mhc_device.cuh"

namespace mhc {

// Split schedule geometry (also sizes its workspace).
constexpr int kSplitTok = 16;    // tokens per CTA of the partial-sum kernel
constexpr int kSplitH = 256;     // hidden elements per chunk
constexpr int kPartStride = 32;  // floats per (token, chunk) record: z[24], square sum, pad

// Bytes at the start of every workspace reserved for the control block
// (device status word, barrier counters).
constexpr size_t kControlBytes = 256;
// 32-bit words of the control block: the length of the redo list (tokens whose streams cancel
// in X, see redo_kernel) and the count of CTAs done (the redo kernel's, or the token-tile
// kernel's); both zero between calls.
constexpr int kRedoCountWord = 32, kRedoDoneWord = 33;
// The small schedule's two 64-bit grid-barrier words start at these 32-bit word offsets (16-17
// and 18-19); each is zero in its low half between launches.
constexpr int kSmallBarrierWord = 16;

// A second stream for the off-critical-path part of a split call: `fork` is recorded on the
// main stream once the records are in, the side stream waits on it, and `join` is recorded on
// the side stream after its work.
struct SideStream {
    cudaStream_t stream;
    cudaEvent_t fork, join;
};

struct SplitArgs {
    const uint16_t *R;  // residual (fused) or already post-updated residual (pre only)
    const uint16_t *Y;
    const float *prev_post, *prev_comb, *phi, *bias, *mix_scales;
    const uint16_t *gamma;
    int64_t T;
    int H;
    Scalars s;
    uint16_t *R_out;  // nullptr: pre only (R already holds R')
    uint16_t *X_out;
    float *pre_out, *post_out, *res_out;
    float *part;  // workspace: [T][ceil(H/256)][32] floats
    MxOut mx;     // MXFP8 layer input (mx.q == nullptr: none)
    const SideStream *side;  // small schedule only: post and residual mixes on a side stream (nullptr: no)
};

inline size_t split_workspace_bytes(int64_t T, int64_t H) {
    const int64_t nchunk = (H + kSplitH - 1) / kSplitH;
    return (size_t)T * (size_t)nchunk * kPartStride * sizeof(float);
}

cudaError_t launch_split(const SplitArgs &a, cudaStream_t stream);

// Arguments of the warp-specialised cluster schedule (kernels_ws.cu).
struct FusedArgs {
    const uint16_t *R;  // residual (fused) or already post-updated residual (pre only)
    const uint16_t *Y;
    const float *prev_post, *prev_comb, *phi, *bias, *mix_scales;
    const uint16_t *gamma;
    int64_t T;
    int H;
    Scalars s;
    uint16_t *R_out;  // nullptr: pre only
    uint16_t *X_out;
    float *pre_out, *post_out, *res_out;
    uint4 *phi_pack;  // ws_pack_bytes(H): the workspace (packed by the call) or the caller's packed phi
    bool prepacked;   // phi_pack already holds the packed phi (no packing launch)
    bool side_follows;  // ws: the token-tile kernel is launched right after it (beside it)
    unsigned int *redo_list;  // [redo_len]: tokens whose layer input the redo pass recomputes
    int64_t redo_len;         // the call's token count (ws may run on fewer, T above)
    MxOut mx;         // MXFP8 layer input (mx.q == nullptr: none)
};

// Warp-specialised pipelined cluster-of-16 schedule (kernels_ws.cu).
int ws_slice(int H);
bool ws_supported(int H);
size_t ws_pack_bytes(int H);
// phi [4H][24] fp32 -> the packed fragments ws reads (ws_pack_bytes(H) bytes at out).
cudaError_t launch_ws_pack(const float *phi, int H, uint4 *out, cudaStream_t stream);
size_t ws_stash_bytes(int64_t T);
cudaError_t launch_ws(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream);
// CTAs of ws resident at once on this device (clusters of 16 that fit, times 16).
cudaError_t ws_resident_ctas(int H, bool post, int &ctas);

// Token-tile schedule (kernels_tile.cu): tiles of 18 tokens, one CTA per SM, no clusters; phi
// read from the ws packed form (a.phi_pack).  It computes tokens [t_begin, a.T) with up to
// `grid` CTAs, alone or beside ws (beside: launched right after ws on the same stream, on the
// SMs ws leaves idle).  The tokens whose streams cancel in X go on the redo list.
bool tile_supported(int64_t T, int64_t H);
int tile_tokens();  // tokens per tile of the token-tile kernel
cudaError_t launch_tile(const FusedArgs &a, int64_t t_begin, unsigned int *status, float *zstash, int grid,
                        bool beside, cudaStream_t stream);

// Small-T schedule (kernels_small.cu): one cooperative launch, one CTA per hidden slice,
// grid barriers on 64-bit words at control-block bytes 64..71 (after the partial sums) and
// 72..79 (the direct square sums of tokens whose streams cancel in X, when there are any).
constexpr int kSmallMaxT = 128;
int small_ctas(int H, int num_sms);
int small_slice(int H, int num_sms, int align);  // align 8, or 32 for the MXFP8 output
bool small_supported(int64_t T, int H, int num_sms, bool mx);
size_t small_workspace_bytes(int64_t T, int H);  // upper bound over SM counts
cudaError_t launch_small(const SplitArgs &a, unsigned int *ctrl, int num_sms, cudaStream_t stream);

// After the ws kernel on the same stream: the layer input (and its MXFP8 form, mx.q != nullptr)
// of the tokens listed in `list` (length in control-block word kRedoCountWord), with sum_h X^2
// summed directly (kernels_redo.cu).  Rp is the R' the main kernel read or wrote.
cudaError_t launch_redo(const uint16_t *Rp, const uint16_t *gamma, float rmsnorm_eps, int64_t T, int H,
                        const float *pre_out, uint16_t *X_out, const MxOut &mx, unsigned int *ctrl,
                        const unsigned int *list, cudaStream_t stream);

// Records the events set by mhc_set_main_kernel_events (if any) on `stream` right before
// (start) and after (stop) the launch of a call's main kernel.
void mark_main_kernel(cudaStream_t stream, bool start);

// The post with an int8 layer output (Yq, x_scales; Y unused) or a bf16 one (Y), and the
// square sum of R' per token when sqrsum != nullptr (kernels_post.cu).  T < 2^31.
cudaError_t launch_post_ex(const uint16_t *R, const uint16_t *Y, const int8_t *Yq, const float *x_scales,
                           const float *prev_post, const float *prev_comb, int64_t T, int H, uint16_t *R_out,
                           float *sqrsum, cudaStream_t stream);

// The MXFP8 form of a bf16 [T][H] layer input already written (kernels_post.cu); H % 32 == 0.
cudaError_t launch_mx_quantize(const uint16_t *X, int64_t T, int H, const MxOut &mx, int num_sms, cudaStream_t stream);

// R_out[t][j] = x[t] for the four streams (kernels_post.cu).
cudaError_t launch_broadcast4(const uint16_t *x, int64_t T, int H, uint16_t *R_out, int num_sms, cudaStream_t stream);

// The first layer's pre from its (T, H) input x, the residual being four copies of x
// (kernels_bcast.cu): one packing launch, then one persistent kernel.
struct BcastArgs {
    const uint16_t *x;  // [T][H]
    const float *phi, *bias, *mix_scales;
    const uint16_t *gamma;
    int64_t T;
    int H;
    Scalars s;
    uint16_t *R_out;  // [T][4][H]: four copies of x
    uint16_t *X_out;
    float *pre_out, *post_out, *res_out;
};
bool bcast_supported(int64_t T, int64_t H);
size_t bcast_workspace_bytes(int64_t T, int64_t H);  // after the control block
cudaError_t launch_bcast_pre(const BcastArgs &a, unsigned int *status, void *scratch, int num_sms, cudaStream_t stream);

cudaError_t launch_post(const uint16_t *R, const uint16_t *Y, const float *prev_post,
                        const float *prev_comb, int64_t T, int H, uint16_t *R_out, int num_sms,
                        cudaStream_t stream);

}  // namespace mhc
