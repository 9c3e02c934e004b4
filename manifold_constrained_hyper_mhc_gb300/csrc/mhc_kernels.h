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

// Cluster schedule (kernels_fused.cu).
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
    uint4 *phi_pack;  // workspace: fused_pack_bytes(H, C)
    int C, G;         // cluster size, tokens per group
    MxOut mx;         // MXFP8 layer input (mx.q == nullptr: none); ws and small schedules only
};

int fused_slice(int H, int C);                     // hidden elements per CTA (multiple of 16)
size_t fused_pack_bytes(int H, int C);             // packed phi fragments
size_t fused_smem_bytes(int H, int C, int G);      // dynamic shared memory per CTA
cudaError_t launch_fused(const FusedArgs &a, cudaStream_t stream);
// phi [4H][24] fp32 -> mma A fragments for a cluster of C CTAs of slice Hs
void launch_pack_phi(const float *phi, int H, int C, int Hs, uint4 *out, int64_t total, cudaStream_t stream);

// Cluster-of-16 schedule with phi resident in tensor memory (kernels_fused_tmem.cu).
int fused_tmem_slice(int H);
bool fused_tmem_supported(int H);
size_t fused_tmem_pack_bytes(int H);
cudaError_t launch_fused_tmem(const FusedArgs &a, unsigned int *status, cudaStream_t stream);

// Pipelined cluster-of-16 schedule (kernels_pipe.cu).
int pipe_slice(int H);
bool pipe_supported(int H);
size_t pipe_pack_bytes(int H);
size_t pipe_stash_bytes(int64_t T);
cudaError_t launch_pipe(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream);

// Pipelined cluster-of-16 schedule with the projection on tcgen05 (kernels_pipe2.cu).
int pipe2_slice(int H);
bool pipe2_supported(int H);
size_t pipe2_pack_bytes(int H);
size_t pipe2_stash_bytes(int64_t T);
cudaError_t launch_pipe2(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream);
// Warp-specialised pipelined cluster-of-16 schedule (kernels_ws.cu).
int ws_slice(int H);
bool ws_supported(int H);
size_t ws_pack_bytes(int H);
size_t ws_stash_bytes(int64_t T);
cudaError_t launch_ws(const FusedArgs &a, unsigned int *status, float *zstash, cudaStream_t stream);

// Small-T schedule (kernels_small.cu): one cooperative launch, one CTA per hidden slice,
// one grid barrier on a 64-bit arrival counter at control-block bytes 64..71.
constexpr int kSmallMaxT = 128;
int small_ctas(int H, int num_sms);
int small_slice(int H, int num_sms, int align);  // align 8, or 32 for the MXFP8 output
bool small_supported(int64_t T, int H, int num_sms, bool mx);
size_t small_workspace_bytes(int64_t T, int H);  // upper bound over SM counts
cudaError_t launch_small(const SplitArgs &a, unsigned int *ctrl, int num_sms, cudaStream_t stream);

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
