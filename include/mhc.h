/*
 * mhc.h -- C ABI of the GB300 (sm_103a) fused mHC post+pre library (libmhc.so).
 *
 * The op.  A DeepSeek-V4-style decoder carries hc_mult = 4 residual streams per
 * token.  At every layer boundary the previous layer's output is folded into
 * the streams ("post") and the next layer's input is formed from them ("pre").
 * The pages this follows:
 *   - "[SM80] Backport mHC fused post + int8 all-reduce; fixes #28, #29",
 *     "What this fixes": the mHC post kernel and its fused square sum.
 *   - "[DSv4.1] Integrate Mega-mHC from DeepGEMM": the fused post+pre op
 *     mhc_shifted_post_pre (Mega-mHC), its scalar tail and naming
 *     ("Style findings", Major 1: rms_eps->hc_norm_eps, hc_post_alpha->
 *     hc_post_scale, norm_eps->rmsnorm_eps, res_mix->comb_res_mix), the
 *     distinct eps values that catch an argument swap ("Verified OK"), the
 *     hc_mult == 4 gate and the 2^20 token bound ("Verified OK"), and the
 *     capture-on-a-fresh-stream hazard of lazily created barrier state
 *     ("Correctness findings", Minor 3).
 *   - "[DSV4.1] Four BS=1 critical-path fixes for DSpark decode": the mHC
 *     statistics and Sinkhorn and the combine+RMSNorm ("What changed" item 3,
 *     "Measured and deliberately left out").
 *
 * Per token t (all tokens are independent), with streams R[t] in [4][H]:
 *   (1) post:    R'[i] = sum_j comb[j][i] * R[j] + post[i] * Y           -> bf16
 *   (2) RMS:     r = 1 / sqrt(mean over the 4H entries of R'^2 + hc_norm_eps)
 *                z = r * (flat(R') @ phi),  flat index k = i*H + h,  24 logits
 *   (3) heads:   pre_mix[i]  = sigmoid(alpha_pre  * z[i]   + bias[i])
 *                post_mix[i] = hc_post_scale * sigmoid(alpha_post * z[4+i] + bias[4+i])
 *                comb_res_mix = Sinkhorn(M),  M[a][c] = exp(alpha_res * z[8+4a+c] + bias[8+4a+c]),
 *                  one iteration = rows /= (row sum + sinkhorn_eps), then
 *                  columns /= (column sum + sinkhorn_eps); sinkhorn_iters iterations
 *   (4) combine: X = sum_i pre_mix[i] * R'[i];  out = X / sqrt(mean_h X^2 + rmsnorm_eps) * gamma -> bf16
 * Steps (2)-(4) consume the bf16-rounded R', so mhc_shifted_post_pre equals
 * mhc_post followed by mhc_pre bit for bit.  comb_res_mix_out is written
 * [a][c] and a following call consumes it as prev_comb_res_mix[j][i].
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer, owned by the caller, row-major and
 *     contiguous, 16-byte aligned.  bf16 data is passed as raw bit patterns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  They never synchronise, never allocate, and keep no lazy per-
 *     stream state, so the first call may happen inside CUDA-graph capture.
 *   - Arguments are validated before anything is launched; on any error nothing
 *     is launched and no output is touched.
 *   - T == 0 is valid and launches nothing.  1 <= T <= MHC_MAX_TOKENS,
 *     8 <= H <= MHC_MAX_HIDDEN, H % 8 == 0 (16-byte bf16 vectors).
 *   - The eps values must be finite and >= 0, hc_post_scale finite,
 *     0 <= sinkhorn_iters <= MHC_MAX_SINKHORN_ITERS.
 *   - residual_out may be the same buffer as residual (in-place update); any
 *     other overlap between an input and an output is rejected.
 *   - The workspace is caller-owned device memory of at least
 *     mhc_workspace_size(T, H) bytes, 256-byte aligned.  Before its first use it
 *     must be zero-filled (e.g. cudaMemsetAsync); every call that completes
 *     leaves it ready for the next call, whatever that call's T and H (after a
 *     device-side timeout, mhc_check_status clears it).  Calls that share one
 *     workspace must be ordered (same stream or explicit events); concurrent
 *     use races.
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MHC_API __attribute__((visibility("default")))
#else
#define MHC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mhc_bf16; /* bfloat16 bit pattern */

#define MHC_HC_MULT 4
#define MHC_NUM_MIX 24
/* the 2^20-token bound of the integrated kernel ("[DSv4.1] Integrate Mega-mHC from DeepGEMM",
 * Verified OK) */
#define MHC_MAX_TOKENS (1 << 20)
#define MHC_MAX_HIDDEN 65536
#define MHC_MAX_SINKHORN_ITERS 64

typedef enum mhc_status {
    MHC_OK = 0,
    MHC_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size, bad scalar, overlap */
    MHC_ERR_UNSUPPORTED = -2,    /* device is not sm_103 / forced schedule cannot run this shape */
    MHC_ERR_WORKSPACE = -3,      /* workspace missing, too small or misaligned */
    MHC_ERR_CUDA = -4,           /* a CUDA runtime call or launch failed (see mhc_last_error) */
    MHC_ERR_DEVICE_TIMEOUT = -5  /* a bounded device-side wait gave up (mhc_check_status) */
} mhc_status;

/* Kernel schedules.  AUTO picks by T, H and the SM count. */
typedef enum mhc_schedule {
    MHC_SCHEDULE_AUTO = 0,
    MHC_SCHEDULE_SPLIT = 1,       /* three launches: post + partial sums, mixes, combine + RMSNorm
                                     (any H; AUTO's choice where ws does not fit, H > 7168, for
                                     T < 448; from 448 tokens AUTO takes the tile schedule there) */
    /* values 2-7 named cluster and pipelined schedules that the ws schedule superseded; they
       were removed and mhc_set_schedule rejects them */
    MHC_SCHEDULE_WS = 8,          /* clusters of 16 CTAs split the hidden dimension (H <= 7168), 8
                                     tokens per group, phi resident in tensor memory; warp-specialised
                                     roles (post, projection + Gram on the tensor cores, owner,
                                     combine) hand groups over through mbarriers, TMA tensor copies
                                     into a 6-deep tile ring, point-to-point DSMEM messages; a
                                     second small launch redoes the layer input of tokens whose
                                     streams cancel in X with a direct square sum (it exits at once
                                     when there are none) */
    MHC_SCHEDULE_SMALL = 9,       /* T <= 128 only (and its shared memory must fit: at H = 7168,
                                     T <= 96): one cooperative launch, one CTA per hidden slice
                                     on up to every SM, one bounded grid barrier between the partial
                                     sums and the combine (latency-bound decode calls) */
    MHC_SCHEDULE_BCAST = 10,      /* mhc_pre_broadcast only (H % 64 == 0): one persistent kernel that
                                     works from x alone, 8 tokens per tile, x read twice (the second
                                     time from L2); the other calls choose as AUTO */
    MHC_SCHEDULE_TILE = 11        /* H % 64 == 0, H > 256: one CTA per SM on tiles of 18 tokens, no
                                     clusters; a tile's row walked twice in chunks (post, R' to HBM
                                     and kept in L2, projection with phi read from L2; then the
                                     combine from R' read back, with the MXFP8 form when asked for).
                                     AUTO runs it beside ws on the SMs that ws's clusters leave idle,
                                     on a share of the tokens (mhc_auto_side_tokens), for calls of
                                     at least 2048 tokens; forced, it takes every SM */
} mhc_schedule;

/* Bytes of workspace the calls below need for T tokens of hidden size H. */
MHC_API size_t mhc_workspace_size(int64_t T, int64_t H);

/* The fused step (1)-(4): mhc_shifted_post_pre / Mega-mHC ("[DSv4.1] Integrate
 * Mega-mHC from DeepGEMM", "Purpose" and "Verified OK").
 *   residual          [T,4,H] bf16   streams before this layer's post
 *   layer_out         [T,H]   bf16   the previous sublayer's output Y
 *   prev_post_mix     [T,4]   fp32   post mix of the previous layer
 *   prev_comb_res_mix [T,4,4] fp32   residual mix of the previous layer, [j][i]
 *   phi               [4H,24] fp32   projection, row k = i*H + h
 *   bias              [24]    fp32   0:4 pre, 4:8 post, 8:24 residual mix (row-major 4x4)
 *   mix_scales        [3]     fp32   alpha_pre, alpha_post, alpha_res
 *   rmsnorm_weight    [H]     bf16   gamma
 * Outputs:
 *   residual_out      [T,4,H] bf16   R'
 *   layer_in_out      [T,H]   bf16   RMSNorm(sum_i pre_mix[i] R'[i]) * gamma
 *   pre_mix_out       [T,4]   fp32
 *   post_mix_out      [T,4]   fp32
 *   comb_res_mix_out  [T,4,4] fp32   [a][c]
 * The scalar tail is in this order: hc_norm_eps, rmsnorm_eps, hc_post_scale,
 * sinkhorn_eps, sinkhorn_iters. */
MHC_API mhc_status mhc_shifted_post_pre(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
    float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *workspace, size_t workspace_bytes, void *stream);

/* The fused step with its off-critical-path part on a second stream ("[DSV4.1] Four BS=1
 * critical-path fixes for DSpark decode", "Measured and deliberately left out": the split
 * path keeps the mHC statistics and Sinkhorn off the main stream).  Arguments and outputs as in
 * mhc_shifted_post_pre, plus:
 *   side_stream   a cudaStream_t other than `stream`
 *   fork_event,   cudaEvent_t handles owned by the caller (cudaEventDisableTiming is fine)
 *   join_event
 * On `stream`: residual_out, layer_in_out and pre_mix_out (everything the next sublayer needs).
 * fork_event is recorded on `stream` once the per-CTA records are in the workspace; side_stream
 * waits on it, computes post_mix_out and comb_res_mix_out (the Sinkhorn) from those records,
 * and join_event is recorded on side_stream after them.  The caller makes whatever reads the
 * post or residual mix, and the next call that uses this workspace, wait on join_event (e.g.
 * cudaStreamWaitEvent(stream, join_event) before the next layer's call; under stream capture
 * this also joins side_stream back).  Results are bit-identical to mhc_shifted_post_pre on the
 * same schedule.  Only the small schedule (AUTO for T <= 32) has a side part; on the others
 * every output is produced on `stream` and the events are still recorded and waited on. */
MHC_API mhc_status mhc_shifted_post_pre_split(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
    float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *workspace, size_t workspace_bytes, void *stream, void *side_stream, void *fork_event,
    void *join_event);

/* MXFP8 block-scale rules for the quantized layer input (the pages name MXFP8 and the
 * UE8M0 scale byte but give no formula; both rules are offered). */
typedef enum mhc_mx_scale_mode {
    MHC_MX_SCALE_FLOOR = 0,  /* E = floor(log2 amax) - 8 (OCP MX): the largest element lands in
                                [256, 512) and saturates to 448 above 448 */
    MHC_MX_SCALE_CEIL = 1    /* the smallest E with amax <= 448 * 2^E: no element saturates */
} mhc_mx_scale_mode;

/* Bytes of the layer input's MXFP8 scale block for T tokens of size H (H % 32 == 0;
 * 0 otherwise): (T rounded up to 128) * (H / 32 rounded up to 4). */
MHC_API size_t mhc_mxfp8_scale_bytes(int64_t T, int64_t H);

/* The fused step (1)-(4) with the layer input also emitted as MXFP8, the quantize that
 * consumes it fused into the combine+RMSNorm epilogue ("[DSV4.1] Four BS=1 critical-path
 * fixes for DSpark decode", "What changed" item 3 and "Correctness").  Arguments and the other
 * outputs as in mhc_shifted_post_pre, plus:
 *   layer_in_out      [T,H] bf16, or NULL to skip the bf16 layer input
 *   layer_in_fp8      [T,H] uint8  E4M3 codes of x / 2^E for each block of 32 consecutive
 *                     values of a token (x = the bf16 layer input; round to nearest even,
 *                     finite values beyond 448 saturate); 16-byte aligned
 *   layer_in_scales   mhc_mxfp8_scale_bytes(T, H) bytes: the byte E + 127 of block k of
 *                     token m at ((m/128)*KT + k/4)*512 + (m%32)*16 + ((m%128)/32)*4 + k%4,
 *                     KT = ceil(H/128) (the 128x4 tile layout of block-scaled tensor-core
 *                     GEMMs); padding bytes (m >= T, k >= H/32) are not written
 *   scale_mode        MHC_MX_SCALE_FLOOR or MHC_MX_SCALE_CEIL; E is clamped to [-127, 127],
 *                     and an all-zero block gets E = -127
 * Needs H % 32 == 0 (MHC_ERR_INVALID_ARG otherwise).  The ws (with the tile kernel beside it,
 * as AUTO splits a plain call), tile and small schedules quantize in their combine epilogue, or,
 * on ws and tile with layer_in_out given, in a second streaming pass over the bf16 layer input
 * (the same bits; cheaper there than the epilogue).  The split schedule always takes the second
 * pass; with layer_in_out NULL it first writes the bf16 layer input into the workspace, which
 * mhc_workspace_size reserves where AUTO can choose split (H > 7168, T < 448); a forced split
 * call elsewhere then returns MHC_ERR_WORKSPACE when the workspace is too small.  The bf16 output
 * and the mixes are bit-identical to mhc_shifted_post_pre's with the same schedule setting. */
MHC_API mhc_status mhc_shifted_post_pre_mxfp8(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
    float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, uint8_t *layer_in_fp8, uint8_t *layer_in_scales, int scale_mode,
    float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out, void *workspace,
    size_t workspace_bytes, void *stream);

/* The fused step (1)-(4) for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.
 * Some callers cannot call cudaMalloc where they run the op: a host framework
 * that owns all device memory and only hands out the tensors it manages, a
 * plugin that must not grow the process's memory footprint, or a hot path where
 * an allocation would synchronise the device.  Such a caller passes inputs and
 * outputs only (arguments and outputs as in mhc_shifted_post_pre, no workspace);
 * the scratch the kernels need is a 4 MiB static device array inside this
 * library, which every GPU that loads the library holds until the process exits.
 *   - Limit: mhc_workspace_size(T, H) must be at most 4 MiB (at H = 7168 up to
 *     1170 tokens); larger calls return MHC_ERR_INVALID_ARG and launch nothing,
 *     with the reason in mhc_last_error().
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; nothing in it needs clearing between calls, whatever
 *     their T and H.  Calls that overlap on the GPU (different streams without
 *     ordering) race on it.
 *   - A bounded device-side wait that gives up sets the array's status word:
 *     mhc_noalloc_check_status reads and clears it.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
MHC_API mhc_status mhc_shifted_post_pre_noalloc(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const float *bias, const float *mix_scales,
    const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
    float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *stream);

/* The allocation-free counterpart of mhc_check_status (the pages have no counterpart of it
 * either): synchronises `stream`, then reads the status word of the static scratch that
 * mhc_shifted_post_pre_noalloc uses on the current device.  MHC_ERR_DEVICE_TIMEOUT if a bounded
 * device-side wait of one of those calls gave up since the last check (the call's outputs are
 * then not to be trusted); it then zero-fills the scratch's control block, so later calls work
 * again.  MHC_ERR_CUDA if the stream reports an error, else MHC_OK.  Allocates nothing. */
MHC_API mhc_status mhc_noalloc_check_status(void *stream);

/* Step (1) alone: the mHC post ("[SM80] Backport mHC fused post + int8
 * all-reduce", "What this fixes").  Needs no workspace. */
MHC_API mhc_status mhc_post(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                    const float *prev_post_mix, const float *prev_comb_res_mix, int64_t T,
                    int64_t H, mhc_bf16 *residual_out, void *stream);

/* Step (1) with the layer output as int8 codes and one fp32 scale per token (the consumer of
 * an int8 all-reduce), plus the fused square sum: "[SM80] Backport mHC fused post + int8
 * all-reduce; fixes #28, #29", "What this fixes" (VLLM_MHC_AR_INT8, VLLM_MHC_POST_FUSE_SQRSUM).
 *   layer_out_q  [T,H] int8   codes q
 *   x_scales     [T]   fp32   the layer output is Y[t][h] = q[t][h] * x_scales[t]
 *   sqrsum_out   [T]   fp32   sum over i, h of R'[i][h]^2 of the bf16 residual_out (NULL: skip);
 *                             fp32 accumulation in a fixed order (deterministic)
 * Other arguments as in mhc_post (residual_out may equal residual).  Needs no workspace. */
MHC_API mhc_status mhc_post_int8(const mhc_bf16 *residual, const int8_t *layer_out_q, const float *x_scales,
                                 const float *prev_post_mix, const float *prev_comb_res_mix, int64_t T,
                                 int64_t H, mhc_bf16 *residual_out, float *sqrsum_out, void *stream);

/* mhc_post with the fused square sum (sqrsum_out [T] fp32, required; see mhc_post_int8).
 * residual_out is bit-identical to mhc_post's. */
MHC_API mhc_status mhc_post_sqrsum(const mhc_bf16 *residual, const mhc_bf16 *layer_out,
                                   const float *prev_post_mix, const float *prev_comb_res_mix, int64_t T,
                                   int64_t H, mhc_bf16 *residual_out, float *sqrsum_out, void *stream);

/* Steps (2)-(4) alone: the mHC pre, from streams that already went through the
 * post (`residual` here is R').  Same arguments and outputs as the fused call. */
MHC_API mhc_status mhc_pre(const mhc_bf16 *residual, const float *phi, const float *bias,
                   const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T,
                   int64_t H, float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                   float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *layer_in_out,
                   float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
                   void *workspace, size_t workspace_bytes, void *stream);

/* phi in the packed form the fused kernels read, made once per weight instead of on every call
 * ("[DSv4.1] Integrate Mega-mHC from DeepGEMM", "Paths on current main that still call DeepGEMM
 * on SM12x" item 1: the hc prenorm GEMM over the flattened hc_mult * hidden row, whose weight
 * phi is constant across calls).  The packed form holds phi^T split into a bf16 high part and a
 * bf16 remainder, in the fragment order of the tensor-core projection; a plain call rebuilds it
 * in its workspace each time (one extra launch).
 *   mhc_packed_phi_bytes(H)  bytes of the packed form (0 for an H the library does not take)
 *   mhc_pack_phi             writes it from phi [4H,24] fp32 into packed_phi (caller-owned device
 *                            memory of at least that many bytes, 16-byte aligned, not
 *                            overlapping phi) on `stream`; asynchronous, one launch
 * The _prepacked calls take the packed form next to phi (packed_phi must be mhc_pack_phi's output
 * for this phi and H, and must not be written while a call that reads it runs); everything else
 * is as in mhc_shifted_post_pre / mhc_pre, and the results are bit-identical to theirs.  Schedules
 * that read phi directly (small, split) ignore packed_phi. */
MHC_API size_t mhc_packed_phi_bytes(int64_t H);
MHC_API mhc_status mhc_pack_phi(const float *phi, int64_t H, void *packed_phi, size_t packed_bytes, void *stream);
MHC_API mhc_status mhc_shifted_post_pre_prepacked(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const void *packed_phi, const float *bias,
    const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps,
    float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out,
    void *workspace, size_t workspace_bytes, void *stream);
MHC_API mhc_status mhc_pre_prepacked(const mhc_bf16 *residual, const float *phi, const void *packed_phi,
                                     const float *bias, const float *mix_scales, const mhc_bf16 *rmsnorm_weight,
                                     int64_t T, int64_t H, float hc_norm_eps, float rmsnorm_eps,
                                     float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters,
                                     mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                                     float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                     void *stream);
/* mhc_shifted_post_pre_mxfp8 with the packed phi (arguments as there, packed_phi after phi);
 * bit-identical to it. */
MHC_API mhc_status mhc_shifted_post_pre_mxfp8_prepacked(
    const mhc_bf16 *residual, const mhc_bf16 *layer_out, const float *prev_post_mix,
    const float *prev_comb_res_mix, const float *phi, const void *packed_phi, const float *bias,
    const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T, int64_t H, float hc_norm_eps,
    float rmsnorm_eps, float hc_post_scale, float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
    mhc_bf16 *layer_in_out, uint8_t *layer_in_fp8, uint8_t *layer_in_scales, int scale_mode,
    float *pre_mix_out, float *post_mix_out, float *comb_res_mix_out, void *workspace,
    size_t workspace_bytes, void *stream);

/* The first layer's pre: the residual does not exist yet and the layer's (T, H) input x is
 * broadcast to the four streams ("[DSv4.1] Integrate Mega-mHC from DeepGEMM", "Paths on current
 * main that still call DeepGEMM on SM12x" item 1, mhc_pre_broadcast; the None pre mix of "Nit"
 * 6 only occurs here).  Writes residual_out [T,4,H] = four copies of x (what the next layer's
 * post reads) and steps (2)-(4) of that residual.  Two paths:
 *   - T > 32 with H % 64 == 0 (or MHC_SCHEDULE_BCAST forced): one kernel that works from x
 *     alone (phi summed over the four streams, x read twice, the second time from L2; 12H bytes
 *     of HBM traffic per token).  Its results match the oracle within the usual tolerances but
 *     are not bit-identical to mhc_pre's (another summation order);
 *   - otherwise (or with another schedule forced): the residual is written first and mhc_pre
 *     runs on it, bit-identical to mhc_pre on that residual.
 * x must not overlap any output. */
MHC_API mhc_status mhc_pre_broadcast(const mhc_bf16 *x, const float *phi, const float *bias,
                                     const float *mix_scales, const mhc_bf16 *rmsnorm_weight, int64_t T,
                                     int64_t H, float hc_norm_eps, float rmsnorm_eps, float hc_post_scale,
                                     float sinkhorn_eps, int sinkhorn_iters, mhc_bf16 *residual_out,
                                     mhc_bf16 *layer_in_out, float *pre_mix_out, float *post_mix_out,
                                     float *comb_res_mix_out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Forces a schedule for every following call of this process (a test hook; the
 * default is MHC_SCHEDULE_AUTO).  Returns MHC_ERR_INVALID_ARG for an unknown value. */
MHC_API mhc_status mhc_set_schedule(int schedule);

/* The schedule AUTO would pick for (T, H) on the current device. */
MHC_API int mhc_auto_schedule(int64_t T, int64_t H);

/* For a call of T tokens, hidden size H on the current device that AUTO runs on the ws schedule
 * (fused != 0: mhc_shifted_post_pre and its variants; fused == 0: mhc_pre): the number of
 * trailing tokens the token-tile kernel takes beside ws, on the SMs ws's 16-CTA clusters leave
 * idle (0 when ws runs alone or AUTO picks another schedule).  Returns -1 when T or H is negative
 * or no CUDA device is current.  Changes nothing; a planning query. */
MHC_API int64_t mhc_auto_side_tokens(int64_t T, int64_t H, int fused);

/* Synchronises `stream`, then reads the device status word kept in the
 * workspace: MHC_ERR_DEVICE_TIMEOUT if a bounded device-side wait gave up since
 * the last check, MHC_ERR_CUDA if the stream reports an error, else MHC_OK.
 * After a timeout it zero-fills the workspace's control block (the status word
 * and the grid-barrier words a wait that gave up may leave mid-count), so the
 * workspace is usable again. */
MHC_API mhc_status mhc_check_status(void *workspace, void *stream);

/* Number of kernels launched by the last call on this thread (0 if it failed
 * or launched nothing). */
MHC_API int mhc_last_launch_count(void);

/* Measurement hook: while set (non-NULL cudaEvent_t handles, passed as void*), every call
 * on this thread records `start` on its stream right before the launch of its main kernel
 * and `stop` right after it (for the ws schedule that excludes the phi packing launch), so
 * cudaEventElapsedTime(start, stop) is that kernel's duration.  Inside a stream capture the
 * records become event-record nodes of the graph.  NULL, NULL turns it off. */
MHC_API void mhc_set_main_kernel_events(void *start, void *stop);

/* Static description of a status code; never NULL. */
MHC_API const char *mhc_status_string(int status);

/* Detail of the last MHC_ERR_CUDA / MHC_ERR_INVALID_ARG on this thread (never NULL). */
MHC_API const char *mhc_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H */
