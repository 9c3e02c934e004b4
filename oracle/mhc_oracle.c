/*
 * CPU oracle for the fused mHC (manifold-constrained hyper-connection)
 * shifted post+pre step.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg call it; the library never does.
 *
 * Plain, slow, obviously correct: every step is computed in double precision
 * (fp64) with straightforward loops, token by token, in the order the
 * definition states.  It shares no code with the CUDA path.  Tokens are
 * independent, so a driver splits them over POSIX threads; the per-token
 * arithmetic does not depend on the split.
 *
 * Sources.  The pages name the pieces but never print the equations:
 *   [P1] "[SM80] Backport mHC fused post + int8 all-reduce; fixes #28, #29"
 *        section "What this fixes": the mHC post kernel and its fused square
 *        sum (VLLM_MHC_POST_FUSE_SQRSUM).
 *   [P2] "[DSv4.1] Integrate Mega-mHC from DeepGEMM": the fused post+pre op
 *        (mhc_shifted_post_pre / mega_mhc), its scalars hc_norm_eps,
 *        rmsnorm_eps, hc_post_scale, sinkhorn_eps and mix_scales, and the
 *        renamed comb_res_mix ("Style findings", Major 1 and Minor 3); the
 *        hc prenorm GEMM over the flattened hc_mult*hidden row ("Paths on
 *        current main that still call DeepGEMM on SM12x", item 1).
 *   [P3] "[DSV4.1] Four BS=1 critical-path fixes for DSpark decode": the mHC
 *        statistics and Sinkhorn ("Measured and deliberately left out") and
 *        the mHC combine+RMSNorm ("What changed", item 3).
 * The equations follow the workload definition of the op, steps (1)-(4):
 *   (1) post:    R'[i] = sum_j comb[j][i] * R[j] + post[i] * Y
 *   (2) RMS:     r = 1/sqrt(mean over 4H of R'^2 + hc_norm_eps)
 *                z = r * (flat(R') @ phi)                       (24 logits)
 *   (3) heads:   pre  = sigmoid(a_pre  * z[0:4]  + b[0:4])
 *                post = hc_post_scale * sigmoid(a_post * z[4:8] + b[4:8])
 *                res  = Sinkhorn(exp(a_res * z[8:24] + b[8:24]) as 4x4,
 *                                sinkhorn_iters iterations, sinkhorn_eps)
 *   (4) combine: X = sum_i pre[i] * R'[i];  out = X / sqrt(mean X^2 + rmsnorm_eps) * gamma
 *
 * Readings where the definition is silent (each is also listed with the design notes):
 *   - R' is rounded to bf16 (round to nearest even) and steps (2)-(4) consume
 *     the rounded values, so the fused op equals post followed by pre.
 *   - the 16 residual-mix logits are reshaped row-major: M[a][c] = z[8+4a+c].
 *   - one Sinkhorn iteration = divide every row by (row sum + eps), then every
 *     column by (column sum + eps); no max-subtraction before exp.
 *   - X is kept unrounded (fp64 here) until the final bf16 rounding of out.
 *   - pre is a plain sigmoid (no scale, no additive eps).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HC 4
#define NMIX 24

/* ---- bfloat16 <-> double (IEEE binary16-brain: 1 sign, 8 exponent, 7 mantissa bits) ---- */

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bfloat16, ties to even.  Works on the value
 * directly: the quantum of the target binade is 2^(e-8) for |x| in
 * [2^(e-1), 2^e), and 2^-133 below the smallest normal 2^-126. */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                        /* a = m * 2^e, m in [0.5, 1) */
    double quantum = (e - 1 < -126) ? ldexp(1.0, -133) : ldexp(1.0, e - 8);
    double q = a / quantum;              /* exact: division by a power of two */
    double r = floor(q);
    double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = r * quantum;
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (v > ldexp(255.0, 120)) return sign | 0x7F80;
    float f = (float)v;                  /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---- step (3), residual mix: Sinkhorn normalisation of a positive 4x4 matrix ---- */

void oracle_sinkhorn(double *M /* [4][4] row-major, in/out */, int iters, double eps)
{
    for (int it = 0; it < iters; ++it) {
        for (int a = 0; a < HC; ++a) {
            double s = 0.0;
            for (int c = 0; c < HC; ++c) s += M[a * HC + c];
            for (int c = 0; c < HC; ++c) M[a * HC + c] /= (s + eps);
        }
        for (int c = 0; c < HC; ++c) {
            double s = 0.0;
            for (int a = 0; a < HC; ++a) s += M[a * HC + c];
            for (int a = 0; a < HC; ++a) M[a * HC + c] /= (s + eps);
        }
    }
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ---- step (1) for one token: R'[i][h] = sum_j comb[j][i] R[j][h] + post[i] Y[h], to bf16 ---- */

static void post_token(const uint16_t *R, const uint16_t *Y, const float *post,
                       const float *comb, int64_t H, uint16_t *Rout)
{
    for (int i = 0; i < HC; ++i) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = (double)post[i] * oracle_bf16_to_double(Y[h]);
            for (int j = 0; j < HC; ++j)
                acc += (double)comb[j * HC + i] * oracle_bf16_to_double(R[j * H + h]);
            Rout[i * H + h] = oracle_double_to_bf16(acc);
        }
    }
}

/* ---- steps (2)-(4) for one token, from the (bf16) post-updated streams Rp ---- */

typedef struct {
    const float *phi, *bias, *mix_scales;
    const uint16_t *gamma;
    int64_t H;
    double hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps;
    int sinkhorn_iters;
} pre_params;

static void pre_token(const pre_params *p, const uint16_t *Rp, uint16_t *Xout,
                      double *pre, double *post, double *res,
                      double *z_dbg, double *r_dbg, double *rstd_dbg)
{
    const int64_t H = p->H, K = HC * H;

    /* (2) square sum and RMS over all 4H entries of the flattened row */
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double v = oracle_bf16_to_double(Rp[k]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)K + p->hc_norm_eps);

    /* (2) projection of the flattened row onto the 24 columns of phi, scaled by r */
    double z[NMIX];
    for (int n = 0; n < NMIX; ++n) z[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double v = oracle_bf16_to_double(Rp[k]);
        for (int n = 0; n < NMIX; ++n) z[n] += v * (double)p->phi[k * NMIX + n];
    }
    for (int n = 0; n < NMIX; ++n) z[n] *= r;

    /* (3) mix heads */
    const double a_pre = p->mix_scales[0], a_post = p->mix_scales[1], a_res = p->mix_scales[2];
    for (int i = 0; i < HC; ++i) {
        pre[i] = sigmoid(a_pre * z[i] + (double)p->bias[i]);
        post[i] = p->hc_post_scale * sigmoid(a_post * z[HC + i] + (double)p->bias[HC + i]);
    }
    double M[HC * HC];
    for (int e = 0; e < HC * HC; ++e)
        M[e] = exp(a_res * z[2 * HC + e] + (double)p->bias[2 * HC + e]);
    oracle_sinkhorn(M, p->sinkhorn_iters, p->sinkhorn_eps);
    for (int e = 0; e < HC * HC; ++e) res[e] = M[e];

    /* (4) combine the streams with pre, then RMSNorm with weight gamma */
    double *X = (double *)malloc(sizeof(double) * (size_t)H);
    double sx = 0.0;
    for (int64_t h = 0; h < H; ++h) {
        double x = 0.0;
        for (int i = 0; i < HC; ++i) x += pre[i] * oracle_bf16_to_double(Rp[i * H + h]);
        X[h] = x;
        sx += x * x;
    }
    double rstd = 1.0 / sqrt(sx / (double)H + p->rmsnorm_eps);
    for (int64_t h = 0; h < H; ++h)
        Xout[h] = oracle_double_to_bf16(X[h] * rstd * oracle_bf16_to_double(p->gamma[h]));
    free(X);

    if (z_dbg) for (int n = 0; n < NMIX; ++n) z_dbg[n] = z[n];
    if (r_dbg) *r_dbg = r;
    if (rstd_dbg) *rstd_dbg = rstd;
}

/* ---- drivers: split tokens over threads ---- */

typedef struct {
    int mode; /* 0 = post only, 1 = pre only, 2 = post then pre */
    const uint16_t *R, *Y;
    const float *prev_post, *prev_comb;
    pre_params pp;
    uint16_t *Rout, *Xout;
    double *pre, *post, *res, *z, *r, *rstd;
    int64_t t0, t1;
} job;

static void *run_job(void *arg)
{
    job *j = (job *)arg;
    const int64_t H = j->pp.H;
    uint16_t *tmp = NULL;
    if (j->mode == 2) tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(HC * H));
    for (int64_t t = j->t0; t < j->t1; ++t) {
        const uint16_t *Rp = j->R + t * HC * H;
        if (j->mode != 1) {
            uint16_t *dst = j->Rout ? j->Rout + t * HC * H : tmp;
            post_token(j->R + t * HC * H, j->Y + t * H, j->prev_post + t * HC,
                       j->prev_comb + t * HC * HC, H, dst);
            Rp = dst;
        }
        if (j->mode != 0)
            pre_token(&j->pp, Rp, j->Xout + t * H, j->pre + t * HC, j->post + t * HC,
                      j->res + t * HC * HC, j->z ? j->z + t * NMIX : NULL,
                      j->r ? j->r + t : NULL, j->rstd ? j->rstd + t : NULL);
    }
    free(tmp);
    return NULL;
}

static int run(job proto, int64_t T, int nthreads)
{
    if (T < 0 || proto.pp.H < 1) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = (int)(T > 0 ? T : 1);
    job *jobs = (job *)calloc((size_t)nthreads, sizeof(job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = proto;
        jobs[w].t0 = T * w / nthreads;
        jobs[w].t1 = T * (w + 1) / nthreads;
    }
    char *joined = (char *)calloc((size_t)nthreads, 1);
    for (int w = 1; w < nthreads; ++w) {
        if (pthread_create(&th[w], NULL, run_job, &jobs[w]) != 0) {
            run_job(&jobs[w]); /* could not start a thread: do its share here */
            joined[w] = 1;
        }
    }
    run_job(&jobs[0]);
    for (int w = 1; w < nthreads; ++w)
        if (!joined[w]) pthread_join(th[w], NULL);
    free(joined);
    free(jobs);
    free(th);
    return 0;
}

/* Step (1) alone (the mHC post).  R [T,4,H], Y [T,H], prev_post [T,4],
 * prev_comb [T,4,4] -> Rout [T,4,H] (bf16). */
int oracle_post(const uint16_t *R, const uint16_t *Y, const float *prev_post,
                const float *prev_comb, int64_t T, int64_t H, uint16_t *Rout, int nthreads)
{
    job j;
    memset(&j, 0, sizeof j);
    j.mode = 0;
    j.R = R; j.Y = Y; j.prev_post = prev_post; j.prev_comb = prev_comb;
    j.pp.H = H;
    j.Rout = Rout;
    return run(j, T, nthreads);
}

/* Steps (2)-(4) (the mHC pre) from already post-updated bf16 streams Rp [T,4,H].
 * Outputs: Xout [T,H] bf16, pre [T,4], post [T,4], res [T,4,4] in fp64.
 * z [T,24], r [T], rstd [T] are optional (NULL to skip) intermediate values. */
int oracle_pre(const uint16_t *Rp, const float *phi, const float *bias, const float *mix_scales,
               const uint16_t *gamma, int64_t T, int64_t H, double hc_norm_eps,
               double rmsnorm_eps, double hc_post_scale, double sinkhorn_eps, int sinkhorn_iters,
               uint16_t *Xout, double *pre, double *post, double *res,
               double *z, double *r, double *rstd, int nthreads)
{
    job j;
    memset(&j, 0, sizeof j);
    j.mode = 1;
    j.R = Rp;
    j.pp = (pre_params){phi, bias, mix_scales, gamma, H, hc_norm_eps, rmsnorm_eps,
                        hc_post_scale, sinkhorn_eps, sinkhorn_iters};
    j.Xout = Xout; j.pre = pre; j.post = post; j.res = res; j.z = z; j.r = r; j.rstd = rstd;
    return run(j, T, nthreads);
}

/* The whole step: post, then pre on the bf16 result.  Rout may be NULL when
 * the updated residual is not wanted (a per-thread scratch row is used). */
int oracle_shifted_post_pre(const uint16_t *R, const uint16_t *Y, const float *prev_post,
                            const float *prev_comb, const float *phi, const float *bias,
                            const float *mix_scales, const uint16_t *gamma, int64_t T, int64_t H,
                            double hc_norm_eps, double rmsnorm_eps, double hc_post_scale,
                            double sinkhorn_eps, int sinkhorn_iters, uint16_t *Rout,
                            uint16_t *Xout, double *pre, double *post, double *res,
                            double *z, double *r, double *rstd, int nthreads)
{
    job j;
    memset(&j, 0, sizeof j);
    j.mode = 2;
    j.R = R; j.Y = Y; j.prev_post = prev_post; j.prev_comb = prev_comb;
    j.pp = (pre_params){phi, bias, mix_scales, gamma, H, hc_norm_eps, rmsnorm_eps,
                        hc_post_scale, sinkhorn_eps, sinkhorn_iters};
    j.Rout = Rout; j.Xout = Xout; j.pre = pre; j.post = post; j.res = res;
    j.z = z; j.r = r; j.rstd = rstd;
    return run(j, T, nthreads);
}

/* ---- MXFP8 quantize of the layer input --------------------------------------------------
 * [P3] "What changed" item 3: the mHC combine+RMSNorm output, written in bf16, was re-read by a
 * separate MXFP8 quantize; the epilogue emits the quantized form directly.  "Correctness": the
 * epilogue's bf16 output, FP8 values and swizzled UE8M0 scale block equal those of the bf16
 * output followed by the separate quantize.  So the quantize consumes the bf16-rounded layer
 * input, 32 consecutive hidden values of one token per block.
 * The pages give no formula.  Readings (listed with the design notes):
 *   - element format E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *     infinities; largest finite 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals
 *     k/8 * 2^-6), conversion by round to nearest even, finite values beyond 448 saturate;
 *   - block scale 2^E stored as the byte E + 127 (UE8M0), with E from the block's largest
 *     magnitude amax by one of two rules: mode 0 E = floor(log2 amax) - 8 (the largest
 *     element lands in [256, 512) and may saturate); mode 1 the smallest E with
 *     amax <= 448 * 2^E (never saturates).  amax == 0 gives E = -127; E is clamped to
 *     [-127, 127];
 *   - element = E4M3(x / 2^E), the division exact;
 *   - scale bytes in the 128 x 4 tile layout: token m, block k at
 *     ((m / 128) * KT + k / 4) * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4 + k % 4,
 *     KT = ceil(H / 128); rows padded to a multiple of 128, blocks to a multiple of 4. */

uint8_t oracle_e4m3_encode(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t s = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a >= 448.0) return s | 0x7E;             /* largest finite, also the saturation value */
    if (a == 0.0) return s;
    int e;
    frexp(a, &e);                                /* a in [2^(e-1), 2^e) */
    int be = e - 1 < -6 ? -6 : e - 1;            /* binade exponent; subnormals share 2^-6's quantum */
    double quantum = ldexp(1.0, be - 3);
    double q = a / quantum;                      /* exact */
    double r = floor(q), frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double val = r * quantum;                    /* <= 448: a < 448 rounds to at most 448 */
    if (val == 0.0) return s;
    int ve;
    frexp(val, &ve);
    int vb = ve - 1;
    if (vb < -6) return s | (uint8_t)(val / ldexp(1.0, -9));      /* subnormal: k * 2^-9 */
    int mant = (int)((val / ldexp(1.0, vb) - 1.0) * 8.0);
    return s | (uint8_t)(((vb + 7) << 3) | mant);
}

double oracle_e4m3_decode(uint8_t b)
{
    double sign = (b & 0x80) ? -1.0 : 1.0;
    int ef = (b >> 3) & 0xF, m = b & 7;
    if (ef == 0xF && m == 7) return NAN;
    if (ef == 0) return sign * ldexp((double)m, -9);
    return sign * ldexp(1.0 + m / 8.0, ef - 7);
}

int oracle_mx_scale_exp(double amax, int mode)
{
    if (!(amax > 0.0)) return -127;
    int e;
    double m = frexp(amax, &e);                  /* amax = (2m) * 2^(e-1), 2m in [1, 2) */
    int fl = e - 1;
    int E = (mode == 0) ? fl - 8 : (2.0 * m <= 1.75 ? fl - 8 : fl - 7);
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    return E;
}

int64_t oracle_mx_scale_offset(int64_t m, int64_t k, int64_t H)
{
    int64_t kt = (H / 32 + 3) / 4;
    return ((m / 128) * kt + k / 4) * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4 + k % 4;
}

int oracle_mxfp8_quantize(const uint16_t *X /* [T][H] bf16 */, int64_t T, int64_t H, int mode,
                          uint8_t *q /* [T][H] */, uint8_t *scales /* tile layout */)
{
    if (H % 32 != 0 || (mode != 0 && mode != 1)) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < H / 32; ++k) {
            const uint16_t *x = X + t * H + k * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(oracle_bf16_to_double(x[i]));
                if (a > amax) amax = a;
            }
            int E = oracle_mx_scale_exp(amax, mode);
            scales[oracle_mx_scale_offset(t, k, H)] = (uint8_t)(E + 127);
            for (int i = 0; i < 32; ++i)
                q[t * H + k * 32 + i] = oracle_e4m3_encode(ldexp(oracle_bf16_to_double(x[i]), -E));
        }
    return 0;
}

/* ---- the mHC post with an int8 layer output and its fused square sum -----------------------
 * [P1] "What this fixes": the int8 TileLang post kernels that consume the int8 all-reduced
 * attention output together with its x_scales (VLLM_MHC_AR_INT8), and the post kernel's fused
 * square sum (VLLM_MHC_POST_FUSE_SQRSUM).  The page gives no formula.  Readings (listed with the
 * design notes): Y[t][h] = q[t][h] * x_scale[t] (one fp32 scale per token, exact in fp64 here),
 * consumed in the post exactly as the bf16 Y is; the square sum of token t is
 * sum over i, h of R'[i][h]^2 over the bf16-rounded R' (the value step (2) takes its mean of). */

static void post_token_y(const uint16_t *R, const double *y, const float *post, const float *comb,
                         int64_t H, uint16_t *Rout, double *sqrsum)
{
    double ss = 0.0;
    for (int i = 0; i < HC; ++i) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = (double)post[i] * y[h];
            for (int j = 0; j < HC; ++j)
                acc += (double)comb[j * HC + i] * oracle_bf16_to_double(R[j * H + h]);
            Rout[i * H + h] = oracle_double_to_bf16(acc);
            double r = oracle_bf16_to_double(Rout[i * H + h]);
            ss += r * r;
        }
    }
    if (sqrsum) *sqrsum = ss;
}

/* Yq [T][H] int8 (or Y [T][H] bf16 when Yq is NULL), x_scales [T] -> Rout [T,4,H] bf16,
 * sqrsum [T] (NULL to skip). */
int oracle_post_ex(const uint16_t *R, const uint16_t *Y, const int8_t *Yq, const float *x_scales,
                   const float *prev_post, const float *prev_comb, int64_t T, int64_t H,
                   uint16_t *Rout, double *sqrsum)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    if (!y) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h)
            y[h] = Yq ? (double)Yq[t * H + h] * (double)x_scales[t] : oracle_bf16_to_double(Y[t * H + h]);
        post_token_y(R + t * HC * H, y, prev_post + t * HC, prev_comb + t * HC * HC, H, Rout + t * HC * H,
                     sqrsum ? sqrsum + t : NULL);
    }
    free(y);
    return 0;
}
