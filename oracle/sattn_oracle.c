/*
 * sattn_oracle.c -- CPU oracle of quantized exact attention with K smoothing.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, scalar, slow C that restates the method
 * step by step.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path never does.  It shares no code,
 * header or constant with the CUDA library.
 *
 * Method source: the "Experiment Log" page (vortex_exact_attention),
 *   entry "Phase 0 Import And Verification": the contract stages, in order:
 *     Q/K preparation, K smoothing, INT8 quantization, QK traversal,
 *     online softmax, FP8 V/P, two-level PV accumulation, final
 *     conversion, ragged-tail contract;
 *   entry "Phase 1 State-Ownership Decision": invariants kept by every
 *     architecture (strict tile order, exact FP8 score bytes, per-tile RO
 *     rescaling, two-level PV accumulation, final conversion);
 *   entry "Phase 2B Fixed Aligned Numerical Prototype": the checked
 *     intermediates (QK, m, d, FP8 probability, rescale, PV, FP32 RO,
 *     reciprocal, BF16 output).
 * The page names the stages but not their formulas.  Readings taken here
 * (each is listed with its reason in the design notes of the repository):
 *   - head dim 128; tensors [B, H, N, 128] contiguous; GQA query head h reads
 *     KV head h / (Hq / Hkv);
 *   - K smoothing subtracts the per-channel mean of K over the Nkv tokens of
 *     one (batch, KV head); the mean is summed in FP32 over 64-token chunks in
 *     ascending token order, chunk sums added in ascending chunk order, then
 *     divided by Nkv (IEEE round-to-nearest);  Q is not smoothed;
 *   - INT8 quantisation per block of 32 consecutive tokens (all 128 channels):
 *     s = amax / 127, code = clamp(rint(x / s), -127, 127), IEEE division,
 *     ties to even; amax = 0 gives s = 0 and codes 0; pad rows hold code 0;
 *   - V to FP8 E4M3 per channel over all tokens: s_v = amax / 448,
 *     code = E4M3(v / s_v) round-to-nearest-even with saturation to +-448;
 *   - score (log2 domain) s2 = float(acc) * ((s_q * s_k) * c0), acc the exact
 *     int32 dot product of the codes, c0 = sm_scale * log2(e) in FP32;
 *   - FP8 P: p8 = E4M3(exp2(s2 - m) * 448); the denominator d and the PV
 *     partials both take the FP8 values (code units), so the factor 448
 *     cancels in the final conversion;
 *   - the inner PV partial of one tile is an FP32 sum (an FP16 partial would
 *     overflow at these magnitudes);
 *   - final: r = 1 / d, out = bf16_rne((RO * r) * s_v[c]).
 * Build with -ffp-contract=off and without fast-math so that every FP32
 * operation rounds once, as written.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HEAD_DIM 128
#define QBLK 32          /* tokens per INT8 quantisation block */
#define MEAN_CHUNK 64    /* tokens per K-mean partial sum */
#define MAX_TILE 256     /* largest KV tile the oracle accepts */

/* ------------------------------------------------------------------------- */
/* storage formats                                                           */
/* ------------------------------------------------------------------------- */

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* FP32 -> BF16, round to nearest, ties to even, done on the bit pattern. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN stays a (quiet) NaN */
        return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* OCP 8-bit floating point, E4M3 ("FN": no infinities, S.1111.111 is NaN):
 * exponent bias 7, normal values (1 + m/8) * 2^(e-7), subnormals m * 2^-9,
 * largest finite 448. */
float oracle_e4m3_to_f32(uint8_t code)
{
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    const float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return s ? -v : v;
}

/* FP32 -> E4M3, round to nearest, ties to even, finite values saturate to
 * +-448 (the "satfinite" behaviour).  The sign of zero is kept. */
uint8_t oracle_f32_to_e4m3(float x)
{
    const uint8_t s = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return 0x7f;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return s | 0x7e;
    int e;
    frexp(a, &e);                      /* a = f * 2^e with 0.5 <= f < 1 */
    int ex = e - 1;                    /* floor(log2(a)) for a > 0 */
    if (ex < -6)
        ex = -6;                       /* subnormal range shares the 2^-9 step */
    const double step = ldexp(1.0, ex - 3);
    const double r = nearbyint(a / step) * step;   /* exact scaling; RNE */
    if (r == 0.0)
        return s;
    int e2;
    const double f2 = frexp(r, &e2);   /* r = f2 * 2^e2 */
    const int biased = e2 - 1 + 7;
    if (biased <= 0)
        return s | (uint8_t)(r / ldexp(1.0, -9));
    const int mant = (int)((f2 * 2.0 - 1.0) * 8.0);
    return s | (uint8_t)(biased << 3) | (uint8_t)mant;
}

/* exp2 of an FP32 value, correctly rounded to FP32 (round to nearest even).
 * The double-precision exp2 of the C library is within about one double ulp
 * of 2^x, so rounding it to FP32 gives the correctly rounded value unless 2^x
 * lies within a few double ulps of a point halfway between two FP32 values.
 * Those rare cases are decided again from exp2l (extended or quadruple
 * precision, depending on the platform).  2^x of an FP32 x that is not an
 * integer is irrational, so it never equals a halfway point. */
static float exp2_rn(float x)
{
    const double d = exp2((double)x);
    const float f = (float)d;
    if (!(d > 0.0) || isinf(d) || d < 0x1p-126)
        return f;
    /* distance from d to the nearest halfway point between FP32 neighbours */
    const double lo = (double)nextafterf(f, 0.0f), hi = (double)nextafterf(f, INFINITY);
    const double mid_lo = 0.5 * ((double)f + lo), mid_hi = 0.5 * ((double)f + hi);
    const double gap = fmin(fabs(d - mid_lo), fabs(d - mid_hi));
    if (gap > 0x1p-45 * d)
        return f;
    const long double e = exp2l((long double)x);
    return (float)e;
}

/* ------------------------------------------------------------------------- */
/* preparation: K smoothing, INT8 Q/K, FP8 V                                 */
/* ------------------------------------------------------------------------- */

/* Per-channel mean of one head's K rows, in the fixed order stated above. */
static void k_mean_head(const float *kf, int n, float *mean)
{
    for (int c = 0; c < HEAD_DIM; ++c) {
        float total = 0.0f;
        for (int t0 = 0; t0 < n; t0 += MEAN_CHUNK) {
            const int t1 = (t0 + MEAN_CHUNK < n) ? t0 + MEAN_CHUNK : n;
            float s = 0.0f;
            for (int t = t0; t < t1; ++t)
                s = s + kf[(size_t)t * HEAD_DIM + c];
            total = total + s;
        }
        mean[c] = total / (float)n;
    }
}

/* INT8 codes of one head, one scale per 32-token block; rows n .. npad-1 get 0. */
static void quant_int8_head(const float *x, int n, int npad, int8_t *codes, float *scales)
{
    for (int t0 = 0; t0 < npad; t0 += QBLK) {
        const int t1 = (t0 + QBLK < n) ? t0 + QBLK : n;
        float amax = 0.0f;
        for (int t = t0; t < t1; ++t)
            for (int c = 0; c < HEAD_DIM; ++c) {
                const float a = fabsf(x[(size_t)t * HEAD_DIM + c]);
                if (a > amax)
                    amax = a;
            }
        const float s = amax / 127.0f;
        scales[t0 / QBLK] = s;
        for (int t = t0; t < t0 + QBLK; ++t)
            for (int c = 0; c < HEAD_DIM; ++c) {
                int8_t code = 0;
                if (t < n && s > 0.0f) {
                    float r = rintf(x[(size_t)t * HEAD_DIM + c] / s);
                    if (r > 127.0f)
                        r = 127.0f;
                    if (r < -127.0f)
                        r = -127.0f;
                    code = (int8_t)r;
                }
                codes[(size_t)t * HEAD_DIM + c] = code;
            }
    }
}

static int pad_to(int n, int m) { return (n + m - 1) / m * m; }

/*
 * oracle_prepare: BF16 Q, K, V (bit patterns) -> codes and scales.
 *   q [B][Hq][Nq][128], k and v [B][Hkv][Nkv][128] (uint16 BF16 bits)
 *   q_codes [B][Hq][Nq32][128] int8, q_scales [B][Hq][Nq32/32] FP32
 *   k_codes [B][Hkv][Nkv32][128] int8, k_scales [B][Hkv][Nkv32/32] FP32
 *   k_mean [B][Hkv][128] FP32 (zeros when smooth == 0)
 *   v_codes [B][Hkv][Nkv][128] E4M3 bytes (token-major), v_scales [B][Hkv][128]
 * NkvX = N rounded up to a multiple of X.  Returns 0, or -1 on bad sizes.
 */
int oracle_prepare(int B, int Hq, int Hkv, int Nq, int Nkv, int smooth,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                   float *k_mean, uint8_t *v_codes, float *v_scales)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Nq < 1 || Nkv < 1)
        return -1;
    const int nq32 = pad_to(Nq, QBLK), nk32 = pad_to(Nkv, QBLK);
    const int nheads = B * Hq + B * Hkv;

#pragma omp parallel for schedule(dynamic, 1)
    for (int job = 0; job < nheads; ++job) {
        if (job < B * Hq) {                       /* one query head */
            const int bh = job;
            float *x = malloc((size_t)Nq * HEAD_DIM * sizeof *x);
            for (size_t e = 0; e < (size_t)Nq * HEAD_DIM; ++e)
                x[e] = oracle_bf16_to_f32(q[(size_t)bh * Nq * HEAD_DIM + e]);
            quant_int8_head(x, Nq, nq32, q_codes + (size_t)bh * nq32 * HEAD_DIM,
                            q_scales + (size_t)bh * (nq32 / QBLK));
            free(x);
        } else {                                  /* one KV head */
            const int bh = job - B * Hq;
            const uint16_t *kh = k + (size_t)bh * Nkv * HEAD_DIM;
            const uint16_t *vh = v + (size_t)bh * Nkv * HEAD_DIM;
            float *x = malloc((size_t)Nkv * HEAD_DIM * sizeof *x);
            float *mean = k_mean + (size_t)bh * HEAD_DIM;
            for (size_t e = 0; e < (size_t)Nkv * HEAD_DIM; ++e)
                x[e] = oracle_bf16_to_f32(kh[e]);
            if (smooth)
                k_mean_head(x, Nkv, mean);
            else
                for (int c = 0; c < HEAD_DIM; ++c)
                    mean[c] = 0.0f;
            for (int t = 0; t < Nkv; ++t)             /* K smoothing */
                for (int c = 0; c < HEAD_DIM; ++c)
                    x[(size_t)t * HEAD_DIM + c] = x[(size_t)t * HEAD_DIM + c] - mean[c];
            quant_int8_head(x, Nkv, nk32, k_codes + (size_t)bh * nk32 * HEAD_DIM,
                            k_scales + (size_t)bh * (nk32 / QBLK));
            /* V: per-channel absolute maximum, scale, E4M3 codes */
            float *sv = v_scales + (size_t)bh * HEAD_DIM;
            for (int c = 0; c < HEAD_DIM; ++c) {
                float amax = 0.0f;
                for (int t = 0; t < Nkv; ++t) {
                    const float a = fabsf(oracle_bf16_to_f32(vh[(size_t)t * HEAD_DIM + c]));
                    if (a > amax)
                        amax = a;
                }
                sv[c] = amax / 448.0f;
            }
            for (int t = 0; t < Nkv; ++t)
                for (int c = 0; c < HEAD_DIM; ++c) {
                    const size_t e = (size_t)t * HEAD_DIM + c;
                    const float vf = oracle_bf16_to_f32(vh[e]);
                    v_codes[(size_t)bh * Nkv * HEAD_DIM + e] =
                        (sv[c] > 0.0f) ? oracle_f32_to_e4m3(vf / sv[c]) : 0;
                }
            free(x);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* forward: the tiled recurrence, quantised (FP32) and exact (FP64) modes    */
/* ------------------------------------------------------------------------- */

typedef struct {
    int B, Hq, Hkv, Nq, Nkv, causal, tile;
    int Nq_pad, Nkv_pad, nbq, nbk;          /* padded token counts and block counts */
    /* quantised inputs */
    const int8_t *qc, *kc;
    const float *qs, *ks, *vs;
    const uint8_t *vc;                      /* token-major E4M3 */
    float c0;                               /* sm_scale * log2(e), FP32 */
    /* exact-mode inputs */
    const double *qx, *kx, *vx, *kmean;     /* kmean NULL: no smoothing */
    double scale_log2;                      /* sm_scale * log2(e), FP64 */
} ctx_t;

/* State of one row's recurrence after a chosen KV tile, and at the end. */
typedef struct {
    int tile, reached;
    double m, alpha, d, ro[HEAD_DIM];
    double d_final, rcp;
} row_rec_t;

static inline float score_q(const ctx_t *cx, int b, int h, int hk, int i, int j)
{
    const int8_t *qi = cx->qc + ((size_t)(b * cx->Hq + h) * cx->Nq_pad + i) * HEAD_DIM;
    const int8_t *kj = cx->kc + ((size_t)(b * cx->Hkv + hk) * cx->Nkv_pad + j) * HEAD_DIM;
    int32_t acc = 0;
    for (int c = 0; c < HEAD_DIM; ++c)
        acc += (int32_t)qi[c] * (int32_t)kj[c];
    const float sq = cx->qs[(size_t)(b * cx->Hq + h) * cx->nbq + i / QBLK];
    const float sk = cx->ks[(size_t)(b * cx->Hkv + hk) * cx->nbk + j / QBLK];
    const float sigma = (sq * sk) * cx->c0;
    return (float)acc * sigma;
}

/* FP8 P: the E4M3 byte of exp2(s2 - m) * 448, every step rounded to FP32:
 * dd = fl(s2 - m), p = fl(exp2(dd)) (correctly rounded), y = fl(p * 448). */
static inline uint8_t p8_of(float s2, float m)
{
    const float dd = s2 - m;
    const float p = exp2_rn(dd);
    return oracle_f32_to_e4m3(p * 448.0f);
}

static inline float prob_q(float p) { return oracle_e4m3_to_f32(oracle_f32_to_e4m3(p * 448.0f)); }

static inline float value_q(const ctx_t *cx, int b, int hk, int j, int c)
{
    return oracle_e4m3_to_f32(cx->vc[((size_t)(b * cx->Hkv + hk) * cx->Nkv + j) * HEAD_DIM + c]);
}

static inline float out_scale_q(const ctx_t *cx, int b, int hk, int c)
{
    return cx->vs[(size_t)(b * cx->Hkv + hk) * HEAD_DIM + c];
}

static inline double score_x(const ctx_t *cx, int b, int h, int hk, int i, int j)
{
    const double *qi = cx->qx + ((size_t)(b * cx->Hq + h) * cx->Nq + i) * HEAD_DIM;
    const double *kj = cx->kx + ((size_t)(b * cx->Hkv + hk) * cx->Nkv + j) * HEAD_DIM;
    const double *mu = cx->kmean ? cx->kmean + (size_t)(b * cx->Hkv + hk) * HEAD_DIM : NULL;
    double acc = 0.0;
    for (int c = 0; c < HEAD_DIM; ++c)
        acc += qi[c] * (mu ? kj[c] - mu[c] : kj[c]);
    return acc * cx->scale_log2;
}

static inline double value_x(const ctx_t *cx, int b, int hk, int j, int c)
{
    return cx->vx[((size_t)(b * cx->Hkv + hk) * cx->Nkv + j) * HEAD_DIM + c];
}

#define ROW_FN attend_row_quant
#define REAL float
#define EXP2(x) exp2_rn(x)
#define SCORE(cx, b, h, hk, i, j) score_q(cx, b, h, hk, i, j)
#define PROB(p) prob_q(p)
#define VALUE(cx, b, hk, j, c) value_q(cx, b, hk, j, c)
#define OUT_SCALE(cx, b, hk, c) out_scale_q(cx, b, hk, c)
#include "attend_row.inc"
#undef ROW_FN
#undef REAL
#undef EXP2
#undef SCORE
#undef PROB
#undef VALUE
#undef OUT_SCALE

#define ROW_FN attend_row_exact
#define REAL double
#define EXP2(x) exp2(x)
#define SCORE(cx, b, h, hk, i, j) score_x(cx, b, h, hk, i, j)
#define PROB(p) (p)
#define VALUE(cx, b, hk, j, c) value_x(cx, b, hk, j, c)
#define OUT_SCALE(cx, b, hk, c) 1.0
#include "attend_row.inc"

static int check_shape(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, int tile)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Nq < 1 || Nkv < 1)
        return -1;
    if (causal && Nq > Nkv)
        return -1;
    if (tile < 1 || tile > MAX_TILE)
        return -1;
    return 0;
}

static void setup_quant(ctx_t *cx, int B, int Hq, int Hkv, int Nq, int Nkv, int causal,
                        float sm_scale, int tile, const int8_t *q_codes, const float *q_scales,
                        const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                        const float *v_scales)
{
    memset(cx, 0, sizeof *cx);
    cx->B = B; cx->Hq = Hq; cx->Hkv = Hkv; cx->Nq = Nq; cx->Nkv = Nkv;
    cx->causal = causal; cx->tile = tile;
    cx->Nq_pad = pad_to(Nq, QBLK); cx->Nkv_pad = pad_to(Nkv, QBLK);
    cx->nbq = cx->Nq_pad / QBLK; cx->nbk = cx->Nkv_pad / QBLK;
    cx->qc = q_codes; cx->qs = q_scales; cx->kc = k_codes; cx->ks = k_scales;
    cx->vc = v_codes; cx->vs = v_scales;
    if (!(sm_scale > 0.0f))
        sm_scale = 1.0f / sqrtf((float)HEAD_DIM);
    cx->c0 = sm_scale * 1.44269504088896340736f;
}

/*
 * oracle_forward: quantised attention for every query row.
 *   codes and scales as written by oracle_prepare; sm_scale <= 0 means
 *   1/sqrt(128); tile = KV tile size (keys per tile).
 *   out_bf16 [B][Hq][Nq][128] (BF16 bits) and/or out_f32 (same shape); either
 *   may be NULL.  nthreads <= 0 uses the OpenMP default.
 */
int oracle_forward(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, float sm_scale, int tile,
                   const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                   const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                   uint16_t *out_bf16, float *out_f32, int nthreads)
{
    if (check_shape(B, Hq, Hkv, Nq, Nkv, causal, tile))
        return -1;
    ctx_t cx;
    setup_quant(&cx, B, Hq, Hkv, Nq, Nkv, causal, sm_scale, tile, q_codes, q_scales, k_codes,
                k_scales, v_codes, v_scales);
    const long nrows = (long)B * Hq * Nq;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 16)
    for (long row = 0; row < nrows; ++row) {
        const int i = (int)(row % Nq), bh = (int)(row / Nq);
        float o[HEAD_DIM];
        attend_row_quant(&cx, bh / Hq, bh % Hq, i, o, NULL);
        for (int c = 0; c < HEAD_DIM; ++c) {
            if (out_f32)
                out_f32[row * HEAD_DIM + c] = o[c];
            if (out_bf16)
                out_bf16[row * HEAD_DIM + c] = oracle_f32_to_bf16(o[c]);
        }
    }
    return 0;
}

/* oracle_first_tile: the checked intermediates of the first KV tile (entry
 * "Phase 2B Fixed Aligned Numerical Prototype": QK, m, FP8 probability, PV)
 * for the query rows q0 .. q0 + 127 of (batch b, query head h).  For row r
 * (query q0 + r; rows >= Nq stay zero) and key j < tile:
 *   acc[r][j]        the exact int32 dot product of the codes (0 for j >= Nkv),
 *                    masked or not
 *   p8[r][j]         the E4M3 byte of exp2(s2 - m) * 448, m the row's maximum
 *                    score over the tile's kept keys (0 for masked keys)
 *   part[r][c]       sum over j of p8_j * v8_j,c in ascending j (FP32), c < 128
 *   part[r][128]     sum over j of p8_j (the tile's contribution to d)
 * These are the first iteration of attend_row's loop (m = -inf before it, so
 * alpha = 0 and RO = part, d = part[128] after it); with Nkv <= tile they are
 * the whole recurrence. */
int oracle_first_tile(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, float sm_scale, int tile,
                      const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                      const float *k_scales, const uint8_t *v_codes, const float *v_scales, int b,
                      int h, int q0, int32_t *acc, uint8_t *p8, float *part)
{
    if (check_shape(B, Hq, Hkv, Nq, Nkv, causal, tile) || b < 0 || b >= B || h < 0 || h >= Hq ||
        q0 < 0 || q0 >= Nq)
        return -1;
    ctx_t cx;
    setup_quant(&cx, B, Hq, Hkv, Nq, Nkv, causal, sm_scale, tile, q_codes, q_scales, k_codes,
                k_scales, v_codes, v_scales);
    const int hk = h / (Hq / Hkv);
    const int n = Nkv < tile ? Nkv : tile;
    memset(acc, 0, sizeof(int32_t) * 128 * (size_t)tile);
    memset(p8, 0, (size_t)128 * tile);
    memset(part, 0, sizeof(float) * 128 * (HEAD_DIM + 1));
    for (int r = 0; r < 128 && q0 + r < Nq; ++r) {
        const int i = q0 + r;
        int last = Nkv - 1;
        if (causal && i + (Nkv - Nq) < last)
            last = i + (Nkv - Nq);
        const int8_t *qi = cx.qc + ((size_t)(b * Hq + h) * cx.Nq_pad + i) * HEAD_DIM;
        float m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            const int8_t *kj = cx.kc + ((size_t)(b * Hkv + hk) * cx.Nkv_pad + j) * HEAD_DIM;
            int32_t a = 0;
            for (int c = 0; c < HEAD_DIM; ++c)
                a += (int32_t)qi[c] * (int32_t)kj[c];
            acc[(size_t)r * tile + j] = a;
            if (j <= last) {
                const float s2 = score_q(&cx, b, h, hk, i, j);
                if (s2 > m)
                    m = s2;
            }
        }
        float w[MAX_TILE], tsum = 0;
        for (int j = 0; j < n; ++j) {
            w[j] = 0;
            if (j <= last) {
                const uint8_t code = p8_of(score_q(&cx, b, h, hk, i, j), m);
                p8[(size_t)r * tile + j] = code;
                w[j] = oracle_e4m3_to_f32(code);
            }
        }
        for (int j = 0; j < n; ++j)
            tsum = tsum + w[j];
        for (int c = 0; c < HEAD_DIM; ++c) {
            float s = 0;
            for (int j = 0; j < n; ++j)
                s = s + w[j] * value_q(&cx, b, hk, j, c);
            part[(size_t)r * (HEAD_DIM + 1) + c] = s;
        }
        part[(size_t)r * (HEAD_DIM + 1) + HEAD_DIM] = tsum;
    }
    return 0;
}

/* oracle_forward_rows: as oracle_forward, for the listed rows only.
 * rows[r] = (b * Hq + h) * Nq + i; outputs are [nrows][128]. */
int oracle_forward_rows(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, float sm_scale,
                        int tile, const int8_t *q_codes, const float *q_scales,
                        const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                        const float *v_scales, long nrows, const int64_t *rows,
                        uint16_t *out_bf16, float *out_f32, int nthreads)
{
    if (check_shape(B, Hq, Hkv, Nq, Nkv, causal, tile))
        return -1;
    ctx_t cx;
    setup_quant(&cx, B, Hq, Hkv, Nq, Nkv, causal, sm_scale, tile, q_codes, q_scales, k_codes,
                k_scales, v_codes, v_scales);
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= (int64_t)B * Hq * Nq)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < nrows; ++r) {
        const int64_t row = rows[r];
        const int i = (int)(row % Nq), bh = (int)(row / Nq);
        float o[HEAD_DIM];
        attend_row_quant(&cx, bh / Hq, bh % Hq, i, o, NULL);
        for (int c = 0; c < HEAD_DIM; ++c) {
            if (out_f32)
                out_f32[r * HEAD_DIM + c] = o[c];
            if (out_bf16)
                out_bf16[r * HEAD_DIM + c] = oracle_f32_to_bf16(o[c]);
        }
    }
    return 0;
}

/*
 * oracle_forward_exact: the same tiled recurrence in FP64 with every
 * quantiser bypassed (scores from the real dot product, weights exp2 values,
 * values V itself, no FP8 / INT8 / BF16 rounding).  smooth != 0 subtracts the
 * exact per-channel K mean first.  q [B][Hq][Nq][128], k, v [B][Hkv][Nkv][128],
 * out [B][Hq][Nq][128].
 */
int oracle_forward_exact(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, double sm_scale,
                         int tile, const double *q, const double *k, const double *v, int smooth,
                         double *out)
{
    if (check_shape(B, Hq, Hkv, Nq, Nkv, causal, tile))
        return -1;
    ctx_t cx;
    memset(&cx, 0, sizeof cx);
    cx.B = B; cx.Hq = Hq; cx.Hkv = Hkv; cx.Nq = Nq; cx.Nkv = Nkv;
    cx.causal = causal; cx.tile = tile;
    cx.qx = q; cx.kx = k; cx.vx = v;
    if (!(sm_scale > 0.0))
        sm_scale = 1.0 / sqrt((double)HEAD_DIM);
    cx.scale_log2 = sm_scale * 1.44269504088896340736;
    double *mean = NULL;
    if (smooth) {
        mean = calloc((size_t)B * Hkv * HEAD_DIM, sizeof *mean);
        for (int bh = 0; bh < B * Hkv; ++bh)
            for (int c = 0; c < HEAD_DIM; ++c) {
                double s = 0.0;
                for (int t = 0; t < Nkv; ++t)
                    s += k[((size_t)bh * Nkv + t) * HEAD_DIM + c];
                mean[(size_t)bh * HEAD_DIM + c] = s / Nkv;
            }
        cx.kmean = mean;
    }
    const long nrows = (long)B * Hq * Nq;
#pragma omp parallel for schedule(dynamic, 16)
    for (long row = 0; row < nrows; ++row) {
        const int i = (int)(row % Nq), bh = (int)(row / Nq);
        attend_row_exact(&cx, bh / Hq, bh % Hq, i, out + row * HEAD_DIM, NULL);
    }
    free(mean);
    return 0;
}

/*
 * oracle_p8_codes: the FP8 P byte of n (acc, sig, m) triples, as the forward
 * computes it (entry "Phase 1 State-Ownership Decision": exact FP8 score
 * bytes): s2 = fl(acc * sig), then E4M3(fl(fl(exp2(fl(s2 - m))) * 448)) with
 * a correctly rounded exp2.  acc holds exact integers (as FP32 values), sig
 * the block scale product, m the running maximum after the tile.
 */
int oracle_p8_codes(long n, const float *acc, const float *sig, const float *m, uint8_t *out)
{
    if (n < 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (long e = 0; e < n; ++e)
        out[e] = p8_of(acc[e] * sig[e], m[e]);
    return 0;
}

/*
 * oracle_tile_state: the checked intermediates after KV tile `tile` (entry
 * "Phase 2B Fixed Aligned Numerical Prototype": m, rescale, d, FP32 RO,
 * reciprocal) for the query rows q0 .. q0 + 127 of (batch b, query head h),
 * from the same per-row recurrence as oracle_forward.  Per row r (query
 * q0 + r; rows >= Nq stay zero):
 *   st[r][0] = m after the tile, st[r][1] = the tile's alpha,
 *   st[r][2] = d after the tile, st[r][3] = d after the last tile,
 *   st[r][4] = the final reciprocal 1 / d, st[r][5] = 1 if the row visited
 *              the tile (rows whose kept keys end earlier do not)
 *   ro[r][c] = RO after the tile.
 */
int oracle_tile_state(int B, int Hq, int Hkv, int Nq, int Nkv, int causal, float sm_scale, int tile,
                      const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                      const float *k_scales, const uint8_t *v_codes, const float *v_scales, int b,
                      int h, int q0, int which, double *st, double *ro)
{
    if (check_shape(B, Hq, Hkv, Nq, Nkv, causal, tile) || b < 0 || b >= B || h < 0 || h >= Hq ||
        q0 < 0 || q0 >= Nq || which < 0)
        return -1;
    ctx_t cx;
    setup_quant(&cx, B, Hq, Hkv, Nq, Nkv, causal, sm_scale, tile, q_codes, q_scales, k_codes,
                k_scales, v_codes, v_scales);
    memset(st, 0, sizeof(double) * 128 * 6);
    memset(ro, 0, sizeof(double) * 128 * HEAD_DIM);
    for (int r = 0; r < 128 && q0 + r < Nq; ++r) {
        row_rec_t rec;
        memset(&rec, 0, sizeof rec);
        rec.tile = which;
        float o[HEAD_DIM];
        attend_row_quant(&cx, b, h, q0 + r, o, &rec);
        st[r * 6 + 0] = rec.m;
        st[r * 6 + 1] = rec.alpha;
        st[r * 6 + 2] = rec.d;
        st[r * 6 + 3] = rec.d_final;
        st[r * 6 + 4] = rec.rcp;
        st[r * 6 + 5] = rec.reached;
        for (int c = 0; c < HEAD_DIM; ++c)
            ro[(size_t)r * HEAD_DIM + c] = rec.ro[c];
    }
    return 0;
}

/* oracle_exp2_rn: FP32 2^x correctly rounded (the exp2 of the P step), for
 * n values. */
int oracle_exp2_rn(long n, const float *x, float *out)
{
    if (n < 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (long e = 0; e < n; ++e)
        out[e] = exp2_rn(x[e]);
    return 0;
}
