/*
 * CSA2 decode hot path: CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no code with the CUDA path.
 *
 * Plain, slow, scalar C11.  Build with -O2 -ffp-contract=off (no contraction
 * of a*b+c into an FMA unless written as fmaf).  Each function names the
 * passage it follows.  Loops over independent units (rows, positions,
 * heads) may be spread over OpenMP threads (orc_set_threads); no unit's
 * arithmetic depends on how they are spread, so results are identical for
 * every thread count.  Sources (web pages about DeepSeek V4.1 Flash):
 *   [HC]   Helmcode, "DeepSeek V4.1 Flash" architecture explainer
 *          (sections "03 · CSA2", "04 · FP4", "07 · compute, memory, bill")
 *   [LB]   Louis Bouchard, "DeepSeek V4.1 Flash: KV cache and writing benchmark"
 *          (sections "What actually changed over V4 Flash", "Share the cache
 *          and the search work")
 *   [MO]   0x0moeen, "DeepSeek V4.1 Flash KV cache" (section "Then every layer
 *          stops asking the same question")
 * The pages name the formats and modes but give no arithmetic; where they are
 * silent the reading taken is stated beside the code.
 *
 * Codec definitions beyond the pages' format names come from the public OCP
 * formats: E2M1 = 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, values
 * {0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3 ("FN") = 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN, max 448.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads for the loops over independent units (1 = single-threaded). */
void orc_set_threads(int32_t n) { omp_set_num_threads(n > 0 ? n : 1); }
int32_t orc_get_threads(void) { return omp_get_max_threads(); }

/* ------------------------------------------------------------------------ */
/* E2M1 (FP4) -- [HC] "04 · FP4": "E2M1 with an E4M3 scale for every 16      */
/* channels"; [MO] same format.                                              */
/* ------------------------------------------------------------------------ */

static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_e2m1_decode(uint32_t code)
{
    float m = E2M1_MAG[code & 7u];
    return (code & 8u) ? -m : m;
}

/* Nearest grid magnitude to |v|; at an exact midpoint the code with an even
 * mantissa bit (even code) wins (round-half-to-even, the IEEE default the pages
 * do not state); |v| >= 6 gives 6 (saturate to the largest finite value).
 * Sign bit = sign bit of v, also when the magnitude rounds to 0. */
uint32_t orc_e2m1_encode(float v)
{
    float a = fabsf(v);
    uint32_t best = 0;
    double best_d = (double)a;
    for (uint32_t c = 1; c < 8; ++c) {
        double d = fabs((double)a - (double)E2M1_MAG[c]);
        if (d < best_d || (d == best_d && (c % 2u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    if (!(a < 6.0f)) best = 7;
    return (signbit(v) ? 8u : 0u) | best;
}

/* ------------------------------------------------------------------------ */
/* E4M3 (FP8)                                                               */
/* ------------------------------------------------------------------------ */

float orc_e4m3_decode(uint32_t code)
{
    uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u) return NAN;
    float mag = (e == 0u) ? ldexpf((float)m, -9) : ldexpf((float)(8u + m), (int)e - 10);
    return s ? -mag : mag;
}

/* Nearest of the 127 non-negative finite magnitudes; midpoint -> even code;
 * beyond 448 -> 448 (saturating). Sign bit = sign bit of v. */
uint32_t orc_e4m3_encode(float v)
{
    float a = fabsf(v);
    uint32_t best = 0;
    double best_d = (double)a;
    for (uint32_t c = 1; c <= 126u; ++c) {
        double d = fabs((double)a - (double)orc_e4m3_decode(c));
        if (d < best_d || (d == best_d && (c % 2u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    if (!(a < 448.0f)) best = 126;
    return (signbit(v) ? 0x80u : 0u) | best;
}

/* ------------------------------------------------------------------------ */
/* Block-scaled FP4 quantisation -- [HC] "04 · FP4": E2M1 values, one E4M3   */
/* scale per 16 channels, no extra global scale ([MO] same).                 */
/* Reading (pages silent): scale = E4M3(absmax / 6) with fp32 division; code */
/* = E2M1(x / scale) with fp32 division; a zero scale gives all-zero codes.  */
/* ------------------------------------------------------------------------ */

static void fp4_block(const float *x, uint8_t *codes /* 8 bytes */, uint8_t *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float y = amax / 6.0f;
    uint32_t sc = orc_e4m3_encode(y);
    float s = orc_e4m3_decode(sc);
    for (int i = 0; i < 8; ++i) {
        uint32_t lo = 0, hi = 0;
        if (s != 0.0f) {
            lo = orc_e2m1_encode(x[2 * i] / s);
            hi = orc_e2m1_encode(x[2 * i + 1] / s);
        }
        codes[i] = (uint8_t)(lo | (hi << 4)); /* channel 2i in the low nibble */
    }
    *scale = (uint8_t)sc;
}

/* n rows of C channels (C % 16 == 0) -> codes [n][C/2], scales [n][C/16]. */
void orc_quant_fp4_rows(const float *x, int64_t n, int32_t C, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int32_t b = 0; b < C / 16; ++b)
            fp4_block(x + r * C + 16 * b, codes + r * (C / 2) + 8 * b, scales + r * (C / 16) + b);
}

/* Dequantised value of channel c: E2M1(code) * E4M3(scale), exact in double. */
void orc_dequant_fp4_rows(const uint8_t *codes, const uint8_t *scales, int64_t n, int32_t C, double *out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int32_t c = 0; c < C; ++c) {
            uint8_t byte = codes[r * (C / 2) + c / 2];
            uint32_t nib = (c & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15u);
            double s = (double)orc_e4m3_decode(scales[r * (C / 16) + c / 16]);
            out[r * C + c] = (double)orc_e2m1_decode(nib) * s;
        }
}

/* ------------------------------------------------------------------------ */
/* FP8 SWA rows -- [HC] "04 · FP4": the sliding-window KV stays in FP8.      */
/* Reading (pages silent): E4M3 codes with one fp32 scale per token,         */
/* scale = absmax / 448 (fp32 division), code = E4M3(x / scale).             */
/* ------------------------------------------------------------------------ */

void orc_quant_fp8_rows(const float *x, int64_t n, int32_t C, uint8_t *codes, float *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const float *xr = x + r * C;
        float amax = 0.0f;
        for (int32_t c = 0; c < C; ++c) {
            float a = fabsf(xr[c]);
            if (a > amax) amax = a;
        }
        float s = amax / 448.0f;
        for (int32_t c = 0; c < C; ++c)
            codes[r * C + c] = (s != 0.0f) ? (uint8_t)orc_e4m3_encode(xr[c] / s) : 0;
        scales[r] = s;
    }
}

void orc_dequant_fp8_rows(const uint8_t *codes, const float *scales, int64_t n, int32_t C, double *out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int32_t c = 0; c < C; ++c)
            out[r * C + c] = (double)orc_e4m3_decode(codes[r * C + c]) * (double)scales[r];
}

/* ------------------------------------------------------------------------ */
/* Indexer score -- [HC] "03 · CSA2": Full and Reindex layers score the      */
/* positions with their own indexer query; [LB] "What actually changed":     */
/* the indexer already used FP4; [MO]: layers share the indexer keys.        */
/* Form (pages silent; stated synthetic choice):                             */
/*   score(p) = sum_h w_h * relu(q_h . k_p)                                  */
/* with the query quantised by the same FP4 rule as the keys, so that        */
/* q_h . k_p = sum_b t_hb where t_hb = sq_hb * sk_b * P_hb is exact          */
/* (P_hb = the block's E2M1 dot product).  Rounding points, in order:        */
/*   s_h   = ((t_h0 + t_h1) + t_h2) + t_h3        (fp32 adds)                */
/*   r_h   = s_h > 0 ? s_h : +0                                              */
/*   score = fma(w3, r3, fma(w2, r2, fma(w1, r1, w0 * r0)))   (fp32)         */
/*   a zero score is +0.                                                     */
/* ------------------------------------------------------------------------ */

void orc_index_scores(const uint8_t *q_codes /* [Hi][Di/2] */, const uint8_t *q_scales /* [Hi][Di/16] */,
                      const float *w /* [Hi] */, int32_t Hi, int32_t Di,
                      const uint8_t *k_codes /* [n][Di/2] */, const uint8_t *k_scales /* [n][Di/16] */,
                      int64_t n, float *scores /* [n] */)
{
    const int32_t nb = Di / 16;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < n; ++p) {
        const uint8_t *kc = k_codes + p * (Di / 2);
        const uint8_t *ks = k_scales + p * nb;
        float score = 0.0f;
        for (int32_t h = 0; h < Hi; ++h) {
            const uint8_t *qc = q_codes + h * (Di / 2);
            const uint8_t *qs = q_scales + h * nb;
            float s = 0.0f;
            for (int32_t b = 0; b < nb; ++b) {
                double P = 0.0;
                for (int32_t c = 16 * b; c < 16 * b + 16; ++c) {
                    uint32_t qn = (c & 1) ? (uint32_t)(qc[c / 2] >> 4) : (uint32_t)(qc[c / 2] & 15u);
                    uint32_t kn = (c & 1) ? (uint32_t)(kc[c / 2] >> 4) : (uint32_t)(kc[c / 2] & 15u);
                    P += (double)orc_e2m1_decode(qn) * (double)orc_e2m1_decode(kn);
                }
                /* exact: at most 4 + 4 + 12 significant bits */
                float t = (float)((double)orc_e4m3_decode(qs[b]) * (double)orc_e4m3_decode(ks[b]) * P);
                s = (b == 0) ? t : s + t;
            }
            float r = (s > 0.0f) ? s : 0.0f;
            score = (h == 0) ? w[0] * r : fmaf(w[h], r, score);
        }
        if (score == 0.0f) score = 0.0f;
        scores[p] = score;
    }
}

/* ------------------------------------------------------------------------ */
/* Top-K -- [HC] "03 · CSA2" (Full: complete search; Reuse: reuse the        */
/* selection); [LB] "Share the cache and the search work": 512 global        */
/* entries per query, a candidate pool of up to 16,384 positions.            */
/* Order: score descending, ties -> lower position (stated choice).  Output: */
/* the first K of that order as ascending positions, padded with -1.         */
/* ------------------------------------------------------------------------ */

typedef struct {
    float s;
    int32_t p;
} cand_t;

static int cand_order(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->p < y->p) ? -1 : (x->p > y->p) ? 1 : 0;
}

static int int_order(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x < y) ? -1 : (x > y) ? 1 : 0;
}

/* scores[i] belongs to position pos[i]; returns the number selected. */
int32_t orc_topk(const float *scores, const int32_t *pos, int64_t n, int32_t K, int32_t *out)
{
    cand_t *c = (cand_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(cand_t));
    for (int64_t i = 0; i < n; ++i) {
        c[i].s = scores[i];
        c[i].p = pos[i];
    }
    qsort(c, (size_t)n, sizeof(cand_t), cand_order);
    int32_t m = (n < K) ? (int32_t)n : K;
    for (int32_t i = 0; i < m; ++i) out[i] = c[i].p;
    qsort(out, (size_t)m, sizeof(int32_t), int_order);
    for (int32_t i = m; i < K; ++i) out[i] = -1;
    free(c);
    return m;
}

/* ------------------------------------------------------------------------ */
/* Attention -- [LB] "Share the cache and the search work": the selected     */
/* global entries alongside a local 128-token window; [HC] "04 · FP4": the   */
/* selected rows are FP4, the window rows FP8.                               */
/* Reading (pages silent): one softmax over the union (as a multiset) of the */
/* selected rows and the window rows, each row serving as key and value,     */
/* logit = q_h . row (the query carries its own 1/sqrt(512)); fp64 here.     */
/* ------------------------------------------------------------------------ */

void orc_attend(const float *q /* [H][D] */, int32_t H, int32_t D, const double *rows /* [n][D] */,
                int64_t n, double *out /* [H][D] */, double *lse /* [H] */)
{
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < H; ++h) {
        double *z = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        const float *qh = q + (int64_t)h * D;
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int32_t c = 0; c < D; ++c) acc += (double)qh[c] * rows[j * D + c];
            z[j] = acc;
            if (acc > m) m = acc;
        }
        double l = 0.0;
        for (int32_t c = 0; c < D; ++c) out[(int64_t)h * D + c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double e = exp(z[j] - m);
            l += e;
            for (int32_t c = 0; c < D; ++c) out[(int64_t)h * D + c] += e * rows[j * D + c];
        }
        if (n > 0) {
            for (int32_t c = 0; c < D; ++c) out[(int64_t)h * D + c] /= l;
            lse[h] = m + log(l);
        } else {
            lse[h] = -INFINITY;
        }
        free(z);
    }
}
