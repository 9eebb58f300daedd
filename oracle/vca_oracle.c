/*
 * vca_oracle.c -- plain, slow CPU oracle for the VC-Attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or constant generator with the
 * CUDA library; every step is written out from the method's published
 * description ("VC-Attention: Value Smoothing and Softmax Casting for Low-bit
 * Attention", agihunt.info/papers/2609.15810, section "method"; and the news
 * summary at feinterview.poetries.top, sections "V-Smooth" and "ExpCast-FP8").
 *
 * Precision: the method's own arithmetic is followed where it decides an integer
 * (the ExpCast FMA is an fp32 fused multiply-add; quantiser inputs are fp32
 * products), everything else is carried in fp64.  Build with -ffp-contract=off
 * so that no a*b+c in this file is silently fused.
 *
 * Readings where the pages are silent (numbered R1..R14 in the design notes):
 *   R1  k-means init: centroid c starts at V row floor((c+1/2) N / k).
 *   R2  ties in the assignment go to the lowest index; an empty cluster keeps
 *       its previous centroid.
 *   R3  `iters` rounds of (assign, update); labels are those of the last assign.
 *   R4  ExpCast code = rne(8 log2 p + 56 + beta), beta = -0.35, one fp32 FMA.
 *   R5  codes below the E4M3 normal range (< 8) flush to 0; codes > 126 -> 126.
 *   R6  P is coded against a reference max m taken from the key blocks 0..b
 *       visited in increasing (permuted) order.  The pages' kernel is built on
 *       FlashAttention-4, which rescales lazily: m moves to the block max only
 *       when that max exceeds m + tau (log2 units; tau = 8 in the kernel,
 *       tau = 0 is the plain running max), and alpha = 2^(m_old - m_new) then
 *       rescales the accumulators.  P values stay below 2^tau.
 *   R7  one E4M3 residual scale per (batch, head, channel) over the sequence.
 *   R8  Q/K: one absmax/448 scale per (batch, head, 128-token block).
 *   R9  NVFP4 residual: 16 consecutive tokens of one channel share an E4M3
 *       scale; a per-(batch, head) fp32 scale g = amax/(6*448) sits above it.
 *   R10 NVFP4 mode: P is NVFP4 as well (per row, per 16 keys, E4M3 scale of
 *       amax16/6, global scale 1).
 *   R11 the per-block row sums are sums of the decoded P that enters PV.
 *   R12 the block mean is stored as bf16; the residual subtracts the rounded mean.
 *   R13 softmax scale 1/sqrt(d) unless given.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLK 128            /* the 128-token hardware block */
#define E4M3_MAX 448.0
#define E2M1_MAX 6.0
#define EXPCAST_OFFSET 55.65f /* 56 + beta, beta = -0.35 */

enum { ORC_P_EXPCAST = 0, ORC_P_EXP = 1, ORC_P_NVFP4 = 2, ORC_P_EXACT = 3 };
enum { ORC_V_E4M3 = 0, ORC_V_NVFP4 = 1 };

/* Threads the parallel loops below run on (OpenMP's limit for this process,
 * e.g. OMP_NUM_THREADS); reported beside the oracle's timings. */
int orc_threads(void) { return omp_get_max_threads(); }

/* ------------------------------------------------------------------------- */
/* Number formats (OCP 8-bit floating point and microscaling specifications). */
/* ------------------------------------------------------------------------- */

/* Round |x| to a binary format with `frac` fraction bits whose smallest normal
 * exponent is `emin` (below 2^emin the grid is the subnormal spacing
 * 2^(emin-frac)).  Ties go to the even neighbour (nearbyint in the default
 * rounding mode).  No upper saturation here. */
static double round_to_format(double x, int frac, int emin)
{
    if (x == 0.0 || !isfinite(x)) return x;
    double a = fabs(x);
    int e;
    frexp(a, &e);           /* a = f * 2^e with f in [0.5, 1) */
    int E = e - 1;          /* floor(log2 a) */
    if (E < emin) E = emin;
    double q = ldexp(1.0, E - frac);          /* spacing of the grid around a */
    double r = nearbyint(a / q) * q;          /* a / q is exact (power of two) */
    return copysign(r, x);
}

/* E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
 * 0x7F / 0xFF are NaN; largest finite 448; smallest normal 2^-6. */
double orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
    double v;
    if ((c & 0x7F) == 0x7F) return NAN;
    if (E == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, E - 7);
    return s ? -v : v;
}

/* Round to nearest even, saturate to +-448 (the "satfinite" behaviour), keep
 * subnormals, keep the sign of zero. */
uint8_t orc_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double r = fabs(round_to_format(x, 3, -6));
    if (r > E4M3_MAX) r = E4M3_MAX;
    if (r == 0.0) return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;
    uint8_t code;
    if (E < -6) {
        code = (uint8_t)(r / ldexp(1.0, -9));              /* subnormal: m * 2^-9 */
    } else {
        int m = (int)((r / ldexp(1.0, E) - 1.0) * 8.0);     /* exact */
        code = (uint8_t)(((E + 7) << 3) | m);
    }
    return sign | code;
}

/* E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t c)
{
    int s = (c >> 3) & 1, E = (c >> 1) & 3, m = c & 1;
    double v = (E == 0) ? m * 0.5 : (1.0 + m / 2.0) * ldexp(1.0, E - 1);
    return s ? -v : v;
}

uint8_t orc_e2m1_encode(double x)
{
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double r = fabs(round_to_format(x, 1, 0));
    if (r > E2M1_MAX) r = E2M1_MAX;
    if (r == 0.0) return sign;
    if (r < 1.0) return sign | 1;                           /* 0.5 */
    int e;
    frexp(r, &e);
    int E = e - 1;                                          /* 0, 1 or 2 */
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 2.0);
    return sign | (uint8_t)(((E + 1) << 1) | m);
}

/* bfloat16: 7 fraction bits, smallest normal 2^-126. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t orc_bf16_round(double x)
{
    float f = (float)round_to_format(x, 7, -126);   /* exactly representable */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* Batch forms for the tests. */
void orc_e4m3_encode_f32(const float *x, int64_t n, uint8_t *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_encode((double)x[i]);
}

/* Every fp32 bit pattern from `start` for `count` patterns (exhaustive sweeps). */
void orc_e4m3_encode_bits(uint32_t start, int64_t count, uint8_t *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; i++) {
        uint32_t u = start + (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        out[i] = orc_e4m3_encode((double)f);
    }
}

void orc_e2m1_encode_f32(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_e2m1_encode((double)x[i]);
}

/* ------------------------------------------------------------------------- */
/* ExpCast-FP8 (paper page, "method"; news page, "ExpCast-FP8").               */
/* The integer value of an E4M3 byte is about 8*log2(v) + 56, so the byte of  */
/* p = 2^(s - m) is written straight from the log2-domain score with one FMA: */
/*   t = fma(S_raw, 8c, (56 + beta) - 8m),  code = rne(t), clipped (R4, R5).  */
/* ------------------------------------------------------------------------- */
uint8_t orc_expcast_code(float s_raw, float c, float m)
{
    float c8 = 8.0f * c;                    /* exact: power-of-two scaling */
    float bias = EXPCAST_OFFSET - 8.0f * m; /* one rounding */
    float t = fmaf(s_raw, c8, bias);        /* the single fused multiply-add */
    float r = nearbyintf(t);                /* round half to even */
    if (!(r >= 8.0f)) return 0;             /* below the normal range: flush */
    if (r > 126.0f) return 126;             /* above 448: clip */
    return (uint8_t)r;
}

void orc_expcast_codes(const float *s_raw, const float *c, const float *m, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_expcast_code(s_raw[i], c[i], m[i]);
}

/* The conventional path ExpCast replaces: fp32 exp2, then convert to E4M3. */
static uint8_t exp_then_convert(float s_raw, float c, float m)
{
    float arg = fmaf(s_raw, c, -m);
    return orc_e4m3_encode(exp2((double)arg));
}

void orc_exp_codes(const float *s_raw, const float *c, const float *m, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = exp_then_convert(s_raw[i], c[i], m[i]);
}

/* ------------------------------------------------------------------------- */
/* V-Smooth "Group": per-(batch, head) k-means on Value tokens, then a stable */
/* permutation of the tokens by cluster label (paper page, "method"; news     */
/* page, "V-Smooth" bullet "Group").                                           */
/* ------------------------------------------------------------------------- */

/* Stable counting sort: perm[i] is the source token placed in slot i, tokens
 * ordered by (label, original index). */
void orc_stable_sort(const int32_t *labels, int BH, int N, int k, int32_t *perm, int32_t *counts)
{
    for (int bh = 0; bh < BH; bh++) {
        const int32_t *lab = labels + (int64_t)bh * N;
        int32_t *cnt = counts + (int64_t)bh * k;
        int32_t *out = perm + (int64_t)bh * N;
        int64_t *next = calloc((size_t)k, sizeof(int64_t));
        memset(cnt, 0, sizeof(int32_t) * (size_t)k);
        for (int j = 0; j < N; j++) cnt[lab[j]]++;
        int64_t acc = 0;
        for (int c = 0; c < k; c++) { next[c] = acc; acc += cnt[c]; }
        for (int j = 0; j < N; j++) out[next[lab[j]]++] = j;
        free(next);
    }
}

/* Lloyd k-means (R1-R3).  Distances in fp64 from fp32 centroids; updates are
 * fp64 means rounded to fp32. */
void orc_kmeans(const uint16_t *V, int BH, int N, int d, int k, int iters,
                int32_t *labels, int32_t *counts, float *centroids)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; bh++) {
        const uint16_t *v = V + (int64_t)bh * N * d;
        int32_t *lab = labels + (int64_t)bh * N;
        float *C = centroids + (int64_t)bh * k * d;
        double *vrow = malloc(sizeof(double) * (size_t)d);
        double *sum = malloc(sizeof(double) * (size_t)k * d);
        int64_t *cnt = malloc(sizeof(int64_t) * (size_t)k);

        for (int c = 0; c < k; c++) {
            int64_t src = ((int64_t)(2 * c + 1) * N) / (2 * (int64_t)k);
            for (int x = 0; x < d; x++) C[(int64_t)c * d + x] = orc_bf16_to_f32(v[src * d + x]);
        }
        for (int it = 0; it < iters; it++) {
            /* assign */
            for (int j = 0; j < N; j++) {
                for (int x = 0; x < d; x++) vrow[x] = orc_bf16_to_f32(v[(int64_t)j * d + x]);
                double best = INFINITY;
                int arg = 0;
                for (int c = 0; c < k; c++) {
                    double dist = 0.0;
                    for (int x = 0; x < d; x++) {
                        double t = vrow[x] - (double)C[(int64_t)c * d + x];
                        dist += t * t;
                    }
                    if (dist < best) { best = dist; arg = c; }   /* strict: lowest index wins ties */
                }
                lab[j] = arg;
            }
            /* update */
            memset(sum, 0, sizeof(double) * (size_t)k * d);
            memset(cnt, 0, sizeof(int64_t) * (size_t)k);
            for (int j = 0; j < N; j++) {
                int c = lab[j];
                cnt[c]++;
                for (int x = 0; x < d; x++) sum[(int64_t)c * d + x] += orc_bf16_to_f32(v[(int64_t)j * d + x]);
            }
            for (int c = 0; c < k; c++) {
                if (cnt[c] == 0) continue;                       /* empty: keep */
                for (int x = 0; x < d; x++) C[(int64_t)c * d + x] = (float)(sum[(int64_t)c * d + x] / (double)cnt[c]);
            }
        }
        int32_t *ct = counts + (int64_t)bh * k;
        for (int c = 0; c < k; c++) ct[c] = 0;
        for (int j = 0; j < N; j++) ct[lab[j]]++;
        free(vrow); free(sum); free(cnt);
    }
}

/* Sum of squared distances of every token to its assigned centroid (fp64). */
double orc_kmeans_sse(const uint16_t *V, int N, int d, const int32_t *labels, const float *centroids)
{
    double s = 0.0;
    for (int j = 0; j < N; j++)
        for (int x = 0; x < d; x++) {
            double t = orc_bf16_to_f32(V[(int64_t)j * d + x]) - (double)centroids[(int64_t)labels[j] * d + x];
            s += t * t;
        }
    return s;
}

/* ------------------------------------------------------------------------- */
/* Fused prep: gather by perm, 128-token block means, residual quantisation,  */
/* Q/K FP8 quantisation (paper page, "method": demean each hardware block,     */
/* quantise only the residual, per-channel E4M3 for 8 bits, NVFP4 for 4 bits;  */
/* 16-bit mean per block).                                                     */
/* Layouts: q8, k8 [BH][N][d]; sq, sk [BH][N/128]; v_mean bf16 [BH][N/128][d]; */
/*   E4M3:  v_res [BH][N/128][d][128], v_scale [BH][d]                          */
/*   NVFP4: v_res [BH][N/128][d][64] (token 2i low nibble, 2i+1 high nibble),   */
/*          v_sf [BH][N/128][d][8] (one E4M3 scale per 16 tokens), v_scale [BH] */
/* ------------------------------------------------------------------------- */

/* Walsh-Hadamard transform of x[0..d) (d a power of two), unnormalised
 * (entries +-1), as fp32 butterflies in a fixed order: for bit k = 0, 1, ...
 * every pair (c, c + 2^k) with bit k of c clear becomes (a + b, a - b).  The
 * order fixes the rounding, so a device that follows it gets the same bits.
 * H is symmetric with H H = d I, so (H q) . (H k) = d (q . k): rotating Q and
 * K leaves QK^T unchanged up to the factor d, while spreading an outlier
 * channel over all channels before the FP8 quantisation (the QK Hadamard of
 * the Q/K prior art the insight page discusses). */
void orc_fwht_f32(float *x, int d)
{
    for (int h = 1; h < d; h <<= 1)
        for (int c = 0; c < d; c++)
            if (!(c & h)) {
                float a = x[c], b = x[c + h];
                x[c] = a + b;
                x[c + h] = a - b;
            }
}

/* Per-block absmax FP8 quantisation of one 128 x d tile (R8).  `rows` lists the
 * source rows (identity for Q, the permutation for K); with `shift` (K
 * smoothing) every value first has its channel's shift subtracted in fp32;
 * with `hadamard` every row is then rotated by orc_fwht_f32.  The stored
 * scale is amax / 448 times `post` (a power of two). */
static void quant_qk_block(const uint16_t *X, const int32_t *rows, int d, const float *shift, int hadamard,
                           float post, uint8_t *out, float *scale)
{
    float *t = malloc(sizeof(float) * (size_t)BLK * d);
    for (int i = 0; i < BLK; i++) {
        for (int x = 0; x < d; x++) {
            t[(int64_t)i * d + x] = orc_bf16_to_f32(X[(int64_t)rows[i] * d + x]);
            if (shift) t[(int64_t)i * d + x] = t[(int64_t)i * d + x] - shift[x];   /* one fp32 rounding */
        }
        if (hadamard) orc_fwht_f32(t + (int64_t)i * d, d);
    }
    float amax = 0.0f;
    for (int64_t i = 0; i < (int64_t)BLK * d; i++) {
        float a = fabsf(t[i]);
        if (a > amax) amax = a;
    }
    float inv = 1.0f, s = 1.0f;
    if (amax > 0.0f) { inv = 448.0f / amax; s = amax / 448.0f; }
    for (int64_t i = 0; i < (int64_t)BLK * d; i++) {
        float prod = t[i] * inv;   /* one fp32 rounding */
        out[i] = orc_e4m3_encode((double)prod);
    }
    *scale = s * post;
    free(t);
}

/* K smoothing (SageAttention's treatment of the keys' channel bias): the
 * channel mean of K over the whole sequence of one (b,h), subtracted from
 * every key before the FP8 quantisation.  Every score of a query row then
 * moves by the same q . mean, which softmax ignores.  The mean is a fixed
 * fp32 computation, so that it can be reproduced exactly: per permuted
 * 128-token block a halving tree (token i plus token i + 64 for i < 64, then
 * i + 32, ..., i + 1), the block sums added in block order, the total divided
 * by N. */
static float tree_sum128(const float *x)
{
    float y[BLK];
    for (int i = 0; i < BLK; i++) y[i] = x[i];
    for (int h = BLK / 2; h >= 1; h >>= 1)
        for (int i = 0; i < h; i++) y[i] = y[i] + y[i + h];
    return y[0];
}

void orc_k_channel_mean(const uint16_t *K, const int32_t *perm, int N, int d, float *mean)
{
    const int nb = N / BLK;
    float col[BLK];
    for (int x = 0; x < d; x++) {
        float total = 0.0f;
        for (int b = 0; b < nb; b++) {
            for (int i = 0; i < BLK; i++) col[i] = orc_bf16_to_f32(K[(int64_t)perm[b * BLK + i] * d + x]);
            total = total + tree_sum128(col);
        }
        mean[x] = total / (float)N;
    }
}

/* flags: ORC_PREP_QK_HADAMARD rotates every Q and K row by the unnormalised
 * Walsh-Hadamard transform before the FP8 quantisation; the key scale then
 * carries the factor 1/d (exact, a power of two) so that sq sk q8 . k8 still
 * approximates q . k.  ORC_PREP_K_SMOOTH subtracts the keys' channel mean
 * (orc_k_channel_mean) first. */
int orc_prep_ex(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
                int BH, int N, int d, int vmode, unsigned flags,
                uint8_t *q8, float *sq, uint8_t *k8, float *sk,
                uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean)
{
    if (N % BLK != 0 || d <= 0) return 1;
    if (flags & ~3u) return 1;
    const int had = (flags & 1u) != 0;
    const int ksmooth = (flags & 2u) != 0;
    if (had && (d & (d - 1))) return 1;
    const float kpost = had ? 1.0f / (float)d : 1.0f;
    const int nb = N / BLK;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; bh++) {
        const uint16_t *q = Q + (int64_t)bh * N * d, *kk = K + (int64_t)bh * N * d, *v = V + (int64_t)bh * N * d;
        const int32_t *pm = perm + (int64_t)bh * N;
        int32_t ident[BLK];
        float *R = malloc(sizeof(float) * (size_t)N * d);   /* residual, permuted order [slot][ch] */

        /* Q (original order) and K (permuted order, smoothed on request) */
        float *kmean = NULL;
        if (ksmooth) {
            kmean = malloc(sizeof(float) * (size_t)d);
            orc_k_channel_mean(kk, pm, N, d, kmean);
        }
        for (int b = 0; b < nb; b++) {
            for (int i = 0; i < BLK; i++) ident[i] = b * BLK + i;
            quant_qk_block(q, ident, d, NULL, had, 1.0f, q8 + ((int64_t)bh * N + (int64_t)b * BLK) * d,
                           sq + (int64_t)bh * nb + b);
            quant_qk_block(kk, pm + (int64_t)b * BLK, d, kmean, had, kpost,
                           k8 + ((int64_t)bh * N + (int64_t)b * BLK) * d, sk + (int64_t)bh * nb + b);
        }
        free(kmean);
        /* block means of the gathered V, and the residual against the rounded mean */
        for (int b = 0; b < nb; b++) {
            for (int x = 0; x < d; x++) {
                double s = 0.0;
                for (int i = 0; i < BLK; i++) s += orc_bf16_to_f32(v[(int64_t)pm[b * BLK + i] * d + x]);
                float mean = (float)s / 128.0f;
                uint16_t mu = orc_bf16_round((double)mean);
                v_mean[((int64_t)bh * nb + b) * d + x] = mu;
                float muf = orc_bf16_to_f32(mu);
                for (int i = 0; i < BLK; i++)
                    R[((int64_t)b * BLK + i) * d + x] = orc_bf16_to_f32(v[(int64_t)pm[b * BLK + i] * d + x]) - muf;
            }
        }
        if (vmode == ORC_V_E4M3) {
            /* one scale per channel over the whole sequence (R7) */
            for (int x = 0; x < d; x++) {
                float a = 0.0f;
                for (int i = 0; i < N; i++) { float t = fabsf(R[(int64_t)i * d + x]); if (t > a) a = t; }
                float inv = 1.0f, s = 1.0f;
                if (a > 0.0f) { inv = 448.0f / a; s = a / 448.0f; }
                v_scale[(int64_t)bh * d + x] = s;
                for (int i = 0; i < N; i++) {
                    int b = i / BLK, j = i % BLK;
                    float prod = R[(int64_t)i * d + x] * inv;
                    v_res[(((int64_t)bh * nb + b) * d + x) * BLK + j] = orc_e4m3_encode((double)prod);
                }
            }
        } else {
            /* NVFP4 (R9): per-(b,h) global scale, per-16-token E4M3 scales */
            float amax = 0.0f;
            for (int64_t i = 0; i < (int64_t)N * d; i++) { float t = fabsf(R[i]); if (t > amax) amax = t; }
            float g = (amax > 0.0f) ? amax / (6.0f * 448.0f) : 1.0f;
            v_scale[bh] = g;
            float g6 = 6.0f * g;
            for (int b = 0; b < nb; b++)
                for (int x = 0; x < d; x++)
                    for (int grp = 0; grp < BLK / 16; grp++) {
                        float a16 = 0.0f;
                        for (int j = 0; j < 16; j++) {
                            float t = fabsf(R[((int64_t)b * BLK + grp * 16 + j) * d + x]);
                            if (t > a16) a16 = t;
                        }
                        uint8_t sf = orc_e4m3_encode((double)(a16 / g6));
                        v_sf[(((int64_t)bh * nb + b) * d + x) * (BLK / 16) + grp] = sf;
                        float inv = 0.0f;
                        if (sf != 0) inv = 1.0f / ((float)orc_e4m3_decode(sf) * g);
                        for (int j = 0; j < 16; j += 2) {
                            int tok = grp * 16 + j;
                            uint8_t lo = orc_e2m1_encode((double)(R[((int64_t)b * BLK + tok) * d + x] * inv));
                            uint8_t hi = orc_e2m1_encode((double)(R[((int64_t)b * BLK + tok + 1) * d + x] * inv));
                            v_res[(((int64_t)bh * nb + b) * d + x) * (BLK / 2) + tok / 2] = (uint8_t)(lo | (hi << 4));
                        }
                    }
        }
        free(R);
    }
    return 0;
}

int orc_prep(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
             int BH, int N, int d, int vmode,
             uint8_t *q8, float *sq, uint8_t *k8, float *sk,
             uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean)
{
    return orc_prep_ex(Q, K, V, perm, BH, N, d, vmode, 0u, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean);
}

/* ------------------------------------------------------------------------- */
/* Attention with V-Smooth restore and ExpCast, emulating the kernel's        */
/* online-softmax schedule (R6): key blocks in increasing permuted order,      */
/* reference max updated lazily (threshold tau),                               */
/* running max, alpha rescale, per-block row sums of the decoded P (R11) and   */
/* the mean restored as one outer product per block (paper page, "method":    */
/* the block means come back through the row sums online softmax already      */
/* accumulates; news page, "V-Smooth" bullet "Restore").                       */
/* mode: ORC_P_EXPCAST / ORC_P_EXP / ORC_P_NVFP4, or ORC_P_EXACT (P kept in   */
/* fp64, unquantised: reduces the schedule to exact softmax over the          */
/* dequantised operands).  vmode: ORC_V_E4M3 or ORC_V_NVFP4 residuals.        */
/* rows: the query rows to compute per (b,h) (nrows of them), or NULL for all; */
/* O: bf16 [BH][nrows][d]; l_out (optional): fp64 row sums [BH][nrows].        */
/* ------------------------------------------------------------------------- */
int orc_attention(const uint8_t *q8, const float *sq, const uint8_t *k8, const float *sk,
                  const uint8_t *v_res, const uint8_t *v_sf, const float *v_scale, const uint16_t *v_mean,
                  int BH, int N, int d, float softmax_scale, float tau, int mode, int vmode,
                  const int32_t *rows, int nrows, uint16_t *O, double *l_out)
{
    if (N % BLK != 0 || d <= 0) return 1;
    const int nb = N / BLK;
    if (softmax_scale <= 0.0f) softmax_scale = (float)(1.0 / sqrt((double)d));
    const float L = (float)((double)softmax_scale * 1.4426950408889634);   /* log2(e) */
    if (rows == NULL) nrows = N;

    for (int bh = 0; bh < BH; bh++) {
        /* decoded operands of this (b,h) */
        double *kd = malloc(sizeof(double) * (size_t)N * d);
        double *vd = malloc(sizeof(double) * (size_t)N * d);   /* [slot][ch]: residual code (times the 16-scale for NVFP4) */
        for (int64_t i = 0; i < (int64_t)N * d; i++) kd[i] = orc_e4m3_decode(k8[(int64_t)bh * N * d + i]);
        for (int b = 0; b < nb; b++)
            for (int x = 0; x < d; x++)
                for (int j = 0; j < BLK; j++) {
                    double val;
                    if (vmode == ORC_V_E4M3) {
                        val = orc_e4m3_decode(v_res[(((int64_t)bh * nb + b) * d + x) * BLK + j]);
                    } else {
                        uint8_t byte = v_res[(((int64_t)bh * nb + b) * d + x) * (BLK / 2) + j / 2];
                        uint8_t nib = (j & 1) ? (byte >> 4) : (byte & 15);
                        uint8_t sf = v_sf[(((int64_t)bh * nb + b) * d + x) * (BLK / 16) + j / 16];
                        val = orc_e2m1_decode(nib) * orc_e4m3_decode(sf);
                    }
                    vd[((int64_t)b * BLK + j) * d + x] = val;
                }

        #pragma omp parallel for schedule(dynamic, 4)
        for (int ri = 0; ri < nrows; ri++) {
            int r = rows ? rows[ri] : ri;
            double *qd = malloc(sizeof(double) * (size_t)d);
            double *acc = calloc((size_t)d, sizeof(double));   /* sum_b P_b . R_b (codes) */
            double *mac = calloc((size_t)d, sizeof(double));   /* sum_b rowsum_b mu_b     */
            float S[BLK];
            double P[BLK];
            for (int x = 0; x < d; x++) qd[x] = orc_e4m3_decode(q8[((int64_t)bh * N + r) * d + x]);
            const float sqr = sq[(int64_t)bh * nb + r / BLK];
            float m = -INFINITY;
            double l = 0.0;
            for (int b = 0; b < nb; b++) {
                const float c = (sqr * sk[(int64_t)bh * nb + b]) * L;
                float bmax = -INFINITY;
                for (int j = 0; j < BLK; j++) {
                    double dot = 0.0;
                    const double *kr = kd + ((int64_t)b * BLK + j) * d;
                    for (int x = 0; x < d; x++) dot += qd[x] * kr[x];
                    S[j] = (float)dot;                         /* fp32 accumulator value */
                    float s = S[j] * c;
                    if (s > bmax) bmax = s;
                }
                /* lazy update of the reference max (R6): fp32 m + tau */
                if (bmax > m + tau) {
                    if (m != -INFINITY) {
                        double alpha = exp2((double)m - (double)bmax);
                        for (int x = 0; x < d; x++) { acc[x] *= alpha; mac[x] *= alpha; }
                        l *= alpha;
                    }
                    m = bmax;
                }
                double rowsum = 0.0;
                if (mode == ORC_P_NVFP4) {
                    for (int g = 0; g < BLK; g += 16) {
                        float p[16], a16 = 0.0f;
                        for (int j = 0; j < 16; j++) {
                            p[j] = (float)exp2((double)fmaf(S[g + j], c, -m));
                            if (p[j] > a16) a16 = p[j];
                        }
                        uint8_t sf = orc_e4m3_encode((double)(a16 / 6.0f));
                        float inv = (sf != 0) ? 1.0f / (float)orc_e4m3_decode(sf) : 0.0f;
                        for (int j = 0; j < 16; j++)
                            P[g + j] = orc_e2m1_decode(orc_e2m1_encode((double)(p[j] * inv))) * orc_e4m3_decode(sf);
                    }
                } else {
                    for (int j = 0; j < BLK; j++) {
                        if (mode == ORC_P_EXPCAST) P[j] = orc_e4m3_decode(orc_expcast_code(S[j], c, m));
                        else if (mode == ORC_P_EXP) P[j] = orc_e4m3_decode(exp_then_convert(S[j], c, m));
                        else P[j] = exp2((double)S[j] * (double)c - (double)m);
                    }
                }
                for (int j = 0; j < BLK; j++) rowsum += P[j];
                l += rowsum;
                const uint16_t *mu = v_mean + ((int64_t)bh * nb + b) * d;
                for (int x = 0; x < d; x++) {
                    double t = 0.0;
                    for (int j = 0; j < BLK; j++) t += P[j] * vd[((int64_t)b * BLK + j) * d + x];
                    acc[x] += t;                                   /* PV on the residual codes */
                    mac[x] += rowsum * (double)orc_bf16_to_f32(mu[x]);   /* rowsum_b (x) mu_b */
                }
            }
            for (int x = 0; x < d; x++) {
                double sv = (vmode == ORC_V_E4M3) ? (double)v_scale[(int64_t)bh * d + x] : (double)v_scale[bh];
                double o = (acc[x] * sv + mac[x]) / l;
                O[((int64_t)bh * nrows + ri) * d + x] = orc_bf16_round((double)(float)o);
            }
            if (l_out) l_out[(int64_t)bh * nrows + ri] = l;
            free(qd); free(acc); free(mac);
        }
        free(kd); free(vd);
    }
    return 0;
}

/* Exact fp64 softmax attention on the bf16 inputs (no quantisation, no
 * permutation): O = softmax(Q K^T * scale) V.  Rows as in orc_attention; the
 * output is fp64 [BH][nrows][d]. */
int orc_attention_exact(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                        int BH, int N, int d, float softmax_scale,
                        const int32_t *rows, int nrows, double *O)
{
    if (softmax_scale <= 0.0f) softmax_scale = (float)(1.0 / sqrt((double)d));
    if (rows == NULL) nrows = N;
    for (int bh = 0; bh < BH; bh++) {
        const uint16_t *q = Q + (int64_t)bh * N * d, *k = K + (int64_t)bh * N * d, *v = V + (int64_t)bh * N * d;
        #pragma omp parallel for schedule(dynamic, 4)
        for (int ri = 0; ri < nrows; ri++) {
            int r = rows ? rows[ri] : ri;
            double *s = malloc(sizeof(double) * (size_t)N);
            double mx = -INFINITY, den = 0.0;
            for (int j = 0; j < N; j++) {
                double dot = 0.0;
                for (int x = 0; x < d; x++)
                    dot += (double)orc_bf16_to_f32(q[(int64_t)r * d + x]) * (double)orc_bf16_to_f32(k[(int64_t)j * d + x]);
                s[j] = dot * (double)softmax_scale;
                if (s[j] > mx) mx = s[j];
            }
            for (int j = 0; j < N; j++) { s[j] = exp(s[j] - mx); den += s[j]; }
            double *o = O + ((int64_t)bh * nrows + ri) * d;
            for (int x = 0; x < d; x++) o[x] = 0.0;
            for (int j = 0; j < N; j++)
                for (int x = 0; x < d; x++) o[x] += s[j] * (double)orc_bf16_to_f32(v[(int64_t)j * d + x]);
            for (int x = 0; x < d; x++) o[x] /= den;
            free(s);
        }
    }
    return 0;
}
