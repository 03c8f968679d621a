/*
 * cbq_oracle.c -- plain, slow, obviously-correct CPU oracle for the 3.25-bit
 * codebook-quantised matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file; only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header or table with the CUDA library.
 *
 * Source of the method: "Hibana: Fast Agentic Inference on Unified-Memory
 * Devices", section "Model surgery / Three-bit weights": each group of 32
 * weights is a 3-bit index into an 8-entry FP8 codebook, plus one 8-bit scale
 * per group, i.e. 3 + 8/32 = 3.25 bits per weight.  The storage format fixed
 * for this library (the pages leave it open):
 *   codes     : one group (n, g = k/32) is 12 bytes, read as a 96-bit
 *               little-endian number with code j = k%32 at bits 3j..3j+2.
 *               Groups are ordered in 128-row tiles: tile t = n/128 holds
 *               rows 128t .. 128t+R-1 (R = min(128, N-128t)) and starts at
 *               byte 128t * 3K/8; inside it, k-tile c = k/128 (four groups,
 *               fewer in a last partial k-tile) is a block of R rows x W
 *               bytes (W = 12 x its groups) at c*R*48, row n%128 at
 *               (n%128)*W, group g%4 at (g%4)*12.  Total 3KN/8 bytes.
 *   scales    : uint8 [N][K/32], E8M0, value 2^(s-127).
 *   codebooks : uint8 [N][8], OCP FP8 E4M3 ("fn") per output row.
 *   a         : uint8 E4M3 [M][K], a_scale fp32 [M]; y fp32 [M][N].
 *   y[m,n] = a_scale[m] * sum_k E4M3(a[m,k]) * E4M3(cb[n][code(n,k)]) * 2^(s[n,k/32]-127)
 *
 * Arithmetic: every decoded value is exact in double; products are exact in
 * double; the sum over k runs in plain k order in double; the result is
 * multiplied by a_scale in double and rounded once to fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- number formats ---------------------------------------------------- */

/* OCP 8-bit E4M3 ("fn" variant): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0; exponent 0 is subnormal 2^-6 * m/8; S.1111.111 is NaN;
 * there is no infinity.  Largest finite value 448. */
double orc_e4m3_value(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);            /* 2^-6 * m/8 */
    else
        v = ldexp((double)(8 + m), e - 10);  /* 2^(e-7) * (1 + m/8) */
    return sign ? -v : v;
}

/* E8M0 scale byte (OCP MX): 2^(s-127); 255 is NaN. */
double orc_e8m0_value(uint8_t s)
{
    if (s == 255)
        return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* Round a double to the nearest E4M3 value, ties to even mantissa,
 * saturating to +-448 (used by the packer when it rounds centroids). */
uint8_t orc_e4m3_round(double x)
{
    uint8_t sign = 0;
    double ax;
    if (x != x)
        return 0x7F;
    if (signbit(x)) {
        sign = 0x80;
        ax = -x;
    } else {
        ax = x;
    }
    if (ax >= 448.0)
        return sign | 0x7E;
    if (ax < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9 */
        double q = ax * 512.0;
        double r = nearbyint(q);             /* default rounding: to even */
        return sign | (uint8_t)r;            /* r == 8 is exactly 2^-6 */
    }
    {
        int ex;
        double f = frexp(ax, &ex);           /* ax = f * 2^ex, f in [0.5,1) */
        int unb = ex - 1;                    /* ax in [2^unb, 2^(unb+1)) */
        double sig = ldexp(f, 4);            /* in [8,16): 1.mmm * 8 */
        double r = nearbyint(sig);
        int biased;
        int bits;
        if (r >= 16.0) {
            r = 8.0;
            unb += 1;
        }
        biased = unb + 7;
        bits = (biased << 3) | ((int)r - 8);
        if (bits > 0x7E)
            bits = 0x7E;
        return sign | (uint8_t)bits;
    }
}

/* ---- bitstream --------------------------------------------------------- */

/* Byte offset of group (n, g) in the code stream (layout in the header). */
int64_t orc_group_offset(int64_t N, int64_t K, int64_t n, int64_t g)
{
    int64_t t = n / 128;                          /* row tile */
    int64_t R = (N - 128 * t < 128) ? N - 128 * t : 128;  /* rows in it */
    int64_t tile_base = 128 * t * (3 * K / 8);
    int64_t c = g / 4;                            /* k-tile of 128 weights */
    int64_t G = K / 32;                           /* groups per row */
    int64_t W = (G - 4 * c < 4) ? 12 * (G - 4 * c) : 48;  /* block row bytes */
    return tile_base + c * R * 48 + (n % 128) * W + (g % 4) * 12;
}

/* Code of weight (n, k): bits 3j..3j+2 of the 96-bit little-endian group,
 * read one bit at a time. */
int orc_code(const uint8_t *codes, int64_t N, int64_t K, int64_t n, int64_t k)
{
    int64_t base = orc_group_offset(N, K, n, k / 32);
    int j = (int)(k % 32);
    int code = 0;
    for (int i = 0; i < 3; i++) {
        int pos = 3 * j + i;
        int bit = (codes[base + pos / 8] >> (pos % 8)) & 1;
        code |= bit << i;
    }
    return code;
}

/* Write code c for weight (n, k) one bit at a time (codes must start zeroed
 * or hold the old value; bits are overwritten). */
void orc_set_code(uint8_t *codes, int64_t N, int64_t K, int64_t n, int64_t k, int c)
{
    int64_t base = orc_group_offset(N, K, n, k / 32);
    int j = (int)(k % 32);
    for (int i = 0; i < 3; i++) {
        int pos = 3 * j + i;
        uint8_t mask = (uint8_t)(1u << (pos % 8));
        if ((c >> i) & 1)
            codes[base + pos / 8] |= mask;
        else
            codes[base + pos / 8] &= (uint8_t)~mask;
    }
}

/* Dequantised weight w[n,k] = E4M3(cb[n][code]) * 2^(s[n,g]-127), exact. */
double orc_weight(const uint8_t *codes, const uint8_t *scales,
                  const uint8_t *codebooks, int64_t N, int64_t K, int64_t n, int64_t k)
{
    int c = orc_code(codes, N, K, n, k);
    return orc_e4m3_value(codebooks[n * 8 + c]) *
           orc_e8m0_value(scales[n * (K / 32) + k / 32]);
}

/* ---- unpack, gemm, grouped gemm ---------------------------------------- */

void orc_unpack(const uint8_t *codes, const uint8_t *scales,
                const uint8_t *codebooks, int64_t N, int64_t K, float *W)
{
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            W[n * K + k] = (float)orc_weight(codes, scales, codebooks, N, K, n, k);
}

/* y[m,n] and the error-bound base B[m,n] = |a_scale[m]| * sum_k |a*w|.
 * Rows n are independent; the OpenMP loop only splits them across threads,
 * each (m, n) sum is still taken in k order. */
void orc_gemm(const uint8_t *a, const float *a_scale,
              const uint8_t *codes, const uint8_t *scales,
              const uint8_t *codebooks, int64_t M, int64_t N, int64_t K,
              float *y, double *bound)
{
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = orc_e4m3_value(a[m * K + k]) *
                           orc_weight(codes, scales, codebooks, N, K, n, k);
                acc += p;
                accabs += fabs(p);
            }
            y[m * N + n] = (float)((double)a_scale[m] * acc);
            if (bound)
                bound[m * N + n] = fabs((double)a_scale[m]) * accabs;
        }
    }
}

/* y for a subset of output rows: y[m][i] for row rows[i] of the N-row
 * matrix (same arithmetic as orc_gemm, row by row). */
void orc_gemm_rows(const uint8_t *a, const float *a_scale,
                   const uint8_t *codes, const uint8_t *scales,
                   const uint8_t *codebooks, int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, int64_t nrows, float *y, double *bound)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; i++) {
        int64_t n = rows[i];
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = orc_e4m3_value(a[m * K + k]) *
                           orc_weight(codes, scales, codebooks, N, K, n, k);
                acc += p;
                accabs += fabs(p);
            }
            y[m * nrows + i] = (float)((double)a_scale[m] * acc);
            if (bound)
                bound[m * nrows + i] = fabs((double)a_scale[m]) * accabs;
        }
    }
}

/* Mixture-of-experts verify round: experts are stacked, expert e owns rows
 * e*N .. e*N+N-1 of one packed matrix.  y[t, j, :] is the product of token t
 * with expert topk_idx[t, j]; no gate weight, no combine.  When read_count is
 * given, read_count[e] is incremented once for every expert whose weights
 * this routine actually reads. */
void orc_grouped_gemm(const uint8_t *a, const float *a_scale,
                      const uint8_t *codes, const uint8_t *scales,
                      const uint8_t *codebooks, int64_t E, const int32_t *topk_idx,
                      int64_t topk, int64_t M, int64_t N, int64_t K,
                      float *y, double *bound, int64_t *read_count)
{
    int64_t gk = K / 32;
    char *touched = (char *)calloc((size_t)E, 1);
    for (int64_t t = 0; t < M; t++) {
        for (int64_t j = 0; j < topk; j++) {
            int64_t e = topk_idx[t * topk + j];
            const uint8_t *ce = codes + e * (3 * K * N / 8);
            const uint8_t *se = scales + e * N * gk;
            const uint8_t *be = codebooks + e * N * 8;
            touched[e] = 1;
            orc_gemm(a + t * K, a_scale + t, ce, se, be, 1, N, K,
                     y + (t * topk + j) * N,
                     bound ? bound + (t * topk + j) * N : NULL);
        }
    }
    if (read_count)
        for (int64_t e = 0; e < E; e++)
            read_count[e] += touched[e];
    free(touched);
}

/* ---- two-bit draft head ------------------------------------------------- */
/*
 * "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
 * surgery / Two-bit draft head": the drafter's vocabulary head is stored in
 * 2 bits, scores every token, keeps a shortlist of 16 and rescores the
 * shortlist with the FP8 head.  The pages fix neither the 2-bit format nor
 * the FP8 head's; the readings taken here mirror the 3-bit format:
 *   codes2     : one group (n, g = k/32) is 8 bytes, read as a 64-bit
 *                little-endian number with code j = k%32 at bits 2j..2j+1;
 *                groups in 128-row tiles as for 3 bits, with 32 bytes per row
 *                and k-tile (8 per group): tile t starts at byte 128t * K/4,
 *                k-tile c of a tile with R rows at c*R*32, row n%128 at
 *                (n%128)*W (W = 8 x the k-tile's groups), group g%4 at (g%4)*8.
 *                Total KN/4 bytes.
 *   scales2    : uint8 [N][K/32], E8M0 (2^(s-127)).
 *   codebooks2 : uint8 [N][4], E4M3.
 *   2 + 8/32 = 2.25 bits per weight.
 *   head8      : the FP8 head, uint8 E4M3 [N][K] row-major, with one fp32
 *                scale per row: w8[n,k] = E4M3(head8[n,k]) * row_scale[n].
 */
int64_t orc_group_offset2(int64_t N, int64_t K, int64_t n, int64_t g)
{
    int64_t t = n / 128;
    int64_t R = (N - 128 * t < 128) ? N - 128 * t : 128;
    int64_t tile_base = 128 * t * (K / 4);
    int64_t c = g / 4;
    int64_t G = K / 32;
    int64_t W = (G - 4 * c < 4) ? 8 * (G - 4 * c) : 32;
    return tile_base + c * R * 32 + (n % 128) * W + (g % 4) * 8;
}

/* Code of weight (n, k): bits 2j, 2j+1 of the 64-bit little-endian group. */
int orc_code2(const uint8_t *codes, int64_t N, int64_t K, int64_t n, int64_t k)
{
    int64_t base = orc_group_offset2(N, K, n, k / 32);
    int j = (int)(k % 32);
    int code = 0;
    for (int i = 0; i < 2; i++) {
        int pos = 2 * j + i;
        int bit = (codes[base + pos / 8] >> (pos % 8)) & 1;
        code |= bit << i;
    }
    return code;
}

/* Dequantised weight of the 2-bit head, exact. */
double orc_weight2(const uint8_t *codes, const uint8_t *scales,
                   const uint8_t *codebooks, int64_t N, int64_t K, int64_t n, int64_t k)
{
    int c = orc_code2(codes, N, K, n, k);
    return orc_e4m3_value(codebooks[n * 4 + c]) *
           orc_e8m0_value(scales[n * (K / 32) + k / 32]);
}

/* Scores of the 2-bit head: s[m,n] = a_scale[m] * sum_k a[m,k] w2[n,k]
 * (sum in k order in double, one rounding to fp32), and the bound base
 * |a_scale| * sum |a w2|, as orc_gemm. */
void orc_gemm2(const uint8_t *a, const float *a_scale,
               const uint8_t *codes, const uint8_t *scales,
               const uint8_t *codebooks, int64_t M, int64_t N, int64_t K,
               float *y, double *bound)
{
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = orc_e4m3_value(a[m * K + k]) *
                           orc_weight2(codes, scales, codebooks, N, K, n, k);
                acc += p;
                accabs += fabs(p);
            }
            y[m * N + n] = (float)((double)a_scale[m] * acc);
            if (bound)
                bound[m * N + n] = fabs((double)a_scale[m]) * accabs;
        }
    }
}

/* FP8 rescoring of chosen rows: for token m and its rows rows[m][i]
 * (i < R), logit = a_scale[m] * row_scale[n] * sum_k a[m,k] E4M3(head8[n,k])
 * (sum in k order in double, then the two scales, one rounding to fp32), and
 * the bound base |a_scale * row_scale| * sum |a w8|. */
void orc_rescore8(const uint8_t *a, const float *a_scale, const uint8_t *head8,
                  const float *row_scale, int64_t M, int64_t N, int64_t K,
                  const int32_t *rows, int64_t R, float *logits, double *bound)
{
    for (int64_t m = 0; m < M; m++) {
        for (int64_t i = 0; i < R; i++) {
            int64_t n = rows[m * R + i];
            double acc = 0.0, accabs = 0.0;
            if (n >= 0 && n < N) {
                for (int64_t k = 0; k < K; k++) {
                    double p = orc_e4m3_value(a[m * K + k]) * orc_e4m3_value(head8[n * K + k]);
                    acc += p;
                    accabs += fabs(p);
                }
            }
            double sc = (double)a_scale[m] * (double)((n >= 0 && n < N) ? row_scale[n] : 0.0f);
            logits[m * R + i] = (float)(sc * acc);
            if (bound)
                bound[m * R + i] = fabs(sc) * accabs;
        }
    }
}

/* ---- pack (quantiser) -------------------------------------------------- */
/*
 * The pages state only that each 32-weight group is mapped onto an 8-entry
 * FP8 codebook derived from the weights; the format puts one codebook on each
 * output row and one E8M0 scale on each group of 32.  The rule taken here,
 * step by step:
 *  1. group scale s = clamp(127 + ceil(log2(max|w|)), 0, 254), s = 127 for
 *     an all-zero group, so that |w| / 2^(s-127) <= 1;
 *  2. u = w / 2^(s-127) for every weight of the row;
 *  3. 1-D Lloyd (k-means) with 8 centroids over the row's u values:
 *     start at the sorted values at index floor((i + 0.5) * K / 8),
 *     16 rounds of (assign to nearest centroid, ties to the lower index;
 *     centroid = mean of its members, summed in k order; an empty cluster
 *     keeps its centroid);
 *  4. round centroids to E4M3 (ties to even, saturate at 448), sort ascending;
 *  5. code = index of the nearest rounded centroid, ties to the lower index;
 *  6. write the bitstream.
 */

static int orc_cmp_double(const void *pa, const void *pb)
{
    double a = *(const double *)pa, b = *(const double *)pb;
    return (a > b) - (a < b);
}

static int orc_cmp_e4m3(const void *pa, const void *pb)
{
    double a = orc_e4m3_value(*(const uint8_t *)pa);
    double b = orc_e4m3_value(*(const uint8_t *)pb);
    return (a > b) - (a < b);
}

/* group scale byte of one group of 32 weights (step 1) */
uint8_t orc_group_scale(const float *w32)
{
    double amax = 0.0;
    int ex, s;
    double f;
    for (int j = 0; j < 32; j++)
        if (fabs((double)w32[j]) > amax)
            amax = fabs((double)w32[j]);
    if (amax == 0.0)
        return 127;
    f = frexp(amax, &ex);                     /* amax = f * 2^ex */
    /* ceil(log2(amax)): ex - 1 when amax is a power of two, else ex */
    s = 127 + ((f == 0.5) ? ex - 1 : ex);
    if (s < 0)
        s = 0;
    if (s > 254)
        s = 254;
    return (uint8_t)s;
}

void orc_pack(const float *W, int64_t N, int64_t K,
              uint8_t *codes, uint8_t *scales, uint8_t *codebooks)
{
    int64_t gk = K / 32;
    double *u = (double *)malloc(sizeof(double) * (size_t)K);
    double *sorted = (double *)malloc(sizeof(double) * (size_t)K);
    memset(codes, 0, (size_t)(N * gk * 12));
    for (int64_t n = 0; n < N; n++) {
        const float *wr = W + n * K;
        double cen[8];
        uint8_t cb[8];
        /* steps 1-2 */
        for (int64_t g = 0; g < gk; g++) {
            uint8_t s = orc_group_scale(wr + g * 32);
            scales[n * gk + g] = s;
            for (int j = 0; j < 32; j++)
                u[g * 32 + j] = (double)wr[g * 32 + j] / orc_e8m0_value(s);
        }
        /* step 3 */
        memcpy(sorted, u, sizeof(double) * (size_t)K);
        qsort(sorted, (size_t)K, sizeof(double), orc_cmp_double);
        for (int i = 0; i < 8; i++)
            cen[i] = sorted[(int64_t)((i + 0.5) * (double)K / 8.0)];
        for (int it = 0; it < 16; it++) {
            double sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            int64_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int64_t k = 0; k < K; k++) {
                int best = 0;
                for (int c = 1; c < 8; c++)
                    if (fabs(u[k] - cen[c]) < fabs(u[k] - cen[best]))
                        best = c;
                sum[best] += u[k];
                cnt[best] += 1;
            }
            for (int c = 0; c < 8; c++)
                if (cnt[c] > 0)
                    cen[c] = sum[c] / (double)cnt[c];
        }
        /* step 4 */
        for (int c = 0; c < 8; c++)
            cb[c] = orc_e4m3_round(cen[c]);
        /* insertion sort by value: stable, so +0 and -0 keep their order */
        for (int i = 1; i < 8; i++) {
            uint8_t key = cb[i];
            int j = i - 1;
            while (j >= 0 && orc_cmp_e4m3(&cb[j], &key) > 0) {
                cb[j + 1] = cb[j];
                j--;
            }
            cb[j + 1] = key;
        }
        memcpy(codebooks + n * 8, cb, 8);
        /* steps 5-6 */
        for (int64_t k = 0; k < K; k++) {
            int best = 0;
            for (int c = 1; c < 8; c++)
                if (fabs(u[k] - orc_e4m3_value(cb[c])) <
                    fabs(u[k] - orc_e4m3_value(cb[best])))
                    best = c;
            orc_set_code(codes, N, K, n, k, best);
        }
    }
    free(u);
    free(sorted);
}

/* Number of OpenMP threads the gemm loop uses (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int orc_num_threads(void) { return omp_get_max_threads(); }
void orc_set_num_threads(int n) { omp_set_num_threads(n); }
#else
int orc_num_threads(void) { return 1; }
void orc_set_num_threads(int n) { (void)n; }
#endif
