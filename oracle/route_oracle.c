/*
 * Route-step oracle: plain, slow, single-threaded CPU definition of what the
 * MoE route step computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg may call it; the product path
 * never does.  It shares no code, header or table with the CUDA library.
 *
 * Sources (all arithmetic below restates them):
 *   [P2-Num]  "Optionally gather the Kimi3 prefill latent instead of reducing
 *             it", Description, Numerics bullet: a latent value is one
 *             FP32-accumulated full-K dot product, rounded once to BF16, and
 *             is more accurate against float64 than the K-split path.
 *   [P2-Cmp]  same page, Description, Compile bullet: the projection is
 *             M = rows, K = 7168; 3584 latent columns in total.
 *   [P2-Body] same page, commit body: the general path rounds each K-slice
 *             partial to BF16, adds the partials in FP32 and rounds the sum
 *             to BF16 again -- two roundings.
 *   [P3]      "Use two row blocks for eight-row Kimi paired gathers", body:
 *             FP32 router logits, 56 per rank at TP16, i.e. 896 experts.
 *   [P1]      "Kimi K3.1 recipe: route 9..20 decode rows through the pushed
 *             pair gather and standalone top-16", commit message: a
 *             standalone top-16 selects each row's experts; routing weights
 *             are compared to within 5 FP32 ULP.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - weights are stored [K, N] row-major (N contiguous);
 *   - the float64 value is rounded to FP32 and then to BF16, both
 *     round-to-nearest-even;
 *   - top-16 ranks by raw FP32 logit, descending; equal logits (with
 *     -0 == +0) go to the lower expert id; output is in rank order;
 *     NaN ranks below every number (below -Inf);
 *   - routing weight w_i = s_i / sum_j s_j with s_i = 1 / (1 + exp(-logit)),
 *     over the 16 picked experts, computed in double, rounded to FP32;
 *   - the latent sum of squares is taken over the BF16 latent values the
 *     step returns (what a following norm reads), rounded once to FP32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- number formats ---------------------------------------------------- */

/* BF16 bit pattern -> the real number it denotes (exactly, via FP32). */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t b) { return (double)bf16_bits_to_float(b); }

/* FP32 -> BF16, round to nearest, ties to even (IEEE default rounding).
 * BF16 keeps the FP32 sign, the 8 exponent bits and the top 7 fraction bits;
 * the low 16 bits are rounded away.  NaN stays a (quiet) NaN. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* may carry into the exponent: correct, rounds up to Inf */
    return (uint16_t)upper;
}

/* double -> FP32 with round-to-nearest-even: the C conversion under the
 * default rounding mode does exactly this. */
float oracle_fp32_rne(double x) { return (float)x; }

/* ---- a1 + a2: the projections [P2-Num], [P2-Cmp], [P3] ----------------- */

/* y[r, n] = sum_{k = 0 .. K-1} h[r, k] * W[k, n], in float64, k ascending.
 * h: BF16 bits [R, K] row-major; W: BF16 bits [K, N] row-major.
 * Every BF16 x BF16 product is exact in double (8-bit significands); only the
 * running double sum rounds.  Loop order r -> k -> n keeps one double
 * accumulator row per r, so each element still sums k ascending. */
void oracle_dot64(const uint16_t *h, const uint16_t *W, int R, int K, int N, double *y)
{
    double *wrow = (double *)malloc(sizeof(double) * (size_t)N);
    for (int r = 0; r < R; ++r) {
        double *acc = y + (size_t)r * N;
        for (int n = 0; n < N; ++n)
            acc[n] = 0.0;
        for (int k = 0; k < K; ++k) {
            double hk = oracle_bf16_to_double(h[(size_t)r * K + k]);
            const uint16_t *w = W + (size_t)k * N;
            for (int n = 0; n < N; ++n)
                wrow[n] = oracle_bf16_to_double(w[n]);
            for (int n = 0; n < N; ++n)
                acc[n] += hk * wrow[n];
        }
    }
    free(wrow);
}

/* The route projection of one layer.
 *   latent[r, n] = bf16_rne(fp32_rne(sum_k h[r,k] * Wl[k,n]))      (a1)
 *   logits[r, e] = fp32_rne(sum_k h[r,k] * Wr[k,e])                (a2)
 * y_lat / y_log (optional, may be NULL) receive the float64 sums.  */
void oracle_latent_router(const uint16_t *h, const uint16_t *Wl, const uint16_t *Wr,
                          int R, int K, int NL, int NR,
                          uint16_t *latent, float *logits, double *y_lat, double *y_log)
{
    double *yl = y_lat ? y_lat : (double *)malloc(sizeof(double) * (size_t)R * NL);
    double *yr = y_log ? y_log : (double *)malloc(sizeof(double) * (size_t)R * NR);
    oracle_dot64(h, Wl, R, K, NL, yl);
    oracle_dot64(h, Wr, R, K, NR, yr);
    for (size_t i = 0; i < (size_t)R * NL; ++i)
        latent[i] = oracle_bf16_rne(oracle_fp32_rne(yl[i]));
    for (size_t i = 0; i < (size_t)R * NR; ++i)
        logits[i] = oracle_fp32_rne(yr[i]);
    if (!y_lat) free(yl);
    if (!y_log) free(yr);
}

/* The general (K-split) path the pages replace [P2-Num], [P2-Body]: the K
 * range is cut into `shards` equal slices, each slice's FP32-accumulated
 * partial is rounded to BF16, the rounded partials are summed in FP32 in shard
 * order and the sum is rounded to BF16 again.  Each slice's sum is taken in
 * float64 and rounded to FP32 (the same per-slice definition as above).
 * Used only to check the direction of the accuracy claim. */
void oracle_latent_ksplit(const uint16_t *h, const uint16_t *W, int R, int K, int N,
                          int shards, uint16_t *out)
{
    int ks = K / shards;
    double *acc = (double *)malloc(sizeof(double) * (size_t)N);
    float *sum = (float *)malloc(sizeof(float) * (size_t)N);
    for (int r = 0; r < R; ++r) {
        for (int n = 0; n < N; ++n)
            sum[n] = 0.0f;
        for (int s = 0; s < shards; ++s) {
            for (int n = 0; n < N; ++n)
                acc[n] = 0.0;
            for (int k = s * ks; k < (s + 1) * ks; ++k) {
                double hk = oracle_bf16_to_double(h[(size_t)r * K + k]);
                for (int n = 0; n < N; ++n)
                    acc[n] += hk * oracle_bf16_to_double(W[(size_t)k * N + n]);
            }
            for (int n = 0; n < N; ++n) {
                float part = bf16_bits_to_float(oracle_bf16_rne(oracle_fp32_rne(acc[n])));
                sum[n] = sum[n] + part;
            }
        }
        for (int n = 0; n < N; ++n)
            out[(size_t)r * N + n] = oracle_bf16_rne(sum[n]);
    }
    free(sum);
    free(acc);
}

/* ---- a3 + a4: standalone top-k selection with routing weights [P1] ----- */

typedef struct {
    float v;
    int id;
} scored;

/* Total order: larger value first; NaN after every number; equal values
 * (IEEE equality, so -0 == +0) by ascending id.  Ids are unique, so no two
 * entries compare equal and the sort result is unique. */
static int rank_cmp(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    int na = isnan(a->v), nb = isnan(b->v);
    if (na != nb)
        return na ? 1 : -1;
    if (!na) {
        if (a->v > b->v) return -1;
        if (a->v < b->v) return 1;
    }
    return (a->id < b->id) ? -1 : 1;
}

/* For each row of logits [R, E]: sort all E (logit, id) pairs with rank_cmp
 * and keep the first k ids, then
 *   s_i = 1 / (1 + exp(-logit_i)),  w_i = fp32_rne(s_i / sum_j s_j)
 * in double, the sum taken over the k picked experts in rank order. */
void oracle_topk(const float *logits, int R, int E, int k, int32_t *ids, float *weights)
{
    scored *buf = (scored *)malloc(sizeof(scored) * (size_t)E);
    double *s = (double *)malloc(sizeof(double) * (size_t)k);
    for (int r = 0; r < R; ++r) {
        for (int e = 0; e < E; ++e) {
            buf[e].v = logits[(size_t)r * E + e];
            buf[e].id = e;
        }
        qsort(buf, (size_t)E, sizeof(scored), rank_cmp);
        double total = 0.0;
        for (int i = 0; i < k; ++i) {
            ids[(size_t)r * k + i] = buf[i].id;
            s[i] = 1.0 / (1.0 + exp(-(double)buf[i].v));
            total += s[i];
        }
        for (int i = 0; i < k; ++i)
            weights[(size_t)r * k + i] = oracle_fp32_rne(s[i] / total);
    }
    free(s);
    free(buf);
}

/* ---- latent sum of squares per row [P2-Rev] ---------------------------- */

/* ss[r] = fp32_rne( sum_{n < N} v[r, n]^2 ), v = the value of the BF16 bits
 * latent[r, n], summed in float64 with n ascending.  A BF16 value has an
 * 8-bit significand, so its square is exact in double; the running double sum
 * is the only rounding before the final one to FP32. */
void oracle_latent_sumsq(const uint16_t *latent, int R, int N, float *ss)
{
    for (int r = 0; r < R; ++r) {
        double acc = 0.0;
        for (int n = 0; n < N; ++n) {
            double v = oracle_bf16_to_double(latent[(size_t)r * N + n]);
            acc += v * v;
        }
        ss[r] = oracle_fp32_rne(acc);
    }
}
