/*
 * Seeded synthetic inputs for the route step (hidden rows and weight banks).
 *
 * This module draws random numbers and shapes them into BF16 inputs.  It
 * holds none of the route step's own arithmetic (no projection, no top-k) and
 * serves both the oracle side and the CUDA side with the same bytes.
 *
 * Random stream: the splitmix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", 2014) applied to a
 * counter.  Draw i of the stream keyed by (seed, bank, tensor) is
 *     mix64(key + (i + 1) * 0x9E3779B97F4A7C15),
 *     key = mix64(mix64(mix64(seed) ^ bank) ^ tensor),
 * so any element can be produced independently and the result does not
 * depend on how the work is split across threads.
 *
 * Normals: Box-Muller on draws 2j and 2j+1 (53-bit uniforms u1 in (0, 1],
 * u2 in [0, 1)); element 2j takes the cosine branch and 2j+1 the sine branch.
 * A value is scaled in double, rounded to FP32 and then to BF16 (both ties to
 * even).  Host libm log/sin/cos may differ in the last bit between host
 * architectures; every consumer generates its inputs on the machine it runs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t bank, uint64_t tensor)
{
    return mix64(mix64(mix64(seed) ^ bank) ^ tensor);
}

uint64_t synth_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static inline double normal_at(uint64_t key, uint64_t i)
{
    uint64_t j = i >> 1;
    uint64_t a = synth_draw(key, 2 * j);
    uint64_t b = synth_draw(key, 2 * j + 1);
    double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586 * u2;
    return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

static inline uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ---- threaded fill ------------------------------------------------------ */

typedef struct {
    uint64_t key;
    uint64_t begin, end;
    double sigma;
    uint16_t *out16;
    double *out64;
} fill_job;

static void *fill_worker(void *p)
{
    fill_job *j = (fill_job *)p;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        double z = normal_at(j->key, i);
        if (j->out16)
            j->out16[i] = to_bf16(j->sigma * z);
        else
            j->out64[i] = j->sigma * z;
    }
    return NULL;
}

static void fill(uint64_t key, uint64_t count, double sigma, uint16_t *out16, double *out64,
                 int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((uint64_t)threads > count / 65536 + 1) threads = (int)(count / 65536 + 1);
    pthread_t tid[256];
    fill_job job[256];
    for (int t = 0; t < threads; ++t) {
        job[t].key = key;
        job[t].begin = count * (uint64_t)t / (uint64_t)threads;
        job[t].end = count * (uint64_t)(t + 1) / (uint64_t)threads;
        job[t].sigma = sigma;
        job[t].out16 = out16;
        job[t].out64 = out64;
    }
    int started = 0;
    for (int t = 1; t < threads; ++t)
        if (pthread_create(&tid[t], NULL, fill_worker, &job[t]) == 0)
            started = t;
        else
            break;
    fill_worker(&job[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
    for (int t = started + 1; t < threads; ++t) /* threads that failed to start */
        fill_worker(&job[t]);
}

/* out[i] = bf16(sigma * N(0,1)_i), i < count. */
void synth_normal_bf16(uint64_t key, uint64_t count, double sigma, uint16_t *out, int threads)
{
    fill(key, count, sigma, out, NULL, threads);
}

/* out[i] = sigma * N(0,1)_i in double. */
void synth_normal_f64(uint64_t key, uint64_t count, double sigma, double *out, int threads)
{
    fill(key, count, sigma, NULL, out, threads);
}

/* Hidden rows with per-row unit RMS: row r is z[r, :] / sqrt(mean(z[r, :]^2))
 * with z ~ N(0, 1) from the stream, then rounded to BF16. */
void synth_hidden_rms_bf16(uint64_t key, int rows, int K, uint16_t *out, int threads)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)rows * K);
    fill(key, (uint64_t)rows * K, 1.0, NULL, z, threads);
    for (int r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int k = 0; k < K; ++k)
            ss += z[(size_t)r * K + k] * z[(size_t)r * K + k];
        double inv = 1.0 / sqrt(ss / K);
        for (int k = 0; k < K; ++k)
            out[(size_t)r * K + k] = to_bf16(z[(size_t)r * K + k] * inv);
    }
    free(z);
}

/* Cancel group: for columns n < ncols of a [K, N] weight, the sign of each
 * entry is replaced so that row d = n mod rows of `hidden` sees K-slices of
 * `slice` entries with alternating sign:
 *     W[k, n] = (-1)^(k / slice) * sign(h[d, k]) * |W[k, n]|
 * (sign(0) taken as +).  Only sign bits change; magnitudes stay the drawn
 * ones. */
void synth_cancel_group(uint16_t *W, int K, int N, int ncols, const uint16_t *hidden,
                        int rows, int slice)
{
    for (int k = 0; k < K; ++k) {
        int neg_slice = (k / slice) & 1;
        for (int n = 0; n < ncols; ++n) {
            int d = n % rows;
            int neg_h = (hidden[(size_t)d * K + k] >> 15) & 1;
            uint16_t mag = W[(size_t)k * N + n] & 0x7FFFu;
            W[(size_t)k * N + n] = (uint16_t)(mag | ((neg_slice ^ neg_h) ? 0x8000u : 0u));
        }
    }
}
