/* A plain C program on the route library's C ABI alone (no Python, no
 * PyTorch): device buffers from the CUDA runtime, one decode step (8 rows)
 * and one prefill step (264 rows: two 256-row blocks, the second ragged)
 * through route_prepare / route_step / route_destroy, the results checked
 * against the oracle (float64 C, linked
 * from oracle/route_oracle.c; test code only):
 *   - ids equal the oracle's top-16 of the library's own logits, weights
 *     within 5 FP32 ULP of the oracle's;
 *   - latent relative RMS error against the float64 sums <= 2e-3;
 *   - |logit - float64 sum| <= 2^-19 * sum_k |h * w| for every logit.
 * Then two decode host steps of one plan on page-locked buffers, in flight
 * together (route_host_step_launch / route_host_step_wait) on two inputs,
 * each result equal bit for bit to route_step's on device buffers.
 * Inputs: a fixed 64-bit LCG, hidden ~ uniform(-1.7, 1.7) (about unit
 * variance), weights ~ uniform scaled to variance 1/7168, rounded to BF16.
 * Exit status 0 when every check passes. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "route.h"

/* oracle/route_oracle.c */
void oracle_latent_router(const uint16_t *h, const uint16_t *Wl, const uint16_t *Wr, int R, int K,
                          int NL, int NR, uint16_t *latent, float *logits, double *y_lat,
                          double *y_log);
void oracle_topk(const float *logits, int R, int E, int k, int32_t *ids, float *weights);
double oracle_bf16_to_double(uint16_t b);

enum { K = 7168, NL = 3584, NE = 896, TOPK = 16 };

static uint64_t g_state = 0x9E3779B97F4A7C15ull;
static double *g_abs_wr; /* |W_router| as doubles, [K][NE] */

static double uniform(void) { /* [0, 1) */
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(g_state >> 11) * (1.0 / 9007199254740992.0);
}

static uint16_t to_bf16(float f) { /* round to nearest even; inputs are finite */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static void fill(uint16_t *x, size_t n, double scale) {
    for (size_t i = 0; i < n; ++i) x[i] = to_bf16((float)((2.0 * uniform() - 1.0) * scale));
}

static int32_t ulp_distance(float a, float b) {
    int32_t ia, ib;
    memcpy(&ia, &a, 4);
    memcpy(&ib, &b, 4);
    if (ia < 0) ia = (int32_t)0x80000000 - ia;
    if (ib < 0) ib = (int32_t)0x80000000 - ib;
    return ia > ib ? ia - ib : ib - ia;
}

#define CUDA_OK(call)                                                                    \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                 \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

static int run_case(int mode, int R, const uint16_t *wl, const uint16_t *wr,
                    void *d_wl, void *d_wr) {
    const char *name = mode == ROUTE_DECODE ? "decode" : "prefill";
    uint16_t *h = malloc(sizeof(uint16_t) * (size_t)R * K);
    uint16_t *lat = malloc(sizeof(uint16_t) * (size_t)R * NL);
    uint16_t *lat_ref = malloc(sizeof(uint16_t) * (size_t)R * NL);
    float *lg = malloc(sizeof(float) * (size_t)R * NE), *lg_ref = malloc(sizeof(float) * (size_t)R * NE);
    double *y_lat = malloc(sizeof(double) * (size_t)R * NL), *y_log = malloc(sizeof(double) * (size_t)R * NE);
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)R * TOPK), *ids_ref = malloc(sizeof(int32_t) * (size_t)R * TOPK);
    float *w = malloc(sizeof(float) * (size_t)R * TOPK), *w_ref = malloc(sizeof(float) * (size_t)R * TOPK);
    fill(h, (size_t)R * K, 1.7320508);

    void *d_h, *d_lat, *d_lg, *d_ids, *d_w;
    CUDA_OK(cudaMalloc(&d_h, sizeof(uint16_t) * (size_t)R * K));
    CUDA_OK(cudaMalloc(&d_lat, sizeof(uint16_t) * (size_t)R * NL));
    CUDA_OK(cudaMalloc(&d_lg, sizeof(float) * (size_t)R * NE));
    CUDA_OK(cudaMalloc(&d_ids, sizeof(int32_t) * (size_t)R * TOPK));
    CUDA_OK(cudaMalloc(&d_w, sizeof(float) * (size_t)R * TOPK));
    CUDA_OK(cudaMemcpy(d_h, h, sizeof(uint16_t) * (size_t)R * K, cudaMemcpyHostToDevice));

    route_plan *plan = NULL;
    route_status st = route_prepare(mode, R, 0, &plan);
    if (st == ROUTE_OK)
        st = route_step(plan, d_h, d_wl, d_wr, d_lat, (float *)d_lg, (int32_t *)d_ids, (float *)d_w,
                        NULL);
    if (st == ROUTE_OK) CUDA_OK(cudaDeviceSynchronize());
    if (st == ROUTE_OK) st = route_device_status(plan);
    if (st != ROUTE_OK) {
        fprintf(stderr, "%s: status %d: %s\n", name, (int)st, route_last_error());
        return 1;
    }
    route_destroy(plan);
    CUDA_OK(cudaMemcpy(lat, d_lat, sizeof(uint16_t) * (size_t)R * NL, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(lg, d_lg, sizeof(float) * (size_t)R * NE, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(ids, d_ids, sizeof(int32_t) * (size_t)R * TOPK, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(w, d_w, sizeof(float) * (size_t)R * TOPK, cudaMemcpyDeviceToHost));

    oracle_latent_router(h, wl, wr, R, K, NL, NE, lat_ref, lg_ref, y_lat, y_log);
    oracle_topk(lg, R, NE, TOPK, ids_ref, w_ref);

    int bad = 0;
    double num = 0.0, den = 0.0;
    for (size_t i = 0; i < (size_t)R * NL; ++i) {
        const double d = oracle_bf16_to_double(lat[i]) - y_lat[i];
        num += d * d;
        den += y_lat[i] * y_lat[i];
    }
    const double rel = sqrt(num / den);
    if (!(rel <= 2e-3)) {
        fprintf(stderr, "%s: latent relative RMS %.3e > 2e-3\n", name, rel);
        bad = 1;
    }
    /* sum_k |h * w| per logit, from |h| and |W_router| as doubles */
    double *ah = malloc(sizeof(double) * K), *sabs = malloc(sizeof(double) * NE);
    for (int r = 0; r < R && !bad; ++r) {
        for (int k = 0; k < K; ++k) ah[k] = fabs(oracle_bf16_to_double(h[(size_t)r * K + k]));
        for (int e = 0; e < NE; ++e) sabs[e] = 0.0;
        for (int k = 0; k < K; ++k)
            for (int e = 0; e < NE; ++e) sabs[e] += ah[k] * g_abs_wr[(size_t)k * NE + e];
        for (int e = 0; e < NE; ++e) {
            const double err = fabs((double)lg[(size_t)r * NE + e] - y_log[(size_t)r * NE + e]);
            if (!(err <= ldexp(sabs[e], -19))) {
                fprintf(stderr, "%s: logit (%d, %d) off by %.3e\n", name, r, e, err);
                bad = 1;
                break;
            }
        }
    }
    free(ah);
    free(sabs);
    for (size_t i = 0; i < (size_t)R * TOPK && !bad; ++i) {
        if (ids[i] != ids_ref[i] || ulp_distance(w[i], w_ref[i]) > 5) {
            fprintf(stderr, "%s: top-16 entry %zu: id %d vs %d, weight %.9g vs %.9g\n", name, i,
                    ids[i], ids_ref[i], w[i], w_ref[i]);
            bad = 1;
        }
    }
    if (!bad) printf("%s %d rows: ok (latent relative RMS %.3e)\n", name, R, rel);
    cudaFree(d_h);
    cudaFree(d_lat);
    cudaFree(d_lg);
    cudaFree(d_ids);
    cudaFree(d_w);
    free(h); free(lat); free(lat_ref); free(lg); free(lg_ref); free(y_lat); free(y_log);
    free(ids); free(ids_ref); free(w); free(w_ref);
    return bad;
}

/* route_step on device buffers: the results copied back into `out`
 * (latent, logits, ids, weights, packed in that order). */
static int device_step(route_plan *plan, const uint16_t *h, int R, void *d_wl, void *d_wr,
                       uint8_t *out) {
    const size_t nh = sizeof(uint16_t) * (size_t)R * K, nl = sizeof(uint16_t) * (size_t)R * NL,
                 ng = sizeof(float) * (size_t)R * NE, nk = sizeof(int32_t) * (size_t)R * TOPK;
    void *d_h, *d_out;
    CUDA_OK(cudaMalloc(&d_h, nh));
    CUDA_OK(cudaMalloc(&d_out, nl + ng + 2 * nk));
    CUDA_OK(cudaMemcpy(d_h, h, nh, cudaMemcpyHostToDevice));
    uint8_t *o = d_out;
    route_status st = route_step(plan, d_h, d_wl, d_wr, o, (float *)(o + nl), (int32_t *)(o + nl + ng),
                                 (float *)(o + nl + ng + nk), NULL);
    if (st == ROUTE_OK) CUDA_OK(cudaDeviceSynchronize());
    if (st == ROUTE_OK) st = route_device_status(plan);
    if (st != ROUTE_OK) {
        fprintf(stderr, "route_step: status %d: %s\n", (int)st, route_last_error());
        return 1;
    }
    CUDA_OK(cudaMemcpy(out, d_out, nl + ng + 2 * nk, cudaMemcpyDeviceToHost));
    cudaFree(d_h);
    cudaFree(d_out);
    return 0;
}

/* Two host steps of one decode plan in flight together: launch A, launch B,
 * wait A, check A, refill A, launch A, wait B, check B, wait A, check A. */
static int run_host_steps(void *d_wl, void *d_wr) {
    enum { R = 8 };
    const size_t nh = sizeof(uint16_t) * (size_t)R * K, nl = sizeof(uint16_t) * (size_t)R * NL,
                 ng = sizeof(float) * (size_t)R * NE, nk = sizeof(int32_t) * (size_t)R * TOPK,
                 nout = nl + ng + 2 * nk;
    uint16_t *h[2];
    uint8_t *want[2];
    route_plan *plan = NULL;
    route_status st = route_prepare(ROUTE_DECODE, R, 0, &plan);
    if (st != ROUTE_OK) {
        fprintf(stderr, "host steps: prepare: %s\n", route_last_error());
        return 1;
    }
    for (int i = 0; i < 2; ++i) {
        h[i] = malloc(nh);
        want[i] = malloc(nout);
        fill(h[i], (size_t)R * K, 1.7320508);
        if (device_step(plan, h[i], R, d_wl, d_wr, want[i])) return 1;
    }
    cudaStream_t s;
    CUDA_OK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    uint16_t *hh[2];
    uint8_t *out[2];
    route_host_step *step[2];
    for (int j = 0; j < 2; ++j) {
        CUDA_OK(cudaHostAlloc((void **)&hh[j], nh, cudaHostAllocDefault));
        CUDA_OK(cudaHostAlloc((void **)&out[j], nout, cudaHostAllocDefault));
        uint8_t *o = out[j];
        st = route_host_step_create(plan, hh[j], d_wl, d_wr, o, (float *)(o + nl),
                                    (int32_t *)(o + nl + ng), (float *)(o + nl + ng + nk), s,
                                    &step[j]);
        if (st != ROUTE_OK) {
            fprintf(stderr, "host steps: create: %s\n", route_last_error());
            return 1;
        }
    }
    /* launch A(0), launch B(1); wait A, check, A(1); wait B, check, B(0);
     * wait A, check; wait B, check */
    int in[2] = {0, 1}, bad = 0;
    memcpy(hh[0], h[0], nh);
    memcpy(hh[1], h[1], nh);
    st = route_host_step_launch(step[0]);
    if (st == ROUTE_OK) st = route_host_step_launch(step[1]);
    for (int k = 0; k < 4 && st == ROUTE_OK; ++k) {
        const int j = k % 2;
        if ((st = route_host_step_wait(step[j])) != ROUTE_OK) break;
        if (memcmp(out[j], want[in[j]], nout) != 0) {
            fprintf(stderr, "host steps: wait %d (step %d, input %d) differs from route_step\n", k,
                    j, in[j]);
            bad = 1;
            break;
        }
        if (k < 2) { /* the other input, launched behind the step still in flight */
            in[j] = 1 - in[j];
            memcpy(hh[j], h[in[j]], nh);
            memset(out[j], 0xFF, nout);
            st = route_host_step_launch(step[j]);
        }
    }
    if (st != ROUTE_OK) {
        fprintf(stderr, "host steps: status %d: %s\n", (int)st, route_last_error());
        bad = 1;
    }
    for (int j = 0; j < 2; ++j) {
        route_host_step_destroy(step[j]);
        cudaFreeHost(hh[j]);
        cudaFreeHost(out[j]);
        free(h[j]);
        free(want[j]);
    }
    route_destroy(plan);
    cudaStreamDestroy(s);
    if (!bad) printf("host steps, two in flight: ok\n");
    return bad;
}

int main(void) {
    uint16_t *wl = malloc(sizeof(uint16_t) * (size_t)K * NL);
    uint16_t *wr = malloc(sizeof(uint16_t) * (size_t)K * NE);
    const double s = sqrt(3.0 / K); /* uniform(-s, s): variance 1/7168 */
    fill(wl, (size_t)K * NL, s);
    fill(wr, (size_t)K * NE, s);
    g_abs_wr = malloc(sizeof(double) * (size_t)K * NE);
    for (size_t i = 0; i < (size_t)K * NE; ++i) g_abs_wr[i] = fabs(oracle_bf16_to_double(wr[i]));
    void *d_wl, *d_wr;
    CUDA_OK(cudaMalloc(&d_wl, sizeof(uint16_t) * (size_t)K * NL));
    CUDA_OK(cudaMalloc(&d_wr, sizeof(uint16_t) * (size_t)K * NE));
    CUDA_OK(cudaMemcpy(d_wl, wl, sizeof(uint16_t) * (size_t)K * NL, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_wr, wr, sizeof(uint16_t) * (size_t)K * NE, cudaMemcpyHostToDevice));
    int bad = run_case(ROUTE_DECODE, 8, wl, wr, d_wl, d_wr);
    bad |= run_case(ROUTE_PREFILL, 264, wl, wr, d_wl, d_wr);  /* two row blocks, ragged */
    bad |= run_host_steps(d_wl, d_wr);
    cudaFree(d_wl);
    cudaFree(d_wr);
    free(wl);
    free(wr);
    free(g_abs_wr);
    return bad;
}
