/*
 * libroute -- the per-MoE-layer route step on one GB300 (sm_103a), C ABI.
 *
 * The route step of one MoE layer, for `rows` token rows:
 *
 *   latent[r, n] = bf16( sum_{k<7168} hidden[r, k] * W_latent[k, n] )   n < 3584
 *   logits[r, e] =       sum_{k<7168} hidden[r, k] * W_router[k, e]    e < 896
 *   ids[r, :]    = the 16 experts with the largest logits, in rank order
 *   weights[r,i] = s_i / sum_j s_j,  s_i = 1 / (1 + exp(-logits[r, ids[r, i]]))
 *
 * Every sum is accumulated in FP32 over the full K = 7168 and rounded once
 * (to BF16 for the latent, kept in FP32 for the logits): "Optionally gather
 * the Kimi3 prefill latent instead of reducing it", Description, Numerics and
 * Compile bullets.  896 experts = 56 router columns x 16 ranks: "Use two row
 * blocks for eight-row Kimi paired gathers", body.  The standalone top-16 and
 * the 1..20-row decode envelope: "Kimi K3.1 recipe: route 9..20 decode rows
 * through the pushed pair gather and standalone top-16", commit message.
 *
 * Conventions for every entry point:
 *  - All tensors are dense, row-major, contiguous, owned by the caller and
 *    resident in device memory of the plan's device (except where a function
 *    says "host").  BF16 tensors are passed as `void*` (IEEE bfloat16 bits).
 *  - Weights are stored [K, N]: W_latent [7168, 3584], W_router [7168, 896],
 *    N contiguous.
 *  - Every device pointer must be 16-byte aligned (TMA and 16-byte vector
 *    accesses); otherwise ROUTE_ERR_ALIGN is returned and nothing is launched.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; no entry point synchronises the device unless it
 *    says so.  Forward calls never allocate and may be captured in a CUDA
 *    graph.
 *  - A plan holds scratch memory (split-K partials or sum-of-squares parts,
 *    and a status word), so one plan must not run on two streams at the same
 *    time.
 *  - Errors are status codes; no C++ exception crosses this interface.
 *    route_last_error() returns a message for the calling thread's last
 *    failure.
 */
#ifndef ROUTE_H
#define ROUTE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ROUTE_K_HIDDEN 7168
#define ROUTE_N_LATENT 3584
#define ROUTE_N_EXPERTS 896
#define ROUTE_TOPK 16
#define ROUTE_DECODE_MAX_ROWS 20
#define ROUTE_PREFILL_MAX_ROWS 65536

typedef enum {
    ROUTE_OK = 0,
    ROUTE_ERR_ROWS = 1,           /* rows outside the mode's envelope */
    ROUTE_ERR_MODE = 2,           /* unknown mode */
    ROUTE_ERR_NULL = 3,           /* a required pointer is NULL */
    ROUTE_ERR_ALIGN = 4,          /* a pointer is not 16-byte aligned */
    ROUTE_ERR_CUDA = 5,           /* a CUDA call failed; see route_last_error() */
    ROUTE_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up waiting and returned */
    ROUTE_ERR_PLAN = 7,           /* the plan cannot run this call */
    ROUTE_ERR_DEVICE = 8,         /* the device is not an sm_103 GPU */
    ROUTE_ERR_DEVICE_BOUNDS = 9   /* (debug library) a kernel computed an index out of
                                     range and skipped that access */
} route_status;

typedef enum {
    ROUTE_DECODE = 0,  /* 1..20 rows: weight streaming with split-K over all SMs */
    ROUTE_PREFILL = 1  /* 1..65536 rows: full-K tensor-core tiles */
} route_mode;

typedef struct route_plan route_plan; /* opaque */

/*
 * route_prepare: validate the row envelope and build a plan on `device`.
 * The plan fixes the launch geometry and the split-K partition (which depend
 * only on the device's SM count, never on the data or on `rows` within the
 * envelope) and owns its scratch memory, allocated here.
 * Decode accepts 1 <= rows <= 20 and rejects anything else with
 * ROUTE_ERR_ROWS before touching the device -- the envelope is checked at
 * preparation, loudly, with no fallback ("Kimi K3.1 recipe ...", commit
 * message: the recipe prepares only 1 to 20 rows and otherwise fails at
 * preparation; Tests: the 21-row envelope rejection).  Prefill accepts
 * 1 <= rows <= 65536.
 * On success *out receives the plan; on failure *out is set to NULL.
 */
route_status route_prepare(int mode, int rows, int device, route_plan **out);

/* route_destroy: free the plan and its scratch memory (synchronises the
 * plan's device).  NULL is accepted and ignored. */
route_status route_destroy(route_plan *plan);

/*
 * latent_router_forward: steps a1 (latent down projection) and a2 (router
 * logits) for the plan's `rows`.
 *   hidden   [rows, 7168] BF16     (read)
 *   W_latent [7168, 3584] BF16     (read)
 *   W_router [7168, 896]  BF16     (read)
 *   latent   [rows, 3584] BF16     (written)  one FP32 full-K sum, rounded once
 *   logits   [rows, 896]  FP32     (written)  FP32 full-K sum
 * Decode plans also use the plan's scratch for split-K partials, which are
 * summed in a fixed order, so results are bitwise reproducible and a row's
 * bits do not depend on `rows`.
 */
route_status latent_router_forward(const route_plan *plan, const void *hidden,
                                   const void *W_latent, const void *W_router, void *latent,
                                   float *logits, void *stream);

/*
 * topk16_select: steps a3 (standalone top-16) and a4 (routing weights).
 *   logits  [rows, 896] FP32 (read)
 *   ids     [rows, 16] int32 (written)  largest logit first; equal logits
 *                                       (-0 == +0) go to the lower expert id;
 *                                       NaN ranks below every number
 *   weights [rows, 16] FP32  (written)  s_i / sum_j s_j, s = sigmoid(logit),
 *                                       in FP32 with compensated (two-float)
 *                                       steps and one final rounding: within
 *                                       5 FP32 ULP of the value in double
 * ("Kimi K3.1 recipe ...", commit message: a standalone top-16 picks each
 * row's experts; the routing-weight formula is this library's convention.)
 */
route_status topk16_select(const route_plan *plan, const float *logits, int32_t *ids,
                           float *weights, void *stream);

/*
 * route_step: the whole route step (a1..a4) for the plan's rows, same
 * arguments and results as latent_router_forward followed by topk16_select.
 * Decode plans run it as two kernels: the weight stream, then one that
 * finishes the split-K sums and runs the top-16 on the router logits it has
 * just summed, without reading them back.
 */
route_status route_step(const route_plan *plan, const void *hidden, const void *W_latent,
                        const void *W_router, void *latent, float *logits, int32_t *ids,
                        float *weights, void *stream);

/*
 * route_step_sumsq: route_step that also writes latent_sumsq [rows] FP32
 * (device, 4-byte aligned, caller-owned): for each row, the sum of the
 * squares of the BF16 latent values this step stores, the per-row statistic
 * the latent's RMS norm needs ("Optionally gather the Kimi3 prefill latent
 * instead of reducing it", Reviewer Notes: an FP32 sum of squares for the
 * latent norm).  The squares are exact in FP32 and are summed as two-floats
 * in a fixed order, then rounded once, so the result is bitwise reproducible.
 * Prefill: the projection's epilogue writes two-float parts of the values it
 * stores and the top-16 kernel adds them; decode: the kernel that finishes
 * the split-K sums runs as one thread-block cluster per row, whose latent
 * CTAs hand their parts to the row's router CTA.  latent, logits, ids and
 * weights are exactly those route_step writes.  NULL latent_sumsq:
 * ROUTE_ERR_NULL.
 */
route_status route_step_sumsq(const route_plan *plan, const void *hidden, const void *W_latent,
                              const void *W_router, void *latent, float *logits, int32_t *ids,
                              float *weights, float *latent_sumsq, void *stream);

/*
 * route_step_host: route_step with the per-step tensors in HOST memory.
 * hidden_host [rows, 7168] BF16 is copied to the device, the step runs, and
 * latent_host, logits_host, ids_host, weights_host receive the results.
 * Weights stay device pointers (they are resident model parameters).  The
 * copies use the plan's device staging buffers (allocated by route_prepare)
 * and are enqueued on `stream`; the call returns after the stream has
 * finished (it synchronises `stream`).  Host pointers need no alignment.
 * Decode plans with every host buffer page-locked and 16-byte aligned skip the
 * copies: a staging kernel reads `hidden_host` through its mapped address and
 * the kernels write the results straight into the host buffers.
 */
route_status route_step_host(const route_plan *plan, const void *hidden_host,
                             const void *W_latent, const void *W_router, void *latent_host,
                             float *logits_host, int32_t *ids_host, float *weights_host,
                             void *stream);

/*
 * route_host_step: route_step_host on fixed buffers, prepared once, for a
 * serving loop that refills the same page-locked `hidden_host` every step and
 * reads the results in place.
 *
 * route_host_step_create takes the arguments of route_step_host.  Decode
 * plans with every host buffer page-locked and 16-byte aligned only (the
 * path that copies nothing); otherwise ROUTE_ERR_PLAN, and the caller uses
 * route_step_host.  A step holds, besides its graph, two device buffers of
 * the hidden rows (2 x rows x 14,336 bytes) and a few device and page-locked
 * words, until route_host_step_destroy or the plan's route_destroy.  The
 * staging, stream and finish kernels are captured once into a CUDA graph (on
 * a stream of the step's own), with a last one-thread kernel that, once they
 * have finished, stores the step's number into a page-locked completion word
 * after a system-scope fence.
 * route_host_step_run is one graph launch on `stream` and a wait (below).
 * route_host_step_launch enqueues the step's kernels one by one on `stream`
 * and returns at once: unlike a graph launch, which starts once everything
 * before it on the stream has finished, they are chained to their
 * predecessor by programmatic dependent launch.  Its staging kernel copies
 * the hidden rows into one of two device buffers of the step's own
 * (alternate launches) and publishes them through a device counter, so that
 * a step launched behind another one streams its weights and reads its rows
 * under the other's tail (it writes the plan's scratch only once the other
 * has finished).
 * route_host_step_wait waits for the number of the step's latest launch in
 * the completion word (not for the stream: the last kernel may still be
 * leaving when it returns) and returns after that launch's results are in
 * the host buffers (at once when no launch is in flight).  Without the
 * number after 4 s it synchronises `stream` and reports its error (or
 * ROUTE_ERR_DEVICE).  Between a step's launch and its wait the caller
 * neither writes its `hidden_host` nor reads its results.  Several steps of
 * one plan may be in flight together (a serving loop with two batches:
 * launch B, wait A, refill A, launch A, wait B, ...) when they were created
 * with the same stream: they share the plan's device scratch, and the
 * stream's order keeps them apart.  A launch or run while another step of
 * the plan, created with another stream, has a launch in flight returns
 * ROUTE_ERR_PLAN and launches nothing.  Both launch forms keep the plan's
 * settings (route_set_latent_ksplit) as they were at creation.  The step
 * belongs to the plan: route_destroy releases its graph and buffers, after
 * which launch, wait and run return ROUTE_ERR_NULL.
 * route_host_step_destroy frees the step (NULL: no-op).  Steps and their
 * plan are not thread-safe.
 */
typedef struct route_host_step route_host_step;

route_status route_host_step_create(route_plan *plan, const void *hidden_host,
                                    const void *W_latent, const void *W_router,
                                    void *latent_host, float *logits_host, int32_t *ids_host,
                                    float *weights_host, void *stream, route_host_step **out);
route_status route_host_step_launch(route_host_step *step);
route_status route_host_step_wait(route_host_step *step);
route_status route_host_step_run(route_host_step *step);
route_status route_host_step_destroy(route_host_step *step);

/*
 * route_device_status: synchronise the plan's device, then report (and clear)
 * the device-side error word that kernels set instead of hanging or
 * faulting: ROUTE_OK, ROUTE_ERR_DEVICE_TIMEOUT (a bounded wait expired) or,
 * in the checked library, ROUTE_ERR_DEVICE_BOUNDS (an index out of range was
 * skipped); the outputs of that launch are invalid.
 */
route_status route_device_status(const route_plan *plan);

/*
 * route_set_overlap: let a plan's projection read `hidden` before the
 * preceding work on the stream has finished.  Every route kernel lets its
 * successor launch early; by default the projection kernels still wait for
 * their predecessor before they read `hidden`.  With enable != 0 they read
 * it at once and wait only before they first write (decode: its scratch;
 * prefill: its outputs), so a decode step's weight stream runs under the
 * previous step's final reduction and top-16, and a prefill GEMM's main loop
 * under the previous step's top-16.  Enable ONLY when `hidden` is never
 * written by the route call issued immediately before on the same stream
 * (it is safe whenever any other kernel or copy produces `hidden`: those do
 * not release their successors early).  route_step_host ignores it.
 * Default: disabled.
 */
route_status route_set_overlap(route_plan *plan, int enable);

/*
 * route_set_latent_ksplit: compute a decode plan's latent with the general
 * (K-split) path's arithmetic instead of one full-K sum: K is cut into eight
 * 896-deep slices, each slice's FP32 partial is rounded to BF16, the eight
 * BF16 partials are summed in FP32 in slice order and the sum is rounded to
 * BF16 again ("Optionally gather the Kimi3 prefill latent instead of reducing
 * it", Description, Numerics bullet and commit body: the path whose numbers
 * existing captured packages were made with).  Logits, ids and weights are
 * unchanged.  Decode plans need their split-K partition to give each CTA
 * exactly one K slice of a latent tile (it does on a 152-SM GB300: 144 CTAs
 * of 14 k-blocks); otherwise ROUTE_ERR_PLAN.  Prefill plans drain and re-start
 * each latent tile's accumulator at every slice boundary (slower: the tensor
 * cores wait for each slice's drain).  Default: disabled (full-K latent).
 */
route_status route_set_latent_ksplit(route_plan *plan, int enable);

/*
 * route_test_stall: TEST HOOK for the bounded-wait path, not for production.
 * With enable != 0, each CTA of the plan's projection kernel skips a copy of
 * its last k-block, so its MMA warp waits for data that never arrives; after
 * timeout_ns the wait gives up, the kernel sets the device status word, drains
 * its in-flight work, frees its tensor memory and returns, and
 * route_device_status() then reports ROUTE_ERR_DEVICE_TIMEOUT.  enable == 0
 * restores normal operation with the default bound (2 s).  Not thread-safe
 * with concurrent use of the plan.
 */
route_status route_test_stall(route_plan *plan, int enable, uint64_t timeout_ns);

/*
 * route_test_poison_scratch: TEST HOOK.  Fill the plan's scratch (decode:
 * the split-K partials; prefill: the latent sum-of-squares parts; column
 * shards keep none: a no-op) with 0xFF bytes on `stream`, so that a test can
 * show that no launch reads scratch it did not write first.  Capturable in a
 * CUDA graph.
 */
route_status route_test_poison_scratch(const route_plan *plan, void *stream);

/*
 * Column shards.  Shard s of W computes, from the full hidden rows, latent
 * columns [3584 s / W, 3584 (s+1) / W) and experts [896 s / W, 896 (s+1) / W)
 * of the layer, and picks its own top-16 of those experts; a merge of the
 * W x 16 candidates finishes the selection.  This is how the step divides
 * over W GPUs with one exchange and no reduction: every rank computes its
 * own latent columns from the full hidden row and the results are gathered
 * ("Optionally gather the Kimi3 prefill latent instead of reducing it",
 * Description: each of 8 ranks computes its own 448 latent columns, then an
 * all-gather), the decode gather pairs each rank's latent and router columns
 * (at TP16, 224 latent and 56 router columns a rank: "Use two row blocks for
 * eight-row Kimi paired gathers", body), and candidate selection and merge
 * are what that page's tests and the first page's tests name.  The exchange
 * itself (an all-gather of the candidates, and of the latent and logit
 * columns where the caller wants them whole) is the caller's collective;
 * this library computes each shard and the merge.  The merged ids and
 * weights are those of the top-16 of the whole logit row the shards computed.
 *
 * route_prepare_shard: a plan for shard `shard` (0 <= shard < num_shards) of
 * `num_shards` W in {1, 2, 4, 7, 8, 14, 16} (W divides 896 experts, with at
 * least 16 experts a shard), for 1 <= rows <= 65536 on `device`.  Up to 20
 * rows it runs the decode weight stream (split-K over the SMs) over the
 * shard's column tiles and a kernel that sums the partials and picks the
 * candidates: the decode path's arithmetic, within the same bounds of the
 * float64 values.  Above 20 rows it runs the prefill kernel over the shard's
 * column tiles, and every result equals the matching columns of route_step
 * on a prefill plan of the same rows (the per-column arithmetic is the
 * same).  Anything else returns ROUTE_ERR_PLAN or ROUTE_ERR_ROWS before
 * touching the device.  A shard plan runs route_shard_step (and the set-up
 * calls route_set_overlap, route_set_latent_ksplit -- above 20 rows only --,
 * route_test_stall, route_device_status); every other step entry point
 * refuses it with ROUTE_ERR_PLAN.
 */
route_status route_prepare_shard(int rows, int device, int shard, int num_shards,
                                 route_plan **out);

/*
 * route_shard_step: steps a1..a3 of one column shard, NL = 3584 / W latent
 * columns and NE = 896 / W experts (device memory, 16-byte aligned):
 *   hidden         [rows, 7168] BF16  (read)   the full hidden rows
 *   W_latent_shard [7168, NL]   BF16  (read)   columns s NL .. of W_latent
 *   W_router_shard [7168, NE]   BF16  (read)   columns s NE .. of W_router
 *   latent_shard   [rows, NL]   BF16  (written)
 *   logits_shard   [rows, NE]   FP32  (written)
 *   cand_ids       [rows, 16]   int32 (written) the shard's top-16, global
 *                                               expert ids (s NE + local id)
 *   cand_logits    [rows, 16]   FP32  (written) their logits
 * Two kernels on `stream`: the projection, then the shard's top-16 (up to
 * 20 rows: the weight stream, then the split-K sums and the top-16).
 */
route_status route_shard_step(const route_plan *plan, const void *hidden,
                              const void *W_latent_shard, const void *W_router_shard,
                              void *latent_shard, float *logits_shard, int32_t *cand_ids,
                              float *cand_logits, void *stream);

/*
 * route_merge_candidates: steps a3 and a4 over the W shards' candidates, on
 * the current device (no plan; one kernel on `stream`):
 *   cand_ids    [W, rows, 16] int32 (read)  shard after shard, as an
 *   cand_logits [W, rows, 16] FP32  (read)  all-gather of route_shard_step's
 *                                           outputs lays them out
 *   ids         [rows, 16]    int32 (written) as topk16_select
 *   weights     [rows, 16]    FP32  (written) as topk16_select
 * rows 1..65536 (ROUTE_ERR_ROWS), W 1..16 (ROUTE_ERR_PLAN), pointers
 * non-NULL and 16-byte aligned.  Candidates must hold distinct ids.
 */
route_status route_merge_candidates(int rows, int num_shards, const int32_t *cand_ids,
                                    const float *cand_logits, int32_t *ids, float *weights,
                                    void *stream);

/*
 * route_step_decode_noalloc: the decode route step (route_step for 1..20
 * rows) without a plan and without allocating any memory.  The pages have no
 * counterpart; this exists for callers that cannot allocate device memory:
 * code running inside a host framework that owns all device memory and hands
 * its plug-ins no allocator, and latency-critical paths where cudaMalloc's
 * device-wide synchronisation is not acceptable.
 *   rows     1..20 (the fixed scratch is sized for 20); anything else returns
 *            ROUTE_ERR_ROWS before touching the device
 *   hidden, W_latent, W_router, latent, logits, ids, weights: as route_step,
 *            device pointers on the CURRENT device, 16-byte aligned
 *   stream   cudaStream_t on the current device
 * Results are the same as route_step's on a plan of the same rows (the same
 * kernels and, on devices with up to 160 SMs, the same split-K partition).
 * Scratch: one file-scope device array per device of about 7.25 MB (partials
 * for 20 rows and up to 160 CTAs, plus a status word), held by every device
 * that loads the library until the process exits.  Every call on a device
 * shares it and it keeps the last call's contents, so calls whose work
 * overlaps on the GPU (other streams, other host threads) race: serialise
 * them, e.g. on one stream.  The first call on a device does a one-time
 * set-up (the array's device address, the kernels' shared-memory limit):
 * make that first call before any stream capture.  A device-side timeout of
 * these calls is read with route_noalloc_status.
 */
route_status route_step_decode_noalloc(int rows, const void *hidden, const void *W_latent,
                                       const void *W_router, void *latent, float *logits,
                                       int32_t *ids, float *weights, void *stream);

/*
 * route_noalloc_status: synchronises `device` and reports whether a kernel of
 * route_step_decode_noalloc on it gave up waiting (ROUTE_ERR_DEVICE_TIMEOUT;
 * the outputs of that call are invalid) since the last query, then clears
 * the fixed array's status word.  ROUTE_OK when nothing failed or no
 * call has run on the device.  device outside 0..63: ROUTE_ERR_DEVICE before
 * any CUDA call.  Allocates nothing.
 */
route_status route_noalloc_status(int device);

/*
 * route_test_noalloc_stall: TEST HOOK, as route_test_stall for the calls of
 * route_step_decode_noalloc on `device` (set up on first use, like a call):
 * with enable != 0 each CTA of the weight stream skips a copy so that its
 * wait gives up after timeout_ns (0: 1 ms) and route_noalloc_status reports
 * ROUTE_ERR_DEVICE_TIMEOUT; enable == 0 restores the default bound (2 s).
 * device outside 0..63: ROUTE_ERR_DEVICE.  Not for concurrent use with calls
 * on the device.
 */
route_status route_test_noalloc_stall(int device, int enable, uint64_t timeout_ns);

/*
 * route_noalloc_grid: the CTA count route_step_decode_noalloc's weight stream
 * uses on `device` (a function of its SM count, capped at 160); the same as
 * route_plan_grid of a decode plan on devices with up to 160 SMs.  -1 when
 * the device cannot be queried.
 */
int route_noalloc_grid(int device);

/* Plan properties: rows, mode, launch grid (CTAs), split-K segments (decode)
 * or tiles (prefill), and the latent columns and experts the plan computes
 * (3584 and 896, or a column shard's share).  -1 for a NULL plan. */
int route_plan_rows(const route_plan *plan);
int route_plan_mode(const route_plan *plan);
int route_plan_grid(const route_plan *plan);
int route_plan_segments(const route_plan *plan);
int route_plan_latent_cols(const route_plan *plan);
int route_plan_experts(const route_plan *plan);

/* Message for the calling thread's most recent failure ("" if none). */
const char *route_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ROUTE_H */
