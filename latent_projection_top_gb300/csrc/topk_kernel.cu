// Standalone top-16 kernel: one warp per token row (steps a3 and a4 of the
// route step; the selection itself lives in topk16.cuh and is shared with the
// decode finish kernel).  Launched with programmatic dependent launch: it
// waits for the logits' producer before reading them.
//
// Optionally the same warp also adds up its row's latent sum-of-squares
// parts into the FP32 statistic a following norm needs ("Optionally gather
// the Kimi3 prefill latent instead of reducing it", Reviewer Notes): the
// projection's epilogue left one two-float part per 32 latent columns (the
// squares of the BF16 values it stored, exact in FP32); the parts are summed
// as two-floats in a fixed order and rounded once.
//
// Column shards.  A shard that owns a range of experts picks its own top-16
// of that range (global ids, with their logits); once every shard's
// candidates are in one place, the merge ranks the W x 16 of them with the
// same keys and computes the weights.  The top 16 of a row lie among its
// shards' local top 16s, so the merged result equals the top-16 of the
// whole logit row.  The pages shard the latent by output column, each rank
// computing its own columns from the full hidden row, and gather the results
// ("Optionally gather the Kimi3 prefill latent instead of reducing it",
// Description); the decode gather pairs each rank's latent and router
// columns ("Use two row blocks for eight-row Kimi paired gathers", body);
// candidate selection and merge are named by that page's tests and the
// first's.
#include <cuda_bf16.h>

#include "common.cuh"
#include "topk16.cuh"
#include "twofloat.cuh"

namespace route {
namespace {

constexpr int kRowsPerBlock = 8;

// A row's sum-of-squares parts in two steps, so that their loads overlap the
// top-16's: lane l loads parts l, l + 32, ... (row_parts_load), then adds
// them in that order and a fixed tree joins the lanes (row_parts_sum).
constexpr int kPartsPerLane = (kSsParts + 31) / 32;  // 4

__device__ __forceinline__ void row_parts_load(const float2 *parts, int lane,
                                               float2 (&p)[kPartsPerLane]) {
#pragma unroll
    for (int j = 0; j < kPartsPerLane; ++j)
        p[j] = lane + 32 * j < kSsParts ? __ldcg(parts + lane + 32 * j) : make_float2(0.f, 0.f);
}

__device__ __forceinline__ float row_parts_sum(const float2 (&p)[kPartsPerLane], int lane) {
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int j = 0; j < kPartsPerLane; ++j)
        if (lane + 32 * j < kSsParts) {
            two_sum_acc(hi, lo, p[j].x);
            lo += p[j].y;
        }
    warp_two_sum(hi, lo);
    return two_float_value(hi, lo);
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    topk16_kernel(const float *__restrict__ logits, int rows, int32_t *__restrict__ ids,
                  float *__restrict__ weights, const float2 *__restrict__ ss_part,
                  float *__restrict__ sumsq) {
    __shared__ uint2 cand[kRowsPerBlock][kCandMax];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the logits' producer has finished
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= rows) return;  // whole warps leave together
    float2 parts[kPartsPerLane];
    if (sumsq != nullptr) row_parts_load(ss_part + (size_t)row * kSsParts, lane, parts);
    topk16_warp(logits + (size_t)row * kExperts, ids + (size_t)row * kTopK,
                weights + (size_t)row * kTopK, lane, cand[warp]);
    if (sumsq != nullptr) {
        const float ss = row_parts_sum(parts, lane);
        if (lane == 0) sumsq[row] = ss;
    }
}

// A column shard's local top-16, one warp per row: global ids and the
// picks' logits (the candidates route_merge_candidates ranks).
// (80 registers at most: under __launch_bounds__ alone it compiled to 64 with
// a spilled word)
__global__ void __maxnreg__(80)
    shard_topk16_kernel(const float *__restrict__ logits, int rows, int n, int id_base,
                        int32_t *__restrict__ cand_ids, float *__restrict__ cand_logits) {
    __shared__ uint2 cand[kRowsPerBlock][kCandMax];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the logits' producer has finished
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= rows) return;
    uint32_t key, id;
    topk16_warp_picks(logits + (size_t)row * n, n, lane, cand[warp], key, id);
    if (lane < kTopK) {
        cand_ids[(size_t)row * kTopK + lane] = id_base + (int32_t)id;
        cand_logits[(size_t)row * kTopK + lane] = key_to_float(key);
    }
}

// The top-16 over num_shards x 16 candidates of each row, one warp per row:
// every candidate's rank among all of them (larger logit first, the lower
// expert id on equal logits; the same keys as the top-16) by counting, the
// ranks 0..15 in order, then the routing weights of those 16.
constexpr int kMergeMax = kMaxShards * kTopK;  // 256

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    merge_kernel(const int32_t *__restrict__ cand_ids, const float *__restrict__ cand_logits, int rows,
                 int num_shards, int32_t *__restrict__ ids, float *__restrict__ weights) {
    __shared__ uint2 cand[kRowsPerBlock][kMergeMax];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the candidates' producers have finished
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= rows) return;
    const int total = num_shards * kTopK;
    uint2 *c = cand[warp];
    for (int i = lane; i < total; i += 32) {
        const int s = i / kTopK, j = i % kTopK;
        const size_t at = ((size_t)s * rows + row) * kTopK + j;
        c[i] = make_uint2(rank_key(cand_logits[at]), (uint32_t)cand_ids[at]);
    }
    __syncwarp();
    uint2 mine[kMergeMax / 32];
    uint32_t rank[kMergeMax / 32];
#pragma unroll
    for (int q = 0; q < kMergeMax / 32; ++q) {
        const int i = lane + 32 * q;
        mine[q] = i < total ? c[i] : make_uint2(0u, 0xFFFFFFFFu);
        rank[q] = 0u;
    }
    for (int j = 0; j < total; ++j) {
        const uint2 o = c[j];
#pragma unroll
        for (int q = 0; q < kMergeMax / 32; ++q)
            rank[q] += (o.x > mine[q].x || (o.x == mine[q].x && o.y < mine[q].y)) ? 1u : 0u;
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < kMergeMax / 32; ++q)
        if (lane + 32 * q < total && rank[q] < (uint32_t)kTopK) c[rank[q]] = mine[q];
    __syncwarp();
    uint32_t key = 0u, id = 0u;
    if (lane < kTopK) {
        key = c[lane].x;
        id = c[lane].y;
    }
    __syncwarp();
    weights16_store(key, id, lane, ids + (size_t)row * kTopK, weights + (size_t)row * kTopK);
}

// One warp per row, rows in blocks of kRowsPerBlock; launched as a
// programmatic dependent of the previous kernel on the stream.
cudaLaunchConfig_t row_warps_config(int rows, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    c.blockDim = dim3(32 * kRowsPerBlock);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return c;
}

}  // namespace

cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        const float2 *ss_part, float *sumsq, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_warps_config(rows, stream, attr);
    return cudaLaunchKernelEx(&c, topk16_kernel, logits, rows, ids, weights, ss_part, sumsq);
}

cudaError_t shard_topk_launch(const float *logits, int rows, int n, int id_base, int32_t *cand_ids,
                              float *cand_logits, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    if (n < kTopK || n > kExpertsTopk) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_warps_config(rows, stream, attr);
    return cudaLaunchKernelEx(&c, shard_topk16_kernel, logits, rows, n, id_base, cand_ids, cand_logits);
}

cudaError_t merge_launch(const int32_t *cand_ids, const float *cand_logits, int rows,
                         int num_shards, int32_t *ids, float *weights, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    if (num_shards < 1 || num_shards > kMaxShards) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_warps_config(rows, stream, attr);
    return cudaLaunchKernelEx(&c, merge_kernel, cand_ids, cand_logits, rows, num_shards, ids, weights);
}

}  // namespace route
