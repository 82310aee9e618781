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
#include <cuda_bf16.h>

#include "common.cuh"
#include "topk16.cuh"
#include "twofloat.cuh"

namespace route {
namespace {

constexpr int kRowsPerBlock = 8;

// Lane l adds parts l, l + 32, ... in order, then a fixed tree over the lanes.
__device__ __forceinline__ float row_sumsq_from_parts(const float2 *parts, int lane) {
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int j = lane; j < kSsParts; j += 32) {
        const float2 p = __ldcg(parts + j);
        two_sum_acc(hi, lo, p.x);
        lo += p.y;
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
    topk16_warp(logits + (size_t)row * kExperts, ids + (size_t)row * kTopK,
                weights + (size_t)row * kTopK, lane, cand[warp]);
    if (sumsq != nullptr) {
        const float ss = row_sumsq_from_parts(ss_part + (size_t)row * kSsParts, lane);
        if (lane == 0) sumsq[row] = ss;
    }
}

}  // namespace

cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        const float2 *ss_part, float *sumsq, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    c.blockDim = dim3(32 * kRowsPerBlock);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, topk16_kernel, logits, rows, ids, weights, ss_part, sumsq);
}

}  // namespace route
