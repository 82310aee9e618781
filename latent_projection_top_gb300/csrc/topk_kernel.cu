// Standalone top-16 kernel: one warp per token row (steps a3 and a4 of the
// route step; the selection itself lives in topk16.cuh and is shared with the
// decode finish kernel).  Launched with programmatic dependent launch: it
// waits for the logits' producer before reading them.
//
// Optionally the same warp also reduces its row of the latent to the FP32 sum
// of squares a following norm needs ("Optionally gather the Kimi3 prefill
// latent instead of reducing it", Reviewer Notes): the squares of the BF16
// values the projection stored (exact in FP32) are summed as two-floats in a
// fixed order and rounded once.
#include <cuda_bf16.h>

#include "common.cuh"
#include "topk16.cuh"
#include "twofloat.cuh"

namespace route {
namespace {

constexpr int kRowsPerBlock = 8;

// Sum of squares of one latent row (3584 BF16 values) by one warp: lane l
// takes the 16-byte groups l, l + 32, ... in order into four two-float
// accumulators (one per 32-bit word of a group, so that four independent
// chains run at once), adds them in order, then a fixed tree over the lanes.
__device__ __forceinline__ float latent_row_sumsq(const uint16_t *row, int lane) {
    const uint4 *v = reinterpret_cast<const uint4 *>(row);
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int j = lane; j < kLatent / 8; j += 32) {
        const uint4 q = __ldcg(v + j);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = __uint_as_float(w[e] << 16);          // low BF16 of the word
            const float b = __uint_as_float(w[e] & 0xFFFF0000u);  // high BF16
            two_sum_acc(hi[e], lo[e], a * a);
            two_sum_acc(hi[e], lo[e], b * b);
        }
    }
#pragma unroll
    for (int e = 1; e < 4; ++e) {
        two_sum_acc(hi[0], lo[0], hi[e]);
        lo[0] += lo[e];
    }
    warp_two_sum(hi[0], lo[0]);
    return two_float_value(hi[0], lo[0]);
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    topk16_kernel(const float *__restrict__ logits, int rows, int32_t *__restrict__ ids,
                  float *__restrict__ weights, const uint16_t *__restrict__ latent,
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
        const float ss = latent_row_sumsq(latent + (size_t)row * kLatent, lane);
        if (lane == 0) sumsq[row] = ss;
    }
}

}  // namespace

cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        const uint16_t *latent, float *sumsq, cudaStream_t stream) {
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
    return cudaLaunchKernelEx(&c, topk16_kernel, logits, rows, ids, weights, latent, sumsq);
}

}  // namespace route
