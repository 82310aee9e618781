// Standalone top-16 kernel: one warp per token row (steps a3 and a4 of the
// route step; the selection itself lives in topk16.cuh and is shared with the
// fused decode tail of the projection kernel).
#include "common.cuh"
#include "topk16.cuh"

namespace route {
namespace {

constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    topk16_kernel(const float *__restrict__ logits, int rows, int32_t *__restrict__ ids,
                  float *__restrict__ weights) {
    __shared__ uint2 cand[kRowsPerBlock][kCandMax];
    const int warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= rows) return;  // whole warps leave together
    topk16_warp(logits + (size_t)row * kExperts, ids + (size_t)row * kTopK,
                weights + (size_t)row * kTopK, threadIdx.x & 31, cand[warp]);
}

}  // namespace

cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    topk16_kernel<<<blocks, 32 * kRowsPerBlock, 0, stream>>>(logits, rows, ids, weights);
    return cudaGetLastError();
}

}  // namespace route
