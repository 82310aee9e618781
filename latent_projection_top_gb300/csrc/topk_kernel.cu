// Standalone top-16 kernel: one warp per token row (steps a3 and a4 of the
// route step; the selection itself lives in topk16.cuh and is shared with the
// decode finish kernel).  Launched with programmatic dependent launch: it
// waits for the logits' producer before reading them.
#include "common.cuh"
#include "topk16.cuh"

namespace route {
namespace {

constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    topk16_kernel(const float *__restrict__ logits, int rows, int32_t *__restrict__ ids,
                  float *__restrict__ weights) {
    __shared__ uint2 cand[kRowsPerBlock][kCandMax];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the logits' producer has finished
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
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    c.blockDim = dim3(32 * kRowsPerBlock);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, topk16_kernel, logits, rows, ids, weights);
}

}  // namespace route
