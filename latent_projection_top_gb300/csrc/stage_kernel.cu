// Copy of one step's hidden rows from page-locked host memory (read by the
// GPU over its host link through the mapped address) into the plan's device
// staging buffer, for route_step_host.  Launched with programmatic dependent
// launch like the route kernels: it lets the next kernel launch at once (the
// decode stream kernel then prefetches its weights while this copy runs) and
// writes the staging buffer only after its own predecessor has completed.
#include "common.cuh"

namespace route {
namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
    stage_in_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the staging buffer's last reader is done
    for (int i = blockIdx.x * kStageThreads + threadIdx.x; i < n16; i += gridDim.x * kStageThreads)
        dst[i] = src[i];
}

}  // namespace

cudaError_t stage_in_launch(const void *src_mapped, void *dst, size_t bytes, cudaStream_t stream) {
    if (bytes == 0 || bytes % 16 != 0) return cudaErrorInvalidValue;
    const int n16 = (int)(bytes / 16);
    int grid = (n16 + kStageThreads - 1) / kStageThreads;
    if (grid > 64) grid = 64;
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3(grid);
    c.blockDim = dim3(kStageThreads);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, stage_in_kernel, static_cast<const uint4 *>(src_mapped),
                              static_cast<uint4 *>(dst), n16);
}

}  // namespace route
