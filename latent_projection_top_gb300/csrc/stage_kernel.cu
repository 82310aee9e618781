// Copy of one step's hidden rows from page-locked host memory (read by the
// GPU over its host link through the mapped address) into the plan's device
// staging buffer, for route_step_host and a host step's graph, and the
// completion kernel of a host step.  Launched with programmatic dependent
// launch like the route kernels: it lets the next kernel launch at once (the
// decode stream kernel then prefetches its weights while this copy runs) and
// writes the staging buffer only after its own predecessor has completed.
// The host rows are written by the caller before the launch, so they are
// read before that wait: the host link's latency passes under it.  A second
// form (stage_publish_kernel) publishes the rows through a device counter
// for a stream kernel that reads them before its own dependency resolves.
#include "common.cuh"
#include "sm103_ptx.cuh"

namespace route {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageAhead = 4;  // 16-byte words a thread reads before the wait

__global__ void __launch_bounds__(kStageThreads)
    stage_in_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int stride = gridDim.x * kStageThreads;
    const int i0 = blockIdx.x * kStageThreads + threadIdx.x;
    uint4 v[kStageAhead];
#pragma unroll
    for (int j = 0; j < kStageAhead; ++j)
        if (i0 + j * stride < n16) v[j] = src[i0 + j * stride];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the staging buffer's last reader is done
#pragma unroll
    for (int j = 0; j < kStageAhead; ++j)
        if (i0 + j * stride < n16) dst[i0 + j * stride] = v[j];
    for (int i = i0 + kStageAhead * stride; i < n16; i += stride) dst[i] = src[i];
}

// The last kernel of a prepared host step: once the step's kernels have
// finished (the grid dependency) it advances the step's device counter and
// stores the new value into a page-locked word that the calling thread
// watches, with a system-scope fence before the store, so that the results
// the finish kernel wrote into host memory are visible first.  It lets the
// next kernel on the stream (another step's staging kernel) launch at once.
__global__ void host_done_kernel(unsigned *counter, unsigned *flag_mapped) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // every kernel of the step has finished
    if (threadIdx.x == 0) {
        const unsigned v = *counter + 1u;
        *counter = v;
        __threadfence_system();
        asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(flag_mapped), "r"(v) : "memory");
    }
}

// The copy for a host step launched behind another step (route_host_step_
// launch): the step's stream kernel reads these rows before its own grid
// dependency resolves, so this kernel publishes them instead of letting its
// completion do it.  Each thread reads its (up to) kPublishAhead words of
// the host rows at once; thread 0 waits until `done_counter` (the step's
// count of finished launches) reaches `need`, i.e. the launch that last read
// `dst` has finished (bounded: after timeout_ns it records a timeout in the
// status word and goes on); the CTA stores its words, and thread 0 adds one
// to `published` after a device-scope fence (the block's stores are ordered
// before it by the barrier).  The stream kernel waits for the sum of all
// CTAs' additions.  Last, the kernel waits for its own predecessor, so that
// its completion -- which the stream kernel's writes of scratch wait for --
// still follows everything before it on the stream.
constexpr int kPublishThreads = 256;
constexpr int kPublishAhead = 10;

__global__ void __launch_bounds__(kPublishThreads)
    stage_publish_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int n16,
                         const unsigned *done_counter, unsigned need, unsigned *published,
                         unsigned *status, unsigned long long timeout_ns) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i0 = blockIdx.x * kPublishThreads * kPublishAhead + threadIdx.x;
    uint4 v[kPublishAhead];
#pragma unroll
    for (int j = 0; j < kPublishAhead; ++j)
        if (i0 + j * kPublishThreads < n16) v[j] = src[i0 + j * kPublishThreads];
    if (threadIdx.x == 0) {
        const uint64_t t0 = ptx::global_timer_ns();
        while ((int)(ptx::ld_acquire_gpu(done_counter) - need) < 0) {
            if (ptx::global_timer_ns() - t0 > timeout_ns) {
                atomicOr(status, kStatusTimeout);
                break;
            }
            __nanosleep(64);
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPublishAhead; ++j)
        if (i0 + j * kPublishThreads < n16) dst[i0 + j * kPublishThreads] = v[j];
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(published, 1u);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t stage_publish_launch(const void *src_mapped, void *dst, size_t bytes,
                                 const unsigned *done_counter, unsigned need, unsigned *published,
                                 unsigned *status, unsigned long long timeout_ns, int *ctas,
                                 cudaStream_t stream) {
    if (bytes == 0 || bytes % 16 != 0 || !ctas) return cudaErrorInvalidValue;
    const int n16 = (int)(bytes / 16);
    const int per_cta = kPublishThreads * kPublishAhead;
    const int grid = (n16 + per_cta - 1) / per_cta;
    *ctas = grid;
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3(grid);
    c.blockDim = dim3(kPublishThreads);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, stage_publish_kernel, static_cast<const uint4 *>(src_mapped),
                              static_cast<uint4 *>(dst), n16, done_counter, need, published,
                              status, timeout_ns);
}

cudaError_t host_done_launch(unsigned *counter, unsigned *flag_mapped, cudaStream_t stream) {
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3(1);
    c.blockDim = dim3(32);
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, host_done_kernel, counter, flag_mapped);
}

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
