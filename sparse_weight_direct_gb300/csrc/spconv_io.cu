// Copies between page-locked host memory and the device workspaces, run on
// the SMs through the host buffer's device mapping (used by
// spconv_forward_host when CUDA maps the buffers).  Next to the forward kernel
// this avoids the switch between the copy engine and the SMs, which measured
// several microseconds per switch on one-image layers; the bandwidth over the
// host link is the same either way.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "spconv_internal.h"

namespace spconv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyMaxBlocks = 4 * 152;

// dst[i] = src[i] for i < n.  A kernel launched after this one with
// programmatic dependent launch may start its prologue at once: it waits for
// this grid to complete before it reads dst.
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(const float *__restrict__ src,
                                                               float *__restrict__ dst, size_t n,
                                                               int vec) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nthreads = (size_t)gridDim.x * blockDim.x;
    size_t done = 0;
    if (vec) {
        const size_t n4 = n / 4;
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
        float4 *d4 = reinterpret_cast<float4 *>(dst);
        for (size_t i = tid; i < n4; i += nthreads) d4[i] = s4[i];
        done = n4 * 4;
    }
    for (size_t i = done + tid; i < n; i += nthreads) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(const float *src, float *dst, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int vec = (((uintptr_t)src | (uintptr_t)dst) & 15) == 0;
    const size_t per_block = (size_t)kCopyThreads * (vec ? 4 : 1);
    size_t blocks = (n + per_block - 1) / per_block;
    if (blocks > (size_t)kCopyMaxBlocks) blocks = kCopyMaxBlocks;
    copy_kernel<<<(unsigned)blocks, kCopyThreads, 0, stream>>>(src, dst, n, vec);
    return cudaGetLastError();
}

}  // namespace spconv
