// spconv_forward_host_noalloc: the host-buffer forward (spconv_forward_host)
// for callers that must not allocate device memory when they run a layer --
// a plugin inside a framework whose allocator owns the GPU's memory, a
// service whose memory is budgeted up front, or a latency-critical caller
// that cannot take cudaMalloc's implicit synchronisation.  Its two device
// workspaces (the staged input and, for outputs above 1 MiB, the staged
// output) live in one file-scope device array that the library declares
// statically, so every GPU that loads this code holds the array until the
// process exits and no call allocates.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "spconv.h"

namespace {

constexpr size_t kScratchFloats = SPCONV_NOALLOC_MAX_BYTES / sizeof(float);
constexpr size_t kAlignFloats = 64;  // 256 bytes between the two workspaces
constexpr int kMaxDevices = 256;

// The workspaces.  In host code this name is only a stand-in for the symbol:
// its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float spconv_noalloc_scratch[kScratchFloats];

std::mutex g_lock;
float *g_scratch[kMaxDevices];  // device address of the array, per device (nullptr: not set up)

// Device address of the array on the current device; looked up on the first
// call on each device (with that device current) and remembered.
int scratch_on_current_device(float **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_lock);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, spconv_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SPCONV_ERR_CUDA;
        }
        g_scratch[dev] = static_cast<float *>(p);
    }
    *out = g_scratch[dev];
    return SPCONV_OK;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int spconv_forward_host_noalloc(
    int N, int C, int H, int W, int M, int R, int S, int stride, int pad, const float *input_host,
    const spconv_packed *packed, const float *bias, int act, float *output_host, void *stream) {
    if (!packed || N < 0 || C < 1 || H < 1 || W < 1 || M < 1 || R < 1 || S < 1 || stride < 1 ||
        pad < 0)
        return SPCONV_ERR_INVALID_ARG;
    const int64_t E = ((int64_t)H + 2 * (int64_t)pad - R) / stride + 1;
    const int64_t F = ((int64_t)W + 2 * (int64_t)pad - S) / stride + 1;
    if ((int64_t)H + 2 * (int64_t)pad < R || (int64_t)W + 2 * (int64_t)pad < S || E < 1 || F < 1)
        return SPCONV_ERR_INVALID_ARG;
    // input workspace first, output workspace 256 bytes aligned after it
    const uint64_t in_floats = (uint64_t)N * C * H * W;
    const uint64_t out_floats = (uint64_t)N * M * E * F;
    const uint64_t in_region = (in_floats + kAlignFloats - 1) / kAlignFloats * kAlignFloats;
    if (in_region > kScratchFloats || out_floats > kScratchFloats - in_region)
        return SPCONV_ERR_UNSUPPORTED;
    float *base = nullptr;
    if (N > 0) {
        const int st = scratch_on_current_device(&base);
        if (st != SPCONV_OK) return st;
    }
    return spconv_forward_host(N, C, H, W, M, R, S, stride, pad, input_host, packed, bias, act,
                               output_host, base, base ? base + in_region : nullptr, stream);
}
