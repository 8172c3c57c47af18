// Launcher of the sparse-weight direct convolution kernel (sm_103a): picks the
// kernel instance, sizes shared memory, and launches it (with a thread-block
// cluster for channel-split layers).  The kernel itself is in spconv_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <utility>

#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

// Exercises the bounded pipeline wait: one warp waits on an mbarrier whose
// phase nothing completes (armed for one arrival that never comes), with a
// short limit; the wait gives up, the kernel records bit 0 in `flags` and
// returns.  A second launch mode arrives first, so the wait succeeds.
__global__ void wait_selftest_kernel(unsigned int *flags, unsigned long long limit_ns,
                                     int arrive) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    __syncwarp();
    if (arrive && threadIdx.x == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&bar)) : "memory");
    __syncwarp();
    const bool ok = mbar_wait_bounded(&bar, 0u, limit_ns);
    if (!ok && threadIdx.x == 0) atomicOr(flags, 1u);
    if (ok && threadIdx.x == 0) atomicOr(flags, 2u);
}

KernelFn pick(int S, int stride, int P, int Q, int LR, bool pairs = false, bool plane = false,
              bool cols = false, int W = 0, bool tight = false) {
    if (tight)
        return (S == 3 && stride == 1 && LR == 1 && !pairs && !plane && !cols) ? pick_tight(P, Q)
                                                                                : nullptr;
    if (cols) {
        if (stride != 1 || plane) return nullptr;
        if (LR == 4 && S == 5) return pick_colpair5(P, Q, pairs);
        if (S != 3 || pairs) return nullptr;
        return LR == 4 ? pick_colpair(P, Q) : pick_cols(P, Q, LR);
    }
    if (pairs) return pick_pairs(S, stride, P, Q, LR);
    if (plane) return (S == 3 && stride == 1 && LR == 2) ? pick_plane(P, Q, W) : nullptr;
    switch (Q) {
        case 1: return pick_q1(S, stride, P, LR);
        case 2: return pick_q2(S, stride, P, LR);
        case 4: return pick_q4(S, stride, P, LR);
        case 8: return pick_q8(S, stride, P, LR);
        default: return nullptr;
    }
}

size_t stage_bytes(const Geometry &g) { return g.in_stage_bytes + g.blob_stage_bytes; }

// The dynamic shared-memory limit is a per-function, per-device attribute:
// raise it once to the largest size any plan uses, and remember that.
cudaError_t raise_smem_limit(const void *fn) {
    constexpr int kMaxDev = 64;
    constexpr int kSlots = 256;
    static std::mutex lock;
    static std::pair<const void *, int> done[kSlots];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(lock);
    for (int i = 0; i < ndone; ++i)
        if (done[i].first == fn && done[i].second == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kern::kMaxDynamicSmem);
    if (e != cudaSuccess) return e;
    if (ndone < kSlots && dev < kMaxDev) done[ndone++] = {fn, dev};
    return cudaSuccess;
}

}  // namespace kern

using namespace kern;

#ifdef SPCONV_TRACE
// Trace build: one record buffer per device, allocated on first use.
static unsigned long long *trace_buffer() {
    constexpr int kMaxDev = 64;
    static std::mutex lock;
    static unsigned long long *bufs[kMaxDev] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lk(lock);
    if (!bufs[dev]) {
        void *ptr = nullptr;
        if (cudaMalloc(&ptr, (size_t)kTraceBlocks * 4 * sizeof(unsigned long long)) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        bufs[dev] = static_cast<unsigned long long *>(ptr);
    }
    return bufs[dev];
}
#endif

int trace_read(void *dst, int64_t bytes) {
#ifdef SPCONV_TRACE
    unsigned long long *b = trace_buffer();
    if (!b) return -5;
    const size_t cap = (size_t)kTraceBlocks * 4 * sizeof(unsigned long long);
    const size_t n = bytes < 0 ? 0 : ((size_t)bytes < cap ? (size_t)bytes : cap);
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(dst, b, n, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return -5;
    }
    return 0;
#else
    (void)dst;
    (void)bytes;
    return -3;
#endif
}

cudaError_t launch_wait_selftest(unsigned int *flags, int arrive, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(flags, 20000000ull /* 20 ms */, arrive);
    return cudaGetLastError();
}

bool dense_taps_supported(int R, int S, int stride, int LR, int Q) {
    return stride == 1 && R == S && (S == 3 || (S == 5 && LR == 1)) && Q <= 4;
}

int forward_variant_supported(int S, int stride, int P, int Q, int LR, bool pairs, bool plane,
                              bool cols, bool tight) {
    return pick(S, stride, P, Q, LR, pairs, plane, cols, 0, tight) ? 0 : -1;
}

bool plane_stage_supported(int H, int W, int R, int S, int stride, int pad, int P, int LR, int Q) {
    return R == 3 && S == 3 && stride == 1 && pad == 1 && LR == 2 && H == 2 * P && W >= 2 &&
           W <= 16 && (W * 4) % 16 != 0 && (H * W) % 4 == 0 &&
           pick(S, stride, P, Q, LR, false, true, false, W);
}

// Shared memory of the stage buffers a block with `split` cluster ranks uses.
static size_t stages_bytes(const Geometry &g, int split) {
    const int per_block = (g.num_chunks + split - 1) / split;
    return (size_t)(per_block > 1 ? 2 : 1) * stage_bytes(g);
}

// Receive buffer of the push-mode cluster reduction: [rank][owned slot][P][32].
static size_t recv_bytes(const Geometry &g, int split) {
    const int nslot = g.warps * g.slots;
    return (size_t)split * ((nslot + split - 1) / split) * g.tile_rows * 32 * sizeof(float);
}

void forward_grid(const Geometry &g, int N, int split, bool group_fast, unsigned *gx,
                  unsigned *gy) {
    const int ti = g.tile_images > 1 ? g.tile_images : 1;
    const int64_t tiles = (int64_t)((N + ti - 1) / ti) * g.tiles_y *
                          g.tiles_x * split;
    *gx = (unsigned)(group_fast ? tiles * g.groups : tiles);
    *gy = group_fast ? 1u : (unsigned)g.groups;
}

bool push_reduction(const Geometry &g, int split) {
    return split > 1 && !g.split_rows && g.slots <= 2 &&  // compiled into Q <= 2 instances
           stages_bytes(g, split) + recv_bytes(g, split) + 128 <= (size_t)kern::kMaxDynamicSmem;
}

size_t forward_smem_bytes(const Geometry &g, int split) {
    size_t bytes = stages_bytes(g, split);
    if (push_reduction(g, split)) {
        bytes += recv_bytes(g, split) + 128;
    } else {
        // room for the partial sums of split rows / a channel-split cluster
        const size_t part = (size_t)g.warps * g.slots * g.tile_rows * 32 * sizeof(float);
        if (part > bytes) bytes = part;
        bytes += 128;  // room to align the stage buffers to 128 bytes
    }
    // plane staging (one-image layers): at most two blocks per SM, as with the
    // padded tile, so the cluster blocks spread over the SMs
    if (g.plane_stage && bytes < 76 * 1024) bytes = 76 * 1024;
    return bytes;
}

cudaError_t launch_forward(const Geometry &g, int N, int split, bool group_fast, bool pdl,
                           const float *x, float *y, const float *bias, int act,
                           const DeviceArrays &d, const CUtensorMap *tmap, cudaStream_t stream) {
    KernelFn fn = pick(g.S, g.stride, g.tile_rows, g.slots, g.lane_rows, g.tap_pairs != 0,
                       g.plane_stage != 0, g.col_blocks != 0, g.W, g.tight != 0);
    if (!fn || split < 1 || split > kMaxSplit || split > g.num_chunks)
        return cudaErrorInvalidConfiguration;
    // tight-pitch tiles have no cp.async path: their tensor map is required
    if (g.tight && !tmap) return cudaErrorInvalidConfiguration;
    const size_t smem = forward_smem_bytes(g, split);
    if (smem > 48 * 1024) {
        cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(fn));
        if (e != cudaSuccess) return e;
    }
    KParams p;
    p.x = x;
    p.y = y;
    p.bias = bias;
    p.act = act;
    p.blobs = d.blobs;
    p.blob_off = d.blob_off;
    p.slot_oc = d.slot_oc;
    p.slot_next = d.slot_next;
    p.group_flags = d.group_flags;
    p.err = d.err;
    p.N = N; p.C = g.C; p.H = g.H; p.W = g.W; p.M = g.M; p.E = g.E; p.F = g.F;
    p.stride = g.stride; p.pad = g.pad;
    p.tiles_y = g.tiles_y; p.tiles_x = g.tiles_x; p.in_rows = g.in_rows; p.in_cols = g.in_cols;
    p.shift = g.shift; p.phase_pitch = g.phase_pitch; p.row_pitch = g.row_pitch;
    p.plane = g.plane; p.chunk = g.chunk; p.num_chunks = g.num_chunks; p.split = split;
    p.hdr_words = g.hdr_words;
    p.dense_mask_words = g.dense_mask_words;
    p.in_stage_bytes = (int)g.in_stage_bytes;
    p.stage_bytes = (int)stage_bytes(g);
    // (image pairs: one box spans both images' sub-tiles)
    p.in_tma_bytes = g.chunk * g.plane * (int)sizeof(float) * (g.tile_images == 2 ? 2 : 1);
    p.use_tma = tmap ? 1 : 0;
    p.fmt = g.format;
    p.blob_stride16 = (uint32_t)g.blob_stride16;
    p.push = push_reduction(g, split) ? 1 : 0;
    p.pairs = (g.stride == 1 && g.W % 2 == 0 && g.row_pitch % 2 == 0 && g.plane % 2 == 0) ? 1 : 0;
    p.recv_off = (int)stages_bytes(g, split);
    p.plane_stage = g.plane_stage;
    p.pair_off = g.tile_images == 2 ? g.pair_off : 0;
    p.num_slots = g.num_slots;
    p.smem_bytes = (int)smem;
    p.blob_bytes = d.blob_bytes;
    p.trace = nullptr;
#ifdef SPCONV_TRACE
    p.trace = trace_buffer();
    if (p.trace) cudaMemsetAsync(p.trace, 0, (size_t)kTraceBlocks * 4 * sizeof(unsigned long long), stream);
#endif
    CUtensorMap dummy;
    if (!tmap) {
        for (int i = 0; i < 16; ++i) dummy.opaque[i] = 0;
        tmap = &dummy;
    }

    cudaLaunchConfig_t cfg = {};
    p.groups = g.groups;
    p.group_fast = group_fast ? 1 : 0;
    unsigned gx = 0, gy = 0;
    forward_grid(g, N, split, group_fast, &gx, &gy);
    cfg.gridDim = dim3(gx, gy, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    // Programmatic dependent launch: the kernel may start while the previous
    // kernel on the stream finishes; it waits (griddepcontrol.wait) before it
    // reads the input or writes the output.
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, fn, p, *tmap);
}

}  // namespace spconv
