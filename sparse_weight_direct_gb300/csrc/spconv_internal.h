// Internal interface between the host library (spconv_host.cpp) and the CUDA
// kernels (spconv_fwd.cu).  Not installed; the public ABI is include/spconv.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#if defined(__CUDACC__)
#define SPCONV_HD __host__ __device__
#else
#define SPCONV_HD
#endif

namespace spconv {

constexpr int kTileCols = 32;  // one output column per lane

// Words of one stride-phase sub-row of a staged input row.  With stride st the
// staged row is split into st sub-rows (column col goes to sub-row col % st at
// position col / st), so lanes reading columns lane*st + s touch consecutive
// words.  For st dividing 32 the pitch is padded to 32/st (mod 32) so the
// st sub-rows start in different banks.  Host planner and kernels share it.
SPCONV_HD constexpr int phase_pitch_for(int S, int stride) {
    const int in_cols = (kTileCols - 1) * stride + S;
    if (stride == 1) return in_cols;
    int pp = (in_cols + stride - 1) / stride;
    if (32 % stride == 0) {
        const int want = (32 / stride) % 32;
        while (pp % 32 != want) ++pp;
    }
    return pp;
}

// Tiling of one layer, fixed at pack time.  The precomputed entry offsets
// depend on it, so forward must use exactly this geometry.
struct Geometry {
    int C, H, W, M, R, S, stride, pad, E, F;
    int tile_rows;    // P: output rows of a tile; each lane carries P rows
    int tiles_y, tiles_x;
    int in_rows;      // (P - 1) * stride + R
    int in_cols;      // (32 - 1) * stride + S
    int phase_pitch;  // words of one stride-phase sub-row
    int row_pitch;    // stride * phase_pitch
    int plane;        // words of one staged channel
    int chunk;        // channels staged per pipeline stage
    int num_chunks;
    int slots;        // Q: output channels a warp carries at once
    int warps;        // warps per block
    int groups;       // output-channel groups (grid y)
    int num_slots;    // groups * warps * slots
    size_t smem_bytes;
};

struct DeviceArrays {
    const float2 *entries;  // {value, int offset bits}
    const int *segptr;      // [num_slots][num_chunks + 1]
    const int *slot_oc;     // [num_slots]
};

// Kernel variants compiled for sm_103a.  Returns 0 if (S, stride, P, Q) has
// an instance, else -1.
int forward_variant_supported(int S, int stride, int P, int Q);

// Enqueues the forward kernel.  Returns cudaSuccess or the launch error.
cudaError_t launch_forward(const Geometry &g, int N, const float *x, float *y,
                           const DeviceArrays &d, cudaStream_t stream);

}  // namespace spconv
