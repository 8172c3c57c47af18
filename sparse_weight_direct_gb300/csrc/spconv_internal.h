// Internal interface between the host library (spconv_host.cpp) and the CUDA
// kernels (spconv_fwd.cu).  Not installed; the public ABI is include/spconv.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#if defined(__CUDACC__)
#define SPCONV_HD __host__ __device__
#else
#define SPCONV_HD
#endif

namespace spconv {

constexpr int kLanes = 32;
constexpr int kWarps = 8;       // warps per block
constexpr int kMaxSplit = 8;    // largest thread-block cluster of the channel split

// Words of one stride-phase sub-row of a staged input row.  With stride st the
// staged row is split into st sub-rows (column col goes to sub-row col % st at
// position col / st), so lanes reading columns lane*st + s touch consecutive
// words.  For st dividing 32 the pitch is padded to 32/st (mod 32) so the
// st sub-rows start in different banks.  Host planner and kernels share it.
SPCONV_HD constexpr int phase_pitch_for(int S, int stride) {
    const int in_cols = (kLanes - 1) * stride + S;
    if (stride == 1) return in_cols;
    int pp = (in_cols + stride - 1) / stride;
    if (32 % stride == 0) {
        const int want = (32 / stride) % 32;
        while (pp % 32 != want) ++pp;
    }
    return pp;
}

// Left shift that brings a stride-1 tile's first staged column down to a
// multiple of 4 words (tile origins are multiples of 32 minus pad), so the
// tile can be fetched by a TMA copy whose x coordinate is 16-byte aligned.
SPCONV_HD constexpr int align_shift_for(int pad, int stride) {
    return stride == 1 ? (4 - pad % 4) % 4 : 0;
}

// Words per staged input row for stride 1 with `lane_rows` lane rows of
// 32 / lane_rows lanes: the tile's columns plus room for the largest alignment
// shift (3), rounded to 4 words (a TMA box row is a multiple of 16 B).  With
// two lane rows (interleaved output rows) the half-warps read rows one pitch
// apart, so the pitch is also made 16 (mod 32) words: the halves then hit
// disjoint banks.  Independent of pad so kernels can fix it at compile time.
SPCONV_HD constexpr int row_pitch_s1(int S, int lane_rows) {
    const int need = (kLanes / lane_rows - 1) + S + 3;
    if (lane_rows == 1) return (need + 3) / 4 * 4;
    int rp = 16;
    while (rp < need) rp += 32;
    return rp;
}

// Tiling of one layer, fixed at pack time.  The precomputed entry offsets
// depend on it, so forward must use exactly this geometry.
struct Geometry {
    int C, H, W, M, R, S, stride, pad, E, F;
    int tile_rows;    // P: output rows each lane carries
    int lane_rows;    // LR: lane rows of a warp (1, or 2 for outputs <= 16 wide)
    int tile_h, tile_w;  // output tile: LR * P rows x 32 / LR columns
    int tiles_y, tiles_x;
    int in_rows;      // (tile_h - 1) * stride + R
    int in_cols;      // (tile_w - 1) * stride + S
    int shift;        // staged column of input column ix0 (stride 1), else 0
    int phase_pitch;  // words of one stride-phase sub-row
    int row_pitch;    // words of one staged row
    int plane;        // words of one staged channel (in_rows * row_pitch)
    int chunk;        // channels staged per pipeline stage (weight-stationary
                      // format: entries per stage)
    int num_chunks;   // (weight-stationary format: most stages of any row)
    int slots;        // Q: output channels a warp carries at once
    int warps;        // warps per block
    int groups;       // output-channel groups (grid y)
    int num_slots;    // groups * warps * slots
    int format;       // 0 = {fp32, int32 offset} entries, 1 = 32-bit packed words,
                      // 2 = weight-stationary rows (one output channel per block)
    int batch_hint;   // batch size the plan targets (0 = unknown)
    int hdr_words;    // words of a sparse blob header (warps * slots + 1, to 4; with
                      // tap pairs + warps * slot pairs + 1)
    int tap_pairs;    // 1: sparse blobs also hold pair entries -- a tap two slots of a
                      // warp share, applied to both from one set of shared loads
    int plane_stage;  // 1: the chunk's raw input planes are staged by one bulk copy
                      // (whole-image tiles whose rows TMA cannot address) and the
                      // padding is applied to the weights (see kPlaneLead)
    int col_blocks;   // 1: column blocks -- lane_rows lane rows of 32 / lane_rows
                      // lanes, each lane holding tile_rows consecutive outputs of
                      // its row (stride 1, widths a multiple of 28, not of 32)
    int tight;        // 1: tight-pitch tiles (a 32-word pitch from column 0, shift -1,
                      // kTightLead zeroed words before each stage's tile)
    int tile_images;  // images side by side in a tile: 2 for image-pair column
                      // blocks (then N counts pairs in the grid), else 1
    int pair_off;     // image pairs: words from a stage's first sub-tile to its
                      // second (so the two halves of a warp hit disjoint banks)
    int dense_groups; // leading groups whose blobs are dense-tap (0 if none)
    int split_rows;   // 1 if any group has rows split into parts (bit 1 of its flags)
    int dense_mask_words;  // words of a dense blob's slot masks (warps * chunk, to 4)
    int blob_stride16;        // blobs at a fixed stride (16-byte units), or 0: blob_off
    size_t in_stage_bytes;    // staged input of one chunk, rounded to 128 B
    size_t blob_stage_bytes;  // largest weight blob, rounded to 128 B
};

struct DeviceArrays {
    const unsigned char *blobs;  // weight blobs, each 16-byte aligned
    const uint32_t *blob_off;    // [groups * num_chunks + 1] in 16-byte units
    const int *slot_oc;          // [num_slots]: head slot -> output channel, else -1
    const int *slot_next;        // [num_slots]: next part (group-local slot) or -1
    const int *group_flags;      // [groups]: bit 0 dense-tap blobs, bit 1 split rows
    unsigned int *err;           // device error flags (bit 0: pipeline wait timed out;
                                 // bit 1: the drain of in-flight copies timed out too;
                                 // bit 2: a check of the bounds-checked build failed)
    int64_t blob_bytes;          // bytes of the blobs array
};

// Kernel variants compiled for sm_103a.  Returns 0 if (S, stride, P, Q, LR)
// has an instance (pairs: with tap-pair segments; plane: with plane staging;
// cols: with column blocks), else -1.
int forward_variant_supported(int S, int stride, int P, int Q, int LR, bool pairs = false,
                              bool plane = false, bool cols = false, bool tight = false);

// Tight-pitch tiles: zeroed words before each stage's tile (kTightLead in the
// kernel; the copy's destination stays 128-byte aligned), and words after it
// (the right tap of the last lanes -- past the image, outputs discarded --
// reaches one word beyond the last row of the last channel).
constexpr int kTightLeadWords = 32;
constexpr int kTightTailWords = 32;

// Plane staging: zeroed words before and after the raw planes of a stage, so
// that taps reaching past the first or last plane read finite values.
constexpr int kPlaneLead = 16;
constexpr int kPlaneTail = 48;

// Whether a plan can stage raw planes: 3 x 3, pad 1, stride 1, two lane rows,
// one tile covering the whole image (H = 2 P rows, W <= 16 columns), rows that
// a TMA tensor map cannot address (4 W not a multiple of 16), and planes that
// start on 16-byte boundaries (H W a multiple of 4).
bool plane_stage_supported(int H, int W, int R, int S, int stride, int pad, int P, int LR, int Q);

// Trace build (-DSPCONV_TRACE=1): copies up to `bytes` of the current
// device's per-block records of the last forward launch to host memory
// (synchronises the device).  0 on success, -3 in other builds, -5 on a CUDA
// error.
int trace_read(void *dst, int64_t bytes);

// Whether a layer shape can use the dense-tap path (output channels with dense
// rows get their K x K blocks applied from a register window).
bool dense_taps_supported(int R, int S, int stride, int LR, int Q);

// Launches the bounded-wait self-test (flags: bit 0 = the wait timed out,
// bit 1 = it completed).  arrive = 0 leaves the barrier incomplete.
cudaError_t launch_wait_selftest(unsigned int *flags, int arrive, cudaStream_t stream);

// Dynamic shared memory a launch needs with `split` blocks per cluster.
size_t forward_smem_bytes(const Geometry &g, int split);

// Grid of a forward launch (x: cluster rank fastest, then tiles [and groups];
// y: groups, or 1 when groups run fastest).
void forward_grid(const Geometry &g, int N, int split, bool group_fast, unsigned *gx,
                  unsigned *gy);

// Whether a launch with `split` cluster ranks reduces by pushing partial sums
// into the owning block (no split rows, and room beside the stage buffers).
bool push_reduction(const Geometry &g, int split);

// Enqueues the forward kernel.  tmap is a tiled tensor map of the input for
// stride-1 layers whose row stride is a multiple of 16 bytes (nullptr:
// stage with cp.async).  group_fast orders blocks so all channel groups of a
// tile run together (they then share the tile's input through L2).  Returns
// cudaSuccess or the launch error.  bias (M floats or nullptr) and act
// (0 identity, 1 ReLU) form the fused epilogue y = act(conv + bias).
// pdl: launch with programmatic stream serialization (the kernel's prologue
// may overlap the previous kernel on the stream).
cudaError_t launch_forward(const Geometry &g, int N, int split, bool group_fast, bool pdl,
                           const float *x, float *y, const float *bias, int act,
                           const DeviceArrays &d, const CUtensorMap *tmap, cudaStream_t stream);

// dst[0, n) = src[0, n) on the SMs (one side the device mapping of a
// page-locked host buffer, the other device memory), after the previous work
// on the stream.  A forward launched next with pdl = true overlaps its
// prologue with the copy and waits for it before reading dst.
cudaError_t launch_copy(const float *src, float *dst, size_t n, cudaStream_t stream);

// Weight-stationary format (one output channel per block, input read in
// place): whether (P, LR) has an instance, the dynamic shared memory of a
// launch, and the launcher (N <= 65535).  d.blobs holds the row entries,
// d.blob_off the [2 * M] (first entry, count) pairs, d.slot_oc the row order.
bool ws_variant_supported(int P, int LR);
size_t ws_smem_bytes(const Geometry &g);
cudaError_t launch_forward_ws(const Geometry &g, int N, const float *x, float *y,
                              const float *bias, int act, const DeviceArrays &d,
                              cudaStream_t stream);

}  // namespace spconv
