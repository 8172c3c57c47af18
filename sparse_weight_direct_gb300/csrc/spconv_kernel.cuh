// Internal: the forward kernel template and its device helpers, shared by the
// per-Q translation units (spconv_fwd_q*.cu) and the launcher (spconv_fwd.cu).
#pragma once
// Forward kernel of the sparse-weight direct convolution (sm_103a).
//
// What it computes: Tuteja et al., "Theoretical and Empirical Analysis of
// Sparse Convolution", Sec. 3 Eq.(3) -- each output is the sum, over the
// nonzeros of its output channel, of value * input at the padding-shifted
// position -- with stride (Escoin, arXiv 1802.10280, Algorithm 2).
//
// Work decomposition.  A block owns one output tile (P rows x 32 columns of one
// image) and one group of 8 * Q output channels; a thread-block cluster of
// `split` blocks shares the tile and splits the input-channel chunks between
// them.  Per chunk, a pipeline stage holds
//   * the input tile plus halo of the chunk's channels (Sec. 5.1 of the first
//     page: each input region is read once per block and reused by all of the
//     block's output channels and rows), fetched by one TMA tensor copy with
//     hardware zero fill for the padding, or by cp.async where the input row
//     stride is not 16-byte aligned (whole-image 3x3 tiles of such inputs
//     instead stage the raw planes with one bulk copy and apply the padding
//     to the weights: kModePlane); and
//   * the chunk's weight blob of the block's channel group (a header of per-warp
//     entry ranges, then 8-byte (value, offset) entries), fetched by one bulk
//     asynchronous copy.
// Both complete on the stage's mbarrier; two stages overlap copy and compute.
// Each warp carries Q output channels; each lane owns one output column and P
// rows in registers.  A warp walks its entries with 16-byte shared-memory
// broadcasts (two entries per load) and does P FMAs per entry, reading
// smem[lane + offset + p * row_step]: consecutive lanes read consecutive words,
// so the reads are conflict free.  Offsets were precomputed per nonzero on the
// host against this tile layout (Escoin's weight stretching).  With split > 1
// the blocks of a cluster add their partial sums through distributed shared
// memory in a fixed rank order (deterministic), then write back; otherwise the
// accumulators are written directly (coalesced along the row, predicated for
// partial tiles: Sec. 5.5 of the first page).
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "spconv_internal.h"

namespace cg = cooperative_groups;

namespace spconv {
namespace kern {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait
constexpr int kMaxDynamicSmem = 200 * 1024;                   // upper bound of any plan

// Raises a kernel's dynamic shared-memory limit to kMaxDynamicSmem, once per
// kernel and device (later calls only look it up: no API call, so launches
// can be captured into a CUDA graph).
cudaError_t raise_smem_limit(const void *fn);

struct KParams {
    const float *x;
    float *y;
    const float *bias;  // [M] or nullptr
    int act;            // 0 identity, 1 ReLU
    const unsigned char *blobs;
    const uint32_t *blob_off;
    const int *slot_oc;      // head slot -> output channel; -1 empty or a later part
    const int *slot_next;    // next part of the same output channel (group-local), -1
    const int *group_flags;  // per group: bit 0 dense-tap blobs, bit 1 split rows
    unsigned int *err;
    int N, C, H, W, M, E, F, stride, pad;
    int tiles_y, tiles_x, in_rows, in_cols, shift, phase_pitch, row_pitch, plane;
    int chunk, num_chunks, split, hdr_words, dense_mask_words;
    int in_stage_bytes, stage_bytes, in_tma_bytes;
    int use_tma;
    int fmt;  // sparse entries: 0 = {fp32 value, int32 offset}, 1 = 32-bit packed word
    int group_fast, groups;  // block order; number of groups
    uint32_t blob_stride16;  // blobs at a fixed stride (16-byte units), or 0: blob_off
    int push;                // cluster reduction by remote stores into the owner's buffer
    int pairs;               // cp.async staging in 8-byte column pairs (stride 1, W even)
    int recv_off;            // byte offset of that receive buffer in shared memory
    int plane_stage;         // raw planes staged by one bulk copy (kModePlane instances)
    int pair_off;            // image-pair column blocks: words from a stage's first
                             // sub-tile (image 2n) to its second (image 2n + 1), else 0;
                             // with TMA one box spans both images (in_tma_bytes)
    int num_slots;           // entries of slot_oc / slot_next (bounds-checked build)
    int smem_bytes;          // dynamic shared memory of the launch (bounds-checked build)
    int64_t blob_bytes;      // bytes of the blobs array (bounds-checked build)
    unsigned long long *trace;  // trace build: kTraceBlocks records of 4 words, else nullptr
};

// ---------------------------------------------------------------- bounds-checked build
//
// Compiled with -DSPCONV_DEBUG=1 (libspconv_debug.so; the stand-in for a
// memory checker), every read of a staged input tile, every weight-blob range,
// shared-memory scratch index, distributed-shared-memory slot and global index
// of the kernels is checked against its extent before the access.  An access
// that would leave its extent is skipped (a read gives 0), and bit 2 of the
// device error word is set; the kernel never traps.  The default build
// compiles every check away.
constexpr unsigned int kErrBounds = 4u;
#ifdef SPCONV_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif

// ---------------------------------------------------------------- trace build
//
// Compiled with -DSPCONV_TRACE=1 (libspconv_trace.so), every block of the
// forward kernel records four words in p.trace[block * 4 ..]: its start, the
// moment its first stage became ready (thread 0), the end of its pipeline
// (all warps out of the chunk loop), each a global-timer value in ns, and
// smid | group << 16 | group flags << 32.  The default build compiles the
// records away.
#ifdef SPCONV_TRACE
constexpr bool kTrace = true;
#else
constexpr bool kTrace = false;
#endif
constexpr int kTraceBlocks = 65536;  // records kept per launch

// [lo, hi) of the staged input of the current stage, and the error word.
struct Span {
    const float *lo, *hi;
    unsigned int *err;
};

// true if `in_range`; otherwise (bounds-checked build) records the failure.
static __device__ __forceinline__ bool dbg_ok(bool in_range, unsigned int *err) {
    if constexpr (kDebug) {
        if (!in_range) {
            atomicOr(err, kErrBounds);
            return false;
        }
    }
    return true;
}

// Shared-memory read of a staged input word.
static __device__ __forceinline__ float sld(const Span &sp, const float *ptr) {
    if constexpr (kDebug) {
        if (ptr < sp.lo || ptr >= sp.hi) {
            atomicOr(sp.err, kErrBounds);
            return 0.f;
        }
    }
    return *ptr;
}

// ---------------------------------------------------------------- PTX helpers

static __device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

static __device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

static __device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

static __device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Waits for the stage's phase with a time limit; false on timeout.
static __device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

static __device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *tmap, int x, int y,
                                            int c, int n, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(c), "r"(n),
        "r"(smem_u32(bar))
        : "memory");
}

static __device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];\n" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

static __device__ __forceinline__ void cp_async_4(float *smem_dst, const float *gsrc, bool pred) {
    const int src_size = pred ? 4 : 0;  // 0 -> the 4 destination bytes are zero-filled
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(src_size)
                 : "memory");
}
static __device__ __forceinline__ void cp_async_8(float *smem_dst, const float *gsrc,
                                                  int src_bytes) {
    // 8-byte copy; the bytes past src_bytes (0, 4 or 8) are zero-filled
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
static __device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
static __device__ __forceinline__ void cp_async_wait_all_but_one() {
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}
static __device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// ---------------------------------------------------------------- staging

// cp.async staging of channels [c0, c0 + cc) of image n: staged element
// (channel cl, row, col) holds input (c0 + cl, iy0 + row, ix0 + col), zero
// outside the image.  A thread owns fixed positions (row, col) of the staged
// plane (its validity and both offsets do not depend on the channel) and walks
// the chunk's channels for each, so the inner loop is two adds and a cp.async;
// consecutive threads take consecutive columns (coalesced per channel).
template <int ST_CT>
static __device__ __forceinline__ void stage_input_cp_async(const KParams &p, float *buf, int n, int c0,
                                                     int cc, int iy0, int ix0) {
    const int st = ST_CT ? ST_CT : p.stride;
    const int in_cols = p.in_cols;
    const int plane_elems = p.in_rows * in_cols;
    const size_t hw = (size_t)p.H * p.W;
    const float *xc0 = p.x + ((size_t)n * p.C + c0) * hw;
    const int T = blockDim.x;
    int row = threadIdx.x / in_cols, col = threadIdx.x - row * in_cols;
    const int drow = T / in_cols, dcol = T - drow * in_cols;
    for (int e = threadIdx.x; e < plane_elems; e += T) {
        const int gy = iy0 + row, gx = ix0 + col;
        const bool ok = (unsigned)gy < (unsigned)p.H && (unsigned)gx < (unsigned)p.W;
        const float *src = ok ? xc0 + (size_t)gy * p.W + gx : p.x;
        const size_t src_step = ok ? hw : 0;
        const int phys = (st == 1) ? col + p.shift : (col % st) * p.phase_pitch + col / st;
        float *dst = buf + row * p.row_pitch + phys;
        for (int cl = 0; cl < cc; ++cl) {
            if (dbg_ok(dst - buf + 1 <= p.in_stage_bytes / 4 &&
                           (!ok || (src >= p.x && src < p.x + (size_t)p.N * p.C * hw)),
                       p.err))
                cp_async_4(dst, src, ok);
            dst += p.plane;
            src += src_step;
        }
        row += drow;
        col += dcol;
        if (col >= in_cols) {
            col -= in_cols;
            ++row;
        }
    }
}

// The same staging with 8-byte copies, for stride 1 with an even input width
// W: then global column x and its staged word x - ix0 + shift have the same
// parity (row starts are even on both sides and ix0 = pad = shift mod 2), so
// each aligned column pair is one copy.  Units u cover staged columns
// 2u - a, 2u - a + 1 with a = pad & 1; the first unit (a = 1) and a unit that
// would run past the staged row copy their one column with 4 bytes, so
// nothing outside the staged row is written.  A pair whose second column is
// past the image copies 4 bytes and zero-fills 4; one wholly outside copies
// none (x is even, so a pair never starts left of the image and ends inside).
static __device__ __forceinline__ void stage_input_cp_async_pairs(const KParams &p, float *buf,
                                                                  int n, int c0, int cc, int iy0,
                                                                  int ix0) {
    const int in_cols = p.in_cols;
    const int a = p.pad & 1;
    const int units = (in_cols + a + 1) / 2;
    const int plane_units = p.in_rows * units;
    const size_t hw = (size_t)p.H * p.W;
    const float *xc0 = p.x + ((size_t)n * p.C + c0) * hw;
    const int T = blockDim.x;
    int row = threadIdx.x / units, u = threadIdx.x - row * units;
    const int drow = T / units, du = T - drow * units;
    for (int e = threadIdx.x; e < plane_units; e += T) {
        const int gy = iy0 + row;
        const int j = 2 * u - a;  // first staged column of the unit
        const bool row_ok = (unsigned)gy < (unsigned)p.H;
        float *dst = buf + row * p.row_pitch + p.shift;
        if (j < 0 || j + 1 >= in_cols) {  // one column
            const int jj = j < 0 ? 0 : j;
            const int gx = ix0 + jj;
            const bool ok = row_ok && (unsigned)gx < (unsigned)p.W;
            const float *src = ok ? xc0 + (size_t)gy * p.W + gx : p.x;
            const size_t step = ok ? hw : 0;
            float *d = dst + jj;
            for (int cl = 0; cl < cc; ++cl) {
                if (dbg_ok(d - buf + 1 <= p.in_stage_bytes / 4 &&
                               (!ok || (src >= p.x && src < p.x + (size_t)p.N * p.C * hw)),
                           p.err))
                    cp_async_4(d, src, ok);
                d += p.plane;
                src += step;
            }
        } else {
            const int gx = ix0 + j;  // even
            const int bytes = !row_ok || gx < 0 || gx >= p.W ? 0 : (gx + 1 < p.W ? 8 : 4);
            const float *src = bytes ? xc0 + (size_t)gy * p.W + gx : p.x;
            const size_t step = bytes ? hw : 0;
            float *d = dst + j;
            for (int cl = 0; cl < cc; ++cl) {
                if (dbg_ok(d - buf + 2 <= p.in_stage_bytes / 4 &&
                               (bytes == 0 ||
                                (src >= p.x && src + bytes / 4 <= p.x + (size_t)p.N * p.C * hw)),
                           p.err))
                    cp_async_8(d, src, bytes);
                d += p.plane;
                src += step;
            }
        }
        row += drow;
        u += du;
        if (u >= units) {
            u -= units;
            ++row;
        }
    }
}

// ---------------------------------------------------------------- compute

// Reads of the per-slot arrays (bounds-checked build: an index past
// num_slots reads as -1, "no channel / no next part").
static __device__ __forceinline__ int slot_oc_at(const KParams &p, int i) {
    if (!dbg_ok((unsigned)i < (unsigned)p.num_slots, p.err)) return -1;
    return p.slot_oc[i];
}
static __device__ __forceinline__ int slot_next_at(const KParams &p, int i) {
    if (!dbg_ok((unsigned)i < (unsigned)p.num_slots, p.err)) return -1;
    return p.slot_next[i];
}

// Fused epilogue: bias, then the activation.
static __device__ __forceinline__ float finish(const KParams &p, int m, float v) {
    if (p.bias) v += __ldg(p.bias + m);
    if (p.act == 1) v = fmaxf(v, 0.f);
    return v;
}

// Kernel instances that carry the dense-tap path: stride 1, K x K with K = 3, 5.
template <int S_CT, int ST_CT>
constexpr bool kDenseTaps = ST_CT == 1 && (S_CT == 3 || S_CT == 5);

template <int P, int ROW_STEP>
static __device__ __forceinline__ void apply_entry(float (&acc)[P], const float *sb, float v, int off,
                                            int row_step, const Span &sp) {
    const float *s = sb + off;
#pragma unroll
    for (int r = 0; r < P; ++r)
        acc[r] = fmaf(v, sld(sp, s + r * (ROW_STEP ? ROW_STEP : row_step)), acc[r]);
}

// UNROLL: iterations (two entries each) unrolled; more shared loads in flight
// per lane, where the registers allow it.
template <int P, int ROW_STEP, int UNROLL>
static __device__ __forceinline__ void run_segment(float (&acc)[P], const float *sb, const float2 *ent,
                                            int j, int j1, int row_step, const Span &sp) {
    if ((j & 1) && j < j1) {  // head: bring j to a 16-byte boundary
        const float2 e = ent[j];
        apply_entry<P, ROW_STEP>(acc, sb, e.x, __float_as_int(e.y), row_step, sp);
        ++j;
    }
#pragma unroll UNROLL
    for (; j + 1 < j1; j += 2) {
        const float4 e = *reinterpret_cast<const float4 *>(ent + j);
        apply_entry<P, ROW_STEP>(acc, sb, e.x, __float_as_int(e.y), row_step, sp);
        apply_entry<P, ROW_STEP>(acc, sb, e.z, __float_as_int(e.w), row_step, sp);
    }
    if (j < j1) {  // tail
        const float2 e = ent[j];
        apply_entry<P, ROW_STEP>(acc, sb, e.x, __float_as_int(e.y), row_step, sp);
    }
}

// Plane staging (whole-image tiles, 3 x 3, pad 1): the stage holds the raw
// input planes, pitch W, after kPlaneLead zeroed words, so a tap's input is at
// lane base + offset + p * row_step with no padding in shared memory.  The
// padding is applied to the weight instead: an entry's low 4 bits flag the
// sides its tap can leave the image by (bit 0 left column, 1 right column, 2
// the row above, 3 the row below); lanebits holds the sides this lane's
// outputs touch (its column is the first / last, its lane row holds the top
// row at p = 0 / the bottom row at p = P - 1), and a tap that leaves the image
// there reads a finite neighbour with weight zero.  RS: the step between the
// lane's outputs (two rows, 2 W words) when the instance fixes it, so the P
// loads take immediate offsets; 0 = row_step at run time.
template <int P, int RS>
static __device__ __forceinline__ void apply_entry_plane(float (&acc)[P], const float *sb, float v,
                                                         uint32_t code, int row_step,
                                                         uint32_t lanebits, const Span &sp) {
    const float *s = sb + (code >> 4);
    const uint32_t hit = code & lanebits;
    const float wc = (hit & 3u) ? 0.f : v;
    const float w0 = (hit & 4u) ? 0.f : wc;
    const float wl = (hit & 8u) ? 0.f : wc;
#pragma unroll
    for (int r = 0; r < P; ++r)
        acc[r] = fmaf(r == 0 ? w0 : (r == P - 1 ? wl : wc), sld(sp, s + r * (RS ? RS : row_step)),
                      acc[r]);
}

template <int P, int RS, int UNROLL>
static __device__ __forceinline__ void run_segment_plane(float (&acc)[P], const float *sb,
                                                         const float2 *ent, int j, int j1,
                                                         int row_step, uint32_t lanebits,
                                                         const Span &sp) {
    if ((j & 1) && j < j1) {  // head: bring j to a 16-byte boundary
        const float2 e = ent[j];
        apply_entry_plane<P, RS>(acc, sb, e.x, __float_as_uint(e.y), row_step, lanebits, sp);
        ++j;
    }
#pragma unroll UNROLL
    for (; j + 1 < j1; j += 2) {
        const float4 e = *reinterpret_cast<const float4 *>(ent + j);
        apply_entry_plane<P, RS>(acc, sb, e.x, __float_as_uint(e.y), row_step, lanebits, sp);
        apply_entry_plane<P, RS>(acc, sb, e.z, __float_as_uint(e.w), row_step, lanebits, sp);
    }
    if (j < j1) {  // tail
        const float2 e = ent[j];
        apply_entry_plane<P, RS>(acc, sb, e.x, __float_as_uint(e.y), row_step, lanebits, sp);
    }
}

// A pair entry: a tap that two of the warp's output channels share.  Its P
// inputs are loaded once and feed both channels' accumulators.
template <int P, int ROW_STEP>
static __device__ __forceinline__ void apply_pair(float (&a)[P], float (&b)[P], const float *sb,
                                                  float va, float vb, int off, int row_step,
                                                  const Span &sp) {
    const float *s = sb + off;
#pragma unroll
    for (int r = 0; r < P; ++r) {
        const float x = sld(sp, s + r * (ROW_STEP ? ROW_STEP : row_step));
        a[r] = fmaf(va, x, a[r]);
        b[r] = fmaf(vb, x, b[r]);
    }
}

// The warp's pair segments, one per slot pair (q1 < q2, lexicographic): hp
// holds their ranges in 8-byte units, each pair entry 16 bytes {w1, w2,
// offset, 0} starting on a 16-byte boundary.
template <int P, int Q, int ROW_STEP>
static __device__ __forceinline__ void run_pairs(float (&acc)[Q][P], const float *sb,
                                                 const uint32_t *hp, const float4 *ent4,
                                                 int row_step, const Span &sp, int ent4_cap) {
#pragma unroll
    for (int q1 = 0; q1 < Q; ++q1)
#pragma unroll
        for (int q2 = q1 + 1; q2 < Q; ++q2) {
            const int k = q1 * Q - q1 * (q1 + 1) / 2 + (q2 - q1 - 1);
            const int j1 = (int)(hp[k + 1] >> 1);
            int j = (int)(hp[k] >> 1);
            if (!dbg_ok(0 <= j && j <= j1 && j1 <= ent4_cap, sp.err)) continue;
#pragma unroll 2
            for (; j < j1; ++j) {
                const float4 e = ent4[j];
                apply_pair<P, ROW_STEP>(acc[q1], acc[q2], sb, e.x, e.y, __float_as_int(e.z),
                                        row_step, sp);
            }
        }
}

// Dense-tap accumulation of one chunk for a warp of dense output channels: the
// channel's input window (LR*(P-1)+K rows x K columns around this lane's output
// column) is loaded into registers once and every tap of every slot of the
// warp is applied to it with compile-time register indices.  The blob holds,
// per (warp, channel), a mask of the slots with any nonzero in that channel
// and, per (warp, channel, slot), the K*K weights (zeros included) padded to a
// multiple of 4 floats.  Useful fraction = density of the channel's K x K
// block; shared-memory reads per FMA drop by about the slot count.
template <int P, int Q, int K, int LR, int RP>
static __device__ __forceinline__ void run_dense_chunk(float (&acc)[Q][P], const float *sb,
                                                const uint32_t *dmask, const float4 *dw,
                                                int warp, int chunk, int cc, int plane,
                                                const Span &sp, const void *blob_end) {
    constexpr int WR = LR * (P - 1) + K;  // window rows
    constexpr int KK4 = (K * K + 3) / 4;  // float4 per weight block
    for (int cl = 0; cl < cc; ++cl) {
        const uint32_t mask = dmask[warp * chunk + cl];
        if (mask == 0) continue;
        const float *s = sb + cl * plane;
        float win[WR][K];
#pragma unroll
        for (int i = 0; i < WR; ++i)
#pragma unroll
            for (int j = 0; j < K; ++j) win[i][j] = sld(sp, s + i * RP + j);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (!(mask & (1u << q))) continue;
            const float4 *wq = dw + ((size_t)(warp * chunk + cl) * Q + q) * KK4;
            if (!dbg_ok((const void *)(wq + KK4) <= blob_end, sp.err)) continue;
            float w[KK4 * 4];
#pragma unroll
            for (int t = 0; t < KK4; ++t) {
                const float4 v = wq[t];
                w[4 * t] = v.x;
                w[4 * t + 1] = v.y;
                w[4 * t + 2] = v.z;
                w[4 * t + 3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < K; ++r)
#pragma unroll
                for (int c = 0; c < K; ++c)
#pragma unroll
                    for (int pr = 0; pr < P; ++pr)
                        acc[q][pr] = fmaf(w[r * K + c], win[LR * pr + r][c], acc[q][pr]);
        }
    }
}

// Dense-tap accumulation for column blocks: a lane's P outputs run along a
// row, so the channel's window is K rows x (P + K - 1) columns starting at the
// lane's first output; tap (r, c) of output p reads window (r, p + c).  Blob
// layout as for run_dense_chunk.
template <int P, int Q, int K>
static __device__ __forceinline__ void run_dense_chunk_cols(float (&acc)[Q][P], const float *sb,
                                                            const uint32_t *dmask, const float4 *dw,
                                                            int warp, int chunk, int cc, int plane,
                                                            int rp, const Span &sp,
                                                            const void *blob_end) {
    constexpr int WC = P + K - 1;         // window columns
    constexpr int KK4 = (K * K + 3) / 4;  // float4 per weight block
    for (int cl = 0; cl < cc; ++cl) {
        const uint32_t mask = dmask[warp * chunk + cl];
        if (mask == 0) continue;
        const float *s = sb + cl * plane;
        float win[K][WC];
#pragma unroll
        for (int r = 0; r < K; ++r)
#pragma unroll
            for (int j = 0; j < WC; ++j) win[r][j] = sld(sp, s + r * rp + j);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (!(mask & (1u << q))) continue;
            const float4 *wq = dw + ((size_t)(warp * chunk + cl) * Q + q) * KK4;
            if (!dbg_ok((const void *)(wq + KK4) <= blob_end, sp.err)) continue;
            float w[KK4 * 4];
#pragma unroll
            for (int t = 0; t < KK4; ++t) {
                const float4 v = wq[t];
                w[4 * t] = v.x;
                w[4 * t + 1] = v.y;
                w[4 * t + 2] = v.z;
                w[4 * t + 3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < K; ++r)
#pragma unroll
                for (int c = 0; c < K; ++c)
#pragma unroll
                    for (int pc = 0; pc < P; ++pc)
                        acc[q][pc] = fmaf(w[r * K + c], win[r][pc + c], acc[q][pc]);
        }
    }
}

// The first page's packed weight word (Tuteja et al., Sec. 5.3, Fig. 4):
// [31:16] FP16 value, [15:8] input channel (here: within the chunk), [7:4]
// kernel column px, [3:0] kernel row py.  The offset into the staged tile is
// rebuilt from (channel, py, px) per entry.
template <int P, int ROW_STEP, int ST_CT>
static __device__ __forceinline__ void apply_word(float (&acc)[P], const float *sb, uint32_t w,
                                           const KParams &p, int row_step, const Span &sp) {
    const float v = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    const int cl = (int)((w >> 8) & 0xffu), px = (int)((w >> 4) & 0xfu), py = (int)(w & 0xfu);
    const int st = ST_CT ? ST_CT : p.stride;
    const int col = (st == 1) ? px + p.shift : (px % st) * p.phase_pitch + px / st;
    apply_entry<P, ROW_STEP>(acc, sb, v, cl * p.plane + py * p.row_pitch + col, row_step, sp);
}

template <int P, int ROW_STEP, int ST_CT>
static __device__ __forceinline__ void run_segment_words(float (&acc)[P], const float *sb,
                                                  const uint32_t *ent, int j, int j1,
                                                  const KParams &p, int row_step, const Span &sp) {
    for (; (j & 3) && j < j1; ++j)  // head: bring j to a 16-byte boundary
        apply_word<P, ROW_STEP, ST_CT>(acc, sb, ent[j], p, row_step, sp);
    for (; j + 3 < j1; j += 4) {
        const uint4 e = *reinterpret_cast<const uint4 *>(ent + j);
        apply_word<P, ROW_STEP, ST_CT>(acc, sb, e.x, p, row_step, sp);
        apply_word<P, ROW_STEP, ST_CT>(acc, sb, e.y, p, row_step, sp);
        apply_word<P, ROW_STEP, ST_CT>(acc, sb, e.z, p, row_step, sp);
        apply_word<P, ROW_STEP, ST_CT>(acc, sb, e.w, p, row_step, sp);
    }
    for (; j < j1; ++j) apply_word<P, ROW_STEP, ST_CT>(acc, sb, ent[j], p, row_step, sp);  // tail
}

// Tight-pitch tiles (3x3, pad 1, one lane row, images up to 31 wide in one
// tile column): the tensor copy starts at column 0 with a 32-word pitch, so
// the columns past the image arrive as the copy's zero fill and a tap left of
// column 0 reads the previous row's last column -- a zero -- instead of a
// staged halo column: 9 x 32 words per channel against the padded tile's
// 9 x 40, so the chunks hold a quarter more channels.  The stage keeps
// kTightLead zeroed words before the tile for the first row's left tap.
constexpr int kTightLead = kTightLeadWords;  // 128 bytes: the copy's destination stays aligned

// P: output rows per lane; Q: output channels per warp; LR: lane rows (1, or 2
// interleaved half-warps of 16 lanes for outputs at most 16 wide); S_CT/ST_CT:
// kernel width and stride when known at compile time (0 = read from p); MODE:
// 0 the shared-memory path, kModePairs the shared-memory path with tap-pair
// segments (blobs of the tap-pair layout).  The pair loop lives in instances
// of its own: compiled into the plain ones it slowed layers that never use it.
constexpr int kModePairs = 2;
constexpr int kModePlane = 3;  // plane staging (see apply_entry_plane)
constexpr int kModeCols = 4;   // column blocks: a lane's P outputs run along a row
constexpr int kModeColsPair = 5;  // column blocks over two images side by side
constexpr int kModeColsPairTaps = 6;  // kModeColsPair with tap-pair segments
template <int P, int Q, int S_CT, int ST_CT, int LR, int MODE = 0, int PLANE_RS = 0>
__global__ void __launch_bounds__(kWarps * 32, 2)
    spconv_fwd_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmap) {
    constexpr bool PAIRS = MODE == kModePairs || MODE == kModeColsPairTaps;
    constexpr bool PLANE = MODE == kModePlane;
    // Column blocks (stride 1): lane (ly, lx) holds outputs (ly, lx*P + r) of
    // an LR x (LC*P) tile, so widths that are multiples of LC*P but not of 32
    // leave no lane idle; a tap's P inputs are consecutive words.
    // Image-pair column blocks (outputs 22..28 wide): four lane rows of eight
    // lanes; lanes 0..3 of a row cover image 2n, lanes 4..7 image 2n + 1,
    // each lane seven consecutive outputs, so a 4 x 28 tile of each image
    // leaves no lane idle (28-wide outputs waste 4 of 32 lanes otherwise).
    // The stage holds the two images' sub-tiles pair_off words apart.
    constexpr bool PAIR = MODE == kModeColsPair || MODE == kModeColsPairTaps;
    constexpr bool COLS = MODE == kModeCols || PAIR;
    static_assert(!COLS || ST_CT == 1, "column blocks: stride 1");
    static_assert(!PAIR || (LR == 4 && P == 7), "image-pair column blocks: 4 x (2 x 28)");
    static_assert(!PLANE || (S_CT == 3 && ST_CT == 1 && LR == 2), "plane staging: 3x3, two lane rows");
    // (MODE 0 with PLANE_RS: the tight-pitch tiles, PLANE_RS their row pitch)
    constexpr bool TIGHT = MODE == 0 && PLANE_RS != 0;
    constexpr int LEAD = TIGHT ? kTightLead : 0;
    static_assert(PLANE || TIGHT || PLANE_RS == 0, "a fixed row step is a plane-staging instance");
    static_assert(!TIGHT || (S_CT == 3 && ST_CT == 1 && LR == 1), "tight pitch: 3x3, one lane row");
    static_assert(!PAIRS || Q == 2 || Q == 4, "tap pairs: 2 or 4 output channels per warp");
    static_assert(Q <= 8, "at most eight output channels per warp (the slot table in shared memory)");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int stage_done[2];  // warps that have released a stage (TMA path)
    __shared__ int issued[2];      // copy phases issued into each stage
    // One-block tiles: the group's slot table (output channel and next part
    // of each slot) for the write-back, so that its lookups cost no global
    // round trips (one per slot and per link of a split row otherwise).
    __shared__ int oc_sh[kWarps * 8], next_sh[kWarps * 8];
    // stage buffers start on a 128-byte boundary (TMA destination)
    unsigned char *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    constexpr int LC = kLanes / LR;  // lanes per lane row = output columns of a tile
    constexpr int ROW_STEP =
        COLS ? 1
             : TIGHT ? PLANE_RS
             : (S_CT && !PLANE) ? LR * (ST_CT == 1 ? row_pitch_s1(S_CT, LR)
                                                   : ST_CT * ST_CT * phase_pitch_for(S_CT, ST_CT))
                                : 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ly = lane / LC, lx = lane % LC;  // lane row / column of this thread
    const int st = ST_CT ? ST_CT : p.stride;
    const int row_step = COLS ? 1 : LR * st * p.row_pitch;  // between this lane's outputs

    // Block order (clusters run along x): channel-split rank fastest, then
    // either the tile (groups in grid y: the heaviest groups, dense ones,
    // start first) or, when the input does not fit in L2, the group (grid y =
    // 1: all groups of a tile run together and share its input through L2).
    const int split = p.split;
    int b = blockIdx.x;
    const int kr = b % split;
    b /= split;
    int group = blockIdx.y;
    if (p.group_fast) {
        group = b % p.groups;
        b /= p.groups;
    }
    const int tx = b % p.tiles_x;
    b /= p.tiles_x;
    const int ty = b % p.tiles_y;
    const int n = b / p.tiles_y;
    const int k_begin = kr * p.num_chunks / split;
    const int k_end = (kr + 1) * p.num_chunks / split;
    const int iy0 = ty * (COLS ? LR : LR * P) * st - p.pad;
    const int ix0 = tx * (PAIR ? (LC / 2) * P : COLS ? LC * P : LC) * st - p.pad;
    // images of the block's tile (image pairs: n counts pairs) and of this lane
    const int img0 = PAIR ? 2 * n : n;
    const int img1 = img0 + 1;  // (image pairs) the second image, if < N
    const int n_out = PAIR ? img0 + (lx >= LC / 2 ? 1 : 0) : n;
    const int nmine = k_end - k_begin;
    const int nslot = kWarps * Q;
    const unsigned int tr_block = blockIdx.y * gridDim.x + blockIdx.x;
    const bool tr_on = kTrace && p.trace != nullptr && tr_block < (unsigned)kTraceBlocks;
    unsigned long long tr_start = 0;
    if (tr_on && threadIdx.x == 0) tr_start = global_ns();

    // Barrier set-up first: its release fence would otherwise wait for the
    // global loads below (a whole memory round trip before the first copy).
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        stage_done[0] = 0;
        stage_done[1] = 0;
        issued[0] = 0;
        issued[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    }
    if constexpr (TIGHT) {
        // the lead words of the block's stages (read by the first row's left
        // taps; a block of one chunk has one stage)
        for (int i = threadIdx.x; i < (nmine > 1 ? 2 : 1) * LEAD; i += blockDim.x)
            reinterpret_cast<float *>(smem + (size_t)(i / LEAD) * p.stage_bytes)[i % LEAD] = 0.f;
    }
    if constexpr (PLANE) {
        // stage input regions start zeroed: the margins (and a last, partial
        // chunk's tail) are read by taps that leave the image, with weight 0
        const int nz = (nmine > 1 ? 2 : 1) * (p.stage_bytes / 16);
        float4 *z = reinterpret_cast<float4 *>(smem);
        for (int i = threadIdx.x; i < nz; i += blockDim.x) {
            const int sidx = i / (p.stage_bytes / 16);
            if ((i - sidx * (p.stage_bytes / 16)) * 16 < p.in_stage_bytes) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the bulk copies (async proxy) later overwrite part of these bytes:
        // each thread orders its own generic-proxy zero stores before them
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    }
    __syncthreads();

    // Loads that nothing computed here feeds, issued before any wait so that
    // their latency overlaps the pipeline: the group's flags, the first
    // blobs' offsets (issuing thread) and the output channel (+ chain link)
    // of this warp's first output item.
    const int gflags =
        dbg_ok(group < p.groups, p.err) ? p.group_flags[group] : 0;
    const bool dense = (gflags & 1) != 0;
    const bool has_parts = (gflags & 2) != 0;
    uint32_t pre_off[3] = {0u, 0u, 0u};
    if (threadIdx.x == 0 && nmine > 0 && p.blob_stride16 == 0 &&
        dbg_ok(group * p.num_chunks + k_end <= p.groups * p.num_chunks, p.err)) {
        const uint32_t *bo = p.blob_off + group * p.num_chunks + k_begin;
        pre_off[0] = bo[0];
        pre_off[1] = bo[1];
        if (nmine > 1) pre_off[2] = bo[2];
    }
    const int item0_slot =
        split == 1 ? warp * Q : kr * nslot / split + warp / P;  // first item's slot
    const bool item0_valid =
        split == 1 ? true : warp < ((kr + 1) * nslot / split - kr * nslot / split) * P;
    int pre_m = -1, pre_next = -1;
    if (item0_valid) {
        pre_m = slot_oc_at(p, group * nslot + item0_slot);
        pre_next = slot_next_at(p, group * nslot + item0_slot);
    }
    // (the last warp copies the slot table while the first stage is in
    // flight; the barrier after the pipeline publishes it)
    if (split == 1 && warp == kWarps - 1)
        for (int i = lane; i < nslot; i += 32) {
            oc_sh[i] = slot_oc_at(p, group * nslot + i);
            next_sh[i] = slot_next_at(p, group * nslot + i);
        }
    // Push-mode cluster reduction: this block announces that it is running;
    // the matching wait comes before its first store into another block.
    const bool push = split > 1 && p.push;
    if (push) asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");

    // Enqueue chunk k into stage s.  `issuer` (one thread) arms the stage's
    // mbarrier and issues the bulk copies; without TMA every thread also
    // stages its share of the input with cp.async.
    // (weights: arm the stage's mbarrier for all its bytes and copy the blob;
    // input: copy the input tile, which completes on the same mbarrier.)
    // (bounds-checked build: the staged input of a chunk fits its region; a
    // copy that would not is skipped)
    auto input_fits = [&](int c0) {
        const size_t in_bytes =
            PLANE ? kPlaneLead * sizeof(float) + (size_t)min(p.chunk, p.C - c0) * p.H * p.W * 4u
                  : (p.use_tma ? (size_t)p.in_tma_bytes + LEAD * sizeof(float) : 0u);
        return !kDebug || in_bytes <= (size_t)p.in_stage_bytes;
    };
    auto issue = [&](int k, int s, bool issuer, bool weights, bool input) {
        unsigned char *base = smem + (size_t)s * p.stage_bytes;
        const int c0 = k * p.chunk;
        const bool in_fits = input_fits(c0);
        if (issuer && weights) {
            ++issued[s];  // one writer per stage at a time (the thread that frees it)
            uint32_t o0, blob_bytes;
            if (p.blob_stride16) {  // fixed-stride blobs: position from the indices alone
                o0 = (uint32_t)(group * p.num_chunks + k) * p.blob_stride16;
                blob_bytes = p.blob_stride16 * 16u;
            } else {
                const int i = k - k_begin;
                o0 = i < 2 ? pre_off[i] : p.blob_off[group * p.num_chunks + k];
                const uint32_t o1 =
                    i < 2 ? pre_off[i + 1] : p.blob_off[group * p.num_chunks + k + 1];
                blob_bytes = (o1 - o0) * 16u;
            }
            if (!dbg_ok(group * p.num_chunks + k < p.groups * p.num_chunks &&
                            (int64_t)o0 * 16 + blob_bytes <= p.blob_bytes &&
                            blob_bytes <= (uint32_t)(p.stage_bytes - p.in_stage_bytes),
                        p.err))
                blob_bytes = 0;  // (bounds-checked build) the copy is skipped
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            const uint32_t in_bytes =
                !in_fits ? 0u
                         : PLANE ? (uint32_t)(min(p.chunk, p.C - c0) * p.H * p.W) * 4u
                                 : (p.use_tma ? (uint32_t)p.in_tma_bytes : 0u);
            if (!in_fits) dbg_ok(false, p.err);
            mbar_expect_tx(&bar[s], blob_bytes + in_bytes);
            if (!kDebug || blob_bytes > 0)
                bulk_load(base + p.in_stage_bytes, p.blobs + (size_t)o0 * 16u, blob_bytes, &bar[s]);
        }
        if constexpr (PLANE) {
            // the chunk's planes are contiguous in the input (and start on a
            // 16-byte boundary: H * W is a multiple of 4)
            if (issuer && input && in_fits) {
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                const size_t hw = (size_t)p.H * p.W;
                bulk_load(base + kPlaneLead * sizeof(float), p.x + ((size_t)n * p.C + c0) * hw,
                          (uint32_t)(min(p.chunk, p.C - c0) * hw * sizeof(float)), &bar[s]);
            }
            return;
        }
        // (image pairs: the box spans both images, the second landing pair_off
        // words after the first -- one 128-byte aligned destination; an image
        // past the batch reads as zeros)
        if (issuer && input && p.use_tma && in_fits)
            tma_load_4d(base + LEAD * sizeof(float), &tmap, ix0 - p.shift, iy0, c0, img0, &bar[s]);
        if (input && !p.use_tma) {
            for (int h = 0; h < (PAIR && img1 < p.N ? 2 : 1); ++h) {
                float *dst = reinterpret_cast<float *>(base) + h * p.pair_off;
                if (ST_CT == 1 && p.pairs)
                    stage_input_cp_async_pairs(p, dst, img0 + h, c0, min(p.chunk, p.C - c0), iy0,
                                               ix0);
                else
                    stage_input_cp_async<ST_CT>(p, dst, img0 + h, c0, min(p.chunk, p.C - c0),
                                                iy0, ix0);
            }
            cp_async_commit();
        }
    };

    float acc[Q][P];
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
        for (int r = 0; r < P; ++r) acc[q][r] = 0.f;

    bool failed = false;
    // The weight blobs do not depend on earlier kernels: their copies start
    // before the wait below, which (with programmatic dependent launch) lets
    // this prologue overlap the previous kernel on the stream.  Past the wait
    // that kernel has completed and its writes are visible, so the input may
    // be read and the output written.
    if (nmine > 0) issue(k_begin, 0, threadIdx.x == 0, true, false);
    if (nmine > 1) issue(k_begin + 1, 1, threadIdx.x == 0, true, false);
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (nmine > 0) issue(k_begin, 0, threadIdx.x == 0, false, true);
    if (nmine > 1) issue(k_begin + 1, 1, threadIdx.x == 0, false, true);
    for (int it = 0; it < nmine && !failed; ++it) {
        const int s = it & 1;
        if (!p.use_tma && !PLANE) {
            if (it + 1 < nmine)
                cp_async_wait_all_but_one();
            else
                cp_async_wait_all();
        }
        const bool ok = mbar_wait_bounded(&bar[s], (uint32_t)((it >> 1) & 1));
        if (p.use_tma || PLANE) {
            // warps run independently; a warp that timed out stops
            failed = !ok;
        } else {
            failed = __syncthreads_or(!ok) != 0;  // cp.async data of all threads
        }
        if (failed) break;
        if (tr_on && it == 0 && threadIdx.x == 0) p.trace[(size_t)tr_block * 4 + 1] = global_ns();
        const unsigned char *base = smem + (size_t)s * p.stage_bytes;
        const float *sb = reinterpret_cast<const float *>(base) + LEAD + ly * st * p.row_pitch +
                          (PAIR ? (lx >= LC / 2 ? p.pair_off : 0) + (lx % (LC / 2)) * P
                                : COLS ? lx * P : lx);
        if constexpr (PLANE) {
            // dense planes: lanes past the image's width read the spare banks
            // 2W .. 31 (finite values, outputs discarded), so the 32 reads of a
            // load stay in distinct banks
            sb = reinterpret_cast<const float *>(base) +
                 (lx < p.W ? ly * p.W + lx : 2 * p.W + ly * (LC - p.W) + (lx - p.W));
        }
        const uint32_t *hdr = reinterpret_cast<const uint32_t *>(base + p.in_stage_bytes);
        // this stage's staged input and the end of its weight blob
        const Span sp{reinterpret_cast<const float *>(base),
                      reinterpret_cast<const float *>(base + p.in_stage_bytes), p.err};
        const unsigned char *blob_end = base + p.stage_bytes;
        if constexpr (kDenseTaps<S_CT, ST_CT> && Q <= 4 && COLS && S_CT == 3) {
            if (dense) {
                const int k = k_begin + it;
                run_dense_chunk_cols<P, Q, S_CT>(
                    acc, sb + p.shift, hdr, reinterpret_cast<const float4 *>(hdr + p.dense_mask_words),
                    warp, p.chunk, min(p.chunk, p.C - k * p.chunk), p.plane, p.row_pitch, sp,
                    blob_end);
            }
        }
        if constexpr (kDenseTaps<S_CT, ST_CT> && Q <= 4 && !PLANE && !COLS) {
            if (dense) {
                const int k = k_begin + it;
                run_dense_chunk<P, Q, S_CT, LR, (TIGHT ? PLANE_RS : row_pitch_s1(S_CT, LR))>(
                    acc, sb + p.shift, hdr, reinterpret_cast<const float4 *>(hdr + p.dense_mask_words),
                    warp, p.chunk, min(p.chunk, p.C - k * p.chunk), p.plane, sp, blob_end);
            }
        }
        if (!dense && p.fmt == 0) {
            const float2 *ent = reinterpret_cast<const float2 *>(hdr + p.hdr_words);
            const int ent_cap = (int)((blob_end - reinterpret_cast<const unsigned char *>(ent)) / 8);
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int j0 = (int)hdr[warp * Q + q];
                const int j1 = (int)hdr[warp * Q + q + 1];
                if (!dbg_ok(0 <= j0 && j0 <= j1 && j1 <= ent_cap, p.err)) continue;
                if constexpr (PLANE) {
                    const uint32_t lanebits = (lx == 0 ? 1u : 0u) | (lx == p.W - 1 ? 2u : 0u) |
                                              (ly == 0 ? 4u : 0u) | (ly == LR - 1 ? 8u : 0u);
                    run_segment_plane<P, PLANE_RS, 4>(acc[q], sb, ent, j0, j1, row_step, lanebits,
                                                      sp);
                } else {
                    // Q = 8 instances are at the register cap: no unrolling there
                    run_segment<P, ROW_STEP, (Q >= 8 ? 1 : 4)>(acc[q], sb, ent, j0, j1, row_step,
                                                               sp);
                }
            }
            if constexpr (PAIRS)
                run_pairs<P, Q, ROW_STEP>(acc, sb, hdr + kWarps * Q + 1 + warp * (Q * (Q - 1) / 2),
                                          reinterpret_cast<const float4 *>(ent), row_step, sp,
                                          ent_cap / 2);
        } else if (!dense) {
            const uint32_t *ent = hdr + p.hdr_words;
            const int ent_cap = (int)((blob_end - reinterpret_cast<const unsigned char *>(ent)) / 4);
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int j0 = (int)hdr[warp * Q + q];
                const int j1 = (int)hdr[warp * Q + q + 1];
                if (!dbg_ok(0 <= j0 && j0 <= j1 && j1 <= ent_cap, p.err)) continue;
                run_segment_words<P, ROW_STEP, ST_CT>(acc[q], sb, ent, j0, j1, p, row_step, sp);
            }
        }
        if (p.use_tma || PLANE) {
            // Release stage s without a block barrier: each warp counts itself
            // out; the warp that completes the count refills the stage (its
            // generic-proxy reads are ordered before the async-proxy copy by
            // the fences).  Faster warps move on to the other stage.
            if (it + 2 < nmine) {
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    const int old = atomicAdd(&stage_done[s], 1);
                    if (old == kWarps - 1) {
                        stage_done[s] = 0;
                        __threadfence_block();
                        issue(k_begin + it + 2, s, true, true, true);
                    }
                }
            }
        } else {
            __syncthreads();  // stage s is free again
            if (it + 2 < nmine) issue(k_begin + it + 2, s, threadIdx.x == 0, true, true);
        }
    }
    // The next kernel on the stream may start launching (it waits for this
    // grid to complete before touching memory that this grid uses).
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    // Every warp is out of the pipeline.  If any gave up waiting, the whole
    // block writes no outputs; its copies still in flight (at most one phase
    // per stage, since a stage is refilled only after it was consumed) are
    // waited for, again with a limit, before shared memory can go away.  A
    // drain that runs out too is recorded apart (bit 1): a copy may then still
    // be writing into shared memory that the SM's next block will own.
    failed = __syncthreads_or(failed) != 0;
    if (tr_on && threadIdx.x == 0) {
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[(size_t)tr_block * 4 + 0] = tr_start;
        p.trace[(size_t)tr_block * 4 + 2] = global_ns();
        p.trace[(size_t)tr_block * 4 + 3] = (unsigned long long)smid |
                                            ((unsigned long long)group << 16) |
                                            ((unsigned long long)(gflags & 0xff) << 32);
    }
    if (failed) {
        if (!p.use_tma && !PLANE) cp_async_wait_all();
        if (threadIdx.x == 0) {
            atomicOr(p.err, 1u);
            for (int st2 = 0; st2 < 2; ++st2)
                if (issued[st2] > 0 &&
                    !mbar_wait_bounded(&bar[st2], (uint32_t)((issued[st2] - 1) & 1)))
                    atomicOr(p.err, 2u);
        }
        __syncthreads();
    }

    // (bounds-checked build) end of the launch's dynamic shared memory
    const unsigned char *smem_end = smem_raw + p.smem_bytes;
    // This lane's outputs r = 0 .. P-1: rows oy0 + LR * r of column ox, or
    // (column blocks) columns ox + r of row oy0.
    const int ox = PAIR ? tx * ((LC / 2) * P) + (lx % (LC / 2)) * P
                        : COLS ? tx * (LC * P) + lx * P : tx * LC + lx;
    const int oy0 = COLS ? ty * LR + ly : ty * (LR * P) + ly;
    const bool lane_out = (COLS ? oy0 < p.E : ox < p.F) && n_out < p.N;  // the lane has outputs
    auto out_ok = [&](int r) { return COLS ? ox + r < p.F : oy0 + LR * r < p.E; };
    auto out_at = [&](int r) {  // offset of output r within its (n, m) plane
        return COLS ? (size_t)oy0 * p.F + ox + r : (size_t)(oy0 + LR * r) * p.F + ox;
    };
    if constexpr (COLS) {
        if (split == 1 && !has_parts) {
            // Column blocks: lane (ly, lx) holds tile positions 7 lane + r
            // (row-major LR x LC*P).  Each warp passes its slots through
            // shared memory (free past the barrier above) so that a store
            // instruction writes 32 consecutive positions of the tile, not
            // 32 scattered ones.
            if (failed) return;
            float *tb = reinterpret_cast<float *>(smem) + (size_t)warp * Q * (P * 32);
            if (!dbg_ok(reinterpret_cast<const unsigned char *>(tb + Q * P * 32) <= smem_end, p.err))
                return;
#pragma unroll
            for (int q = 0; q < Q; ++q)
#pragma unroll
                for (int r = 0; r < P; ++r) tb[q * (P * 32) + lane * P + r] = acc[q][r];
            __syncwarp();
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int m = oc_sh[warp * Q + q];
                if (m < 0) continue;
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    // tile position t: row t / (LC*P); with image pairs the row's
                    // first half is image 2n, its second half image 2n + 1
                    const int t = i * 32 + lane;
                    const int oy = ty * LR + t / (LC * P);
                    const int col = t % (LC * P);
                    const int half = PAIR ? col / ((LC / 2) * P) : 0;
                    const int oxt = PAIR ? tx * ((LC / 2) * P) + col % ((LC / 2) * P)
                                         : tx * (LC * P) + col;
                    const int img = img0 + half;
                    if (oy < p.E && oxt < p.F && img < p.N && dbg_ok(m < p.M, p.err))
                        p.y[(((size_t)img * p.M + m) * p.E + oy) * p.F + oxt] =
                            finish(p, m, tb[q * (P * 32) + t]);
                }
            }
            return;
        }
    }
    if (split == 1 && !has_parts) {
        if (failed || !lane_out) return;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int m = oc_sh[warp * Q + q];
            if (m < 0) continue;
            float *yo = p.y + ((size_t)n_out * p.M + m) * p.E * p.F;
#pragma unroll
            for (int r = 0; r < P; ++r)
                if (out_ok(r) && dbg_ok(m < p.M, p.err)) yo[out_at(r)] = finish(p, m, acc[q][r]);
        }
        return;
    }

    if constexpr (Q <= 2) {  // push mode is planned for narrow instances only
        if (push) {
            // ---- cluster reduction by pushing (groups without split rows).  Each
            // block stores its partial sums straight into the receive buffer of
            // the block that owns the slot (distributed shared memory, a region
            // apart from the stage buffers, so an owner still computing is not
            // disturbed); one cluster barrier publishes them; each owner adds its
            // slots' partials in rank order -- the pull path's order, so the
            // results are identical -- from its own shared memory, and needs no
            // barrier after that because no other block reads it.
            float *recv = reinterpret_cast<float *>(smem + p.recv_off);  // [rank][own][P][32]
            const int own = (nslot + split - 1) / split;  // most slots a rank owns
            // (bounds-checked build) every rank's buffer ends inside its shared memory
            const bool recv_ok = dbg_ok(
                reinterpret_cast<const unsigned char *>(recv + split * own * P * 32) <= smem_end,
                p.err);
            cg::cluster_group cluster = cg::this_cluster();
            asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");  // all blocks started
            if (!failed && recv_ok) {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int sl = warp * Q + q;
                    int o = split - 1;  // owner: the last rank whose range starts at or before sl
                    while (o > 0 && o * nslot / split > sl) --o;
                    if (!dbg_ok(sl - o * nslot / split < own, p.err)) continue;
                    float *dst = cluster.map_shared_rank(recv, o) +
                                 ((kr * own + (sl - o * nslot / split)) * P) * 32 + lane;
#pragma unroll
                    for (int r = 0; r < P; ++r) dst[r * 32] = acc[q][r];
                }
            }
            asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
            asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
            if (failed || !lane_out || !recv_ok) return;
            const int s_begin = kr * nslot / split, s_end = (kr + 1) * nslot / split;
            const int items = (s_end - s_begin) * P;
            for (int item = warp; item < items; item += kWarps) {
                const int li = item / P, r = item % P;
                const int m = item == warp ? pre_m : slot_oc_at(p, group * nslot + s_begin + li);
                if (m < 0) continue;
                float v[kMaxSplit];
#pragma unroll
                for (int j = 0; j < kMaxSplit; ++j)
                    v[j] = j < split ? recv[((j * own + li) * P + r) * 32 + lane] : 0.f;
                float sum = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxSplit; ++j)
                    if (j < split) sum += v[j];
                if (out_ok(r) && dbg_ok(m < p.M, p.err))
                    p.y[((size_t)n_out * p.M + m) * p.E * p.F + out_at(r)] = finish(p, m, sum);
            }
            return;
        }
    }

    // ---- partial sums through shared memory: parts of split rows (summed in
    // chain order) and/or the blocks of a channel-split cluster (summed in rank
    // order, through distributed shared memory).  Both orders are fixed, so the
    // result is deterministic.  The stage buffers are free: every issued copy
    // has been consumed.
    float *part = reinterpret_cast<float *>(smem);  // [warp * Q + q][P][32]
    if (!dbg_ok(reinterpret_cast<const unsigned char *>(part + kWarps * Q * P * 32) <= smem_end,
                p.err))
        failed = true;  // (bounds-checked build) no room: write nothing
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
        for (int r = 0; r < P; ++r)
            if (!kDebug || !failed) part[((warp * Q + q) * P + r) * 32 + lane] = acc[q][r];
    if (split == 1) {
        __syncthreads();
        if (failed || !lane_out) return;
        for (int q = 0; q < Q; ++q) {
            const int sl = warp * Q + q;
            const int m = oc_sh[sl];
            if (m < 0) continue;
            const int next0 = next_sh[sl];
            float *yo = p.y + ((size_t)n_out * p.M + m) * p.E * p.F;
            for (int r = 0; r < P; ++r) {
                float sum = part[(sl * P + r) * 32 + lane];
                for (int c = next0; c >= 0 && dbg_ok(c < nslot, p.err); c = next_sh[c])
                    sum += part[(c * P + r) * 32 + lane];
                if (out_ok(r) && dbg_ok(m < p.M, p.err)) yo[out_at(r)] = finish(p, m, sum);
            }
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int s_begin = kr * nslot / split, s_end = (kr + 1) * nslot / split;
    if constexpr (Q <= 2) {
        if (!failed && lane_out) {
            // (slot, output row) items spread over all warps; the ranks' partials
            // of one item are loaded back to back, then added in rank order
            const int items = (s_end - s_begin) * P;
            for (int item = warp; item < items; item += kWarps) {
                const int sl = s_begin + item / P, r = item % P;
                const bool first = item == warp;
                const int m = first ? pre_m : slot_oc_at(p, group * nslot + sl);
                if (m < 0) continue;
                float sum = 0.f;
                for (int c = sl, next = first ? pre_next : slot_next_at(p, group * nslot + sl);
                     c >= 0 && dbg_ok(c < nslot, p.err);
                     c = next, next = c >= 0 ? slot_next_at(p, group * nslot + c) : -1) {
                    float v[kMaxSplit];
#pragma unroll
                    for (int j = 0; j < kMaxSplit; ++j)
                        v[j] = j < split ? cluster.map_shared_rank(part, j)[(c * P + r) * 32 + lane]
                                         : 0.f;
#pragma unroll
                    for (int j = 0; j < kMaxSplit; ++j)
                        if (j < split) sum += v[j];
                }
                if (out_ok(r) && dbg_ok(m < p.M, p.err))
                    p.y[((size_t)n_out * p.M + m) * p.E * p.F + out_at(r)] = finish(p, m, sum);
            }
        }
    } else {
        // wide instances: one warp per slot, ranks and rows in sequence (compact
        // code; these instances carry the register-heavy dense-tap path)
        if (!failed && lane_out) {
            for (int sl = s_begin + warp; sl < s_end; sl += kWarps) {
                const int m = slot_oc_at(p, group * nslot + sl);
                if (m < 0) continue;
                float *yo = p.y + ((size_t)n_out * p.M + m) * p.E * p.F;
                for (int r = 0; r < P; ++r) {
                    float sum = 0.f;
                    for (int c = sl; c >= 0 && dbg_ok(c < nslot, p.err);
                         c = slot_next_at(p, group * nslot + c))
                        for (int j = 0; j < split; ++j)
                            sum += cluster.map_shared_rank(part, j)[(c * P + r) * 32 + lane];
                    if (out_ok(r) && dbg_ok(m < p.M, p.err)) yo[out_at(r)] = finish(p, m, sum);
                }
            }
        }
    }
    cluster.sync();  // partials stay readable until every block is done
}

using KernelFn = void (*)(const KParams, const CUtensorMap);

// Instances of one output-channel-per-warp count Q (one translation unit each,
// compiled in parallel): the kernel for (S, stride, P, LR), or nullptr.
KernelFn pick_q1(int S, int stride, int P, int LR);
KernelFn pick_q2(int S, int stride, int P, int LR);
KernelFn pick_q4(int S, int stride, int P, int LR);
KernelFn pick_q8(int S, int stride, int P, int LR);
// Tap-pair instances (Q = 4, one lane row; 3x3 and 5x5 stride 1, 11x11 stride 4).
KernelFn pick_pairs(int S, int stride, int P, int Q, int LR);
// Plane-staging instances (3x3 stride 1, two lane rows, Q in {1, 2}); 14-wide
// images (row step 28 words) have their own, with immediate load offsets.
KernelFn pick_plane(int P, int Q, int W);
KernelFn pick_cols(int P, int Q, int LR);
// Image-pair column-block instances (3x3 stride 1, four lane rows of eight),
// and those of 5x5 layers, with or without tap-pair segments.
KernelFn pick_colpair(int P, int Q);
KernelFn pick_colpair5(int P, int Q, bool pairs);
// Tight-pitch instances (3x3 stride 1 pad 1, one lane row, a 32-word pitch).
KernelFn pick_tight(int P, int Q);

// Instantiates the kernels of one Q for the supported kernel widths, strides,
// rows per lane and lane rows.
template <int Q>
KernelFn pick_instances(int S, int stride, int P, int LR) {
    auto by_p = [&](auto pc) -> KernelFn {
        constexpr int PP = decltype(pc)::value;
        if (LR == 2) {
            if (stride != 1) return nullptr;
            if (S == 3) return spconv_fwd_kernel<PP, Q, 3, 1, 2>;
            return spconv_fwd_kernel<PP, Q, 0, 1, 2>;
        }
        if (LR != 1) return nullptr;
        if (S == 3 && stride == 1) return spconv_fwd_kernel<PP, Q, 3, 1, 1>;
        if (S == 5 && stride == 1) return spconv_fwd_kernel<PP, Q, 5, 1, 1>;
        if (S == 11 && stride == 4) return spconv_fwd_kernel<PP, Q, 11, 4, 1>;
        if (stride == 1) return spconv_fwd_kernel<PP, Q, 0, 1, 1>;
        return spconv_fwd_kernel<PP, Q, 0, 0, 1>;
    };
    switch (P) {
        case 7: return by_p(std::integral_constant<int, 7>{});
        case 8: return by_p(std::integral_constant<int, 8>{});
        default: return nullptr;
    }
}

}  // namespace kern
}  // namespace spconv
