// Forward kernel of the sparse-weight direct convolution (sm_103a).
//
// What it computes: Tuteja et al., "Theoretical and Empirical Analysis of
// Sparse Convolution", Sec. 3 Eq.(3) -- each output is the sum, over the
// nonzeros of its output channel, of value * input at the padding-shifted
// position -- with stride (Escoin, arXiv 1802.10280, Algorithm 2).
//
// How (one block = one output tile of P rows x 32 columns of one image, for a
// group of 8 * Q output channels):
//   1. stage: the input tile plus halo of a chunk of input channels is copied
//      into shared memory with cp.async (zero-filled outside the image, so the
//      padding needs no branch in the hot loop), double-buffered across chunks
//      (the shared-memory tiling of Sec. 5.1 of the first page);
//   2. accumulate: every warp carries Q output channels; lanes own one output
//      column each and P rows in registers.  A warp walks its channels'
//      packed (value, offset) entries with warp-uniform 16-byte loads (two
//      entries per load, broadcast to all lanes) and, per entry, does P FMAs
//      reading smem[lane_base + offset + p * row_step] -- consecutive lanes read
//      consecutive words, so the reads are bank-conflict free;
//   3. write back: coalesced stores along the output row, predicated for
//      partial tiles (Sec. 5.5 of the first page).
// Offsets are precomputed on the host per nonzero (Escoin's weight stretching),
// against the shared-memory tile layout, so the kernel never decodes (c, r, s).
#include <cuda_runtime.h>

#include <cstdint>

#include "spconv_internal.h"

namespace spconv {
namespace {

struct KParams {
    const float *__restrict__ x;
    float *__restrict__ y;
    const float2 *__restrict__ entries;
    const int *__restrict__ segptr;
    const int *__restrict__ slot_oc;
    int N, C, H, W, M, E, F, stride, pad;
    int tiles_y, tiles_x, in_rows, in_cols, phase_pitch, row_pitch, plane, chunk, num_chunks;
};

__device__ __forceinline__ void cp_async_4(float *smem_dst, const float *gsrc, bool pred) {
    const unsigned saddr = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    const int src_size = pred ? 4 : 0;  // 0 -> the 4 destination bytes are zero-filled
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(saddr), "l"(gsrc),
                 "r"(src_size)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int K>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(K) : "memory");
}

// Stage channels [c0, c0 + cc) of image n, input rows iy0.., columns ix0..
// into buf with the tile layout [channel][row][phase][col / stride].
template <int ST_CT>
__device__ __forceinline__ void stage_chunk(const KParams &p, float *buf, int n, int c0, int cc,
                                            int iy0, int ix0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int st = ST_CT ? ST_CT : p.stride;
    const int rows = cc * p.in_rows;
    for (int rr = warp; rr < rows; rr += nw) {
        const int cl = rr / p.in_rows;
        const int row = rr - cl * p.in_rows;
        const int gy = iy0 + row;
        const bool rowok = gy >= 0 && gy < p.H;
        const float *src = p.x + (((size_t)n * p.C + (c0 + cl)) * p.H + (rowok ? gy : 0)) * p.W;
        float *dst = buf + cl * p.plane + row * p.row_pitch;
        for (int col = lane; col < p.in_cols; col += 32) {
            const int gx = ix0 + col;
            const bool ok = rowok && gx >= 0 && gx < p.W;
            const int phys = (st == 1) ? col : (col % st) * p.phase_pitch + col / st;
            cp_async_4(dst + phys, ok ? src + gx : p.x, ok);
        }
    }
}

template <int P, int ROW_STEP>
__device__ __forceinline__ void apply_entry(float (&acc)[P], const float *sb, float v, int off,
                                            int row_step) {
    const float *s = sb + off;
#pragma unroll
    for (int r = 0; r < P; ++r)
        acc[r] = fmaf(v, s[r * (ROW_STEP ? ROW_STEP : row_step)], acc[r]);
}

// P: output rows per lane; Q: output channels per warp; S_CT/ST_CT: kernel
// width and stride when known at compile time (0 = read from p).
template <int P, int Q, int S_CT, int ST_CT>
__global__ void __launch_bounds__(256, 2) spconv_fwd_kernel(const KParams p) {
    extern __shared__ __align__(16) float smem[];
    constexpr int ROW_STEP = S_CT ? ST_CT * ST_CT * phase_pitch_for(S_CT, ST_CT) : 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int t = blockIdx.x;
    const int tx = t % p.tiles_x;
    t /= p.tiles_x;
    const int ty = t % p.tiles_y;
    const int n = t / p.tiles_y;
    const int st = ST_CT ? ST_CT : p.stride;
    const int row_step = st * p.row_pitch;
    const int slot0 = (blockIdx.y * nw + warp) * Q;
    const int nch = p.num_chunks;
    const int buf_words = p.chunk * p.plane;
    const int iy0 = ty * P * st - p.pad;
    const int ix0 = tx * kTileCols * st - p.pad;

    float acc[Q][P];
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
        for (int r = 0; r < P; ++r) acc[q][r] = 0.f;

    stage_chunk<ST_CT>(p, smem, n, 0, min(p.chunk, p.C), iy0, ix0);
    cp_async_commit();
    for (int k = 0; k < nch; ++k) {
        if (k + 1 < nch) {
            const int c1 = (k + 1) * p.chunk;
            stage_chunk<ST_CT>(p, smem + ((k + 1) & 1) * buf_words, n, c1, min(p.chunk, p.C - c1),
                               iy0, ix0);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *sb = smem + (k & 1) * buf_words + lane;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int *sp = p.segptr + (size_t)(slot0 + q) * (nch + 1) + k;
            int j = __ldg(sp);
            const int j1 = __ldg(sp + 1);
            if ((j & 1) && j < j1) {  // head: bring j to a 16-byte boundary
                const float2 e = __ldg(p.entries + j);
                apply_entry<P, ROW_STEP>(acc[q], sb, e.x, __float_as_int(e.y), row_step);
                ++j;
            }
            for (; j + 1 < j1; j += 2) {
                const float4 e = __ldg(reinterpret_cast<const float4 *>(p.entries + j));
                apply_entry<P, ROW_STEP>(acc[q], sb, e.x, __float_as_int(e.y), row_step);
                apply_entry<P, ROW_STEP>(acc[q], sb, e.z, __float_as_int(e.w), row_step);
            }
            if (j < j1) {  // tail
                const float2 e = __ldg(p.entries + j);
                apply_entry<P, ROW_STEP>(acc[q], sb, e.x, __float_as_int(e.y), row_step);
            }
        }
        __syncthreads();  // buffer (k & 1) is restaged two chunks later
    }

    const int ox = tx * kTileCols + lane;
    if (ox >= p.F) return;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int m = __ldg(p.slot_oc + slot0 + q);
        if (m < 0) continue;
        float *yo = p.y + ((size_t)n * p.M + m) * p.E * p.F + ox;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const int oy = ty * P + r;
            if (oy < p.E) yo[(size_t)oy * p.F] = acc[q][r];
        }
    }
}

using KernelFn = void (*)(const KParams);

template <int P, int Q>
KernelFn pick_sst(int S, int stride) {
    if (S == 3 && stride == 1) return spconv_fwd_kernel<P, Q, 3, 1>;
    if (S == 5 && stride == 1) return spconv_fwd_kernel<P, Q, 5, 1>;
    if (S == 11 && stride == 4) return spconv_fwd_kernel<P, Q, 11, 4>;
    if (stride == 1) return spconv_fwd_kernel<P, Q, 0, 1>;
    return spconv_fwd_kernel<P, Q, 0, 0>;
}

template <int P>
KernelFn pick_q(int S, int stride, int Q) {
    switch (Q) {
        case 1: return pick_sst<P, 1>(S, stride);
        case 2: return pick_sst<P, 2>(S, stride);
        case 4: return pick_sst<P, 4>(S, stride);
        default: return nullptr;
    }
}

KernelFn pick(int S, int stride, int P, int Q) {
    switch (P) {
        case 7: return pick_q<7>(S, stride, Q);
        case 8: return pick_q<8>(S, stride, Q);
        default: return nullptr;
    }
}

}  // namespace

int forward_variant_supported(int S, int stride, int P, int Q) {
    return pick(S, stride, P, Q) ? 0 : -1;
}

cudaError_t launch_forward(const Geometry &g, int N, const float *x, float *y,
                           const DeviceArrays &d, cudaStream_t stream) {
    KernelFn fn = pick(g.S, g.stride, g.tile_rows, g.slots);
    if (!fn) return cudaErrorInvalidConfiguration;
    if (g.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)g.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    KParams p;
    p.x = x;
    p.y = y;
    p.entries = d.entries;
    p.segptr = d.segptr;
    p.slot_oc = d.slot_oc;
    p.N = N; p.C = g.C; p.H = g.H; p.W = g.W; p.M = g.M; p.E = g.E; p.F = g.F;
    p.stride = g.stride; p.pad = g.pad;
    p.tiles_y = g.tiles_y; p.tiles_x = g.tiles_x; p.in_rows = g.in_rows; p.in_cols = g.in_cols;
    p.phase_pitch = g.phase_pitch; p.row_pitch = g.row_pitch; p.plane = g.plane;
    p.chunk = g.chunk; p.num_chunks = g.num_chunks;
    const dim3 grid((unsigned)((int64_t)N * g.tiles_y * g.tiles_x), (unsigned)g.groups, 1);
    fn<<<grid, g.warps * 32, g.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spconv
