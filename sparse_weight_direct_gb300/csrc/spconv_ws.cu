// Weight-stationary forward kernel: one output channel per thread block.
//
// The mapping of Escoin (arXiv 1802.10280), Figs. 5-7 and its data-placement
// discussion: a thread block owns one output channel (one row of the sparse
// M x CRS weight matrix) and keeps that row's weights on chip while it streams
// the input; every nonzero multiplies a window of consecutive input elements,
// consecutive threads own consecutive output positions (so input reads and
// output writes are coalesced), and partial sums stay in registers.  Each
// weight read from shared memory is applied to every output the block owns.
//
// On sm_103a:
//   * the row's entries (fp32 value + a 32-bit word holding the stretched
//     offset c*H*W + r*W + s and the tap (r, s)) are fetched into shared memory
//     by bulk asynchronous copies, two pipeline stages of `piece` entries, each
//     completing on an mbarrier (bounded wait);
//   * the input is read in place through the read-only data path (L1), not
//     staged: the whole image-channel window of a tap is what the block reads,
//     so the 256 KB L1 of the SM plays the role of Escoin's texture cache;
//   * no padded copy of the input is made.  Each thread keeps bit masks of the
//     kernel rows and columns that land inside the image for its outputs and
//     predicates its loads on them; warps whose outputs see no padding at all
//     take a loop without the tests;
//   * a lane owns one output column and P output rows, so one entry read feeds
//     P loads and P FMAs; grid = (output channels, heaviest row first) x
//     (spatial tiles) x (images).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

struct WsParams {
    const float *x;
    float *y;
    const float *bias;  // [M] or nullptr
    int act;            // 0 identity, 1 ReLU
    const unsigned char *ent;  // entries {float value, uint32 word}, rows 16-byte aligned
    const uint32_t *row_info;  // [2 * M]: first entry, entry count of output channel m
    const int *row_order;      // [M]: output channel of grid column x (heaviest first)
    unsigned int *err;
    int C, H, W, M, E, F, R, S, stride, pad;
    int tiles_x;  // spatial tiles along F (grid y = tiles_y * tiles_x)
    int piece;    // entries per pipeline stage (even)
    int64_t ent_bytes;  // bytes of the entries array (bounds-checked build)
};

static __device__ __forceinline__ float ws_finish(const WsParams &p, int m, float v) {
    if (p.bias) v += __ldg(p.bias + m);
    if (p.act == 1) v = fmaxf(v, 0.f);
    return v;
}

// One entry applied to this thread's P outputs.  word = off << 8 | r << 4 | s
// with off = c*H*W + r*W + s; base[i] = iy0_i*W + ix0 of output row i, so
// base[i] + off indexes input (c, iy0_i + r, ix0 + s) of the image.
// Read of input element i of the image (bounds-checked build: i inside the
// image's C*H*W elements, else the read is skipped and gives 0).
static __device__ __forceinline__ float ws_ld(const WsParams &p, const float *xn, int i) {
    if (!dbg_ok((unsigned)i < (unsigned)(p.C * p.H * p.W), p.err)) return 0.f;
    return __ldg(xn + i);
}

template <int P, bool CHECK>
static __device__ __forceinline__ void ws_apply(const WsParams &p, float (&acc)[P], const float *xn,
                                                const int (&base)[P], const uint32_t (&rmask)[P],
                                                uint32_t cmask, float v, uint32_t word) {
    const int off = (int)(word >> 8);
    if constexpr (CHECK) {
        const uint32_t r = (word >> 4) & 15u, s = word & 15u;
        const uint32_t cv = (cmask >> s) & 1u;
#pragma unroll
        for (int i = 0; i < P; ++i)
            if ((rmask[i] >> r) & cv) acc[i] = fmaf(v, ws_ld(p, xn, base[i] + off), acc[i]);
    } else {
#pragma unroll
        for (int i = 0; i < P; ++i) acc[i] = fmaf(v, ws_ld(p, xn, base[i] + off), acc[i]);
    }
}

// Entries [0, len) of a staged piece (16-byte aligned, two entries per load).
template <int P, bool CHECK>
static __device__ __forceinline__ void ws_run(const WsParams &p, float (&acc)[P], const float *xn,
                                              const int (&base)[P], const uint32_t (&rmask)[P],
                                              uint32_t cmask, const float2 *e, int len) {
    int j = 0;
#pragma unroll 2
    for (; j + 1 < len; j += 2) {
        const float4 q = *reinterpret_cast<const float4 *>(e + j);
        ws_apply<P, CHECK>(p, acc, xn, base, rmask, cmask, q.x, __float_as_uint(q.y));
        ws_apply<P, CHECK>(p, acc, xn, base, rmask, cmask, q.z, __float_as_uint(q.w));
    }
    if (j < len) {
        const float2 q = e[j];
        ws_apply<P, CHECK>(p, acc, xn, base, rmask, cmask, q.x, __float_as_uint(q.y));
    }
}

// P: output rows per lane; LR: lane rows (2 for outputs at most 16 wide).
template <int P, int LR>
__global__ void __launch_bounds__(kWarps * 32)
    spconv_ws_kernel(const __grid_constant__ WsParams p) {
    extern __shared__ __align__(16) unsigned char ws_smem_raw[];
    __shared__ __align__(8) uint64_t bar[2];
    // stage buffers start on a 16-byte boundary (bulk-copy destination)
    unsigned char *ws_smem = ws_smem_raw + ((16u - (smem_u32(ws_smem_raw) & 15u)) & 15u);
    constexpr int LC = kLanes / LR;          // output columns of a tile
    constexpr int ROWS = kWarps * LR;        // output rows covered by one step of i
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ly = lane / LC, lx = lane % LC;
    const int m0 = dbg_ok(blockIdx.x < (unsigned)p.M, p.err) ? p.row_order[blockIdx.x] : 0;
    const int m = dbg_ok((unsigned)m0 < (unsigned)p.M, p.err) ? m0 : 0;
    const int tx = blockIdx.y % p.tiles_x, ty = blockIdx.y / p.tiles_x;
    const int n = blockIdx.z;
    const uint32_t first = p.row_info[2 * m], count = p.row_info[2 * m + 1];

    // This thread's outputs: column ox, rows oy0 + i * ROWS.  Positions past
    // the layer's edge are clamped onto it for the loads and never stored.
    const int ox = tx * LC + lx;
    const int oy0 = ty * (ROWS * P) + warp * LR + ly;
    const int ix0 = min(ox, p.F - 1) * p.stride - p.pad;
    const uint32_t full_s = (1u << p.S) - 1u, full_r = (1u << p.R) - 1u;
    uint32_t cmask = 0;  // bit s: input column ix0 + s lies inside the image
    for (int s = 0; s < p.S; ++s)
        if ((unsigned)(ix0 + s) < (unsigned)p.W) cmask |= 1u << s;
    bool inside = cmask == full_s;
    int base[P];
    uint32_t rmask[P];
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int iy0 = min(oy0 + i * ROWS, p.E - 1) * p.stride - p.pad;
        uint32_t rm = 0;
        for (int r = 0; r < p.R; ++r)
            if ((unsigned)(iy0 + r) < (unsigned)p.H) rm |= 1u << r;
        rmask[i] = rm;
        inside = inside && rm == full_r;
        base[i] = iy0 * p.W + ix0;
    }
    const bool interior = __all_sync(0xffffffffu, inside);
    const float *xn = p.x + (size_t)n * p.C * p.H * p.W;

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    }
    __syncthreads();

    const int npieces = (int)((count + (uint32_t)p.piece - 1) / (uint32_t)p.piece);
    // Piece k of the row into stage k & 1 (issuing thread).  Rows start on an
    // even entry and pieces are even, so the copy starts 16-byte aligned; its
    // length is rounded up to whole 16 bytes (the entry after an odd row end
    // is padding or the next row, copied but not used).
    auto issue = [&](int k) {
        const uint32_t j0 = first + (uint32_t)k * (uint32_t)p.piece;
        const uint32_t len = min((uint32_t)p.piece, count - (uint32_t)k * (uint32_t)p.piece);
        uint32_t bytes = ((len + 1u) & ~1u) * 8u;
        // (bounds-checked build) the piece lies inside the entries and its stage
        if (!dbg_ok((int64_t)j0 * 8 + bytes <= p.ent_bytes && bytes <= (uint32_t)p.piece * 8u &&
                        (unsigned)m < (unsigned)p.M,
                    p.err))
            bytes = 0;
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        mbar_expect_tx(&bar[k & 1], bytes);
        if (!kDebug || bytes > 0)
            bulk_load(ws_smem + (size_t)(k & 1) * p.piece * 8, p.ent + (size_t)j0 * 8, bytes,
                      &bar[k & 1]);
    };
    if (threadIdx.x == 0) {
        if (npieces > 0) issue(0);
        if (npieces > 1) issue(1);
    }

    float acc[P];
#pragma unroll
    for (int i = 0; i < P; ++i) acc[i] = 0.f;
    bool failed = false;
    int k = 0;
    for (; k < npieces; ++k) {
        const bool ok = mbar_wait_bounded(&bar[k & 1], (uint32_t)((k >> 1) & 1));
        failed = __syncthreads_or(!ok) != 0;
        if (failed) break;
        const float2 *e = reinterpret_cast<const float2 *>(ws_smem + (size_t)(k & 1) * p.piece * 8);
        const int len = (int)min((uint32_t)p.piece, count - (uint32_t)k * (uint32_t)p.piece);
        if (interior)
            ws_run<P, false>(p, acc, xn, base, rmask, cmask, e, len);
        else
            ws_run<P, true>(p, acc, xn, base, rmask, cmask, e, len);
        __syncthreads();  // stage k & 1 is free again
        if (threadIdx.x == 0 && k + 2 < npieces) issue(k + 2);
    }
    if (failed) {
        // Let the copies still in flight (pieces k and k + 1, if issued) land
        // before the block's shared memory goes away, again with a limit.
        // A drain that runs out too is recorded apart (bit 1): a copy may then
        // still be writing into shared memory that the SM's next block will own.
        if (threadIdx.x == 0) {
            atomicOr(p.err, 1u);
            for (int j = k; j < min(k + 2, npieces); ++j)
                if (!mbar_wait_bounded(&bar[j & 1], (uint32_t)((j >> 1) & 1))) atomicOr(p.err, 2u);
        }
        return;
    }
    if (ox >= p.F) return;
    float *yo = p.y + ((size_t)n * p.M + m) * p.E * p.F + ox;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int oy = oy0 + i * ROWS;
        if (oy < p.E && dbg_ok((unsigned)m < (unsigned)p.M, p.err))
            yo[(size_t)oy * p.F] = ws_finish(p, m, acc[i]);
    }
}

using WsKernelFn = void (*)(const WsParams);

template <int LR>
static WsKernelFn ws_pick_lr(int P) {
    switch (P) {
        case 1: return spconv_ws_kernel<1, LR>;
        case 2: return spconv_ws_kernel<2, LR>;
        case 4: return spconv_ws_kernel<4, LR>;
        case 7: return spconv_ws_kernel<7, LR>;
        case 8: return spconv_ws_kernel<8, LR>;
        default: return nullptr;
    }
}

static WsKernelFn ws_pick(int P, int LR) {
    return LR == 1 ? ws_pick_lr<1>(P) : LR == 2 ? ws_pick_lr<2>(P) : nullptr;
}

}  // namespace kern

bool ws_variant_supported(int P, int LR) { return kern::ws_pick(P, LR) != nullptr; }

size_t ws_smem_bytes(const Geometry &g) {
    return (size_t)(g.num_chunks > 1 ? 2 : 1) * g.chunk * 8 + 16;  // + alignment room
}

cudaError_t launch_forward_ws(const Geometry &g, int N, const float *x, float *y,
                              const float *bias, int act, const DeviceArrays &d,
                              cudaStream_t stream) {
    kern::WsKernelFn fn = kern::ws_pick(g.tile_rows, g.lane_rows);
    if (!fn || N < 1 || N > 65535 || g.tiles_y * g.tiles_x > 65535)
        return cudaErrorInvalidConfiguration;
    const size_t smem = ws_smem_bytes(g);
    if (smem > 48 * 1024) {
        if (smem > (size_t)kern::kMaxDynamicSmem) return cudaErrorInvalidConfiguration;
        cudaError_t e = kern::raise_smem_limit(reinterpret_cast<const void *>(fn));
        if (e != cudaSuccess) return e;
    }
    kern::WsParams p;
    p.x = x;
    p.y = y;
    p.bias = bias;
    p.act = act;
    p.ent = d.blobs;
    p.row_info = d.blob_off;
    p.row_order = d.slot_oc;
    p.err = d.err;
    p.C = g.C; p.H = g.H; p.W = g.W; p.M = g.M; p.E = g.E; p.F = g.F;
    p.R = g.R; p.S = g.S; p.stride = g.stride; p.pad = g.pad;
    p.tiles_x = g.tiles_x;
    p.piece = g.chunk;
    p.ent_bytes = d.blob_bytes;
    const dim3 grid((unsigned)g.M, (unsigned)(g.tiles_y * g.tiles_x), (unsigned)N);
    fn<<<grid, kWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spconv
