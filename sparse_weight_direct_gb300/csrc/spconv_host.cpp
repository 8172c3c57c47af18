// Host side of libspconv: argument validation, the packing of CSR weights into
// the kernel's layout (weight stretching + output-channel binning), device
// upload, and the C ABI declared in include/spconv.h.
//
// Packing follows Escoin (arXiv 1802.10280), "Sparse convolution": dynamic
// indexing with the layout function f(c, y, x) and its shift property
// f(c, y + r, x + s) = f(c, y, x) + f(0, r, s), so each nonzero's column
// (c, r, s) is rewritten once ("weight stretching") into an offset that the
// kernel adds to a per-output-pixel base.  Here f is the layout of the
// shared-memory input tile the kernel stages (channel plane, row, stride
// phase, column), not of the global array.  The per-output-channel ranges
// play the role of the offset array of Tuteja et al., "Theoretical and
// Empirical Analysis of Sparse Convolution", Sec. 5.3.
#include "../../include/spconv.h"

#include <algorithm>
#include <cstring>
#include <new>
#include <numeric>
#include <queue>
#include <vector>

#include "spconv_internal.h"

namespace {

struct HostEntry {
    float value;
    int32_t off;
};
static_assert(sizeof(HostEntry) == 8, "entry must be 8 bytes");

}  // namespace

struct spconv_packed {
    spconv::Geometry g{};
    int64_t nnz = 0;
    int64_t max_warp_nnz = 0, mean_warp_nnz = 0;
    std::vector<HostEntry> entries;
    std::vector<int32_t> segptr;   // [num_slots][num_chunks + 1]
    std::vector<int32_t> slot_oc;  // [num_slots]
    int device = -1;
    void *dev_block = nullptr;
    size_t dev_bytes = 0;
    spconv::DeviceArrays d{};
};

namespace {

constexpr int kWarps = 8;
constexpr size_t kStageBudget = 96 * 1024;  // bytes of staged input per block

int out_extent(int in, int k, int stride, int pad) {
    const long num = (long)in + 2L * pad - k;
    if (num < 0) return 0;
    return (int)(num / stride + 1);
}

int validate_shape(int C, int H, int W, int M, int R, int S, int stride, int pad) {
    if (C < 1 || H < 1 || W < 1 || M < 1 || R < 1 || S < 1 || stride < 1 || pad < 0)
        return SPCONV_ERR_INVALID_ARG;
    if (out_extent(H, R, stride, pad) < 1 || out_extent(W, S, stride, pad) < 1)
        return SPCONV_ERR_INVALID_ARG;
    // keep every index the host computes inside int32 / int64 comfortably
    if ((int64_t)C * R * S >= (int64_t)1 << 31) return SPCONV_ERR_UNSUPPORTED;
    if (pad > 4096 || stride > 64 || R > 64 || S > 64) return SPCONV_ERR_UNSUPPORTED;
    return SPCONV_OK;
}

int validate_csr(int M, int64_t CRS, const int32_t *rowptr, const int32_t *colidx,
                 const float *value, int64_t *nnz_out) {
    if (!rowptr) return SPCONV_ERR_INVALID_ARG;
    if (rowptr[0] != 0) return SPCONV_ERR_BAD_CSR;
    for (int m = 0; m < M; ++m)
        if (rowptr[m + 1] < rowptr[m]) return SPCONV_ERR_BAD_CSR;
    const int64_t nnz = rowptr[M];
    if (nnz > 0 && (!colidx || !value)) return SPCONV_ERR_INVALID_ARG;
    for (int64_t j = 0; j < nnz; ++j)
        if (colidx[j] < 0 || colidx[j] >= CRS) return SPCONV_ERR_BAD_CSR;
    *nnz_out = nnz;
    return SPCONV_OK;
}

// Choose the tiling.  Returns SPCONV_OK or SPCONV_ERR_UNSUPPORTED.
int plan(spconv::Geometry &g, int C, int H, int W, int M, int R, int S, int stride, int pad) {
    g.C = C; g.H = H; g.W = W; g.M = M; g.R = R; g.S = S; g.stride = stride; g.pad = pad;
    g.E = out_extent(H, R, stride, pad);
    g.F = out_extent(W, S, stride, pad);
    // rows per tile: the instance (7 or 8) that wastes the fewest rows
    int best_p = 8, best_waste = 1 << 30;
    for (int P : {8, 7}) {
        const int waste = (g.E + P - 1) / P * P - g.E;
        if (waste < best_waste) { best_waste = waste; best_p = P; }
    }
    g.tile_rows = best_p;
    g.tiles_y = (g.E + best_p - 1) / best_p;
    g.tiles_x = (g.F + spconv::kTileCols - 1) / spconv::kTileCols;
    g.in_rows = (best_p - 1) * stride + R;
    g.in_cols = (spconv::kTileCols - 1) * stride + S;
    g.phase_pitch = spconv::phase_pitch_for(S, stride);
    g.row_pitch = stride * g.phase_pitch;
    g.plane = g.in_rows * g.row_pitch;
    const size_t plane_bytes = (size_t)g.plane * sizeof(float);
    if ((size_t)C * plane_bytes <= kStageBudget) {
        g.chunk = C;
        g.num_chunks = 1;
        g.smem_bytes = (size_t)C * plane_bytes;
    } else {
        g.chunk = (int)(kStageBudget / (2 * plane_bytes));
        if (g.chunk < 1) return SPCONV_ERR_UNSUPPORTED;
        // even out the chunks so the last is not a sliver
        g.num_chunks = (C + g.chunk - 1) / g.chunk;
        g.chunk = (C + g.num_chunks - 1) / g.num_chunks;
        g.smem_bytes = 2 * (size_t)g.chunk * plane_bytes;
    }
    g.warps = kWarps;
    // output channels per warp: four when that still leaves >= 4 groups
    g.slots = M >= 4 * kWarps * 4 ? 4 : (M >= 4 * kWarps * 2 ? 2 : 1);
    g.groups = (M + kWarps * g.slots - 1) / (kWarps * g.slots);
    g.num_slots = g.groups * kWarps * g.slots;
    if (g.groups > 65535) return SPCONV_ERR_UNSUPPORTED;
    if (spconv::forward_variant_supported(S, stride, g.tile_rows, g.slots) != 0)
        return SPCONV_ERR_UNSUPPORTED;
    if (g.smem_bytes > 200 * 1024) return SPCONV_ERR_UNSUPPORTED;
    return SPCONV_OK;
}

// Builds the host arrays of a handle.  Returns a status.
int build_layout(spconv_packed &P, const int32_t *rowptr, const int32_t *colidx,
                 const float *value) {
    const spconv::Geometry &g = P.g;
    const int RS = g.R * g.S;
    // --- bin output channels onto warps: longest row first onto the warp
    //     with the least work that still has a free slot
    std::vector<int> order(g.M);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        return rowptr[a + 1] - rowptr[a] > rowptr[b + 1] - rowptr[b];
    });
    const int nwarps = g.groups * g.warps;
    using Item = std::pair<int64_t, int>;  // (load, warp)
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
    for (int w = 0; w < nwarps; ++w) heap.push({0, w});
    std::vector<int> fill(nwarps, 0);
    std::vector<int64_t> load(nwarps, 0);
    P.slot_oc.assign(g.num_slots, -1);
    for (int m : order) {
        Item it = heap.top();
        heap.pop();
        const int w = it.second;
        P.slot_oc[(size_t)w * g.slots + fill[w]] = m;
        ++fill[w];
        load[w] += rowptr[m + 1] - rowptr[m];
        if (fill[w] < g.slots) heap.push({load[w], w});
    }
    int64_t mx = 0, sum = 0, used = 0;
    for (int w = 0; w < nwarps; ++w) {
        mx = std::max(mx, load[w]);
        if (fill[w]) { sum += load[w]; ++used; }
    }
    P.max_warp_nnz = mx;
    P.mean_warp_nnz = used ? sum / used : 0;

    // --- entries: per slot, per chunk, columns ascending ((c, r, s) order)
    const int nch = g.num_chunks;
    P.segptr.assign((size_t)g.num_slots * (nch + 1), 0);
    P.entries.clear();
    P.entries.reserve((size_t)P.nnz);
    std::vector<int32_t> cols;
    std::vector<int64_t> idx;
    for (int slot = 0; slot < g.num_slots; ++slot) {
        int32_t *sp = &P.segptr[(size_t)slot * (nch + 1)];
        const int m = P.slot_oc[slot];
        if (m < 0) {
            for (int k = 0; k <= nch; ++k) sp[k] = (int32_t)P.entries.size();
            continue;
        }
        const int64_t lo = rowptr[m], hi = rowptr[m + 1];
        idx.resize(hi - lo);
        std::iota(idx.begin(), idx.end(), lo);
        std::sort(idx.begin(), idx.end(),
                  [&](int64_t a, int64_t b) { return colidx[a] < colidx[b]; });
        for (size_t t = 1; t < idx.size(); ++t)
            if (colidx[idx[t]] == colidx[idx[t - 1]]) return SPCONV_ERR_BAD_CSR;
        size_t t = 0;
        for (int k = 0; k < nch; ++k) {
            sp[k] = (int32_t)P.entries.size();
            const int c_end = std::min(g.C, (k + 1) * g.chunk);
            for (; t < idx.size(); ++t) {
                const int col = colidx[idx[t]];
                const int c = col / RS;
                if (c >= c_end) break;
                const int r = (col / g.S) % g.R;
                const int s = col % g.S;
                const int cl = c - k * g.chunk;
                HostEntry e;
                e.value = value[idx[t]];
                e.off = cl * g.plane + r * g.row_pitch + (s % g.stride) * g.phase_pitch +
                        s / g.stride;
                P.entries.push_back(e);
            }
        }
        sp[nch] = (int32_t)P.entries.size();
    }
    return (int64_t)P.entries.size() == P.nnz ? SPCONV_OK : SPCONV_ERR_BAD_CSR;
}

int make_handle(int C, int H, int W, int M, int R, int S, int stride, int pad,
                const int32_t *rowptr, const int32_t *colidx, const float *value,
                spconv_packed **out) {
    if (!out) return SPCONV_ERR_INVALID_ARG;
    int st = validate_shape(C, H, W, M, R, S, stride, pad);
    if (st) return st;
    int64_t nnz = 0;
    st = validate_csr(M, (int64_t)C * R * S, rowptr, colidx, value, &nnz);
    if (st) return st;
    if (nnz >= ((int64_t)1 << 31) - 16) return SPCONV_ERR_UNSUPPORTED;
    spconv_packed *P = new (std::nothrow) spconv_packed();
    if (!P) return SPCONV_ERR_ALLOC;
    P->nnz = nnz;
    st = plan(P->g, C, H, W, M, R, S, stride, pad);
    if (!st) st = build_layout(*P, rowptr, colidx, value);
    if (st) {
        delete P;
        return st;
    }
    *out = P;
    return SPCONV_OK;
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

int upload(spconv_packed *P, cudaStream_t stream) {
    if (cudaGetDevice(&P->device) != cudaSuccess) return SPCONV_ERR_CUDA;
    const size_t b_entries = align256(std::max<size_t>(P->entries.size(), 2) * sizeof(HostEntry));
    const size_t b_segptr = align256(P->segptr.size() * sizeof(int32_t));
    const size_t b_slot = align256(P->slot_oc.size() * sizeof(int32_t));
    P->dev_bytes = b_entries + b_segptr + b_slot;
    void *blk = nullptr;
    if (cudaMalloc(&blk, P->dev_bytes) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_ALLOC;
    }
    P->dev_block = blk;
    char *base = static_cast<char *>(blk);
    bool ok = cudaMemsetAsync(base, 0, b_entries, stream) == cudaSuccess;
    ok = ok && (P->entries.empty() ||
                cudaMemcpyAsync(base, P->entries.data(), P->entries.size() * sizeof(HostEntry),
                                cudaMemcpyHostToDevice, stream) == cudaSuccess);
    ok = ok && cudaMemcpyAsync(base + b_entries, P->segptr.data(),
                               P->segptr.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                               stream) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(base + b_entries + b_segptr, P->slot_oc.data(),
                               P->slot_oc.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                               stream) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(stream) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    P->d.entries = reinterpret_cast<const float2 *>(base);
    P->d.segptr = reinterpret_cast<const int *>(base + b_entries);
    P->d.slot_oc = reinterpret_cast<const int *>(base + b_entries + b_segptr);
    return SPCONV_OK;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int spconv_pack_host(
    int C, int H, int W, int M, int R, int S, int stride, int pad, const int32_t *rowptr,
    const int32_t *colidx, const float *value, spconv_packed **out) {
    try {
        return make_handle(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, out);
    } catch (...) {
        return SPCONV_ERR_ALLOC;
    }
}

__attribute__((visibility("default"))) int spconv_pack(
    int C, int H, int W, int M, int R, int S, int stride, int pad, const int32_t *rowptr,
    const int32_t *colidx, const float *value, void *stream, spconv_packed **out) {
    try {
        spconv_packed *P = nullptr;
        int st = make_handle(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, &P);
        if (st) return st;
        st = upload(P, static_cast<cudaStream_t>(stream));
        if (st) {
            spconv_packed_free(P);
            return st;
        }
        *out = P;
        return SPCONV_OK;
    } catch (...) {
        return SPCONV_ERR_ALLOC;
    }
}

__attribute__((visibility("default"))) int spconv_forward(
    int N, int C, int H, int W, int M, int R, int S, int stride, int pad, const float *input,
    const spconv_packed *packed, float *output, void *stream) {
    if (!packed || N < 0) return SPCONV_ERR_INVALID_ARG;
    const spconv::Geometry &g = packed->g;
    if (C != g.C || H != g.H || W != g.W || M != g.M || R != g.R || S != g.S ||
        stride != g.stride || pad != g.pad)
        return SPCONV_ERR_MISMATCH;
    if (!packed->dev_block) return SPCONV_ERR_MISMATCH;
    if (N == 0) return SPCONV_OK;
    if (!input || !output) return SPCONV_ERR_INVALID_ARG;
    if (((uintptr_t)input & 15) || ((uintptr_t)output & 3)) return SPCONV_ERR_INVALID_ARG;
    const int64_t tiles = (int64_t)N * g.tiles_y * g.tiles_x;
    if (tiles > 0x7fffffffLL) return SPCONV_ERR_UNSUPPORTED;
    const size_t in_bytes = (size_t)N * C * H * W * sizeof(float);
    const size_t out_bytes = (size_t)N * M * g.E * g.F * sizeof(float);
    if (ranges_overlap(input, in_bytes, output, out_bytes)) return SPCONV_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPCONV_ERR_CUDA;
    if (dev != packed->device) return SPCONV_ERR_MISMATCH;
    cudaError_t e = spconv::launch_forward(g, N, input, output, packed->d,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    return SPCONV_OK;
}

__attribute__((visibility("default"))) void spconv_packed_free(spconv_packed *p) {
    if (!p) return;
    if (p->dev_block) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != p->device) cudaSetDevice(p->device);
        cudaFree(p->dev_block);
        if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    }
    delete p;
}

__attribute__((visibility("default"))) const char *spconv_status_string(int status) {
    switch (status) {
        case SPCONV_OK: return "ok";
        case SPCONV_ERR_INVALID_ARG: return "invalid argument";
        case SPCONV_ERR_BAD_CSR: return "malformed CSR weights";
        case SPCONV_ERR_UNSUPPORTED: return "unsupported layer shape";
        case SPCONV_ERR_ALLOC: return "allocation failed";
        case SPCONV_ERR_CUDA: return "CUDA error";
        case SPCONV_ERR_MISMATCH: return "shape or device differs from the packed weights";
        default: return "unknown status";
    }
}

__attribute__((visibility("default"))) int spconv_packed_info_get(const spconv_packed *p,
                                                                  spconv_packed_info *info) {
    if (!p || !info) return SPCONV_ERR_INVALID_ARG;
    const spconv::Geometry &g = p->g;
    std::memset(info, 0, sizeof(*info));
    info->C = g.C; info->H = g.H; info->W = g.W; info->M = g.M;
    info->R = g.R; info->S = g.S; info->stride = g.stride; info->pad = g.pad;
    info->E = g.E; info->F = g.F;
    info->nnz = p->nnz;
    info->entries = (int64_t)p->entries.size();
    info->tile_rows = g.tile_rows;
    info->tile_cols = spconv::kTileCols;
    info->tiles_y = g.tiles_y;
    info->tiles_x = g.tiles_x;
    info->in_rows = g.in_rows;
    info->in_cols = g.in_cols;
    info->phase_pitch = g.phase_pitch;
    info->row_pitch = g.row_pitch;
    info->plane = g.plane;
    info->chunk = g.chunk;
    info->num_chunks = g.num_chunks;
    info->slots_per_warp = g.slots;
    info->warps = g.warps;
    info->groups = g.groups;
    info->num_slots = g.num_slots;
    info->on_device = p->dev_block ? 1 : 0;
    info->device_bytes = (int64_t)p->dev_bytes;
    info->smem_bytes = (int64_t)g.smem_bytes;
    info->max_warp_nnz = p->max_warp_nnz;
    info->mean_warp_nnz = p->mean_warp_nnz;
    return SPCONV_OK;
}

__attribute__((visibility("default"))) int spconv_packed_copy_array(
    const spconv_packed *p, int which, void *dst, int64_t dst_bytes, int64_t *needed) {
    if (!p) return SPCONV_ERR_INVALID_ARG;
    const void *src = nullptr;
    int64_t n = 0;
    switch (which) {
        case SPCONV_ARRAY_ENTRIES:
            src = p->entries.data();
            n = (int64_t)(p->entries.size() * sizeof(HostEntry));
            break;
        case SPCONV_ARRAY_SEGPTR:
            src = p->segptr.data();
            n = (int64_t)(p->segptr.size() * sizeof(int32_t));
            break;
        case SPCONV_ARRAY_SLOT_OC:
            src = p->slot_oc.data();
            n = (int64_t)(p->slot_oc.size() * sizeof(int32_t));
            break;
        default: return SPCONV_ERR_INVALID_ARG;
    }
    if (needed) *needed = n;
    if (!dst) return SPCONV_OK;
    if (dst_bytes < n) return SPCONV_ERR_INVALID_ARG;
    if (n) std::memcpy(dst, src, (size_t)n);
    return SPCONV_OK;
}

}  // extern "C"
