// Host side of libspconv: argument validation, the packing of CSR weights into
// the kernel's layout (weight stretching + output-channel binning), device
// upload, tensor-map encoding, and the C ABI declared in include/spconv.h.
//
// Packing follows Escoin (arXiv 1802.10280), "Sparse convolution": dynamic
// indexing with the layout function f(c, y, x) and its shift property
// f(c, y + r, x + s) = f(c, y, x) + f(0, r, s), so each nonzero's column
// (c, r, s) is rewritten once ("weight stretching") into an offset that the
// kernel adds to a per-output-pixel base.  Here f is the layout of the
// shared-memory input tile the kernel stages (channel plane, row, stride
// phase, column), not of the global array.  The per-slot entry ranges in each
// blob header play the role of the offset array of Tuteja et al.,
// "Theoretical and Empirical Analysis of Sparse Convolution", Sec. 5.3.
#include "../../include/spconv.h"

#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
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

struct TmapCacheEntry {
    const void *x = nullptr;
    int N = -1;
    CUtensorMap map;
};

}  // namespace

struct spconv_packed {
    spconv::Geometry g{};
    int64_t nnz = 0;
    int64_t max_warp_nnz = 0, mean_warp_nnz = 0;
    std::vector<unsigned char> blobs;  // concatenated (group, chunk) blobs
    std::vector<uint32_t> blob_off;    // [groups * num_chunks + 1], 16-byte units
    std::vector<int32_t> slot_oc;      // [num_slots]: head slot -> output channel, else -1
    std::vector<int32_t> slot_next;    // [num_slots]: next part (group-local slot) or -1
    std::vector<int32_t> group_flags;  // [groups]: bit 0 dense, bit 1 split rows
    std::vector<std::vector<int64_t>> slot_entries;  // CSR indices per slot, column order
    int device = -1;
    void *dev_block = nullptr;
    size_t dev_bytes = 0;
    spconv::DeviceArrays d{};
    mutable std::mutex tmap_lock;
    mutable TmapCacheEntry tmap_cache[4];
    mutable unsigned tmap_next = 0;
};

namespace {

constexpr size_t kSmemBudget = 110 * 1024;  // two resident blocks per SM
constexpr int kSMs = 152;                   // GB300 SM count, for the grid heuristics
// Rows at least this dense take the dense-tap path where the shape allows it:
// it issues K*K FMAs per (slot, channel) block with zeros included, about four
// times cheaper per FMA than a shared-memory load per FMA.
constexpr double kDenseRowMin = 0.30;
constexpr int64_t kMinPart = 32;  // smallest part a split row is cut into
// spconv_forward_host: outputs up to this size are written by the forward
// straight into the mapped host buffer, larger ones copied out after it.
constexpr size_t kDirectOutBytes = 1 << 20;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

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
    if ((int64_t)H * W >= (int64_t)1 << 31 || (int64_t)M * C >= (int64_t)1 << 40)
        return SPCONV_ERR_UNSUPPORTED;
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

// Tile shape and channel group size (everything but the chunking).
int plan_tiles(spconv::Geometry &g, int C, int H, int W, int M, int R, int S, int stride,
               int pad, int64_t nnz, double dense_share) {
    g.C = C; g.H = H; g.W = W; g.M = M; g.R = R; g.S = S; g.stride = stride; g.pad = pad;
    g.E = out_extent(H, R, stride, pad);
    g.F = out_extent(W, S, stride, pad);
    // two interleaved lane rows of 16 lanes for outputs at most 16 wide
    g.lane_rows = (stride == 1 && g.F <= 16) ? 2 : 1;
    g.tile_w = spconv::kLanes / g.lane_rows;
    // rows per lane: the instance (7 or 8) that wastes the fewest rows
    int best_p = 8, best_waste = 1 << 30;
    for (int P : {8, 7}) {
        const int h = P * g.lane_rows;
        const int waste = (g.E + h - 1) / h * h - g.E;
        if (waste < best_waste) { best_waste = waste; best_p = P; }
    }
    g.tile_rows = best_p;
    g.tile_h = best_p * g.lane_rows;
    g.tiles_y = (g.E + g.tile_h - 1) / g.tile_h;
    g.tiles_x = (g.F + g.tile_w - 1) / g.tile_w;
    g.in_rows = (g.tile_h - 1) * stride + R;
    g.in_cols = (g.tile_w - 1) * stride + S;
    g.shift = spconv::align_shift_for(pad, stride);
    if (stride == 1) {
        g.phase_pitch = spconv::row_pitch_s1(S, g.lane_rows);
        g.row_pitch = g.phase_pitch;
    } else {
        g.phase_pitch = spconv::phase_pitch_for(S, stride);
        g.row_pitch = stride * g.phase_pitch;
    }
    // Column blocks (3x3, stride 1): eight lane rows of four lanes, each lane
    // holding seven consecutive outputs of its row, tile 8 x 28 -- where that
    // covers fewer output positions than the column-per-lane tiles (widths a
    // multiple of 28 but not of 32, e.g. 56 and 112, leave no lane idle).  The
    // staged row pitch is 4 mod 8 words, so the 32 lanes' first inputs
    // (ly * pitch + 7 lx) fall in distinct banks.
    g.col_blocks = 0;
    g.tight = 0;
    g.tile_images = 1;
    g.pair_off = 0;
    const bool tile_fmt = g.format == SPCONV_FORMAT_F32 || g.format == SPCONV_FORMAT_PACKED32;
    if (stride == 1 && R == 3 && S == 3 && tile_fmt && g.lane_rows == 1) {
        const int64_t area = (int64_t)g.tiles_y * g.tile_h * g.tiles_x * g.tile_w;
        const int64_t area_cb = (int64_t)((g.E + 7) / 8) * 8 * ((g.F + 27) / 28) * 28;
        if (area_cb * 100 < area * 97) {
            g.col_blocks = 1;
            g.lane_rows = 8;
            g.tile_rows = 7;
            g.tile_h = 8;
            g.tile_w = 28;
            g.tiles_y = (g.E + g.tile_h - 1) / g.tile_h;
            g.tiles_x = (g.F + g.tile_w - 1) / g.tile_w;
            g.in_rows = g.tile_h - 1 + R;
            g.in_cols = g.tile_w - 1 + S;
            int rp = (int)round_up((size_t)(g.shift + g.in_cols), 4);
            if (rp % 8 == 0) rp += 4;
            g.phase_pitch = rp;
            g.row_pitch = rp;
        }
    }
    // Image-pair column blocks (3x3, stride 1, outputs 22..28 wide, batches of
    // two or more): four lane rows of eight lanes, lanes 0..3 of a row on image
    // 2n and 4..7 on image 2n + 1, each lane seven consecutive outputs -- a
    // 4 x 28 tile of each of two images, so 28-wide outputs leave no lane idle
    // (a column-per-lane tile leaves 4 of 32).  Same pitch rule as column
    // blocks: the first image's 16 lanes start in 16 distinct banks, and the
    // second image's sub-tile starts 16 words later (mod 32), in the other 16.
    // The four-row tiles stage a fifth more input per channel, so chunks are
    // smaller and per-chunk costs grow: measured on GB300 (the lognormal
    // 512-channel 28 x 28 layers) they paid only where dense-tap rows hold most
    // of the nonzeros (50 % sparse: 630 -> 584 us), and lost where sparse rows
    // dominate (90 %: 244 -> 250, 95 %: 117 -> 123, 99 %: 38.6 -> 46.1 us).
    // Taken when they cover at least 3 % fewer output positions and dense-tap
    // rows hold at least three quarters of the nonzeros.  5x5 layers take them
    // on the area alone: the 5x5 instances have no dense-tap path in this
    // layout, and their sparse loop keeps its tap pairs.
    const bool pair_kernel = (R == 3 && S == 3 && dense_share >= 0.75) || (R == 5 && S == 5);
    if (stride == 1 && pair_kernel && tile_fmt && !g.col_blocks && g.lane_rows == 1 &&
        g.F > 21 && g.F <= 28 && g.batch_hint >= 2) {
        const int64_t nb = g.batch_hint;
        const int64_t area = nb * g.tiles_y * g.tile_h * g.tiles_x * g.tile_w;
        const int64_t area_p = (nb + 1) / 2 * 2 * ((g.E + 3) / 4) * 4 * 28;
        if (area_p * 100 < area * 97) {
            g.col_blocks = 1;
            g.tile_images = 2;
            g.lane_rows = 4;
            g.tile_rows = 7;
            g.tile_h = 4;
            g.tile_w = 28;
            g.tiles_y = (g.E + g.tile_h - 1) / g.tile_h;
            g.tiles_x = (g.F + g.tile_w - 1) / g.tile_w;
            g.in_rows = g.tile_h - 1 + R;
            g.in_cols = g.tile_w - 1 + S;
            int rp = (int)round_up((size_t)(g.shift + g.in_cols), 4);
            if (rp % 8 == 0) rp += 4;
            g.phase_pitch = rp;
            g.row_pitch = rp;
            // A tensor copy puts the second image's sub-tile chunk x plane
            // words after the first, which must be 16 mod 32 words: with 8
            // staged rows (5x5) every plane is a multiple of 32, so stage a
            // ninth row (read as zeros or ignored) when the rows are
            // 16-byte aligned.  cp.async staging pads the gap instead.
            if ((size_t)g.in_rows * rp % 32 == 0 && (W * sizeof(float)) % 16 == 0) ++g.in_rows;
        }
    }
    g.plane = g.in_rows * g.row_pitch;
    g.warps = spconv::kWarps;
    // output channels per warp: the largest Q in {4, 2, 1} whose one-image
    // grid, with the channels split over a full cluster, still gives ~1.5
    // blocks per SM (small layers trade per-warp reuse for parallelism)
    // blocks of one launch per channel group, at the planned batch size
    const int64_t spatial = (int64_t)g.tiles_y * g.tiles_x *
                            ((std::max(1, g.batch_hint) + g.tile_images - 1) / g.tile_images);
    auto groups_of = [&](int Q) {
        return (M + (int64_t)spconv::kWarps * Q - 1) / ((int64_t)spconv::kWarps * Q);
    };
    g.slots = 1;
    for (int Q : {4, 2}) {
        if (spatial * groups_of(Q) * spconv::kMaxSplit * 2 >= (int64_t)kSMs * 3) {
            g.slots = Q;
            break;
        }
    }
    // Very sparse layers are bound by staging: every channel group re-stages
    // the whole input.  Eight channels per warp halve the groups when there
    // are many (>= 8 at four per warp) and the estimated staging time (L2 ->
    // shared at ~7 TB/s) exceeds the compute time (the sparse path's ~18 % of
    // fp32 peak), per image.
    if (g.slots == 4 && groups_of(4) >= 8 &&
        spatial * groups_of(8) * spconv::kMaxSplit * 2 >= (int64_t)kSMs * 3) {
        const double staged = (double)groups_of(4) * g.tiles_y * g.tiles_x * g.plane * C * sizeof(float);
        const double staging_s = staged / 7.0e12;
        const double compute_s = 2.0 * nnz * g.E * g.F / (0.18 * kSMs * 128 * 2 * 2.07e9);
        if (staging_s > compute_s) g.slots = 8;
    }
    g.groups = (M + spconv::kWarps * g.slots - 1) / (spconv::kWarps * g.slots);
    g.num_slots = g.groups * spconv::kWarps * g.slots;
    g.hdr_words = (int)round_up((size_t)spconv::kWarps * g.slots + 1, 4);
    if (g.groups > 65535) return SPCONV_ERR_UNSUPPORTED;
    if (spconv::forward_variant_supported(S, stride, g.tile_rows, g.slots, g.lane_rows, false, false,
                                          g.col_blocks != 0) != 0)
        return SPCONV_ERR_UNSUPPORTED;
    // Tight pitch (3x3, pad 1, one lane row, the whole width in one tile
    // column, rows a tensor copy can address, 16-byte-aligned widths up to
    // 31): the copy starts at column 0 with a 32-word pitch; the columns past
    // the image arrive as zeros and stand in for the right halo, and the left
    // halo of row r is the last (zero) column of row r - 1 (a lead of zeroed
    // words before the tile covers the first row).  9 x 32 words per channel
    // against 9 x 40 for the padded tile: the chunks hold a quarter more
    // channels.
    if (stride == 1 && R == 3 && S == 3 && pad == 1 && tile_fmt && !g.col_blocks &&
        g.lane_rows == 1 && g.tiles_x == 1 && W % 4 == 0 && W <= 31 &&
        spconv::forward_variant_supported(S, stride, g.tile_rows, g.slots, g.lane_rows, false,
                                          false, false, true) == 0) {
        g.tight = 1;
        g.shift = -1;
        g.in_cols = 32;
        g.phase_pitch = 32;
        g.row_pitch = 32;
        g.plane = g.in_rows * g.row_pitch;
    }
    // Whole-image tiles of images whose rows TMA cannot address: one bulk copy
    // of the chunk's raw planes (dense, pitch W) instead of per-element
    // cp.async into a padded tile; the kernel applies the padding to the
    // weights of the taps that leave the image.
    g.plane_stage = 0;
    // (F32 entries only: decoding a 32-bit word into a plane offset and side
    // flags measured slower than the padded tile on the one-image layer)
    if (g.format == SPCONV_FORMAT_F32 &&
        spconv::plane_stage_supported(H, W, R, S, stride, pad, g.tile_rows, g.lane_rows, g.slots)) {
        g.plane_stage = 1;
        g.in_rows = H;
        g.in_cols = W;
        g.shift = 0;
        g.phase_pitch = W;
        g.row_pitch = W;
        g.plane = H * W;
    }
    return SPCONV_OK;
}

// Output channels whose rows are dense enough go to leading "dense" groups
// (densest first, dealt round-robin over the warps).  The rest are sparse:
// they are spread over the sparse groups longest row first onto the group with
// the least work that has room; a row heavier than 1.1x (1.5x for short
// warps) a warp's fair share is split into parts (its column-ordered nonzeros
// dealt round-robin, so every part spans all chunks), and inside each group
// the parts are bound to warp slots longest first onto the least-loaded warp
// with a free slot.  The parts of one row stay in one group and are summed in
// the epilogue.  Sets groups, num_slots, slot_oc, slot_next, group_flags and
// the per-slot entry lists.
int bin_channels(spconv_packed &P, const int32_t *rowptr, const int32_t *colidx) {
    spconv::Geometry &g = P.g;
    const int per_group = g.warps * g.slots;
    const double crs = (double)g.C * g.R * g.S;
    auto nnz_of = [&](int m) { return (int64_t)rowptr[m + 1] - rowptr[m]; };
    std::vector<int> dense, sparse;
    const bool can_dense = !g.plane_stage &&
                           spconv::dense_taps_supported(g.R, g.S, g.stride, g.lane_rows, g.slots);
    for (int m = 0; m < g.M; ++m)
        (can_dense && nnz_of(m) / crs >= kDenseRowMin ? dense : sparse).push_back(m);
    std::stable_sort(dense.begin(), dense.end(), [&](int a, int b) { return nnz_of(a) > nnz_of(b); });
    // a dense group less than half full is not worth a group of its own
    const int tail = (int)dense.size() % per_group;
    if (tail && tail * 2 < per_group) {
        sparse.insert(sparse.end(), dense.end() - tail, dense.end());
        dense.resize(dense.size() - tail);
    }
    // Dense-tap groups or none.  A dense-tap block does all its rows' work
    // over all channels, so with few dense groups it can outlast the whole
    // rest of the launch; the same rows on the sparse path (split into parts)
    // keep every block equally long but cost more shared-memory loads.
    // Estimate both launches and keep the shorter.  Model, fitted to
    // per-block timelines on GB300 (the lognormal 512-channel layers): sparse
    // work moves P + 1/2 shared-memory wavefronts per entry and output tile at
    // ~0.88 per clock per SM; a dense-tap warp takes ~2 ns per instruction,
    // (window rows x K + 1) loads per channel plus (3 + K*K*P + 5) per row and
    // channel; two blocks per SM.
    if (!dense.empty()) {
        int64_t dense_nnz = 0, all_nnz = 0;
        for (int m : dense) dense_nnz += nnz_of(m);
        for (int m = 0; m < g.M; ++m) all_nnz += nnz_of(m);
        const int ti = std::max(1, g.tile_images);
        const double tiles = (double)g.tiles_y * g.tiles_x *
                             ((std::max(1, g.batch_hint) + ti - 1) / ti);
        const double lsu = 0.88 * kSMs * 2.07e9;  // wavefronts per second
        const double wf = g.tile_rows + 0.5;
        const double t_sparse_all = (double)all_nnz * tiles * wf / lsu;
        const int gd = (int)((dense.size() + per_group - 1) / per_group);
        const double rows_per_warp = (double)dense.size() / ((double)gd * g.warps);
        const double win = (double)(g.col_blocks ? g.R * (g.tile_rows + g.S - 1)
                                                 : (g.lane_rows * (g.tile_rows - 1) + g.R) * g.S) +
                           1.0;
        const double t_dense_block =
            (double)g.C * (win + rows_per_warp * (8.0 + (double)g.R * g.S * g.tile_rows)) * 2.0e-9;
        const double t_with_dense =
            std::max(t_dense_block, gd * tiles * t_dense_block / (2.0 * kSMs) +
                                        (double)(all_nnz - dense_nnz) * tiles * wf / lsu);
        if (t_sparse_all < t_with_dense) {
            sparse.insert(sparse.end(), dense.begin(), dense.end());
            dense.clear();
        }
    }
    std::stable_sort(sparse.begin(), sparse.end(), [&](int a, int b) { return nnz_of(a) > nnz_of(b); });
    const int gd = ((int)dense.size() + per_group - 1) / per_group;

    // parts per sparse row: rows above the mean warp load are split.  With
    // eight slots per warp a full group forces coarse warp loads, so those
    // plans keep ~10 % of the slots free.
    const int64_t want0 = g.slots >= 8 ? (int64_t)sparse.size() + (int64_t)sparse.size() / 10
                                       : (int64_t)sparse.size();
    int gs = std::max((int)((want0 + per_group - 1) / per_group), sparse.empty() ? 0 : 1);
    int64_t total = 0;
    for (int m : sparse) total += nnz_of(m);
    std::vector<int> parts(g.M, 1);
    for (int iter = 0; iter < 4 && gs > 0; ++iter) {
        const int64_t cap = std::max<int64_t>(1, (total + (int64_t)gs * g.warps - 1) / ((int64_t)gs * g.warps));
        int64_t nparts = 0;
        for (int m : sparse) {
            // rows well above the fair share are split (into parts of at least
            // kMinPart entries): above 1.1x where warps are long (a warp's load
            // sets its block's end; 90 % lognormal layer, 1.5x 229 us, 1.2x
            // 214, 1.1x 213), above 1.5x where they are short (fair share
            // under 512 entries: the parts' sums cost more than they save)
            parts[m] = (cap >= 512 ? nnz_of(m) * 10 > cap * 11 : nnz_of(m) * 2 > cap * 3)
                           ? (int)std::min<int64_t>({(nnz_of(m) + cap - 1) / cap, g.warps,
                                                     std::max<int64_t>(1, nnz_of(m) / kMinPart)})
                           : 1;
            nparts += parts[m];
        }
        // with split rows keep ~10 % of the slots free so the group-level
        // balancing is not forced by capacity
        const int64_t want = nparts > (int64_t)sparse.size() ? nparts + nparts / 10 : nparts;
        const int need = (int)((want + per_group - 1) / per_group);
        if (need <= gs) break;
        gs = need;
    }
    g.dense_groups = gd;
    g.groups = std::max(1, gd + gs);
    if (g.groups > 65535) return SPCONV_ERR_UNSUPPORTED;
    g.num_slots = g.groups * per_group;
    P.slot_oc.assign(g.num_slots, -1);
    P.slot_next.assign(g.num_slots, -1);
    P.group_flags.assign(g.groups, 0);
    P.slot_entries.assign(g.num_slots, {});
    auto sorted_entries = [&](int m) {
        std::vector<int64_t> idx(nnz_of(m));
        std::iota(idx.begin(), idx.end(), (int64_t)rowptr[m]);
        std::sort(idx.begin(), idx.end(), [&](int64_t a, int64_t b) { return colidx[a] < colidx[b]; });
        return idx;
    };

    // dense groups: the i-th densest channel goes to warp i % warps_total, slot i / warps_total
    for (int grp = 0; grp < gd; ++grp) P.group_flags[grp] = 1;
    const int dwarps = gd * g.warps;
    for (size_t i = 0; i < dense.size(); ++i) {
        const int slot = (int)(i % dwarps) * g.slots + (int)(i / dwarps);
        P.slot_oc[slot] = dense[i];
        P.slot_entries[slot] = sorted_entries(dense[i]);
    }

    // sparse rows onto groups (least load with room for the row's parts)
    std::vector<std::vector<int>> members(gs);
    std::vector<int64_t> gload(gs, 0);
    std::vector<int> gfree(gs, per_group);
    for (int m : sparse) {
        int best = -1;
        for (int q = 0; q < gs; ++q)
            if (gfree[q] >= parts[m] && (best < 0 || gload[q] < gload[best])) best = q;
        if (best < 0) {  // no group has room for all parts: use the roomiest
            best = 0;
            for (int q = 1; q < gs; ++q)
                if (gfree[q] > gfree[best]) best = q;
            parts[m] = std::max(1, gfree[best]);
        }
        members[best].push_back(m);
        gload[best] += nnz_of(m);
        gfree[best] -= parts[m];
    }
    // inside each group: parts onto warps, longest first onto the least-loaded
    int64_t mx = 0, sum = 0, used = 0;
    for (int q = 0; q < gs; ++q) {
        const int grp = gd + q;
        struct Part { int m, k, n; int64_t load; };
        std::vector<Part> plist;
        for (int m : members[q])
            for (int k = 0; k < parts[m]; ++k)
                plist.push_back({m, k, parts[m], (nnz_of(m) - k + parts[m] - 1) / parts[m]});
        std::stable_sort(plist.begin(), plist.end(),
                         [](const Part &a, const Part &b) { return a.load > b.load; });
        using Item = std::pair<int64_t, int>;  // (load, warp)
        std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
        for (int w = 0; w < g.warps; ++w) heap.push({0, w});
        std::vector<int> fill(g.warps, 0);
        std::vector<int64_t> load(g.warps, 0);
        std::vector<std::vector<int>> part_slot(g.M);
        for (const Part &pt : plist) {
            if (heap.empty()) return SPCONV_ERR_UNSUPPORTED;  // cannot happen: sized above
            const Item it = heap.top();
            heap.pop();
            const int w = it.second;
            const int local = w * g.slots + fill[w];
            ++fill[w];
            load[w] += pt.load;
            if (fill[w] < g.slots) heap.push({load[w], w});
            if (part_slot[pt.m].empty()) part_slot[pt.m].assign(pt.n, -1);
            part_slot[pt.m][pt.k] = local;
        }
        for (int m : members[q]) {
            const std::vector<int> &ps = part_slot[m];
            const std::vector<int64_t> idx = sorted_entries(m);
            for (size_t k = 0; k < ps.size(); ++k) {
                const int slot = grp * per_group + ps[k];
                if (k == 0) P.slot_oc[slot] = m;
                if (k + 1 < ps.size()) P.slot_next[slot] = ps[k + 1];
                std::vector<int64_t> &mine = P.slot_entries[slot];
                for (size_t t = k; t < idx.size(); t += ps.size()) mine.push_back(idx[t]);
            }
            if (ps.size() > 1) {
                P.group_flags[grp] |= 2;
                g.split_rows = 1;
            }
        }
        for (int w = 0; w < g.warps; ++w) {
            mx = std::max(mx, load[w]);
            if (fill[w]) { sum += load[w]; ++used; }
        }
    }
    P.max_warp_nnz = mx;
    P.mean_warp_nnz = used ? sum / used : 0;
    return SPCONV_OK;
}

size_t entry_bytes(const spconv::Geometry &g) { return g.format == 1 ? 4 : 8; }

// FP16 rounding used by the 32-bit packed format (round to nearest even).
float to_half_and_back(float v) { return __half2float(__float2half_rn(v)); }

size_t dense_blob_bytes(const spconv::Geometry &g, int chunk) {
    const size_t mask_words = round_up((size_t)g.warps * chunk, 4);
    const size_t kk4 = round_up((size_t)g.R * g.S, 4);
    return mask_words * 4 + (size_t)g.warps * chunk * g.slots * kk4 * 4;
}

// Chunk size: the largest that keeps two pipeline stages (staged input plus
// the largest weight blob) within the shared-memory budget, and small enough
// that a one-image launch can split the chunks over a cluster to fill the GPU.
int plan_chunks(spconv::Geometry &g, const std::vector<int64_t> &gpre) {
    // gpre[(group) * (C + 1) + c]: entries of the group in channels [0, c)
    const int C = g.C;
    const int64_t base_blocks = (int64_t)g.tiles_y * g.tiles_x * g.groups *
                                ((std::max(1, g.batch_hint) + g.tile_images - 1) / g.tile_images);
    int want_split = base_blocks >= kSMs
                         ? 1
                         : (int)std::min<int64_t>(spconv::kMaxSplit,
                                                  (2 * kSMs + base_blocks - 1) / base_blocks);
    want_split = std::max(want_split, 1);
    // Plane-staged plans aim at one block per SM: their small stages hold twice
    // the channels, and the one-image ResNet-style layer measured 5.98 us with
    // 4-block clusters of 64-channel chunks (128 blocks) against 6.47 us with
    // 8-block clusters of 32 channels (256 blocks, two on most SMs).
    if (g.plane_stage && base_blocks < kSMs)
        want_split = (int)std::max<int64_t>(1, std::min<int64_t>(spconv::kMaxSplit, kSMs / base_blocks));
    int cap = std::min(C, 256);  // TMA box extent limit
    // Chunks small enough for the split (not below 32 channels; plane staging,
    // whose stages are small, always: its layers are the one-image ones)
    if (want_split > 1 && (C / want_split >= 32 || g.plane_stage))
        cap = std::min(cap, (C + want_split - 1) / want_split);
    // When the planned launch (known batch size) splits the chunks over a
    // cluster with one chunk per block, a single stage is enough: allow it up
    // to 200 KB (larger batches of the same plan then run two stages, one
    // block per SM).
    const bool one_per_block =
        g.batch_hint > 0 && want_split > 1 && (int64_t)cap * want_split >= C;
    // Image pairs: the second image's sub-tile starts pair_off words after the
    // first, 16 mod 32 so that the two halves of a warp load from disjoint
    // banks.  A tensor copy writes it right after the first (pair_off = chunk
    // x plane), so with rows a tensor map can address only chunks with chunk x
    // plane = 16 mod 32 qualify: start from the first such chunk at or above
    // the cap (a chunk past C reads zeros for the missing channels).  cp.async
    // staging places the second sub-tile itself: any chunk, the gap padded.
    const bool tma_pairs = g.tile_images == 2 && (g.W * sizeof(float)) % 16 == 0;
    if (tma_pairs)
        while (cap < 256 && (size_t)cap * g.plane % 32 != 16) ++cap;
    for (int chunk = cap; chunk >= 1; --chunk) {
        const int nch = (C + chunk - 1) / chunk;
        const size_t hdr_bytes = (size_t)g.hdr_words * 4;
        if (tma_pairs && (size_t)chunk * g.plane % 32 != 16) continue;
        const size_t pair_off =
            g.tile_images == 2 ? (size_t)chunk * g.plane + (48 - (size_t)chunk * g.plane % 32) % 32
                               : 0;
        const size_t in_stage = round_up(
            (pair_off + (size_t)chunk * g.plane +
             (g.plane_stage ? spconv::kPlaneLead + spconv::kPlaneTail : 0) +
             (g.tight ? spconv::kTightLeadWords + spconv::kTightTailWords : 0)) * sizeof(float),
            128);
        size_t blob_max = g.dense_groups ? dense_blob_bytes(g, chunk) : 0;
        for (int grp = g.dense_groups; grp < g.groups; ++grp) {
            const int64_t *pre = &gpre[(size_t)grp * (C + 1)];
            for (int k = 0; k < nch; ++k) {
                const int c0 = k * chunk, c1 = std::min(C, c0 + chunk);
                const size_t bytes =
                    hdr_bytes + round_up((size_t)(pre[c1] - pre[c0]) * entry_bytes(g) +
                                             (g.tap_pairs ? 8 : 0), 16);
                blob_max = std::max(blob_max, bytes);
            }
        }
        const size_t stage = in_stage + round_up(blob_max, 128);
        const size_t total = (nch > 1 ? 2 : 1) * stage + 128;
        const bool fits_split = one_per_block && chunk * want_split >= C &&
                                2 * stage + 128 <= 200 * 1024;
        if (total <= kSmemBudget || fits_split || (chunk == 1 && total <= 200 * 1024)) {
            g.chunk = chunk;
            g.num_chunks = nch;
            g.pair_off = (int)pair_off;
            g.dense_mask_words = (int)round_up((size_t)g.warps * chunk, 4);
            g.in_stage_bytes = in_stage;
            g.blob_stage_bytes = round_up(blob_max, 128);
            return SPCONV_OK;
        }
    }
    return SPCONV_ERR_UNSUPPORTED;
}

// Output-channel pairs per warp on the tap-pair layout: Q (Q - 1) / 2.
int slot_pairs(int Q) { return Q * (Q - 1) / 2; }

// Index of the slot pair (q1 < q2) among a warp's pairs, lexicographic.
int pair_index(int Q, int q1, int q2) { return q1 * Q - q1 * (q1 + 1) / 2 + (q2 - q1 - 1); }

// Tap pairs: a tap (c, r, s) that two output channels of one warp both use is
// stored once as a pair entry {w1, w2, offset}; the warp loads the tap's P
// inputs once and updates both channels, so such nonzeros cost half the
// shared-memory loads.  Used where the kernel has tap-pair instances (4 output
// channels per warp, one lane row; 8 leave no registers, 1 has no pairs),
// sparse F32 blobs, and only where pairs remove at
// least a fifth of the shared loads: the pair segments' loops cost enough that
// smaller savings measured slower on GB300 (VGG-style 95 %: 6 % fewer loads,
// 11 % slower; lognormal 80 %: 14 % fewer, 8 % slower), while the 80 % 5x5 and
// 11x11 layers (23 % fewer) ran 16 % and 11 % faster.
void choose_tap_pairs(spconv::Geometry &g, const std::vector<int32_t> &group_flags,
                      const std::vector<std::vector<int64_t>> &order, const int32_t *colidx) {
    g.tap_pairs = 0;
    if (g.format != SPCONV_FORMAT_F32 || g.plane_stage || (g.col_blocks && g.tile_images != 2) ||
        spconv::forward_variant_supported(g.S, g.stride, g.tile_rows, g.slots, g.lane_rows,
                                          true, false, g.col_blocks != 0, g.tight != 0) != 0)
        return;
    int64_t pairs = 0, total = 0;
    std::vector<int32_t> cols;
    for (int grp = 0; grp < g.groups; ++grp) {
        if (group_flags[grp] & 1) continue;
        for (int w = 0; w < g.warps; ++w) {
            cols.clear();
            for (int q = 0; q < g.slots; ++q)
                for (int64_t j : order[((size_t)grp * g.warps + w) * g.slots + q])
                    cols.push_back(colidx[j]);
            std::sort(cols.begin(), cols.end());
            for (size_t i = 0; i < cols.size();) {
                size_t k = i;
                while (k < cols.size() && cols[k] == cols[i]) ++k;
                pairs += (int64_t)(k - i) / 2;
                i = k;
            }
            total += (int64_t)cols.size();
        }
    }
    if (total > 0 && pairs * 5 >= total) {
        g.tap_pairs = 1;
        g.hdr_words = (int)round_up(
            (size_t)g.warps * g.slots + 1 + (size_t)g.warps * slot_pairs(g.slots) + 1, 4);
    }
}

// A column given twice in one row is malformed CSR.
int check_duplicates(int M, const int32_t *rowptr, const int32_t *colidx) {
    std::vector<int32_t> cols;
    for (int m = 0; m < M; ++m) {
        cols.assign(colidx + rowptr[m], colidx + rowptr[m + 1]);
        std::sort(cols.begin(), cols.end());
        if (std::adjacent_find(cols.begin(), cols.end()) != cols.end()) return SPCONV_ERR_BAD_CSR;
    }
    return SPCONV_OK;
}

// Offset of a nonzero (c, r, s) of chunk k in the staged tile.
int32_t tile_offset(const spconv::Geometry &g, int cl, int r, int s) {
    if (g.stride == 1) return cl * g.plane + r * g.row_pitch + s + g.shift;
    return cl * g.plane + r * g.row_pitch + (s % g.stride) * g.phase_pitch + s / g.stride;
}

// One sparse blob of the tap-pair layout: hdr[0 .. warps*Q] single-entry
// ranges (slot w*Q+q spans [hdr[w*Q+q], hdr[w*Q+q+1]), 8-byte entries), then
// hdr[warps*Q + 1 ..] pair ranges (warp w's pair p spans [hp[w*NP+p],
// hp[w*NP+p+1]) in 8-byte units, 16 bytes per pair entry {w1, w2, offset, 0},
// starting on a 16-byte boundary).
void write_pair_blob(const spconv::Geometry &g, int grp, int k, int c_end,
                     const std::vector<std::vector<int64_t>> &order, const int32_t *colidx,
                     const float *value, std::vector<size_t> &cursor, uint32_t *hdr,
                     HostEntry *ent) {
    const int RS = g.R * g.S, Q = g.slots, NP = slot_pairs(Q);
    uint32_t *hp = hdr + g.warps * Q + 1;
    struct Item { int32_t col; int q; float v; };
    std::vector<std::vector<Item>> singles((size_t)g.warps * Q);
    std::vector<std::vector<std::pair<Item, Item>>> pairs((size_t)g.warps * NP);
    std::vector<Item> items;
    for (int w = 0; w < g.warps; ++w) {
        items.clear();
        for (int q = 0; q < Q; ++q) {
            const int slot = (grp * g.warps + w) * Q + q;
            const std::vector<int64_t> &idx = order[slot];
            size_t &t = cursor[slot];
            for (; t < idx.size() && colidx[idx[t]] / RS < c_end; ++t)
                items.push_back({colidx[idx[t]], q, value[idx[t]]});
        }
        // by column, then slot: equal columns are adjacent, paired two by two
        std::stable_sort(items.begin(), items.end(),
                         [](const Item &a, const Item &b) { return a.col < b.col; });
        for (size_t i = 0; i < items.size();) {
            size_t j = i;
            while (j < items.size() && items[j].col == items[i].col) ++j;
            size_t a = i;
            for (; a + 1 < j; a += 2)
                pairs[(size_t)w * NP + pair_index(Q, items[a].q, items[a + 1].q)].push_back(
                    {items[a], items[a + 1]});
            if (a < j) singles[(size_t)w * Q + items[a].q].push_back(items[a]);
            i = j;
        }
    }
    auto offset_of = [&](int32_t col) {
        const int c = col / RS, r = (col / g.S) % g.R, s = col % g.S;
        return tile_offset(g, c - k * g.chunk, r, s);
    };
    uint32_t e = 0;
    for (int ls = 0; ls < g.warps * Q; ++ls) {
        hdr[ls] = e;
        for (const Item &it : singles[ls]) ent[e++] = HostEntry{it.v, offset_of(it.col)};
    }
    hdr[g.warps * Q] = e;
    e = (e + 1) & ~1u;  // pairs start on a 16-byte boundary
    for (int lp = 0; lp < g.warps * NP; ++lp) {
        hp[lp] = e;
        for (const auto &pr : pairs[lp]) {
            float *f = reinterpret_cast<float *>(ent + e);
            f[0] = pr.first.v;
            f[1] = pr.second.v;
            const int32_t off = offset_of(pr.first.col);
            std::memcpy(&f[2], &off, sizeof(off));
            f[3] = 0.f;
            e += 2;
        }
    }
    hp[g.warps * NP] = e;
}

// Builds the host arrays of a handle.  Returns a status.
int build_layout(spconv_packed &P, const int32_t *rowptr, const int32_t *colidx,
                 const float *value) {
    spconv::Geometry &g = P.g;
    const int RS = g.R * g.S;
    // duplicate columns are rejected before anything else
    if (int st = check_duplicates(g.M, rowptr, colidx)) return st;
    int bst = bin_channels(P, rowptr, colidx);
    if (bst) return bst;
    const std::vector<std::vector<int64_t>> &order = P.slot_entries;
    choose_tap_pairs(g, P.group_flags, order, colidx);
    std::vector<int64_t> gpre((size_t)g.groups * (g.C + 1), 0);
    const int slots_per_group = g.warps * g.slots;
    for (int slot = 0; slot < g.num_slots; ++slot) {
        int64_t *pre = &gpre[(size_t)(slot / slots_per_group) * (g.C + 1)];
        for (int64_t j : order[slot]) pre[colidx[j] / RS + 1] += 1;
    }
    for (int grp = 0; grp < g.groups; ++grp) {
        int64_t *pre = &gpre[(size_t)grp * (g.C + 1)];
        for (int c = 0; c < g.C; ++c) pre[c + 1] += pre[c];
    }
    int st = plan_chunks(g, gpre);
    if (st) return st;

    // blobs, in (group, chunk) order
    const int nch = g.num_chunks;
    const size_t nblobs = (size_t)g.groups * nch;
    std::vector<size_t> bsize(nblobs);
    size_t total = 0, largest = 0;
    for (int grp = 0; grp < g.groups; ++grp) {
        const int64_t *pre = &gpre[(size_t)grp * (g.C + 1)];
        for (int k = 0; k < nch; ++k) {
            const int c0 = k * g.chunk, c1 = std::min(g.C, c0 + g.chunk);
            size_t b = (P.group_flags[grp] & 1)
                           ? dense_blob_bytes(g, g.chunk)
                           : (size_t)g.hdr_words * 4 +
                                 round_up((size_t)(pre[c1] - pre[c0]) * entry_bytes(g) +
                                              (g.tap_pairs ? 8 : 0), 16);
            bsize[(size_t)grp * nch + k] = b;
            total += b;
            largest = std::max(largest, b);
        }
    }
    // Nearly equal blobs are stored at a fixed stride (each padded to the
    // largest): a block then finds its blob without first reading blob_off,
    // one dependent global load less before its first stage can start.
    g.blob_stride16 = (largest * nblobs <= total + total / 4) ? (int)(largest / 16) : 0;
    P.blob_off.assign(nblobs + 1, 0);
    size_t at = 0;
    for (size_t b = 0; b < nblobs; ++b) {
        P.blob_off[b] = (uint32_t)(at / 16);
        at += g.blob_stride16 ? largest : bsize[b];
    }
    total = at;
    P.blob_off[nblobs] = (uint32_t)(total / 16);
    if (total / 16 >= ((size_t)1 << 32)) return SPCONV_ERR_UNSUPPORTED;
    P.blobs.assign(total, 0);
    const int kk4 = (int)round_up((size_t)RS, 4);
    std::vector<size_t> cursor(g.num_slots, 0);  // next sorted entry of each slot
    for (int grp = 0; grp < g.groups; ++grp) {
        for (int k = 0; k < nch; ++k) {
            unsigned char *blob = P.blobs.data() + (size_t)P.blob_off[(size_t)grp * nch + k] * 16;
            const int c_end = std::min(g.C, (k + 1) * g.chunk);
            if (P.group_flags[grp] & 1) {
                // [warp][channel] slot masks, then [warp][channel][slot][R*S (to 4)] weights
                uint32_t *mask = reinterpret_cast<uint32_t *>(blob);
                float *wts = reinterpret_cast<float *>(blob + (size_t)g.dense_mask_words * 4);
                for (int w = 0; w < g.warps; ++w)
                    for (int q = 0; q < g.slots; ++q) {
                        const int slot = (grp * g.warps + w) * g.slots + q;
                        const std::vector<int64_t> &idx = order[slot];
                        size_t &t = cursor[slot];
                        for (; t < idx.size(); ++t) {
                            const int col = colidx[idx[t]];
                            const int c = col / RS;
                            if (c >= c_end) break;
                            const int cl = c - k * g.chunk;
                            mask[w * g.chunk + cl] |= 1u << q;
                            const float v = g.format == 1 ? to_half_and_back(value[idx[t]])
                                                          : value[idx[t]];
                            wts[((size_t)(w * g.chunk + cl) * g.slots + q) * kk4 + col % RS] = v;
                        }
                    }
                continue;
            }
            uint32_t *hdr = reinterpret_cast<uint32_t *>(blob);
            HostEntry *ent = reinterpret_cast<HostEntry *>(blob + (size_t)g.hdr_words * 4);
            uint32_t *word = reinterpret_cast<uint32_t *>(blob + (size_t)g.hdr_words * 4);
            if (g.tap_pairs) {
                write_pair_blob(g, grp, k, c_end, order, colidx, value, cursor, hdr, ent);
                continue;
            }
            uint32_t e = 0;
            for (int ls = 0; ls < slots_per_group; ++ls) {
                const int slot = grp * slots_per_group + ls;
                hdr[ls] = e;
                const std::vector<int64_t> &idx = order[slot];
                size_t &t = cursor[slot];
                for (; t < idx.size(); ++t) {
                    const int col = colidx[idx[t]];
                    const int c = col / RS;
                    if (c >= c_end) break;
                    const int r = (col / g.S) % g.R;
                    const int s = col % g.S;
                    const int cl = c - k * g.chunk;
                    if (g.format == 1) {
                        // [31:16] FP16 value, [15:8] channel, [7:4] px (column), [3:0] py (row)
                        const __half hv = __float2half_rn(value[idx[t]]);
                        const uint32_t bits = (uint32_t)__half_as_ushort(hv);
                        word[e++] = (bits << 16) | ((uint32_t)cl << 8) | ((uint32_t)s << 4) |
                                    (uint32_t)r;
                        continue;
                    }
                    HostEntry h;
                    h.value = value[idx[t]];
                    if (g.plane_stage) {
                        // raw planes after the lead margin; bits 3:0 flag the
                        // taps that can leave the image: bit 0 left column,
                        // bit 1 right column, bit 2 top row, bit 3 bottom row
                        const int32_t off = spconv::kPlaneLead + cl * g.plane + (r - 1) * g.W + (s - 1);
                        const int32_t flags = (s == 0 ? 1 : 0) | (s == 2 ? 2 : 0) |
                                              (r == 0 ? 4 : 0) | (r == 2 ? 8 : 0);
                        h.off = (off << 4) | flags;
                    } else if (g.stride == 1) {
                        h.off = cl * g.plane + r * g.row_pitch + s + g.shift;
                    } else {
                        h.off = cl * g.plane + r * g.row_pitch +
                                (s % g.stride) * g.phase_pitch + s / g.stride;
                    }
                    ent[e++] = h;
                }
            }
            hdr[slots_per_group] = e;
        }
    }
    for (int slot = 0; slot < g.num_slots; ++slot)
        if (cursor[slot] != order[slot].size()) return SPCONV_ERR_BAD_CSR;
    P.slot_entries.clear();
    P.slot_entries.shrink_to_fit();
    return SPCONV_OK;
}

// ---- weight-stationary format (Escoin, arXiv 1802.10280, Figs. 5-7: one
// output channel per thread block, its weights kept on chip, the input read
// in place through the read-only cache, one output per thread position)

constexpr int64_t kWsMaxOffset = (int64_t)1 << 24;  // stretched offsets fit 24 bits
constexpr int kWsMaxPiece = 4096;                   // entries per stage (32 KB)

// Tile of one block: 32 / LR columns, 8 warps x LR lane rows x P rows.
int plan_ws(spconv::Geometry &g, int C, int H, int W, int M, int R, int S, int stride, int pad,
            const int32_t *rowptr) {
    g.C = C; g.H = H; g.W = W; g.M = M; g.R = R; g.S = S; g.stride = stride; g.pad = pad;
    g.E = out_extent(H, R, stride, pad);
    g.F = out_extent(W, S, stride, pad);
    g.lane_rows = g.F <= 16 ? 2 : 1;
    const int rows_per_step = spconv::kWarps * g.lane_rows;
    g.tile_w = spconv::kLanes / g.lane_rows;
    g.tiles_x = (g.F + g.tile_w - 1) / g.tile_w;
    // fewest tiles of at most 8 rows per lane, then the smallest instance P
    // that covers the layer's rows with that many tiles
    const int ty = (g.E + rows_per_step * 8 - 1) / (rows_per_step * 8);
    const int need = (g.E + ty * rows_per_step - 1) / (ty * rows_per_step);
    static const int kP[] = {1, 2, 4, 7, 8};
    g.tile_rows = 8;
    for (int cand : kP)
        if (cand >= need) {
            g.tile_rows = cand;
            break;
        }
    if (!spconv::ws_variant_supported(g.tile_rows, g.lane_rows)) return SPCONV_ERR_UNSUPPORTED;
    g.tile_h = rows_per_step * g.tile_rows;
    g.tiles_y = (g.E + g.tile_h - 1) / g.tile_h;
    if ((int64_t)g.tiles_y * g.tiles_x > 65535) return SPCONV_ERR_UNSUPPORTED;
    int64_t longest = 0;
    for (int m = 0; m < M; ++m) longest = std::max<int64_t>(longest, rowptr[m + 1] - rowptr[m]);
    g.chunk = (int)std::min<int64_t>(kWsMaxPiece, std::max<int64_t>(2, round_up(longest, 2)));
    g.num_chunks = (int)std::max<int64_t>(1, (longest + g.chunk - 1) / g.chunk);
    g.warps = spconv::kWarps;
    g.slots = 1;
    g.groups = 0;
    g.num_slots = M;
    return SPCONV_OK;
}

// Row m's entries in column order, each {value, off << 8 | r << 4 | s} with
// off = c*H*W + r*W + s (weight stretching against the input tensor itself);
// every row starts on an even entry (16 bytes) and the array ends on one.
int build_layout_ws(spconv_packed &P, const int32_t *rowptr, const int32_t *colidx,
                    const float *value) {
    spconv::Geometry &g = P.g;
    if (int st = check_duplicates(g.M, rowptr, colidx)) return st;
    const int RS = g.R * g.S;
    const int64_t HW = (int64_t)g.H * g.W;
    std::vector<HostEntry> ent;
    ent.reserve((size_t)P.nnz + 2 * (size_t)g.M + 2);
    P.blob_off.assign(2 * (size_t)g.M, 0);
    std::vector<int64_t> order;
    for (int m = 0; m < g.M; ++m) {
        const int64_t j0 = rowptr[m], j1 = rowptr[m + 1];
        order.assign((size_t)(j1 - j0), 0);
        std::iota(order.begin(), order.end(), j0);
        std::sort(order.begin(), order.end(),
                  [&](int64_t a, int64_t b) { return colidx[a] < colidx[b]; });
        P.blob_off[2 * (size_t)m] = (uint32_t)ent.size();
        P.blob_off[2 * (size_t)m + 1] = (uint32_t)(j1 - j0);
        for (int64_t j : order) {
            const int col = colidx[j];
            const int c = col / RS, r = (col % RS) / g.S, s = col % g.S;
            const int64_t off = c * HW + (int64_t)r * g.W + s;
            HostEntry e;
            e.value = value[j];
            e.off = (int32_t)(((uint32_t)off << 8) | ((uint32_t)r << 4) | (uint32_t)s);
            ent.push_back(e);
        }
        if (ent.size() & 1) ent.push_back(HostEntry{0.f, 0});
    }
    if (ent.empty()) ent.push_back(HostEntry{0.f, 0});
    if (ent.size() & 1) ent.push_back(HostEntry{0.f, 0});
    if (ent.size() >= ((size_t)1 << 32)) return SPCONV_ERR_UNSUPPORTED;
    P.blobs.resize(ent.size() * sizeof(HostEntry));
    std::memcpy(P.blobs.data(), ent.data(), P.blobs.size());
    // heaviest rows first: the hardware hands out blocks in grid order
    P.slot_oc.resize(g.M);
    std::iota(P.slot_oc.begin(), P.slot_oc.end(), 0);
    std::stable_sort(P.slot_oc.begin(), P.slot_oc.end(), [&](int a, int b) {
        return rowptr[a + 1] - rowptr[a] > rowptr[b + 1] - rowptr[b];
    });
    P.slot_next.clear();
    P.group_flags.clear();
    int64_t longest = 0;
    for (int m = 0; m < g.M; ++m) longest = std::max<int64_t>(longest, rowptr[m + 1] - rowptr[m]);
    P.max_warp_nnz = longest;
    P.mean_warp_nnz = g.M ? P.nnz / g.M : 0;
    return SPCONV_OK;
}

int make_handle(int C, int H, int W, int M, int R, int S, int stride, int pad,
                const int32_t *rowptr, const int32_t *colidx, const float *value, int format,
                int batch_hint, spconv_packed **out) {
    if (!out) return SPCONV_ERR_INVALID_ARG;
    if (format != SPCONV_FORMAT_F32 && format != SPCONV_FORMAT_PACKED32 &&
        format != SPCONV_FORMAT_WS)
        return SPCONV_ERR_INVALID_ARG;
    if (batch_hint < 0) return SPCONV_ERR_INVALID_ARG;
    int st = validate_shape(C, H, W, M, R, S, stride, pad);
    if (st) return st;
    if ((format == SPCONV_FORMAT_PACKED32 || format == SPCONV_FORMAT_WS) && (R > 16 || S > 16))
        return SPCONV_ERR_UNSUPPORTED;
    if (format == SPCONV_FORMAT_WS &&
        (int64_t)C * H * W + (int64_t)R * W + S > kWsMaxOffset)
        return SPCONV_ERR_UNSUPPORTED;
    int64_t nnz = 0;
    st = validate_csr(M, (int64_t)C * R * S, rowptr, colidx, value, &nnz);
    if (st) return st;
    if (nnz >= ((int64_t)1 << 31) - 16) return SPCONV_ERR_UNSUPPORTED;
    spconv_packed *P = new (std::nothrow) spconv_packed();
    if (!P) return SPCONV_ERR_ALLOC;
    P->nnz = nnz;
    P->g.format = format;
    P->g.batch_hint = batch_hint > 0 ? batch_hint : 0;
    if (format == SPCONV_FORMAT_WS) {
        st = plan_ws(P->g, C, H, W, M, R, S, stride, pad, rowptr);
        if (!st) st = build_layout_ws(*P, rowptr, colidx, value);
    } else {
        // share of the nonzeros in rows dense enough for the dense-tap path
        int64_t dense_nnz = 0;
        const double crs = (double)C * R * S;
        for (int m = 0; m < M; ++m) {
            const int64_t k = (int64_t)rowptr[m + 1] - rowptr[m];
            if (k / crs >= kDenseRowMin) dense_nnz += k;
        }
        st = plan_tiles(P->g, C, H, W, M, R, S, stride, pad, nnz,
                        nnz > 0 ? (double)dense_nnz / nnz : 0.0);
        if (!st) st = build_layout(*P, rowptr, colidx, value);
    }
    if (st) {
        delete P;
        return st;
    }
    *out = P;
    return SPCONV_OK;
}

int upload(spconv_packed *P, cudaStream_t stream) {
    if (cudaGetDevice(&P->device) != cudaSuccess) return SPCONV_ERR_CUDA;
    const size_t b_blobs = round_up(std::max<size_t>(P->blobs.size(), 16), 256);
    const size_t b_off = round_up(P->blob_off.size() * sizeof(uint32_t), 256);
    const size_t b_slot = round_up(P->slot_oc.size() * sizeof(int32_t), 256);
    const size_t b_next = round_up(P->slot_next.size() * sizeof(int32_t), 256);
    const size_t b_gd = round_up(P->group_flags.size() * sizeof(int32_t), 256);
    const size_t b_err = 256;
    P->dev_bytes = b_blobs + b_off + b_slot + b_next + b_gd + b_err;
    void *blk = nullptr;
    if (cudaMalloc(&blk, P->dev_bytes) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_ALLOC;
    }
    P->dev_block = blk;
    char *base = static_cast<char *>(blk);
    bool ok = cudaMemsetAsync(base, 0, P->dev_bytes, stream) == cudaSuccess;
    ok = ok && (P->blobs.empty() ||
                cudaMemcpyAsync(base, P->blobs.data(), P->blobs.size(), cudaMemcpyHostToDevice,
                                stream) == cudaSuccess);
    auto put = [&](size_t at, const void *src, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(base + at, src, bytes, cudaMemcpyHostToDevice,
                                             stream) == cudaSuccess;
    };
    ok = ok && put(b_blobs, P->blob_off.data(), P->blob_off.size() * sizeof(uint32_t));
    ok = ok && put(b_blobs + b_off, P->slot_oc.data(), P->slot_oc.size() * sizeof(int32_t));
    ok = ok && put(b_blobs + b_off + b_slot, P->slot_next.data(),
                   P->slot_next.size() * sizeof(int32_t));
    ok = ok && put(b_blobs + b_off + b_slot + b_next, P->group_flags.data(),
                   P->group_flags.size() * sizeof(int32_t));
    ok = ok && cudaStreamSynchronize(stream) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    P->d.blobs = reinterpret_cast<const unsigned char *>(base);
    P->d.blob_off = reinterpret_cast<const uint32_t *>(base + b_blobs);
    P->d.slot_oc = reinterpret_cast<const int *>(base + b_blobs + b_off);
    P->d.slot_next = reinterpret_cast<const int *>(base + b_blobs + b_off + b_slot);
    P->d.group_flags = reinterpret_cast<const int *>(base + b_blobs + b_off + b_slot + b_next);
    P->d.err = reinterpret_cast<unsigned int *>(base + b_blobs + b_off + b_slot + b_next + b_gd);
    P->d.blob_bytes = (int64_t)P->blobs.size();
    return SPCONV_OK;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

// ---- device mapping of page-locked host buffers (spconv_forward_host)

using PointerAttrFn = CUresult (*)(void *, CUpointer_attribute, CUdeviceptr);

PointerAttrFn pointer_attr_fn() {
    static PointerAttrFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PointerAttrFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// The address through which kernels on the current device reach the host
// buffer [host, host + bytes), or nullptr when there is none: the buffer must
// be page-locked memory that CUDA maps for this device, and the allocation
// CUDA reports for it must hold all `bytes`.  Anything else (pageable memory,
// a range CUDA cannot confirm) gets nullptr, and the caller copies with
// cudaMemcpyAsync instead.
void *mapped_view(const void *host, size_t bytes) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer || !a.hostPointer) return nullptr;
    PointerAttrFn get = pointer_attr_fn();
    if (!get) return nullptr;
    CUdeviceptr start = 0;
    size_t size = 0;
    const CUdeviceptr dp = (CUdeviceptr)(uintptr_t)a.devicePointer;
    if (get(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
        get(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS)
        return nullptr;
    if (dp < start || dp - start > size || size - (dp - start) < bytes) return nullptr;
    return a.devicePointer;
}

// ---- TMA tensor map of the input (stride-1 layers with 16-byte row stride)

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool tma_eligible(const spconv::Geometry &g) {
    return g.stride == 1 && (g.W * sizeof(float)) % 16 == 0 && g.row_pitch <= 256 &&
           g.in_rows <= 256 && g.chunk <= 256;
}

// Returns a tensor map for (x, N), or nullptr if TMA staging is not possible.
const CUtensorMap *input_tmap(const spconv_packed *P, const float *x, int N, CUtensorMap &tmp) {
    const spconv::Geometry &g = P->g;
    if (!tma_eligible(g)) return nullptr;
    {
        std::lock_guard<std::mutex> lk(P->tmap_lock);
        for (const TmapCacheEntry &e : P->tmap_cache)
            if (e.x == x && e.N == N) {
                tmp = e.map;
                return &tmp;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return nullptr;
    cuuint64_t dims[4] = {(cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.C, (cuuint64_t)N};
    cuuint64_t strides[3] = {(cuuint64_t)g.W * 4, (cuuint64_t)g.H * g.W * 4,
                             (cuuint64_t)g.C * g.H * g.W * 4};
    // (image pairs: the box spans two images, the second sub-tile right after
    // the first -- chunk * plane words later, which the planner makes 16 mod 32)
    cuuint32_t box[4] = {(cuuint32_t)g.row_pitch, (cuuint32_t)g.in_rows, (cuuint32_t)g.chunk,
                         (cuuint32_t)(g.tile_images == 2 ? 2 : 1)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(&tmp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lk(P->tmap_lock);
    TmapCacheEntry &slot = P->tmap_cache[P->tmap_next++ % 4];
    slot.x = x;
    slot.N = N;
    slot.map = tmp;
    return &tmp;
}

// Whether to run all channel groups of a tile together.  With tiles first
// (the default order) every group streams the whole input from HBM once the
// input exceeds L2; with groups first the tile's input is read from HBM once
// and shared through L2, but all groups then hit the same lines at once.
// Groups first wins when re-streaming the input would take longer than a
// quarter of the layer's compute at the sparse path's rate (~18 % of fp32
// peak); the quarter is the crossover measured on GB300 over the first
// page's 256 x 256 sweep (90 % sparse: tiles first; 98 %: groups first).
bool choose_group_fast(const spconv::Geometry &g, int N, int64_t nnz) {
    const double in_bytes = 4.0 * N * g.C * g.H * g.W;
    if (g.groups < 2 || in_bytes < 64.0 * (1 << 20)) return false;
    const double hbm_bps = 6.7e12, sparse_flops = 0.18 * kSMs * 128 * 2 * 2.07e9;
    const double restream_s = (g.groups - 1) * in_bytes / hbm_bps;
    const double compute_s = 2.0 * nnz * N * g.E * g.F / sparse_flops;
    return restream_s * 4.0 > compute_s;
}

// Programmatic dependent launch hides a launch's start-up behind the previous
// kernel's tail: worth most for the short one-wave launches of small layers
// (one-image ResNet layer 8.6 -> 7.3 us back to back).  Measured to cost 4 %
// on a multi-wave layer with dense-tap groups (lognormal sweep, 80 %), so
// those launch without it.
bool choose_pdl(const spconv::Geometry &g, int N, int split, bool group_fast) {
    unsigned gx = 0, gy = 0;
    spconv::forward_grid(g, N, split, group_fast, &gx, &gy);
    return !(g.dense_groups > 0 && (int64_t)gx * gy > 2 * kSMs);
}

// Blocks per cluster along the channel chunks: none when the grid already
// fills the GPU (splitting it further measured slower on every batched layer),
// else enough for about two blocks per SM
// (measured best on the one-image ResNet-style layer).
int choose_split(const spconv::Geometry &g, int N) {
    const int64_t blocks = (int64_t)((N + g.tile_images - 1) / g.tile_images) * g.tiles_y *
                           g.tiles_x * g.groups;
    // Plans of two to four waves whose groups are mostly dense-tap: those
    // blocks are FMA-bound and run ~2x longer than the sparse ones, so the
    // launch ends with them; splitting every tile's chunks over a two-block
    // cluster halves them at the price of the cluster reduction.  Measured on
    // the 50 % lognormal layer (10 of 17 groups dense): 582 -> 543 us; where
    // sparse groups dominate the same split is slower (90 %: 210 -> 237 us,
    // 80 % with 3 of 16 dense: 349 -> 377).
    if (blocks >= 2 * kSMs && blocks <= 4 * kSMs && g.num_chunks >= 4 &&
        g.dense_groups * 2 >= g.groups)
        return 2;
    if (blocks >= kSMs) return 1;
    int s = (int)std::min<int64_t>(spconv::kMaxSplit, (2 * kSMs + blocks - 1) / blocks);
    return std::max(1, std::min(s, g.num_chunks));
}

// Checks of a forward call, before anything is enqueued: the handle, the
// shape, the device pointers' alignment and overlap, the current device.
int check_forward(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                  const float *input, const spconv_packed *packed, const float *bias, int act,
                  const float *output) {
    if (!packed || N < 0) return SPCONV_ERR_INVALID_ARG;
    if (act != SPCONV_ACT_NONE && act != SPCONV_ACT_RELU) return SPCONV_ERR_INVALID_ARG;
    const spconv::Geometry &g = packed->g;
    if (C != g.C || H != g.H || W != g.W || M != g.M || R != g.R || S != g.S ||
        stride != g.stride || pad != g.pad)
        return SPCONV_ERR_MISMATCH;
    if (!packed->dev_block) return SPCONV_ERR_MISMATCH;
    if (N == 0) return SPCONV_OK;
    if (!input || !output) return SPCONV_ERR_INVALID_ARG;
    if (((uintptr_t)input & 15) || ((uintptr_t)output & 3) || ((uintptr_t)bias & 3))
        return SPCONV_ERR_INVALID_ARG;
    const int64_t tiles = (int64_t)N * g.tiles_y * g.tiles_x * spconv::kMaxSplit * g.groups;
    if (tiles > 0x7fffffffLL) return SPCONV_ERR_UNSUPPORTED;
    if (g.format == SPCONV_FORMAT_WS && N > 65535) return SPCONV_ERR_UNSUPPORTED;  // grid z
    const size_t in_bytes = (size_t)N * C * H * W * sizeof(float);
    const size_t out_bytes = (size_t)N * M * g.E * g.F * sizeof(float);
    if (ranges_overlap(input, in_bytes, output, out_bytes)) return SPCONV_ERR_INVALID_ARG;
    if (bias && ranges_overlap(bias, (size_t)M * sizeof(float), output, out_bytes))
        return SPCONV_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPCONV_ERR_CUDA;
    if (dev != packed->device) return SPCONV_ERR_MISMATCH;
    return SPCONV_OK;
}

// Launches a forward whose arguments check_forward accepted (N > 0).  The
// launch mode (programmatic dependent launch or not) is choose_pdl's, also
// behind the host-buffer forward's copy kernel: the forward waits for the
// previous kernel either way before it reads its input.
int enqueue_forward(int N, const float *input, const spconv_packed *packed, const float *bias,
                    int act, float *output, cudaStream_t stream) {
    const spconv::Geometry &g = packed->g;
    if (g.format == SPCONV_FORMAT_WS) {
        cudaError_t e =
            spconv::launch_forward_ws(g, N, input, output, bias, act, packed->d, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return SPCONV_ERR_CUDA;
        }
        return SPCONV_OK;
    }
    try {
        CUtensorMap tmp;
        const CUtensorMap *tmap = input_tmap(packed, input, N, tmp);
        const int split = choose_split(g, N);
        const bool group_fast = choose_group_fast(g, N, packed->nnz);
        const bool pdl = choose_pdl(g, N, split, group_fast);
        cudaError_t e = spconv::launch_forward(g, N, split, group_fast, pdl, input, output, bias,
                                               act, packed->d, tmap, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return SPCONV_ERR_CUDA;
        }
    } catch (...) {
        return SPCONV_ERR_ALLOC;
    }
    return SPCONV_OK;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int spconv_pack_ex(
    int C, int H, int W, int M, int R, int S, int stride, int pad, const int32_t *rowptr,
    const int32_t *colidx, const float *value, int format, int batch_hint, int host_only,
    void *stream, spconv_packed **out) {
    try {
        spconv_packed *P = nullptr;
        int st = make_handle(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, format,
                             batch_hint, &P);
        if (st) return st;
        if (!host_only) {
            st = upload(P, static_cast<cudaStream_t>(stream));
            if (st) {
                spconv_packed_free(P);
                return st;
            }
        }
        *out = P;
        return SPCONV_OK;
    } catch (...) {
        return SPCONV_ERR_ALLOC;
    }
}

__attribute__((visibility("default"))) int spconv_pack_host(
    int C, int H, int W, int M, int R, int S, int stride, int pad, const int32_t *rowptr,
    const int32_t *colidx, const float *value, spconv_packed **out) {
    return spconv_pack_ex(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, SPCONV_FORMAT_F32,
                          0, 1, nullptr, out);
}

__attribute__((visibility("default"))) int spconv_pack(
    int C, int H, int W, int M, int R, int S, int stride, int pad, const int32_t *rowptr,
    const int32_t *colidx, const float *value, void *stream, spconv_packed **out) {
    return spconv_pack_ex(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, SPCONV_FORMAT_F32,
                          0, 0, stream, out);
}

__attribute__((visibility("default"))) int spconv_forward_ex(
    int N, int C, int H, int W, int M, int R, int S, int stride, int pad, const float *input,
    const spconv_packed *packed, const float *bias, int act, float *output, void *stream) {
    const int st = check_forward(N, C, H, W, M, R, S, stride, pad, input, packed, bias, act, output);
    if (st != SPCONV_OK || N == 0) return st;
    return enqueue_forward(N, input, packed, bias, act, output, static_cast<cudaStream_t>(stream));
}

__attribute__((visibility("default"))) int spconv_forward_host(
    int N, int C, int H, int W, int M, int R, int S, int stride, int pad, const float *input_host,
    const spconv_packed *packed, const float *bias, int act, float *output_host,
    float *dev_input, float *dev_output, void *stream) {
    int st = check_forward(N, C, H, W, M, R, S, stride, pad, dev_input, packed, bias, act,
                           dev_output);
    if (st != SPCONV_OK || N == 0) return st;
    if (!input_host || !output_host || ((uintptr_t)output_host & 3)) return SPCONV_ERR_INVALID_ARG;
    const size_t n_in = (size_t)N * C * H * W;
    const size_t in_bytes = n_in * sizeof(float);
    const size_t out_bytes = (size_t)N * M * packed->g.E * packed->g.F * sizeof(float);
    if (ranges_overlap(input_host, in_bytes, output_host, out_bytes)) return SPCONV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Page-locked buffers that CUDA maps for this device: the input is copied
    // by the SMs; a small Y is written by the forward straight into the host
    // buffer (its write-back is plain stores, each output once), a large one
    // goes to dev_output and is copied out by the SMs in 16-byte vectors (the
    // forward's row segments make poorer writes over the host link).
    // Otherwise: copy engine in, forward into dev_output, copy engine out.
    const float *in_view = static_cast<const float *>(mapped_view(input_host, in_bytes));
    float *out_view = static_cast<float *>(mapped_view(output_host, out_bytes));
    if (in_view && out_view) {
        if (spconv::launch_copy(in_view, dev_input, n_in, s) != cudaSuccess) {
            cudaGetLastError();
            return SPCONV_ERR_CUDA;
        }
        const bool direct = out_bytes <= kDirectOutBytes;
        st = enqueue_forward(N, dev_input, packed, bias, act, direct ? out_view : dev_output, s);
        if (st != SPCONV_OK || direct) return st;
        if (spconv::launch_copy(dev_output, out_view, out_bytes / sizeof(float), s) !=
            cudaSuccess) {
            cudaGetLastError();
            return SPCONV_ERR_CUDA;
        }
        return SPCONV_OK;
    }
    if (cudaMemcpyAsync(dev_input, input_host, in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    st = enqueue_forward(N, dev_input, packed, bias, act, dev_output, s);
    if (st != SPCONV_OK) return st;
    if (cudaMemcpyAsync(output_host, dev_output, out_bytes, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    return SPCONV_OK;
}

__attribute__((visibility("default"))) int spconv_forward(
    int N, int C, int H, int W, int M, int R, int S, int stride, int pad, const float *input,
    const spconv_packed *packed, float *output, void *stream) {
    return spconv_forward_ex(N, C, H, W, M, R, S, stride, pad, input, packed, nullptr,
                             SPCONV_ACT_NONE, output, stream);
}

__attribute__((visibility("default"))) int spconv_device_status(const spconv_packed *p,
                                                                void *stream, int32_t *flags) {
    if (!p || !p->dev_block) return SPCONV_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return SPCONV_ERR_CUDA;
    if (cur != p->device) return SPCONV_ERR_MISMATCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, p->d.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(p->d.err, 0, sizeof(word)) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    if (flags) *flags = (int32_t)word;
    return word ? SPCONV_ERR_DEVICE : SPCONV_OK;
}

__attribute__((visibility("default"))) int spconv_trace_read(void *host_dst, int64_t bytes) {
    if (!host_dst || bytes < 0) return SPCONV_ERR_INVALID_ARG;
    return spconv::trace_read(host_dst, bytes);
}

__attribute__((visibility("default"))) int spconv_selftest_wait(int complete, void *stream,
                                                                int32_t *flags) {
    if (!flags) return SPCONV_ERR_INVALID_ARG;
    unsigned int *d = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMalloc(&d, sizeof(unsigned int)) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_ALLOC;
    }
    unsigned int word = 0;
    bool ok = cudaMemsetAsync(d, 0, sizeof(unsigned int), s) == cudaSuccess &&
              spconv::launch_wait_selftest(d, complete ? 1 : 0, s) == cudaSuccess &&
              cudaMemcpyAsync(&word, d, sizeof(word), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
              cudaStreamSynchronize(s) == cudaSuccess;
    cudaFree(d);
    if (!ok) {
        cudaGetLastError();
        return SPCONV_ERR_CUDA;
    }
    *flags = (int32_t)word;
    return (word & 1u) ? SPCONV_ERR_DEVICE : SPCONV_OK;
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
        case SPCONV_ERR_DEVICE: return "a kernel reported a device-side failure";
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
    info->entries = p->nnz;
    info->tile_rows = g.tile_rows;
    info->shift = g.shift;
    info->tile_cols = g.tile_w;
    info->lane_rows = g.lane_rows;
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
    info->smem_bytes = (int64_t)(g.format == SPCONV_FORMAT_WS ? spconv::ws_smem_bytes(g)
                                                               : spconv::forward_smem_bytes(g, 1));
    info->max_warp_nnz = p->max_warp_nnz;
    info->mean_warp_nnz = p->mean_warp_nnz;
    info->hdr_words = g.hdr_words;
    info->blob_stage_bytes = (int32_t)g.blob_stage_bytes;
    info->in_stage_bytes = (int32_t)g.in_stage_bytes;
    info->dense_groups = g.dense_groups;
    info->format = g.format;
    info->batch_hint = g.batch_hint;
    info->dense_mask_words = g.dense_mask_words;
    info->blob_stride = g.blob_stride16 * 16;
    info->tap_pairs = g.tap_pairs;
    info->plane_stage = g.plane_stage;
    info->col_blocks = g.col_blocks;
    info->tile_images = g.tile_images;
    info->pair_off = g.pair_off;
    return SPCONV_OK;
}

__attribute__((visibility("default"))) int spconv_launch_info_get(const spconv_packed *p, int N,
                                                                  spconv_launch_info *info) {
    if (!p || !info || N < 1) return SPCONV_ERR_INVALID_ARG;
    const spconv::Geometry &g = p->g;
    std::memset(info, 0, sizeof(*info));
    info->block_threads = spconv::kWarps * 32;
    if (g.format == SPCONV_FORMAT_WS) {
        if (N > 65535) return SPCONV_ERR_UNSUPPORTED;
        info->kernel = 1;
        info->grid_x = g.M;
        info->grid_y = g.tiles_y * g.tiles_x;
        info->grid_z = N;
        info->cluster = 1;
        info->smem_bytes = (int64_t)spconv::ws_smem_bytes(g);
        return SPCONV_OK;
    }
    const int64_t tiles = (int64_t)N * g.tiles_y * g.tiles_x * spconv::kMaxSplit * g.groups;
    if (tiles > 0x7fffffffLL) return SPCONV_ERR_UNSUPPORTED;
    const int split = choose_split(g, N);
    const bool group_fast = choose_group_fast(g, N, p->nnz);
    unsigned gx = 0, gy = 0;
    spconv::forward_grid(g, N, split, group_fast, &gx, &gy);
    info->kernel = 0;
    info->grid_x = (int32_t)gx;
    info->grid_y = (int32_t)gy;
    info->grid_z = 1;
    info->cluster = split;
    info->push = spconv::push_reduction(g, split) ? 1 : 0;
    info->group_fast = group_fast ? 1 : 0;
    info->pdl = choose_pdl(g, N, split, group_fast) ? 1 : 0;
    info->tma = tma_eligible(g) ? 1 : 0;
    info->smem_bytes = (int64_t)spconv::forward_smem_bytes(g, split);
    return SPCONV_OK;
}

__attribute__((visibility("default"))) int spconv_packed_copy_array(
    const spconv_packed *p, int which, void *dst, int64_t dst_bytes, int64_t *needed) {
    if (!p) return SPCONV_ERR_INVALID_ARG;
    const void *src = nullptr;
    int64_t n = 0;
    switch (which) {
        case SPCONV_ARRAY_BLOBS:
            src = p->blobs.data();
            n = (int64_t)p->blobs.size();
            break;
        case SPCONV_ARRAY_BLOB_OFF:
            src = p->blob_off.data();
            n = (int64_t)(p->blob_off.size() * sizeof(uint32_t));
            break;
        case SPCONV_ARRAY_SLOT_OC:
            src = p->slot_oc.data();
            n = (int64_t)(p->slot_oc.size() * sizeof(int32_t));
            break;
        case SPCONV_ARRAY_SLOT_NEXT:
            src = p->slot_next.data();
            n = (int64_t)(p->slot_next.size() * sizeof(int32_t));
            break;
        case SPCONV_ARRAY_GROUP_FLAGS:
            src = p->group_flags.data();
            n = (int64_t)(p->group_flags.size() * sizeof(int32_t));
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
