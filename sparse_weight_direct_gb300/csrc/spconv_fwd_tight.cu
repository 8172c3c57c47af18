// Kernel instances with tight-pitch tiles: 3x3 stride-1 pad-1 layers up to 31
// outputs wide in one column-per-lane tile column, staged at a 32-word pitch
// from column 0 (the copy's zero fill stands in for the halo columns); seven
// rows per lane, 1, 2, 4 or 8 output channels per warp.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_tight(int P, int Q) {
    // (eight rows per lane never plans tight: where it would, the 8 x 28
    // column blocks cover the same rows with fewer idle lanes)
    if (P != 7) return nullptr;
    switch (Q) {
        case 1: return spconv_fwd_kernel<7, 1, 3, 1, 1, 0, 32>;
        case 2: return spconv_fwd_kernel<7, 2, 3, 1, 1, 0, 32>;
        case 4: return spconv_fwd_kernel<7, 4, 3, 1, 1, 0, 32>;
        case 8: return spconv_fwd_kernel<7, 8, 3, 1, 1, 0, 32>;
        default: return nullptr;
    }
}

}  // namespace kern
}  // namespace spconv
