// Kernel instances with image-pair column blocks: 3x3 stride-1 layers 22..28
// outputs wide.  Four lane rows of eight lanes, each lane holding seven
// consecutive outputs of its row; lanes 0..3 of a row cover image 2n and
// lanes 4..7 image 2n + 1, so a 4 x 28 tile of each of two images leaves no
// lane idle; 1, 2, 4 or 8 output channels per warp.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_colpair(int P, int Q) {
    if (P != 7) return nullptr;
    switch (Q) {
        case 1: return spconv_fwd_kernel<7, 1, 3, 1, 4, kModeColsPair>;
        case 2: return spconv_fwd_kernel<7, 2, 3, 1, 4, kModeColsPair>;
        case 4: return spconv_fwd_kernel<7, 4, 3, 1, 4, kModeColsPair>;
        case 8: return spconv_fwd_kernel<7, 8, 3, 1, 4, kModeColsPair>;
        default: return nullptr;
    }
}

}  // namespace kern
}  // namespace spconv
