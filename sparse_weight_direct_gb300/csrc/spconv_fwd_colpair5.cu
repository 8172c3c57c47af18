// Kernel instances with image-pair column blocks for 5x5 stride-1 layers 22..28
// outputs wide (the layout of the 3x3 instances: four lane rows of eight
// lanes, lanes 0..3 of a row on image 2n and 4..7 on image 2n + 1, seven
// consecutive outputs each), with and without tap-pair segments.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_colpair5(int P, int Q, bool pairs) {
    if (P != 7) return nullptr;
    if (pairs) return Q == 4 ? spconv_fwd_kernel<7, 4, 5, 1, 4, kModeColsPairTaps> : nullptr;
    switch (Q) {
        case 1: return spconv_fwd_kernel<7, 1, 5, 1, 4, kModeColsPair>;
        case 2: return spconv_fwd_kernel<7, 2, 5, 1, 4, kModeColsPair>;
        case 4: return spconv_fwd_kernel<7, 4, 5, 1, 4, kModeColsPair>;
        case 8: return spconv_fwd_kernel<7, 8, 5, 1, 4, kModeColsPair>;
        default: return nullptr;
    }
}

}  // namespace kern
}  // namespace spconv
