// Kernel instances with plane staging: whole-image tiles of 3x3 stride-1
// layers with two lane rows (outputs at most 16 wide) whose input rows a TMA
// tensor map cannot address; 1 or 2 output channels per warp.  14-wide images
// (the common 14 x 14 case) get instances with the lane's row step (2 W = 28
// words) fixed at compile time, so each nonzero's P shared loads use immediate
// offsets (measured 5.95 -> 5.63 us on the one-image ResNet-style layer); other
// widths take it at run time.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_plane(int P, int Q, int W) {
    if (W == 14) {
        if (P == 7 && Q == 1) return spconv_fwd_kernel<7, 1, 3, 1, 2, kModePlane, 28>;
        if (P == 7 && Q == 2) return spconv_fwd_kernel<7, 2, 3, 1, 2, kModePlane, 28>;
    }
    if (P == 7 && Q == 1) return spconv_fwd_kernel<7, 1, 3, 1, 2, kModePlane>;
    if (P == 8 && Q == 1) return spconv_fwd_kernel<8, 1, 3, 1, 2, kModePlane>;
    if (P == 7 && Q == 2) return spconv_fwd_kernel<7, 2, 3, 1, 2, kModePlane>;
    if (P == 8 && Q == 2) return spconv_fwd_kernel<8, 2, 3, 1, 2, kModePlane>;
    return nullptr;
}

}  // namespace kern
}  // namespace spconv
