// Kernel instances with plane staging: whole-image tiles of 3x3 stride-1
// layers with two lane rows (outputs at most 16 wide) whose input rows a TMA
// tensor map cannot address; 1 or 2 output channels per warp.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_plane(int P, int Q) {
    if (P == 7 && Q == 1) return spconv_fwd_kernel<7, 1, 3, 1, 2, kModePlane>;
    if (P == 8 && Q == 1) return spconv_fwd_kernel<8, 1, 3, 1, 2, kModePlane>;
    if (P == 7 && Q == 2) return spconv_fwd_kernel<7, 2, 3, 1, 2, kModePlane>;
    if (P == 8 && Q == 2) return spconv_fwd_kernel<8, 2, 3, 1, 2, kModePlane>;
    return nullptr;
}

}  // namespace kern
}  // namespace spconv
