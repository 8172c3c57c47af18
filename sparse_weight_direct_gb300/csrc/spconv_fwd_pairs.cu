// Kernel instances with tap-pair segments: 4 output channels per warp, one
// lane row of 32 output columns, for the kernel shapes with compile-time
// widths (3x3 and 5x5 stride 1, 11x11 stride 4).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_pairs(int S, int stride, int P, int Q, int LR) {
    if (Q != 4 || LR != 1 || (P != 7 && P != 8)) return nullptr;
    const bool p8 = P == 8;
    if (S == 3 && stride == 1)
        return p8 ? spconv_fwd_kernel<8, 4, 3, 1, 1, kModePairs> : spconv_fwd_kernel<7, 4, 3, 1, 1, kModePairs>;
    if (S == 5 && stride == 1)
        return p8 ? spconv_fwd_kernel<8, 4, 5, 1, 1, kModePairs> : spconv_fwd_kernel<7, 4, 5, 1, 1, kModePairs>;
    if (S == 11 && stride == 4)
        return p8 ? spconv_fwd_kernel<8, 4, 11, 4, 1, kModePairs> : spconv_fwd_kernel<7, 4, 11, 4, 1, kModePairs>;
    return nullptr;
}

}  // namespace kern
}  // namespace spconv
