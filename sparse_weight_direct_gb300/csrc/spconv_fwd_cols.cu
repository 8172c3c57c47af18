// Kernel instances with column blocks: 3x3 stride-1 layers whose output width
// is a multiple of 28 but not of 32 (56, 112, ...).  Eight lane rows of four
// lanes, each lane holding seven consecutive outputs of its row, cover an
// 8 x 28 tile with no idle lane; 1, 2, 4 or 8 output channels per warp.
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_cols(int P, int Q, int LR) {
    if (P != 7 || LR != 8) return nullptr;
    switch (Q) {
        case 1: return spconv_fwd_kernel<7, 1, 3, 1, 8, kModeCols>;
        case 2: return spconv_fwd_kernel<7, 2, 3, 1, 8, kModeCols>;
        case 4: return spconv_fwd_kernel<7, 4, 3, 1, 8, kModeCols>;
        case 8: return spconv_fwd_kernel<7, 8, 3, 1, 8, kModeCols>;
        default: return nullptr;
    }
}

}  // namespace kern
}  // namespace spconv
