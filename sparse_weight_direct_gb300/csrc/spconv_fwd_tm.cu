// Kernel instances of the tensor-memory window path (3 x 3, stride 1, one
// lane row of 32 output columns; 4 or 8 output channels per warp).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_tm(int P, int Q) {
    if (P == 7 && Q == 4) return spconv_fwd_kernel<7, 4, 3, 1, 1, 1>;
    if (P == 8 && Q == 4) return spconv_fwd_kernel<8, 4, 3, 1, 1, 1>;
    if (P == 7 && Q == 8) return spconv_fwd_kernel<7, 8, 3, 1, 1, 1>;
    if (P == 8 && Q == 8) return spconv_fwd_kernel<8, 8, 3, 1, 1, 1>;
    return nullptr;
}

}  // namespace kern
}  // namespace spconv
