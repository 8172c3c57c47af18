// Kernel instances with 8 output channel(s) per warp (one translation unit per
// count so the instances compile in parallel).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_q8(int S, int stride, int P, int LR) { return pick_instances<8>(S, stride, P, LR); }

}  // namespace kern
}  // namespace spconv
