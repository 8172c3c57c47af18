// Kernel instances with 4 output channel(s) per warp (one translation unit per
// count so the instances compile in parallel).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_q4(int S, int stride, int P, int LR) { return pick_instances<4>(S, stride, P, LR); }

}  // namespace kern
}  // namespace spconv
