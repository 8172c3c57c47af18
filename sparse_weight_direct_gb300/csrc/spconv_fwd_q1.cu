// Kernel instances with 1 output channel(s) per warp (one translation unit per
// count so the instances compile in parallel).
#include "spconv_kernel.cuh"

namespace spconv {
namespace kern {

KernelFn pick_q1(int S, int stride, int P, int LR) { return pick_instances<1>(S, stride, P, LR); }

}  // namespace kern
}  // namespace spconv
