// Backward-pass GEMM instantiations: down dgrad (+ SwiGLU backward and router
// weight gradient), gate/up dgrad (+ scatter) and the router weight gradient.
#include "kernels.h"
#include "problems_bwd.cuh"

namespace moe {

cudaError_t launch_down_dgrad(int bn, const GemmArgs& a, int grid, cudaStream_t s) {
  if (bn == 256) return launch_gemm<DownDgradProblem<256>>(a, grid, s);
  if (bn == 128) return launch_gemm<DownDgradProblem<128>>(a, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gate_up_dgrad(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpDgradProblem>(a, grid, s);
}

cudaError_t launch_router_wgrad(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<RouterWgradProblem>(a, grid, s);
}

}  // namespace moe
