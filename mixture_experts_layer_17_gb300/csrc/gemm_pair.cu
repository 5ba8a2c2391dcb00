// CTA-pair (cta_group::2) expert GEMM instantiations.
#include "kernels.h"
#include "problems_pair.cuh"

namespace moe {

cudaError_t launch_gate_up_fwd_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpFwdPairProblem>(a, grid, s);
}
cudaError_t launch_down_fwd_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownFwdPairProblem>(a, grid, s);
}
cudaError_t launch_down_dgrad_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownDgradPairProblem>(a, grid, s);
}
cudaError_t launch_gate_up_dgrad_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpDgradPairProblem>(a, grid, s);
}
cudaError_t launch_down_wgrad_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradPairProblem<DownWgradProblem>>(a, grid, s);
}
cudaError_t launch_gate_up_wgrad_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradPairProblem<GateUpWgradProblem>>(a, grid, s);
}

}  // namespace moe
