// MXFP8 CTA-pair GEMM instantiations (block-scaled cta_group::2 MMA).
#include "kernels.h"
#include "problems_mx_pair.cuh"

namespace moe {

cudaError_t launch_gate_up_fwd_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpFwdMXPairProblem>(a, grid, s);
}
cudaError_t launch_down_fwd_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownFwdMXPairProblem>(a, grid, s);
}
cudaError_t launch_gate_up_dgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpDgradMXPairProblem>(a, grid, s);
}
cudaError_t launch_down_wgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradMXPairProblem<false>>(a, grid, s);
}
cudaError_t launch_gate_up_wgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradMXPairProblem<true>>(a, grid, s);
}
cudaError_t launch_dense_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DenseMXPairProblem>(a, grid, s);
}
cudaError_t launch_down_dgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownDgradMXPairProblem>(a, grid, s);
}

}  // namespace moe
