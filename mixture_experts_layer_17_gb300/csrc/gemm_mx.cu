// MXFP8 GEMM instantiations (block-scaled tcgen05 MMA, E4M3 operands).
#include "kernels.h"
#include "problems_mx.cuh"

namespace moe {

cudaError_t launch_gate_up_fwd_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpFwdMXProblem>(a, grid, s);
}
cudaError_t launch_down_fwd_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownFwdMXProblem>(a, grid, s);
}
cudaError_t launch_down_dgrad_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownDgradMXProblem<128, true>>(a, grid, s);
}
cudaError_t launch_gate_up_dgrad_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpDgradMXProblem>(a, grid, s);
}
cudaError_t launch_down_wgrad_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradMXProblem<false>>(a, grid, s);
}
cudaError_t launch_gate_up_wgrad_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<WgradMXProblem<true>>(a, grid, s);
}
cudaError_t launch_dense_mx(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DenseMXProblem>(a, grid, s);
}

}  // namespace moe
