// Expert weight-gradient GEMMs over ragged per-expert token counts, and the
// dense test GEMM.
#include "kernels.h"
#include "problems_bwd.cuh"

namespace moe {

cudaError_t launch_down_wgrad(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownWgradProblem>(a, grid, s);
}

cudaError_t launch_gate_up_wgrad(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpWgradProblem>(a, grid, s);
}

cudaError_t launch_dense(bool a_mn, bool b_mn, const GemmArgs& a, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return launch_gemm<DenseProblem<false, false>>(a, grid, s);
  if (!a_mn && b_mn) return launch_gemm<DenseProblem<false, true>>(a, grid, s);
  if (a_mn && !b_mn) return launch_gemm<DenseProblem<true, false>>(a, grid, s);
  return launch_gemm<DenseProblem<true, true>>(a, grid, s);
}

}  // namespace moe
