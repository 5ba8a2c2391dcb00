// Forward-pass GEMM instantiations: router (+ top-k), gate/up (+ SwiGLU),
// down (+ weighted scatter).
#include "kernels.h"
#include "problems.cuh"

namespace moe {

cudaError_t launch_router_fwd(int bn, const GemmArgs& a, int grid, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_gemm<RouterProblem<16>>(a, grid, s);
    case 32: return launch_gemm<RouterProblem<32>>(a, grid, s);
    case 64: return launch_gemm<RouterProblem<64>>(a, grid, s);
    case 128: return launch_gemm<RouterProblem<128>>(a, grid, s);
    case 256: return launch_gemm<RouterProblem<256>>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gate_up_fwd(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpFwdProblem>(a, grid, s);
}

cudaError_t launch_down_fwd(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownFwdProblem>(a, grid, s);
}

}  // namespace moe
