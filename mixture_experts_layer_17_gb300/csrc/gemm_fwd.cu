// Forward-pass GEMM instantiations: router (+ top-k), gate/up (+ SwiGLU),
// down (+ weighted scatter).
#include "kernels.h"
#include "problems.cuh"

namespace moe {

template <int kSlots>
cudaError_t launch_router_slots(int bn, const GemmArgs& a, int grid, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_gemm<RouterProblem<16, kSlots>>(a, grid, s);
    case 32: return launch_gemm<RouterProblem<32, kSlots>>(a, grid, s);
    case 64: return launch_gemm<RouterProblem<64, kSlots>>(a, grid, s);
    case 128: return launch_gemm<RouterProblem<128, kSlots>>(a, grid, s);
    case 256: return launch_gemm<RouterProblem<256, kSlots>>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_router_fwd(int bn, const GemmArgs& a, int grid, cudaStream_t s) {
  // the top-k list holds 8 entries when top_k <= 8 (the inner loop of the
  // epilogue runs over all of them for every logit)
  return a.top_k <= 8 ? launch_router_slots<8>(bn, a, grid, s)
                      : launch_router_slots<16>(bn, a, grid, s);
}

cudaError_t launch_gate_up_fwd(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<GateUpFwdProblem>(a, grid, s);
}

cudaError_t launch_down_fwd(const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm<DownFwdProblem>(a, grid, s);
}

}  // namespace moe
