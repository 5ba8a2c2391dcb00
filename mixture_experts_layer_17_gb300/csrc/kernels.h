// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.cuh"

namespace moe {

// tcgen05 GEMMs (gemm_*.cu); `grid` CTAs of kThreads threads, persistent.
cudaError_t launch_router_fwd(int bn, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_fwd(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_fwd(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_dgrad(int bn, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_dgrad(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_wgrad(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_wgrad(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_router_wgrad(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_dense(bool a_mn, bool b_mn, const GemmArgs& a, int grid, cudaStream_t s);

// CTA-pair GEMMs (gemm_pair.cu): grid must be even
cudaError_t launch_gate_up_fwd_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_fwd_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_dgrad_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_dgrad_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_wgrad_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_wgrad_pair(const GemmArgs& a, int grid, cudaStream_t s);

// MXFP8 GEMMs (gemm_mx.cu)
cudaError_t launch_gate_up_fwd_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_fwd_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_dgrad_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_dgrad_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_wgrad_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_wgrad_mx(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_dense_mx(const GemmArgs& a, int grid, cudaStream_t s);
// MXFP8 CTA-pair GEMMs (grid must be even)
cudaError_t launch_gate_up_fwd_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_fwd_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_dgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down_wgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gate_up_wgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_dense_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);
// 256 x 192 tiles, two accumulators per CTA (F a multiple of 192)
cudaError_t launch_down_dgrad_mx_pair(const GemmArgs& a, int grid, cudaStream_t s);

// MXFP8 quantisers (mx_quant.cu): E4M3 data + 512-byte scale atoms.  Rows
// quantiser: sf (128-row atoms) and/or sf192 (192-row blocks of two atoms, R
// a multiple of 192), each written when not null.
cudaError_t launch_quant_rows_dense(const uint16_t* src, int64_t R, int C, uint8_t* dst,
                                    uint8_t* sf, cudaStream_t s, uint8_t* sf192 = nullptr);
cudaError_t launch_quant_cols_weights(const uint16_t* src, int E, int R, int C, uint8_t* dst,
                                      uint8_t* sf, cudaStream_t s);
cudaError_t launch_quant_cols_gate_up(const uint16_t* W_gate, const uint16_t* W_up, int E, int H,
                                      int F, uint8_t* dst, uint8_t* sf, cudaStream_t s);
// Dispatch of an activation [T, C] straight into its two MXFP8 copies: along
// the tokens (token layout, 128-row expert segments) and along C (padded
// permuted rows); no bf16 copy is written.
cudaError_t launch_dispatch_quant(const uint16_t* src, const int* perm_token, const int* offsets,
                                  const int* poff, const int* counts, const int* mtile_off,
                                  int64_t max_ktiles, int E, int C, uint8_t* dst_t, uint8_t* sf_t,
                                  uint8_t* dst_r, uint8_t* sf_r, cudaStream_t s);
cudaError_t launch_quant_cols_tokens(const uint16_t* src, int64_t max_ktiles, int C, uint8_t* dst,
                                     uint8_t* sf, const int* poff, const int* counts,
                                     const int* mtile_off, int E, cudaStream_t s);

// memory-bound kernels (elementwise.cu)
cudaError_t launch_transpose_bf16(const uint16_t* in, uint16_t* out, int rows, int cols,
                                  cudaStream_t s);
cudaError_t launch_scan(const int* hist, int ntiles, int E, int* counts, int* offsets,
                        int* poff, int* block_base, int* mtile_off, int* mtile2_off,
                        int* group_order, cudaStream_t s);
cudaError_t launch_permute(const int* idx, const float* w, const int* block_base,
                           const int* offsets, const int* poff, int64_t T, int k, int E,
                           int* perm_token, int* slot_row, int* slot_pad, int* row_slot,
                           float* w_row, DeviceStatus* st, cudaStream_t s);
// dst[slot_row[t, j]] = src[t] for every slot, and the tail rows of each
// expert's padded segment ([poff[e] + counts[e], poff[e+1])) zeroed
cudaError_t launch_gather_rows(const uint16_t* src, const int* slot_row, uint16_t* dst,
                               int64_t T, int H, int k, const int* poff, const int* counts, int E,
                               int64_t Pa, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* scratch, uint16_t* y, int64_t T, int H, int k,
                           cudaStream_t s);
cudaError_t launch_router_bwd(const float* dw_part, int nparts, const int* slot_row,
                              const float* w, const int* idx, int64_t T, int k, int E, int64_t Pa,
                              float* dl, uint16_t* dlT, int64_t T_pad, DeviceStatus* st,
                              cudaStream_t s);
cudaError_t launch_unpermute(const uint16_t* scratch, const float* dl, const int* idx,
                             const uint16_t* WrT, uint16_t* dx, int64_t T, int H, int k, int E,
                             int sms, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_wr_reduce(const float* part, int S, int E, int H, void* dWr, bool accum_f32,
                             cudaStream_t s);

// Launches `kernel` with programmatic stream serialization (see
// grid_dependency_wait): it may start while the stream's previous kernel
// drains, and waits for it in its first instructions.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Launches gemm_kernel<P>, raising the dynamic shared-memory limit once per
// device; programmatic stream serialization as launch_pdl.
template <class P>
cudaError_t launch_gemm(const GemmArgs& a, int grid, cudaStream_t s) {
  constexpr size_t smem = gemm_smem_bytes<P>();
  static_assert(smem <= 232448, "shared memory per CTA exceeds 227 KB");
  static unsigned long long configured = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  if constexpr (IsPair<P>::value) {
    // clusters of two CTAs (grid is even)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(gemm_threads<P>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, gemm_kernel<P>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  } else {
    return launch_pdl(gemm_kernel<P>, dim3(static_cast<unsigned>(grid)), dim3(gemm_threads<P>()),
                      smem, s, a);
  }
}

}  // namespace moe
