// MXFP8 (OCP Microscaling v1.0) quantisers: E4M3 elements with one E8M0
// power-of-two scale per 32 consecutive elements along a GEMM's reduction
// dimension.  Scale = 2^(floor(log2 amax) - 8), elements rounded to nearest
// even and saturated to +-448; an all-zero block gets scale 2^-127.
//
// Scale factors are written straight into the layout the block-scaled
// tcgen05 MMA reads: 512-byte atoms covering 128 MN-rows x 4 K-blocks, row r
// and K-block kb at byte 16*(r%32) + 4*(r/32) + kb.
#include "kernels.h"

namespace moe {

namespace {

// --------------------------------------------------------------------------
// Along the contiguous dimension (K-major operand [R, C], K = C).
//   kRowsDense:    atom group of row = row / 128, r = row % 128 (weights).
//   kRowsPermuted: rows of the padded expert-major layout (offsets = padded
//                  segment starts); the atom group is the row's grouped-GEMM
//                  m-tile, mtile_off[e] + (row - offsets[e]) / 128, and r its
//                  row inside that tile.
// Atom index = group * (C / 128) + k / 128.  One warp per row.
// --------------------------------------------------------------------------
enum RowMode { kRowsDense = 0, kRowsPermuted = 1 };

template <int MODE>
__global__ void quant_rows_kernel(const uint16_t* __restrict__ src, int64_t R, int C,
                                  uint8_t* __restrict__ dst, uint8_t* __restrict__ sf,
                                  const int* __restrict__ offsets,
                                  const int* __restrict__ mtile_off, int E) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= R) return;
  const int lane = threadIdx.x & 31;
  int64_t group;
  int r;
  if (MODE == kRowsDense) {
    group = row >> 7;
    r = static_cast<int>(row & 127);
  } else {
    if (row >= __ldg(offsets + E)) return;   // rows past the last padded segment
    int lo = 0, hi = E - 1;     // largest e with offsets[e] <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(offsets + mid) <= row) lo = mid; else hi = mid - 1;
    }
    const int64_t local = row - __ldg(offsets + lo);
    group = __ldg(mtile_off + lo) + (local >> 7);
    r = static_cast<int>(local & 127);
  }
  const int KT = C >> 7;
  const uint16_t* s = src + row * C;
  uint8_t* d = dst + row * C;
  for (int b = lane; b < (C >> 5); b += 32) {
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = ld_global_nc_v4(s + b * 32 + q * 8);
      unpack_bf16x2(u.x, v[8 * q + 0], v[8 * q + 1]);
      unpack_bf16x2(u.y, v[8 * q + 2], v[8 * q + 3]);
      unpack_bf16x2(u.z, v[8 * q + 4], v[8 * q + 5]);
      unpack_bf16x2(u.w, v[8 * q + 6], v[8 * q + 7]);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int X = mx_exponent(amax);
    const float inv = ldexpf(1.0f, -X);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = to_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
    st_global_v4(d + b * 32, w[0], w[1], w[2], w[3]);
    st_global_v4(d + b * 32 + 16, w[4], w[5], w[6], w[7]);
    sf[(group * KT + (b >> 2)) * 512 + sf_atom_offset(r, b & 3)] = static_cast<uint8_t>(X + 127);
  }
}

// --------------------------------------------------------------------------
// Along rows (MN-major operand, K = rows, MN = columns).  A CTA quantises one
// 128-row K-tile x 128 columns; the K-tiles are:
//   kColsWeights:  E experts x (R / 128) tiles of a [E, R, C] tensor.
//   kColsGateUp:   as kColsWeights over R = H rows, but the output [E, H, 2F]
//                  interleaves W_gate and W_up in 64-column halves of every
//                  128-column tile (gate columns 64j.., then up columns 64j..).
//   kColsTokens:   the expert-major token rows (segments starting at the
//                  padded offsets, counts[e] valid rows), each expert's
//                  segment padded to whole 128-row tiles (tile g of expert e
//                  is output rows 128*(mtile_off[e] + g) ..); rows past the
//                  segment are zero.
// Atom index = (k-tile) * (C_out / 128) + column tile for the token layout,
// (expert * (C_out / 128) + column tile) * (R / 128) + k-tile for weights.
// --------------------------------------------------------------------------
enum ColMode { kColsWeights = 0, kColsGateUp = 1, kColsTokens = 2 };

template <int MODE>
__global__ void __launch_bounds__(64) quant_cols_kernel(const uint16_t* __restrict__ src0,
                                  const uint16_t* __restrict__ src1, int R, int C_in,
                                  uint8_t* __restrict__ dst, uint8_t* __restrict__ sf,
                                  const int* __restrict__ offsets,
                                  const int* __restrict__ counts,
                                  const int* __restrict__ mtile_off, int E) {
  // 64 threads: thread = (32-row block rb in 0..3, group of 8 columns cg in 0..15);
  // each reads 32 rows x 16 bytes, keeps 8 running maxima, writes 32 x 8 bytes.
  const int kg = blockIdx.x;           // K-tile (global)
  const int ct = blockIdx.y;           // 128-column tile of the output
  const int cg = threadIdx.x & 15;
  const int rb = threadIdx.x >> 4;
  const int C_out = (MODE == kColsGateUp) ? 2 * C_in : C_in;
  int64_t src_row0, dst_row0;
  int valid;                           // valid rows of this K-tile
  int64_t atom;
  const uint16_t* src = src0;
  int src_col;
  if (MODE == kColsTokens) {
    if (kg >= __ldg(mtile_off + E)) return;   // the grid is sized for the worst case
    int lo = 0, hi = E - 1;            // largest e with mtile_off[e] <= kg
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(mtile_off + mid) <= kg) lo = mid; else hi = mid - 1;
    }
    const int g = kg - __ldg(mtile_off + lo);
    src_row0 = static_cast<int64_t>(__ldg(offsets + lo)) + 128 * g;
    valid = min(128, __ldg(counts + lo) - 128 * g);
    dst_row0 = 128ll * kg;
    atom = static_cast<int64_t>(kg) * (C_out >> 7) + ct;
    src_col = ct * 128 + cg * 8;
  } else {
    const int kt_per = R >> 7;
    const int e = kg / kt_per;
    const int kt = kg - e * kt_per;
    src_row0 = static_cast<int64_t>(e) * R + 128 * kt;
    dst_row0 = src_row0;
    valid = 128;
    atom = (static_cast<int64_t>(e) * (C_out >> 7) + ct) * kt_per + kt;
    if (MODE == kColsGateUp) {
      src = (cg < 8) ? src0 : src1;    // output columns 0..63 gate, 64..127 up
      src_col = ct * 64 + (cg & 7) * 8;
    } else {
      src_col = ct * 128 + cg * 8;
    }
  }
  const int out_col = ct * 128 + cg * 8;
  // pass 1: column maxima of the 32-row block; pass 2 re-reads the same
  // 512 bytes per thread (cache-resident) and converts
  float amax[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* base = src + src_row0 * C_in + src_col;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    const int rr = rb * 32 + i;
    if (rr < valid) {
      const uint4 u = ld_global_v4(base + static_cast<int64_t>(rr) * C_in);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float lo, hi;
        unpack_bf16x2(w[q], lo, hi);
        amax[2 * q] = fmaxf(amax[2 * q], fabsf(lo));
        amax[2 * q + 1] = fmaxf(amax[2 * q + 1], fabsf(hi));
      }
    }
  }
  float inv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int X = mx_exponent(amax[j]);
    inv[j] = ldexpf(1.0f, -X);
    sf[atom * 512 + sf_atom_offset(cg * 8 + j, rb)] = static_cast<uint8_t>(X + 127);
  }
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    const int rr = rb * 32 + i;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (rr < valid) u = ld_global_v4(base + static_cast<int64_t>(rr) * C_in);
    float v[8];
    unpack_bf16x2(u.x, v[0], v[1]);
    unpack_bf16x2(u.y, v[2], v[3]);
    unpack_bf16x2(u.z, v[4], v[5]);
    unpack_bf16x2(u.w, v[6], v[7]);
    const uint32_t lo = to_e4m3x4(v[0] * inv[0], v[1] * inv[1], v[2] * inv[2], v[3] * inv[3], 1.0f);
    const uint32_t hi = to_e4m3x4(v[4] * inv[4], v[5] * inv[5], v[6] * inv[6], v[7] * inv[7], 1.0f);
    *reinterpret_cast<uint2*>(dst + (dst_row0 + rb * 32 + i) * C_out + out_col) = make_uint2(lo, hi);
  }
}

}  // namespace

cudaError_t launch_quant_rows_dense(const uint16_t* src, int64_t R, int C, uint8_t* dst,
                                    uint8_t* sf, cudaStream_t s) {
  quant_rows_kernel<kRowsDense><<<static_cast<unsigned>((R + 7) / 8), 256, 0, s>>>(
      src, R, C, dst, sf, nullptr, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_permuted(const uint16_t* src, int64_t P, int C, uint8_t* dst,
                                       uint8_t* sf, const int* offsets, const int* mtile_off,
                                       int E, cudaStream_t s) {
  quant_rows_kernel<kRowsPermuted><<<static_cast<unsigned>((P + 7) / 8), 256, 0, s>>>(
      src, P, C, dst, sf, offsets, mtile_off, E);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols_weights(const uint16_t* src, int E, int R, int C, uint8_t* dst,
                                      uint8_t* sf, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(E * (R / 128)), static_cast<unsigned>(C / 128));
  quant_cols_kernel<kColsWeights><<<grid, 64, 0, s>>>(src, nullptr, R, C, dst, sf, nullptr,
                                                      nullptr, nullptr, E);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols_gate_up(const uint16_t* W_gate, const uint16_t* W_up, int E, int H,
                                      int F, uint8_t* dst, uint8_t* sf, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(E * (H / 128)), static_cast<unsigned>(2 * F / 128));
  quant_cols_kernel<kColsGateUp><<<grid, 64, 0, s>>>(W_gate, W_up, H, F, dst, sf, nullptr,
                                                     nullptr, nullptr, E);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols_tokens(const uint16_t* src, int64_t max_ktiles, int C, uint8_t* dst,
                                     uint8_t* sf, const int* poff, const int* counts,
                                     const int* mtile_off, int E, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(max_ktiles), static_cast<unsigned>(C / 128));
  quant_cols_kernel<kColsTokens><<<grid, 64, 0, s>>>(src, nullptr, 0, C, dst, sf, poff, counts,
                                                     mtile_off, E);
  return cudaGetLastError();
}

}  // namespace moe
