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
// Along the contiguous dimension (K-major operand [R, C], K = C; weights).
// One warp per row.  Two scale layouts, each written when its pointer is set:
//   sf:    128-row atoms: atom (row / 128) * (C / 128) + k / 128, atom row
//          row % 128;
//   sf192: 192-row blocks of two atoms (rows 0..127 of the block, then rows
//          128..191 in the first 64 rows of the second; its other 64 rows are
//          never read): atom ((row / 192) * 2 + half) * (C / 128) + k / 128.
// --------------------------------------------------------------------------
__global__ void quant_rows_kernel(const uint16_t* __restrict__ src, int64_t R, int C,
                                  uint8_t* __restrict__ dst, uint8_t* __restrict__ sf,
                                  uint8_t* __restrict__ sf192) {
  grid_dependency_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= R) return;
  const int lane = threadIdx.x & 31;
  const int64_t group = row >> 7;
  const int r = static_cast<int>(row & 127);
  const int64_t b192 = row / 192;
  const int r192 = static_cast<int>(row - 192 * b192);
  const int64_t group192 = 2 * b192 + (r192 >> 7);
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
    const float inv = mx_inv_scale(X);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = to_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
    st_global_v4(d + b * 32, w[0], w[1], w[2], w[3]);
    st_global_v4(d + b * 32 + 16, w[4], w[5], w[6], w[7]);
    if (sf != nullptr)
      sf[(group * KT + (b >> 2)) * 512 + sf_atom_offset(r, b & 3)] = static_cast<uint8_t>(X + 127);
    if (sf192 != nullptr)
      sf192[(group192 * KT + (b >> 2)) * 512 + sf_atom_offset(r192 & 127, b & 3)] =
          static_cast<uint8_t>(X + 127);
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

constexpr int kColThreads = 256;

// Expert of k-tile kg: the largest e with mtile_off[e] <= kg, or -1 for a
// k-tile past mtile_off[E] (the grids are sized for the worst case).  The
// E + 1 prefix entries stay in L1 after the first block on an SM.
__device__ __forceinline__ int ktile_expert(const int* __restrict__ mtile_off, int E, int kg) {
  if (kg >= __ldg(mtile_off + E)) return -1;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(mtile_off + mid) <= kg) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Shared-memory tiles of 128 rows x 128 bf16 columns hold their 16-byte
// chunks swizzled: logical chunk c of row r sits at c ^ ((c >> 3) << 1) ^ (r & 1).
// Row-wise 16-byte stores, column-pair reads and the (row, 32-column block)
// reads of the quantiser along C are all free of bank conflicts that way.
__device__ __forceinline__ int tile_chunk(int row, int c) { return c ^ ((c >> 3) << 1) ^ (row & 1); }

// The 128 x 128 bf16 tile quantised along its rows' direction (blocks of 32
// rows per column) into qtile, scales into the 512-byte atom sfa: 256
// threads, thread t takes the column pair (2 (t % 64), 2 (t % 64) + 1) of
// 32-row block t / 64.  |max| of each column by a bf16x2 max (exact); the
// E4M3 values are written as byte pairs of one row.
__device__ __forceinline__ void quant_tile_cols(const uint16_t (&tile)[128][128],
                                                uint8_t (&qtile)[128][128], uint8_t* sfa) {
  const int cp = threadIdx.x & 63;
  const int kb = threadIdx.x >> 6;
  __nv_bfloat162 amax2 = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int j = 0; j < 32; ++j)
    amax2 = __hmax2(amax2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(
                               &tile[kb * 32 + j][tile_chunk(kb * 32 + j, cp >> 2) * 8 + (2 * cp & 7)])));
  const int X0 = mx_exponent(__low2float(amax2));
  const int X1 = mx_exponent(__high2float(amax2));
  const float inv0 = mx_inv_scale(X0), inv1 = mx_inv_scale(X1);
  sfa[sf_atom_offset(2 * cp, kb)] = static_cast<uint8_t>(X0 + 127);
  sfa[sf_atom_offset(2 * cp + 1, kb)] = static_cast<uint8_t>(X1 + 127);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(
        &tile[kb * 32 + j][tile_chunk(kb * 32 + j, cp >> 2) * 8 + (2 * cp & 7)]);
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(&qtile[kb * 32 + j][2 * cp]) =
        __nv_cvt_float2_to_fp8x2(make_float2(lo * inv0, hi * inv1), __NV_SATFINITE, __NV_E4M3);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kColThreads) quant_cols_kernel(
    const uint16_t* __restrict__ src0, const uint16_t* __restrict__ src1, int R, int C_in,
    uint8_t* __restrict__ dst, uint8_t* __restrict__ sf, const int* __restrict__ offsets,
    const int* __restrict__ counts, const int* __restrict__ mtile_off, int E) {
  grid_dependency_wait();
  // One pass: the 128-row x 128-column bf16 tile is read once into shared
  // memory (coalesced 16-byte loads), each thread turns two (column, 32-row
  // block) units into a scale and 32 E4M3 bytes, and the E4M3 tile leaves
  // through shared memory as coalesced 16-byte row stores.
  __shared__ __align__(16) uint16_t tile[128][128];
  __shared__ __align__(16) uint8_t qtile[128][128];
  const int kg = blockIdx.x;           // K-tile (global)
  const int ct = blockIdx.y;           // 128-column tile of the output
  const int tid = threadIdx.x;
  const int C_out = (MODE == kColsGateUp) ? 2 * C_in : C_in;
  int64_t src_row0, dst_row0;
  int valid;                           // valid rows of this K-tile
  int64_t atom;
  if (MODE == kColsTokens) {
    const int lo = ktile_expert(mtile_off, E, kg);
    if (lo < 0) return;
    const int g = kg - __ldg(mtile_off + lo);
    src_row0 = static_cast<int64_t>(__ldg(offsets + lo)) + 128 * g;
    valid = min(128, __ldg(counts + lo) - 128 * g);
    dst_row0 = 128ll * kg;
    atom = static_cast<int64_t>(kg) * (C_out >> 7) + ct;
  } else {
    const int kt_per = R >> 7;
    const int e = kg / kt_per;
    const int kt = kg - e * kt_per;
    src_row0 = static_cast<int64_t>(e) * R + 128 * kt;
    dst_row0 = src_row0;
    valid = 128;
    atom = (static_cast<int64_t>(e) * (C_out >> 7) + ct) * kt_per + kt;
  }
  // load: 16 threads per row, 16 bytes (8 columns) each; rows >= valid are zero
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int chunk = tid + kColThreads * i;   // 0 .. 2047
    const int row = chunk >> 4;
    const int c8 = (chunk & 15) * 8;           // output column of the chunk
    uint4 u = make_uint4(0, 0, 0, 0);
    if (row < valid) {
      const uint16_t* src = src0;
      int col = ct * 128 + c8;
      if (MODE == kColsGateUp) {               // output columns 0..63 gate, 64..127 up
        src = c8 < 64 ? src0 : src1;
        col = ct * 64 + (c8 & 63);
      }
      u = ld_global_nc_v4(src + (src_row0 + row) * C_in + col);
    }
    *reinterpret_cast<uint4*>(&tile[row][tile_chunk(row, c8 >> 3) * 8]) = u;
  }
  __syncthreads();
  // convert: a thread takes the column pair (2 cp, 2 cp + 1) of 32-row block kb
  quant_tile_cols(tile, qtile, sf + atom * 512);
  __syncthreads();
  // store: 8 threads per 128-byte output row
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int chunk = tid + kColThreads * i;   // 0 .. 1023
    const int row = chunk >> 3;
    const int c16 = (chunk & 7) * 16;
    const uint4 q = *reinterpret_cast<const uint4*>(&qtile[row][c16]);
    st_global_v4(dst + (dst_row0 + row) * C_out + ct * 128 + c16, q.x, q.y, q.z, q.w);
  }
}

// Dispatch of an activation [T, C] (x, dY) straight into both MXFP8 copies the
// expert GEMMs read, one 128-row k-tile of the token layout x 128 columns per
// CTA.  The k-tile's rows are the expert's tokens (perm_token of the unpadded
// permuted layout), gathered into shared memory; rows past the expert's count
// are zero.  Then
//   along the tokens (unless dst_t is null): the E4M3 tile at token-layout
//     rows 128*kg + i with its scale atom kg * (C/128) + ct (as
//     quant_cols_kernel<kColsTokens>);
//   along C (unless dst_r is null): E4M3 rows at the padded rows poff[e] + 128*g + i that lie inside
//     the expert's padded segment, scale atom (mtile_off[e] + g) * (C/128) + ct
//     (the layout the grouped-M GEMMs read along K).
__global__ void __launch_bounds__(kColThreads) dispatch_quant_kernel(
    const uint16_t* __restrict__ src, const int* __restrict__ perm_token,
    const int* __restrict__ offsets, const int* __restrict__ poff, const int* __restrict__ counts,
    const int* __restrict__ mtile_off, int E, int C, uint8_t* __restrict__ dst_t,
    uint8_t* __restrict__ sf_t, uint8_t* __restrict__ dst_r, uint8_t* __restrict__ sf_r) {
  grid_dependency_wait();
  __shared__ __align__(16) uint16_t tile[128][128];
  __shared__ __align__(16) uint8_t qtile[128][128];
  const int kg = blockIdx.x;
  const int ct = blockIdx.y;
  const int tid = threadIdx.x;
  const int e = ktile_expert(mtile_off, E, kg);
  if (e < 0) return;
  const int g = kg - __ldg(mtile_off + e);
  const int local0 = 128 * g;
  const int valid = min(128, __ldg(counts + e) - local0);
  const int seg = min(128, __ldg(poff + e + 1) - __ldg(poff + e) - local0);
  const int* toks = perm_token + __ldg(offsets + e) + local0;
  // gather: 16 threads per row, 16 bytes each
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int chunk = tid + kColThreads * i;
    const int row = chunk >> 4;
    const int c8 = (chunk & 15) * 8;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (row < valid) {
      const int64_t tok = __ldg(toks + row);
      u = ld_global_nc_v4(src + tok * C + ct * 128 + c8);
    }
    *reinterpret_cast<uint4*>(&tile[row][tile_chunk(row, c8 >> 3) * 8]) = u;
  }
  __syncthreads();
  // along the tokens (dst_t may be null: not wanted): a thread takes the
  // column pair (2 cp, 2 cp + 1) of 32-row block kb; |max| of each column by
  // bf16x2 max (exact), E4M3 written as byte pairs of one row
  if (dst_t != nullptr) quant_tile_cols(tile, qtile, sf_t + (static_cast<int64_t>(kg) * (C >> 7) + ct) * 512);
  // along C (unless dst_r is null): a lane takes one 32-column block of a
  // row (no shuffles), four lanes per row, eight rows per warp step
  if (dst_r != nullptr) {
    const int warp = tid >> 5, lane = tid & 31;
    const int blk = lane & 3;
    const int64_t prow0 = static_cast<int64_t>(__ldg(poff + e)) + local0;
    uint8_t* sfr = sf_r + (static_cast<int64_t>(__ldg(mtile_off + e) + g) * (C >> 7) + ct) * 512;
    uint8_t* dr = dst_r + prow0 * C + ct * 128 + blk * 32;
#pragma unroll 1
    for (int row = 8 * warp + (lane >> 2); row < seg; row += kColThreads / 4) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u =
            *reinterpret_cast<const uint4*>(&tile[row][tile_chunk(row, 4 * blk + q) * 8]);
        unpack_bf16x2(u.x, v[8 * q + 0], v[8 * q + 1]);
        unpack_bf16x2(u.y, v[8 * q + 2], v[8 * q + 3]);
        unpack_bf16x2(u.z, v[8 * q + 4], v[8 * q + 5]);
        unpack_bf16x2(u.w, v[8 * q + 6], v[8 * q + 7]);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const int X = mx_exponent(amax);
      const float inv = mx_inv_scale(X);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = to_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
      uint8_t* d = dr + static_cast<int64_t>(row) * C;
      st_global_v4(d, w[0], w[1], w[2], w[3]);
      st_global_v4(d + 16, w[4], w[5], w[6], w[7]);
      sfr[sf_atom_offset(row, blk)] = static_cast<uint8_t>(X + 127);
    }
  }
  __syncthreads();
  if (dst_t == nullptr) return;
  // the along-tokens tile leaves as whole rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int chunk = tid + kColThreads * i;
    const int row = chunk >> 3;
    const int c16 = (chunk & 7) * 16;
    const uint4 q = *reinterpret_cast<const uint4*>(&qtile[row][c16]);
    st_global_v4(dst_t + (128ll * kg + row) * C + ct * 128 + c16, q.x, q.y, q.z, q.w);
  }
}

}  // namespace

cudaError_t launch_quant_rows_dense(const uint16_t* src, int64_t R, int C, uint8_t* dst,
                                    uint8_t* sf, cudaStream_t s, uint8_t* sf192) {
  if (sf192 != nullptr && R % 192 != 0) return cudaErrorInvalidValue;
  return launch_pdl(quant_rows_kernel, dim3(static_cast<unsigned>((R + 7) / 8)), dim3(256), 0, s,
                    src, R, C, dst, sf, sf192);
}

cudaError_t launch_quant_cols_weights(const uint16_t* src, int E, int R, int C, uint8_t* dst,
                                      uint8_t* sf, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(E * (R / 128)), static_cast<unsigned>(C / 128));
  return launch_pdl(quant_cols_kernel<kColsWeights>, grid, dim3(kColThreads), 0, s, src, nullptr, R,
                    C, dst, sf, nullptr, nullptr, nullptr, E);
}

cudaError_t launch_quant_cols_gate_up(const uint16_t* W_gate, const uint16_t* W_up, int E, int H,
                                      int F, uint8_t* dst, uint8_t* sf, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(E * (H / 128)), static_cast<unsigned>(2 * F / 128));
  return launch_pdl(quant_cols_kernel<kColsGateUp>, grid, dim3(kColThreads), 0, s, W_gate, W_up, H,
                    F, dst, sf, nullptr, nullptr, nullptr, E);
}

cudaError_t launch_quant_cols_tokens(const uint16_t* src, int64_t max_ktiles, int C, uint8_t* dst,
                                     uint8_t* sf, const int* poff, const int* counts,
                                     const int* mtile_off, int E, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(max_ktiles), static_cast<unsigned>(C / 128));
  return launch_pdl(quant_cols_kernel<kColsTokens>, grid, dim3(kColThreads), 0, s, src, nullptr, 0,
                    C, dst, sf, poff, counts, mtile_off, E);
}

cudaError_t launch_dispatch_quant(const uint16_t* src, const int* perm_token, const int* offsets,
                                  const int* poff, const int* counts, const int* mtile_off,
                                  int64_t max_ktiles, int E, int C, uint8_t* dst_t, uint8_t* sf_t,
                                  uint8_t* dst_r, uint8_t* sf_r, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(max_ktiles), static_cast<unsigned>(C / 128));
  return launch_pdl(dispatch_quant_kernel, grid, dim3(kColThreads), 0, s, src, perm_token, offsets,
                    poff, counts, mtile_off, E, C, dst_t, sf_t, dst_r, sf_r);
}

}  // namespace moe
