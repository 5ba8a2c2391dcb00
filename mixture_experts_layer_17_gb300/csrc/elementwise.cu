// Memory-bound kernels of the MoE layer: expert counts and offsets (scan),
// the deterministic expert-major permutation, the token -> row gathers
// (dispatch of x and dY), the k-way combine, the router softmax/top-k
// backward, the un-permute with the router's input gradient, and two small
// transposes.  Every index result is deterministic.
#include <algorithm>

#include "kernels.h"

namespace moe {

namespace {

// ---------------------------------------------------------------- transpose

// out[c, r] = in[r, c] for a bf16 matrix [rows, cols]
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                      int rows, int cols) {
  grid_dependency_wait();
  __shared__ uint16_t tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = in[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[static_cast<int64_t>(c) * rows + r] = tile[threadIdx.x][i];
  }
}

// ---------------------------------------------------------------- F3/F4: scan

// One block of 256 threads (thread = expert).  From the per-tile histograms
// hist[tiles, E] it writes counts[E], offsets[E+1] (exclusive prefix sum),
// poff[E+1] (the same over counts rounded up to 64: the internal permuted
// layout gives every expert a 64-row aligned segment whose tail rows are
// zero), block_base[tiles, E] (first unpadded row of each tile's tokens inside
// each expert's segment), mtile_off[E+1] / mtile2_off[E+1] (prefixes of
// ceil(count / 128) and ceil(count / 256): the grouped-GEMM m-tiles of one CTA
// and of a CTA pair) and group_order[E] (experts by descending count, ties by
// id).
__global__ void scan_kernel(const int* __restrict__ hist, int ntiles, int E,
                            int* __restrict__ counts, int* __restrict__ offsets,
                            int* __restrict__ poff, int* __restrict__ block_base,
                            int* __restrict__ mtile_off, int* __restrict__ mtile2_off,
                            int* __restrict__ group_order) {
  grid_dependency_wait();
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  __shared__ int s_poff[257];
  __shared__ int s_mt[257];
  __shared__ int s_mt2[257];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    for (int b = 0; b < ntiles; ++b) {
      const int h = hist[static_cast<int64_t>(b) * E + e];
      block_base[static_cast<int64_t>(b) * E + e] = run;
      run += h;
    }
  }
  s_cnt[e] = (e < E) ? run : 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0, acc_p = 0, acc_mt = 0, acc_mt2 = 0;
    for (int i = 0; i < E; ++i) {
      s_off[i] = acc;
      s_poff[i] = acc_p;
      s_mt[i] = acc_mt;
      s_mt2[i] = acc_mt2;
      acc += s_cnt[i];
      acc_p += (s_cnt[i] + 63) / 64 * 64;
      acc_mt += (s_cnt[i] + 127) / 128;
      acc_mt2 += (s_cnt[i] + 255) / 256;
    }
    s_off[E] = acc;
    s_poff[E] = acc_p;
    s_mt[E] = acc_mt;
    s_mt2[E] = acc_mt2;
  }
  __syncthreads();
  if (e < E) {
    counts[e] = run;
    offsets[e] = s_off[e];
    poff[e] = s_poff[e];
    mtile_off[e] = s_mt[e];
    mtile2_off[e] = s_mt2[e];
    for (int b = 0; b < ntiles; ++b) block_base[static_cast<int64_t>(b) * E + e] += s_off[e];
    int rank = 0;
    for (int i = 0; i < E; ++i) rank += (s_cnt[i] > run) || (s_cnt[i] == run && i < e);
    group_order[rank] = e;
  }
  if (e == 0) {
    offsets[E] = s_off[E];
    poff[E] = s_poff[E];
    mtile_off[E] = s_mt[E];
    mtile2_off[E] = s_mt2[E];
  }
}

// ---------------------------------------------------------------- F5: permutation

// Block = the 128 tokens of one router tile.  A (token, slot) pair routed to
// expert e goes to row block_base[tile, e] + (number of earlier tokens of the
// tile routed to e); per-warp lane masks give that count without atomics on
// global memory, so rows are expert-major with ascending token inside an
// expert.  The same row shifted to the expert's padded segment (slot_pad) is
// the row the kernels use internally.
// An expert id outside [0, E) (which the router never writes) is recorded in
// the status word and its (token, slot) skipped rather than used as an index.
__global__ void permute_kernel(const int* __restrict__ idx, const float* __restrict__ w,
                               const int* __restrict__ block_base,
                               const int* __restrict__ offsets, const int* __restrict__ poff,
                               int64_t T, int k, int E, int* __restrict__ perm_token,
                               int* __restrict__ slot_row, int* __restrict__ slot_pad,
                               int* __restrict__ row_slot, float* __restrict__ w_row,
                               DeviceStatus* st) {
  grid_dependency_wait();
  __shared__ unsigned mask[4][256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 4 * 256; i += blockDim.x) (&mask[0][0])[i] = 0u;
  __syncthreads();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 128 + tid;
  const bool valid = t < T;
  if (valid) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      if (in_range(e, E))
        atomicOr(&mask[warp][e], 1u << lane);
      else
        record_bad_index(st, kCheckPermuteExpert, e);
    }
  }
  __syncthreads();
  if (!valid) return;
  const unsigned lt = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = idx[t * k + j];
    if (!in_range(e, E)) continue;
    int before = __popc(mask[warp][e] & lt);
    for (int q = 0; q < warp; ++q) before += __popc(mask[q][e]);
    const int r = block_base[static_cast<int64_t>(blockIdx.x) * E + e] + before;
    const int pr = r - offsets[e] + poff[e];     // row of the padded internal layout
    perm_token[r] = static_cast<int>(t);
    slot_row[t * k + j] = r;
    slot_pad[t * k + j] = pr;
    row_slot[pr] = static_cast<int>(t * k + j);
    w_row[pr] = w[t * k + j];
  }
}

// ---------------------------------------------------------------- F6/B1: dispatch

// dst[slot_row[t, j]] = src[t] for every slot j: one warp per token reads the
// token's row once (16-byte vectors) and writes its k copies.  The E blocks
// after the token blocks zero the tail rows [poff[e] + counts[e], poff[e+1])
// of each expert's padded segment (one block per expert); no token row lies
// there.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ src, const int* __restrict__ slot_row,
                                   uint16_t* __restrict__ dst, int64_t T, int H, int k,
                                   const int* __restrict__ poff, const int* __restrict__ counts,
                                   unsigned token_blocks, int64_t Pa, DeviceStatus* st) {
  grid_dependency_wait();
  if (blockIdx.x >= token_blocks) {
    const int e = static_cast<int>(blockIdx.x - token_blocks);
    const int64_t r0 = static_cast<int64_t>(__ldg(poff + e)) + __ldg(counts + e);
    const int64_t r1 = __ldg(poff + e + 1);
    const int cpr = H >> 3;
    for (int64_t i = threadIdx.x; i < (r1 - r0) * cpr; i += blockDim.x) {
      const int64_t row = r0 + i / cpr;
      const int c = static_cast<int>(i % cpr) * 8;
      st_global_v4(dst + row * H + c, 0u, 0u, 0u, 0u);
    }
    return;
  }
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  int64_t rows[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    rows[j] = -1;   // no copy
    if (j < k) {
      const int r = slot_row[t * k + j];
      rows[j] = static_cast<int64_t>(r) * H;
      MOE_CHECK_INDEX(st, kCheckGatherRow, r, Pa, rows[j] = -1);
    }
  }
  const uint16_t* s = src + t * H;
  const int nchunks = H >> 3;
#pragma unroll 4
  for (int c = lane; c < nchunks; c += 32) {
    const uint4 v = ld_global_nc_v4(s + c * 8);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < k && rows[j] >= 0) st_global_v4(dst + rows[j] + c * 8, v.x, v.y, v.z, v.w);
  }
}

MOE_DEV void add_bf16x8(const uint4& v, float (&acc)[8], float scale = 1.0f) {
  float a, b;
  unpack_bf16x2(v.x, a, b); acc[0] = fmaf(scale, a, acc[0]); acc[1] = fmaf(scale, b, acc[1]);
  unpack_bf16x2(v.y, a, b); acc[2] = fmaf(scale, a, acc[2]); acc[3] = fmaf(scale, b, acc[3]);
  unpack_bf16x2(v.z, a, b); acc[4] = fmaf(scale, a, acc[4]); acc[5] = fmaf(scale, b, acc[5]);
  unpack_bf16x2(v.w, a, b); acc[6] = fmaf(scale, a, acc[6]); acc[7] = fmaf(scale, b, acc[7]);
}

// ---------------------------------------------------------------- F10: combine

// y[t] = sum_j scratch[t*k + j]; scratch rows already carry the router weight.
__global__ void combine_kernel(const uint16_t* __restrict__ scratch, uint16_t* __restrict__ y,
                               int64_t T, int H, int k) {
  grid_dependency_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int cpr = H >> 3;
  if (i >= T * cpr) return;
  const int64_t t = i / cpr;
  const int c = static_cast<int>(i - t * cpr) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* base = scratch + t * k * H + c;
  for (int j = 0; j < k; ++j) add_bf16x8(ld_global_nc_v4(base + static_cast<int64_t>(j) * H), acc);
  st_global_v4(y + t * H + c, pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

// ---------------------------------------------------------------- B9: router backward

// dw[t, j] = sum of the down-dgrad epilogue partials of row slot_row[t, j];
// dl[t, j] = w_j (dw_j - sum_i w_i dw_i) (gradient of the renormalised softmax
// at the selected logits); dlT[e, t] = dl for the dense router weight GEMM.
__global__ void router_bwd_kernel(const float* __restrict__ dw_part, int nparts,
                                  const int* __restrict__ slot_row, const float* __restrict__ w,
                                  const int* __restrict__ idx, int64_t T, int k, int E, int64_t Pa,
                                  float* __restrict__ dl, uint16_t* __restrict__ dlT, int64_t T_pad,
                                  DeviceStatus* st) {
  grid_dependency_wait();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float dwv[16], wv[16];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    dwv[j] = 0.f;
    wv[j] = 0.f;
    if (j < k) {
      const int64_t r = slot_row[t * k + j];
      float d = 0.f;
      bool ok = true;
      MOE_CHECK_INDEX(st, kCheckRouterRow, r, Pa, ok = false);
      if (ok)
        for (int n = 0; n < nparts; ++n) d += dw_part[r * nparts + n];
      dwv[j] = d;
      wv[j] = w[t * k + j];
      s = fmaf(wv[j], d, s);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < k) {
      const float g = wv[j] * (dwv[j] - s);
      dl[t * k + j] = g;
      __nv_bfloat16 b = __float2bfloat16_rn(g);
      const int e = idx[t * k + j];
      MOE_CHECK_INDEX(st, kCheckUnpermuteExpert, e, E, continue);
      dlT[static_cast<int64_t>(e) * T_pad + t] = *reinterpret_cast<uint16_t*>(&b);
    }
  }
}

// ---------------------------------------------------------------- B7: un-permute

// dx[t] = sum_j scratch[t*k + j] + sum_j dl[t, j] * W_r^T[idx[t, j]]
// (the expert input gradients plus the router's input gradient dl · W_r^T,
// whose only non-zero terms are the k selected experts).
// A CTA owns a CW-column slice of dx and first copies that slice of W_r^T for
// every expert (E x CW bf16, at most 64 KB) into shared memory, so the k
// router terms of a chunk come from shared memory instead of L2.  Each warp
// walks tokens, CW/8 lanes per token and 16 bytes per lane: all k slot loads
// are issued before the sums (the first token's before the copy), and the
// sums keep the order of the plain definition (slot j's expert gradient,
// then its router term).
template <int CW, int KMAX>
__global__ void __launch_bounds__(256) unpermute_kernel(
    const uint16_t* __restrict__ scratch, const float* __restrict__ dl,
    const int* __restrict__ idx, const uint16_t* __restrict__ WrT, uint16_t* __restrict__ dx,
    int64_t T, int H, int k, int E, DeviceStatus* st) {
  grid_dependency_wait();
  extern __shared__ __align__(16) uint16_t wr_s[];   // [E][CW]
  constexpr int kChunks = CW / 8;                    // 16-byte chunks per row = lanes per token
  constexpr int kTokPerWarp = 32 / kChunks;
  const int c0 = blockIdx.x * CW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cl = (lane % kChunks) * 8;
  const int64_t step = static_cast<int64_t>(gridDim.y) * (blockDim.x >> 5) * kTokPerWarp;
  const int64_t t0 = (static_cast<int64_t>(blockIdx.y) * (blockDim.x >> 5) + warp) * kTokPerWarp +
                     lane / kChunks;
  // the first token's slot loads are in flight while the slice of W_r^T is copied
  uint4 v[KMAX];
  if (t0 < T) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) v[j] = ld_global_nc_v4(scratch + (t0 * k + j) * H + c0 + cl);
  }
  for (int i = threadIdx.x; i < E * kChunks; i += blockDim.x) {
    const int e = i / kChunks, c = (i % kChunks) * 8;
    *reinterpret_cast<uint4*>(wr_s + e * CW + c) =
        ld_global_nc_v4(WrT + static_cast<int64_t>(e) * H + c0 + c);
  }
  __syncthreads();
  for (int64_t t = t0; t < T; t += step) {
    if (t != t0) {
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) v[j] = ld_global_nc_v4(scratch + (t * k + j) * H + c0 + cl);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        add_bf16x8(v[j], acc);
        const int e = __ldg(idx + t * k + j);
        MOE_CHECK_INDEX(st, kCheckUnpermuteExpert, e, E, continue);
        add_bf16x8(*reinterpret_cast<const uint4*>(wr_s + e * CW + cl), acc, __ldg(dl + t * k + j));
      }
    }
    st_global_v4(dx + t * H + c0 + cl, pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                 pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// ---------------------------------------------------------------- B10: dW_r

// dW_r[h, e] = sum over splits of part[s, e, h] (fp32), written as bf16 [H, E].
// dW_r[h, e] = sum over splits of part[split, e, h]: bf16 output, or (kAccum)
// added into an fp32 [H, E] buffer
template <bool kAccum>
__global__ void wr_reduce_kernel(const float* __restrict__ part, int S, int E, int H,
                                 void* __restrict__ out) {
  grid_dependency_wait();
  __shared__ float tile[32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int e = e0 + i, h = h0 + threadIdx.x;
    float s = 0.f;
    if (e < E && h < H)
      for (int sp = 0; sp < S; ++sp) s += part[(static_cast<int64_t>(sp) * E + e) * H + h];
    tile[i][threadIdx.x] = s;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int h = h0 + i, e = e0 + threadIdx.x;
    if (h < H && e < E) {
      const int64_t o = static_cast<int64_t>(h) * E + e;
      if (kAccum) {
        static_cast<float*>(out)[o] += tile[threadIdx.x][i];
      } else {
        __nv_bfloat16 b = __float2bfloat16_rn(tile[threadIdx.x][i]);
        static_cast<uint16_t*>(out)[o] = *reinterpret_cast<uint16_t*>(&b);
      }
    }
  }
}

inline unsigned blocks_for(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

cudaError_t launch_transpose_bf16(const uint16_t* in, uint16_t* out, int rows, int cols,
                                  cudaStream_t s) {
  dim3 grid(blocks_for(cols, 32), blocks_for(rows, 32));
  return launch_pdl(transpose_bf16_kernel, grid, dim3(32, 8), 0, s, in, out, rows, cols);
}

cudaError_t launch_scan(const int* hist, int ntiles, int E, int* counts, int* offsets,
                        int* poff, int* block_base, int* mtile_off, int* mtile2_off,
                        int* group_order, cudaStream_t s) {
  return launch_pdl(scan_kernel, dim3(1), dim3(256), 0, s, hist, ntiles, E, counts, offsets, poff,
                    block_base, mtile_off, mtile2_off, group_order);
}

cudaError_t launch_permute(const int* idx, const float* w, const int* block_base,
                           const int* offsets, const int* poff, int64_t T, int k, int E,
                           int* perm_token, int* slot_row, int* slot_pad, int* row_slot,
                           float* w_row, DeviceStatus* st, cudaStream_t s) {
  return launch_pdl(permute_kernel, dim3(blocks_for(T, 128)), dim3(128), 0, s, idx, w, block_base,
                    offsets, poff, T, k, E, perm_token, slot_row, slot_pad, row_slot, w_row, st);
}

cudaError_t launch_gather_rows(const uint16_t* src, const int* slot_row, uint16_t* dst,
                               int64_t T, int H, int k, const int* poff, const int* counts, int E,
                               int64_t Pa, DeviceStatus* st, cudaStream_t s) {
  const unsigned token_blocks = blocks_for(T, 8);
  if (token_blocks + E == 0) return cudaSuccess;
  return launch_pdl(gather_rows_kernel, dim3(token_blocks + static_cast<unsigned>(E)), dim3(256), 0,
                    s, src, slot_row, dst, T, H, k, poff, counts, token_blocks, Pa, st);
}

cudaError_t launch_combine(const uint16_t* scratch, uint16_t* y, int64_t T, int H, int k,
                           cudaStream_t s) {
  return launch_pdl(combine_kernel, dim3(blocks_for(T * (H / 8), 256)), dim3(256), 0, s, scratch, y,
                    T, H, k);
}

cudaError_t launch_router_bwd(const float* dw_part, int nparts, const int* slot_row,
                              const float* w, const int* idx, int64_t T, int k, int E, int64_t Pa,
                              float* dl, uint16_t* dlT, int64_t T_pad, DeviceStatus* st,
                              cudaStream_t s) {
  return launch_pdl(router_bwd_kernel, dim3(blocks_for(T, 128)), dim3(128), 0, s, dw_part, nparts,
                    slot_row, w, idx, T, k, E, Pa, dl, dlT, T_pad, st);
}

namespace {

// grid: H / CW column slices x token groups, one wave of resident CTAs (as
// many per SM as the E x CW slice of W_r^T in shared memory leaves room for)
template <int CW, int KMAX>
cudaError_t launch_unpermute_cw(const uint16_t* scratch, const float* dl, const int* idx,
                                const uint16_t* WrT, uint16_t* dx, int64_t T, int H, int k, int E,
                                int sms, DeviceStatus* st, cudaStream_t s) {
  constexpr int kSmemMax = 65536;
  static unsigned long long configured = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(unpermute_kernel<CW, KMAX>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  const size_t smem = static_cast<size_t>(E) * CW * 2;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, unpermute_kernel<CW, KMAX>, 256, smem);
  if (e != cudaSuccess) return e;
  const int slices = H / CW;
  const int64_t tok_per_cta = 8 * (32 / (CW / 8));
  const int64_t want = static_cast<int64_t>(std::max(per_sm, 1)) * (sms > 0 ? sms : 1) / slices;
  const int64_t groups = std::max<int64_t>(1, std::min<int64_t>(want, (T + tok_per_cta - 1) / tok_per_cta));
  dim3 grid(static_cast<unsigned>(slices), static_cast<unsigned>(groups));
  return launch_pdl(unpermute_kernel<CW, KMAX>, grid, dim3(256), smem, s, scratch, dl, idx, WrT,
                    dx, T, H, k, E, st);
}

}  // namespace

cudaError_t launch_unpermute(const uint16_t* scratch, const float* dl, const int* idx,
                             const uint16_t* WrT, uint16_t* dx, int64_t T, int H, int k, int E,
                             int sms, DeviceStatus* st, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // 128-column slices: E <= 256 gives at most 64 KB of W_r^T per CTA, and CW
  // divides H.  Each warp then covers two tokens, twice the loads in flight
  // per warp of 256-column slices: 0.218 -> 0.195-0.199 ms at the 235B shape
  // (0.82 -> 0.90-0.92 of the HBM copy rate), 0.039 -> 0.034 ms at 30B.
  return k <= 8 ? launch_unpermute_cw<128, 8>(scratch, dl, idx, WrT, dx, T, H, k, E, sms, st, s)
                : launch_unpermute_cw<128, 16>(scratch, dl, idx, WrT, dx, T, H, k, E, sms, st, s);
}

cudaError_t launch_wr_reduce(const float* part, int S, int E, int H, void* dWr, bool accum_f32,
                             cudaStream_t s) {
  dim3 grid(blocks_for(H, 32), blocks_for(E, 32));
  if (accum_f32)
    return launch_pdl(wr_reduce_kernel<true>, grid, dim3(32, 8), 0, s, part, S, E, H, dWr);
  else
    return launch_pdl(wr_reduce_kernel<false>, grid, dim3(32, 8), 0, s, part, S, E, H, dWr);
}

}  // namespace moe
