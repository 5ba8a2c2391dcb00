// The GEMMs of the MoE layer as policies of the tcgen05 engine (gemm.cuh).
//
// Notation: T tokens, H hidden, F expert width, E experts, k = top_k,
// P = T * k rows of the expert-major permuted layout.  Operand tiles are
// loaded by TMA with the 128-byte swizzle, either K-major (box 64 x rows) or
// MN-major (chunks of 64 MN-elements x 64 K-rows, 8 KB each).
#pragma once

#include "gemm.cuh"

namespace moe {

// named barrier 1 over the epilogue warps (nthreads: 128 per warpgroup)
template <int kThreads = 128>
MOE_DEV void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// ------------------------------------------------------------------------
// Coalesced row stores.  An epilogue thread owns one output row, so a direct
// store instruction of a warp touches 32 rows (32 cache lines).  Instead each
// epilogue warp stages 32 rows x 128 bytes in its own 4 KB of shared memory
// (16-byte chunks XOR-swizzled by row: neither the row-wise writes nor the
// line-wise reads conflict on banks), then writes 4 whole 128-byte lines per
// store instruction, every row to the destination its owner thread names
// (nullptr: the row is skipped).  Every lane of the warp takes part.
// ------------------------------------------------------------------------
constexpr int kStageWarpBytes = 4096;
constexpr size_t kStageSmem = 8 * kStageWarpBytes;   // two epilogue warpgroups of 4 warps

MOE_DEV uint8_t* stage_of(uint8_t* extra, int r, int group) {
  return extra + (group * 4 + (r >> 5)) * kStageWarpBytes;
}
MOE_DEV int stage_off(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// 16 fp32 values as bf16 into 32-byte piece q (0..3) of this lane's staged row
MOE_DEV void stage_bf16x16(uint8_t* st, int lane, int q, const float (&v)[16]) {
  uint32_t u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(st + stage_off(lane, 2 * q)) = make_uint4(u[0], u[1], u[2], u[3]);
  *reinterpret_cast<uint4*>(st + stage_off(lane, 2 * q + 1)) = make_uint4(u[4], u[5], u[6], u[7]);
}

// 16 fp32 values into 64-byte piece q (0..1) of this lane's staged row
MOE_DEV void stage_f32x16(uint8_t* st, int lane, int q, const float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint4*>(st + stage_off(lane, 4 * q + i)) =
        make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                   __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
}

// Writes the warp's 32 staged rows: row i (lane i's) to lane i's dst.
MOE_DEV void stage_flush(const uint8_t* st, int lane, void* dst) {
  __syncwarp();
  const unsigned long long d = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = 4 * i + (lane >> 3), chunk = lane & 7;
    const unsigned long long p = __shfl_sync(0xffffffffu, d, row);
    const uint4 v = *reinterpret_cast<const uint4*>(st + stage_off(row, chunk));
    if (p != 0ull) st_global_v4(reinterpret_cast<char*>(p) + 16 * chunk, v.x, v.y, v.z, v.w);
  }
  __syncwarp();
}

// Half-size stage for kernels with less shared memory to spare (MXFP8): 32
// rows x 64 bytes per warp, chunk j of row r at r * 64 + 16 * (j ^ ((r >> 1) & 3))
// (a quarter-warp's eight rows x one chunk, or two rows x four chunks, hit
// eight distinct bank groups); a store instruction writes 8 half-lines.
constexpr int kStage64WarpBytes = 2048;
constexpr size_t kStage64Smem = 8 * kStage64WarpBytes;

MOE_DEV uint8_t* stage64_of(uint8_t* extra, int r, int group) {
  return extra + (group * 4 + (r >> 5)) * kStage64WarpBytes;
}
MOE_DEV int stage64_off(int row, int chunk) { return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4); }

// 16 fp32 values as bf16 into 32-byte piece q (0..1) of this lane's staged row
MOE_DEV void stage64_bf16x16(uint8_t* st, int lane, int q, const float* v) {
  uint32_t u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(st + stage64_off(lane, 2 * q)) = make_uint4(u[0], u[1], u[2], u[3]);
  *reinterpret_cast<uint4*>(st + stage64_off(lane, 2 * q + 1)) = make_uint4(u[4], u[5], u[6], u[7]);
}

// 16 fp32 values into this lane's staged row (all four chunks)
MOE_DEV void stage64_f32x16(uint8_t* st, int lane, const float* v) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint4*>(st + stage64_off(lane, i)) =
        make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                   __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
}

// Writes the warp's 32 staged 64-byte rows (fp32 rows added to dst when add)
MOE_DEV void stage64_flush(const uint8_t* st, int lane, void* dst, bool add) {
  __syncwarp();
  const unsigned long long d = reinterpret_cast<unsigned long long>(dst);
  const int chunk = lane & 3;
  unsigned long long p[4];
  uint4 o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p[i] = __shfl_sync(0xffffffffu, d, 8 * i + (lane >> 2));
    o[i] = (add && p[i] != 0ull) ? ld_global_v4(reinterpret_cast<char*>(p[i]) + 16 * chunk)
                                 : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (p[i] == 0ull) continue;
    uint4 v = *reinterpret_cast<const uint4*>(st + stage64_off(8 * i + (lane >> 2), chunk));
    if (add)
      v = make_uint4(__float_as_uint(__uint_as_float(o[i].x) + __uint_as_float(v.x)),
                     __float_as_uint(__uint_as_float(o[i].y) + __uint_as_float(v.y)),
                     __float_as_uint(__uint_as_float(o[i].z) + __uint_as_float(v.z)),
                     __float_as_uint(__uint_as_float(o[i].w) + __uint_as_float(v.w)));
    st_global_v4(reinterpret_cast<char*>(p[i]) + 16 * chunk, v.x, v.y, v.z, v.w);
  }
  __syncwarp();
}

// As stage_flush for fp32 rows, adding them to what dst holds (dst += staged);
// the eight loads of the old values are issued before any of them is used.
MOE_DEV void stage_flush_add_f32(const uint8_t* st, int lane, float* dst) {
  __syncwarp();
  const unsigned long long d = reinterpret_cast<unsigned long long>(dst);
  const int chunk = lane & 7;
  unsigned long long p[8];
  uint4 o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    p[i] = __shfl_sync(0xffffffffu, d, 4 * i + (lane >> 3));
    o[i] = p[i] != 0ull ? ld_global_v4(reinterpret_cast<char*>(p[i]) + 16 * chunk)
                        : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (p[i] == 0ull) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(st + stage_off(4 * i + (lane >> 3), chunk));
    st_global_v4(reinterpret_cast<char*>(p[i]) + 16 * chunk,
                 __float_as_uint(__uint_as_float(o[i].x) + __uint_as_float(v.x)),
                 __float_as_uint(__uint_as_float(o[i].y) + __uint_as_float(v.y)),
                 __float_as_uint(__uint_as_float(o[i].z) + __uint_as_float(v.z)),
                 __float_as_uint(__uint_as_float(o[i].w) + __uint_as_float(v.w)));
  }
  __syncwarp();
}

// ------------------------------------------------------------------------
// F1 + F2 (+ histogram): router logits x·W_r (+ logit_bias), top-k selection
// with ties to the lower expert id, softmax weights renormalised over the
// selected experts, and the expert histogram of this 128-token tile.
//   mapA  = x [T, H] K-major, box {64, 128}
//   mapB0 = W_r^T [E, H] K-major, box {64, BN}  (rows >= E read as zero)
//   in0 = logit_bias f32 [E] or null;  out0 = logits f32 [T, E] or null
//   out1 = topk_idx i32 [T, k];  out2 = topk_w f32 [T, k];  out3 = hist i32 [tiles, E]
// ------------------------------------------------------------------------
template <int BN_, int kSlots = 16>
struct RouterProblem {
  static constexpr int BN = BN_;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  // four warpgroups each keep the sorted top-k list of a quarter of the
  // experts (narrow routers: one); the lists meet in shared memory
  static constexpr int kEpiGroups = BN >= 64 ? 4 : 1;
  static constexpr int kCols = BN / kEpiGroups;
  // length of the per-token sorted lists: every logit is inserted through all
  // of it, so it is sized at compile time (8 when top_k <= 8, else 16)
  static constexpr int kMaxK = kSlots;
  static constexpr size_t kListBytes = kEpiGroups > 1 ? size_t(128) * kEpiGroups * kMaxK * 8 : 0;
  static constexpr size_t kExtraSmem = 256 * sizeof(int) + kListBytes;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return dense_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return dense_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t* extra) {
    int* h = reinterpret_cast<int*>(extra);
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  }
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    tma_load_2d(sA, &a.mapA, kb * kBK, ti.m0, bar);
    tma_load_2d(sB, &a.mapB0, kb * kBK, 0, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}

  // (cv, ci) into the list ordered by (-logit, expert id), the last entry
  // falling off.  Its position p (the number of entries that stay ahead of it)
  // comes from k independent comparisons, and every slot then takes its new
  // entry by a select: no chain of compare-and-swap steps through the list.
  MOE_DEV static void insert(float (&topv)[kMaxK], int (&topi)[kMaxK], int k, float cv, int ci) {
    unsigned ahead = 0u;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s)
      if (s < k && ((topv[s] > cv) || (topv[s] == cv && topi[s] < ci))) ahead |= 1u << s;
    const int p = __popc(ahead);   // the list is sorted: the entries ahead are a prefix
#pragma unroll
    for (int s = kMaxK - 1; s >= 0; --s) {
      if (s < k) {
        const float pv = s > 0 ? topv[s > 0 ? s - 1 : 0] : cv;
        const int pi = s > 0 ? topi[s > 0 ? s - 1 : 0] : ci;
        topv[s] = s > p ? pv : (s == p ? cv : topv[s]);
        topi[s] = s > p ? pi : (s == p ? ci : topi[s]);
      }
    }
  }

  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    int* hist = reinterpret_cast<int*>(extra);
    float2* lists = reinterpret_cast<float2*>(extra + 256 * sizeof(int));   // [row][group][slot]
    const int E = a.E;
    const int k = a.top_k;
    const bool valid = r < ti.rows;
    const int64_t t = static_cast<int64_t>(ti.m0) + r;
    const float* bias = static_cast<const float*>(a.in0);
    float* logits = static_cast<float*>(a.out0);
    float topv[kMaxK];
    int topi[kMaxK];
#pragma unroll
    for (int i = 0; i < kMaxK; ++i) {
      topv[i] = -INFINITY;
      topi[i] = 0x7fffffff;
    }
#pragma unroll 1
    for (int c = group * kCols; c < (group + 1) * kCols; c += 16) {
      float v[16];
      tmem_ld16(taddr + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = c + i;
        if (e < E) {
          float l = v[i];
          if (bias != nullptr) l += __ldg(bias + e);
          v[i] = l;
          // a NaN logit (a token whose input holds NaN or Inf) ranks as -inf:
          // every slot then still receives a valid expert id, the lower ids
          // first by the tie rule
          insert(topv, topi, k, isnan(l) ? -INFINITY : l, e);
        }
      }
      if (valid && logits != nullptr) {
        float* dst = logits + t * E + c;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c + i < E) dst[i] = v[i];
      }
    }
    if constexpr (kEpiGroups > 1) {
      // merge: every group leaves its list, group 0 folds the others into its own
      float2* mine = lists + (static_cast<size_t>(r) * kEpiGroups + group) * kMaxK;
      if (group != 0) {
#pragma unroll
        for (int i = 0; i < kMaxK; ++i)
          if (i < k) mine[i] = make_float2(topv[i], __int_as_float(topi[i]));
      }
      epi_bar_sync<128 * kEpiGroups>();
      if (group == 0) {
#pragma unroll 1
        for (int g = 1; g < kEpiGroups; ++g) {
          const float2* other = lists + (static_cast<size_t>(r) * kEpiGroups + g) * kMaxK;
#pragma unroll 1
          for (int i = 0; i < k; ++i) {
            const float2 o = other[i];
            insert(topv, topi, k, o.x, __float_as_int(o.y));
          }
        }
      }
    }
    if (group == 0 && valid) {
      // m = -inf only when every logit of the token is -inf or NaN; the
      // weights are then NaN, as the softmax over such logits is
      const float m = topv[0];
      float ex[kMaxK];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        ex[j] = (j < k) ? expf(topv[j] - m) : 0.f;
        sum += ex[j];
      }
      const float inv = 1.0f / sum;
      int* idx_out = static_cast<int*>(a.out1) + t * k;
      float* w_out = static_cast<float*>(a.out2) + t * k;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          idx_out[j] = topi[j];
          w_out[j] = ex[j] * inv;
          if (in_range(topi[j], E))
            atomicAdd(hist + topi[j], 1);
          else
            record_bad_index(a.status, kCheckRouterExpert, topi[j]);
        }
      }
    }
    epi_bar_sync<128 * kEpiGroups>();
    int* hist_out = static_cast<int*>(a.out3) + static_cast<int64_t>(ti.mt) * E;
    for (int e = group * 128 + r; e < E; e += 128 * kEpiGroups) {
      hist_out[e] = hist[e];
      hist[e] = 0;
    }
    epi_bar_sync<128 * kEpiGroups>();
  }
};


// ------------------------------------------------------------------------
// F7 + F8: expert gate/up GEMM with the SwiGLU epilogue.
//   Tile = 128 permuted rows x (128 gate columns | 128 up columns) of expert e.
//   mapA  = x_perm [P, H] K-major, box {64, 128}
//   mapB0 = W_gate as [E*H, F] MN-major, box {64, 64};  mapB1 = W_up, same
//   out0 = a [P, F] bf16 (silu(h_g) * h_u);  out1 = h [P, 2F] bf16 (h_g | h_u)
//   ld0 = F;  K = H;  n_tiles = F / 128;  b_group_rows = H
// ------------------------------------------------------------------------
struct GateUpFwdProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = true;
  static constexpr size_t kExtraSmem = kStageSmem;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile(a, t, 128); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + k0;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    tma_load_2d(sB, &a.mapB0, ti.n0, brow, bar);
    tma_load_2d(sB + kChunkBytes, &a.mapB0, ti.n0 + 64, brow, bar);
    tma_load_2d(sB + 2 * kChunkBytes, &a.mapB1, ti.n0, brow, bar);
    tma_load_2d(sB + 3 * kChunkBytes, &a.mapB1, ti.n0 + 64, brow, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  // Three sweeps over the group's 64 gate and 64 up accumulator columns, one
  // per output (h_gate, h_up, a), each leaving through the warp's stage.
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int lane = r & 31;
    uint8_t* st = stage_of(extra, r, group);
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    const int F = a.ld0;
    const int cb = group * 64;
    __nv_bfloat16* act = valid ? static_cast<__nv_bfloat16*>(a.out0) + row * F + ti.n0 + cb : nullptr;
    __nv_bfloat16* hg = valid ? static_cast<__nv_bfloat16*>(a.out1) + row * 2 * F + ti.n0 + cb : nullptr;
    __nv_bfloat16* hu = valid ? hg + F : nullptr;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float g[16];
      tmem_ld16(taddr + cb + 16 * q, g);
      tmem_ld_wait();
      stage_bf16x16(st, lane, q, g);
    }
    stage_flush(st, lane, hg);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float u[16];
      tmem_ld16(taddr + 128 + cb + 16 * q, u);
      tmem_ld_wait();
      stage_bf16x16(st, lane, q, u);
    }
    stage_flush(st, lane, hu);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      float g[16], u[16];
      tmem_ld16(taddr + cb + 16 * q, g);
      tmem_ld16(taddr + 128 + cb + 16 * q, u);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) g[i] = g[i] * sigmoidf_fast(g[i]) * u[i];
      stage_bf16x16(st, lane, q, g);
    }
    stage_flush(st, lane, act);
  }
};

// ------------------------------------------------------------------------
// F9 + F10 (first half): expert down GEMM; the epilogue scales each row by its
// router weight and scatters it to the (token, slot)-ordered scratch, which
// the combine kernel then sums over the k slots.
//   mapA  = a [P, F] K-major, box {64, 128}
//   mapB0 = W_down as [E*F, H] MN-major, box {64, 64}
//   in0 = w_row f32 [P];  in1 = row_slot i32 [P];  out0 = scratch bf16 [P, H]
//   ld0 = H;  K = F;  n_tiles = H / 256;  b_group_rows = F
// ------------------------------------------------------------------------
struct DownFwdProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = true;
  static constexpr size_t kExtraSmem = kStageSmem;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + k0;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_2d(sB + c * kChunkBytes, &a.mapB0, ti.n0 + 64 * c, brow, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int lane = r & 31;
    uint8_t* st = stage_of(extra, r, group);
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    float w = 0.f;
    __nv_bfloat16* dst = nullptr;
    if (valid) {
      w = __ldg(static_cast<const float*>(a.in0) + row);
      const int slot = __ldg(static_cast<const int*>(a.in1) + row);
      dst = static_cast<__nv_bfloat16*>(a.out0) + static_cast<int64_t>(slot) * a.ld0 + ti.n0;
      MOE_CHECK_INDEX(a.status, kCheckScatterRow, slot, a.T * a.top_k, dst = nullptr);
    }
#pragma unroll 1
    for (int c0 = group * (BN / 2); c0 < (group + 1) * (BN / 2); c0 += 64) {
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float v[16];
        tmem_ld16(taddr + c0 + 16 * q, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= w;
        stage_bf16x16(st, lane, q, v);
      }
      stage_flush(st, lane, valid ? dst + c0 : nullptr);
    }
  }
};

}  // namespace moe
