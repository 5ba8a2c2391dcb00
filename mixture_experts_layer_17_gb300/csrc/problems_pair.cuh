// CTA-pair (cta_group::2) versions of the expert GEMMs: a cluster of two CTAs
// computes a 256-row tile; CTA `rank` TMA-loads rows [128*rank, 128*rank+128)
// of A and N-rows [BN/2*rank, BN/2*rank + BN/2) of B into its own shared
// memory, completing on the leader's full barrier.  Epilogues are the
// single-CTA ones (the engine hands each CTA its 128-row half of the tile).
#pragma once

#include "problems_bwd.cuh"

namespace moe {

// F7 + F8: the leader stages the 128 gate columns, its peer the 128 up columns.
struct GateUpFwdPairProblem : GateUpFwdProblem {
  static constexpr bool kPair = true;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair(a, t, 128); }
  MOE_DEV static void load_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                uint8_t* sA, uint8_t* sB, uint32_t bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + k0;
    const CUtensorMap* mb = rank ? &a.mapB1 : &a.mapB0;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, mb, ti.n0, brow, bar);
    tma_load_2d_pair(sB + kChunkBytes, mb, ti.n0 + 64, brow, bar);
  }
};

// F9 (+ F10 scatter): B MN-major, 64-column chunks 2*rank and 2*rank + 1.
struct DownFwdPairProblem : DownFwdProblem {
  static constexpr bool kPair = true;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair(a, t, BN); }
  MOE_DEV static void load_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                uint8_t* sA, uint8_t* sB, uint32_t bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + k0;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      tma_load_2d_pair(sB + j * kChunkBytes, &a.mapB0, ti.n0 + 64 * (2 * rank + j), brow, bar);
  }
};

// B2-B4: B K-major (box {64, 128}), N-rows 128*rank ...
struct DownDgradPairProblem : DownDgradProblem<256, true> {
  static constexpr bool kPair = true;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair(a, t, BN); }
  MOE_DEV static void load_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                uint8_t* sA, uint8_t* sB, uint32_t bar) {
    const int k0 = kb * kBK;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, &a.mapB0, k0, ti.e * a.b_group_rows + ti.n0 + 128 * rank, bar);
  }
};

// B6: B K-major (box {64, 128}) from W_gate, then W_up, along K.
struct GateUpDgradPairProblem : GateUpDgradProblem {
  static constexpr bool kPair = true;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair(a, t, BN); }
  MOE_DEV static void load_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                uint8_t* sA, uint8_t* sB, uint32_t bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + ti.n0 + 128 * rank;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    if (k0 < a.k_half)
      tma_load_2d_pair(sB, &a.mapB0, k0, brow, bar);
    else
      tma_load_2d_pair(sB, &a.mapB1, k0 - a.k_half, brow, bar);
  }
};

// Weight gradients over the padded token segments: A and B MN-major.
template <class Base>
struct WgradPairProblem : Base {
  static constexpr bool kPair = true;
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) {
    return grouped_k_tile_pair(a, t, Base::BN);
  }
  MOE_DEV static void load_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                uint8_t* sA, uint8_t* sB, uint32_t bar) {
    const int krow = ti.krow0 + kb * kBK;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      tma_load_2d_pair(sA + j * kChunkBytes, &a.mapA, ti.m0 + kBM * rank + 64 * j, krow, bar);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      tma_load_2d_pair(sB + j * kChunkBytes, &a.mapB0, ti.n0 + 64 * (2 * rank + j), krow, bar);
  }
};

}  // namespace moe
