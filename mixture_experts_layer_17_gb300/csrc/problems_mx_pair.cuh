// CTA-pair (cta_group::2) versions of the MXFP8 expert GEMMs: a cluster of
// two CTAs computes a 256 x 256 tile with M = 256 block-scaled MMAs; CTA
// `rank` TMA-loads its 128 rows of A and one 128-row half of B (K = 128 E4M3
// per stage) and the scale atoms its tensor core reads, all completing on the
// leader's full barrier.  The scale atoms come through [atoms, 128] u32
// tensor maps (mapSFA, mapSFB, mapSFB1), one 512-byte atom per load.  Each
// CTA holds in TMEM the scales of its own 128 rows of A and of the B columns
// its tensor core multiplies (kPairSFBFull: both 128-column halves of the
// tile's B; else its own half).  Epilogues are the single-CTA ones: the
// engine hands each CTA its 128-row half of the tile and its m-tile index.
#pragma once

#include "problems_mx.cuh"

namespace moe {

// Which B scale atoms each CTA of a pair keeps in TMEM (see above).
constexpr bool kPairSFBFull = true;
constexpr int kPairSFAtoms = kPairSFBFull ? 3 : 2;

// loads one 512-byte scale atom (row `atom` of an [atoms, 128] u32 map)
MOE_DEV void load_atom_pair(uint8_t* dst, const CUtensorMap* map, int64_t atom, uint32_t bar) {
  tma_load_2d_pair(dst, map, 0, static_cast<int32_t>(atom), bar);
}

// The B atoms of a 256-column tile whose halves' atom rows are b0 and b0 + 1
// (stride 1) or b0 and b0 + stride: both, or this CTA's half.
MOE_DEV void load_b_atoms_pair(uint8_t* sSF, const CUtensorMap* map, int64_t b0, int64_t stride,
                               int rank, uint32_t bar) {
  if constexpr (kPairSFBFull) {
    load_atom_pair(sSF + 512, map, b0, bar);
    load_atom_pair(sSF + 1024, map, b0 + stride, bar);
  } else {
    load_atom_pair(sSF + 512, map, b0 + rank * stride, bar);
  }
}

// grouped-M pair tile with 128-element (fp8) K stages
MOE_DEV TileInfo grouped_m_tile_pair_mx(const GemmArgs& a, int t, int nstep) {
  TileInfo ti = grouped_m_tile_pair(a, t, nstep);
  ti.num_kb = a.K / 128;
  return ti;
}

// atom row of A's scales for this CTA's 128-row m-tile of pair tile ti
MOE_DEV int64_t a_atom_row_pair(const GemmArgs& a, const TileInfo& ti, int rank) {
  return static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + 2 * ti.mt + rank;
}

// F7 + F8: each CTA loads one interleaved [64 gate | 64 up] block of B.
struct GateUpFwdMXPairProblem : GateUpFwdMXProblem {
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = kPairSFAtoms;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair_mx(a, t, 128); }
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    const int k0 = kb * 128;
    const int nb = ti.n0 / 64;                // first interleaved 128-column block
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, &a.mapB0, (nb + rank) * 128, ti.e * a.b_group_rows + k0, bar);
    load_atom_pair(sSF, &a.mapSFA, a_atom_row_pair(a, ti, rank) * a.kt_a + kb, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + nb;
    load_b_atoms_pair(sSF, &a.mapSFB, wrow * a.kt_b + kb, a.kt_b, rank, bar);
  }
};

// F9 (+ F10 scatter): B = W_down along F, MN-major, columns n0 + 128 * rank.
struct DownFwdMXPairProblem : DownFwdMXProblem {
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = kPairSFAtoms;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair_mx(a, t, BN); }
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    const int k0 = kb * 128;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, &a.mapB0, ti.n0 + 128 * rank, ti.e * a.b_group_rows + k0, bar);
    load_atom_pair(sSF, &a.mapSFA, a_atom_row_pair(a, ti, rank) * a.kt_a + kb, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + ti.n0 / 128;
    load_b_atoms_pair(sSF, &a.mapSFB, wrow * a.kt_b + kb, a.kt_b, rank, bar);
  }
};

// B6: B = W_gate then W_up along F (K-major), rows n0 + 128 * rank.
struct GateUpDgradMXPairProblem : GateUpDgradMXProblem {
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = kPairSFAtoms;
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair_mx(a, t, BN); }
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    const int k0 = kb * 128;
    const bool up = k0 >= a.k_half;
    const int kbw = up ? kb - a.kt_b : kb;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, up ? &a.mapB1 : &a.mapB0, up ? k0 - a.k_half : k0,
                     ti.e * a.b_group_rows + ti.n0 + 128 * rank, bar);
    load_atom_pair(sSF, &a.mapSFA, a_atom_row_pair(a, ti, rank) * a.kt_a + kb, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + ti.n0 / 128;
    load_b_atoms_pair(sSF, up ? &a.mapSFB1 : &a.mapSFB, wrow * a.kt_b + kbw, a.kt_b, rank, bar);
  }
};

// Weight gradients (A and B MN-major, K = the expert's 128-row token tiles):
// 256-row M tiles; CTA `rank` loads M columns m0 + 128 * rank and N columns
// n0 + 128 * rank.  a.m_tiles counts the 256-row tiles; A's atoms are laid
// out per 128 M columns: row k-tile * a.kt_a + (128-column tile).
template <bool kGateUp>
struct WgradMXPairProblem : WgradMXProblem<kGateUp> {
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = kPairSFAtoms;
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) {
    TileInfo ti = grouped_k_tile_mx(a, t, 256);
    ti.m0 = ti.mt * 2 * kBM;
    ti.rows = min(2 * kBM, a.M - ti.m0);
    ti.rows_pad = ti.rows;
    return ti;
  }
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    const int kt = ti.kb0 + kb;
    const int krow = 128 * kt;
    tma_load_2d_pair(sA, &a.mapA, ti.m0 + kBM * rank, krow, bar);
    tma_load_2d_pair(sB, &a.mapB0, ti.n0 + 128 * rank, krow, bar);
    load_atom_pair(sSF, &a.mapSFA, static_cast<int64_t>(kt) * a.kt_a + 2 * ti.mt + rank, bar);
    load_b_atoms_pair(sSF, &a.mapSFB, static_cast<int64_t>(kt) * (2 * a.n_tiles) + ti.n0 / 128, 1,
                      rank, bar);
  }
};

// Dense MXFP8 GEMM on 256 x 256 CTA-pair tiles for moe_gemm_mxfp8 (N a
// multiple of 256): A [M, K] and B [N, K] E4M3, K-major; A's atoms (128-row
// m-tile * kt + k-tile), B's (128-row n-tile * kt + k-tile); D fp32 [M, N].
struct DenseMXPairProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kMX = true;
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = kPairSFAtoms;
  static constexpr size_t kExtraSmem = 0;
  static constexpr int kEpiGroups = 2;
  struct Frag {
    float v[128];
  };

  MOE_DEV static int num_tiles(const GemmArgs& a) { return ((a.M + 255) / 256) * a.n_tiles; }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) {
    const int mt = t / a.n_tiles;
    const int nt = t - mt * a.n_tiles;
    TileInfo ti;
    ti.e = -1;
    ti.m0 = mt * 2 * kBM;
    ti.n0 = nt * BN;
    ti.rows = min(2 * kBM, a.M - ti.m0);
    ti.rows_pad = ti.rows;
    ti.kb0 = 0;
    ti.num_kb = a.K / 128;
    ti.k_last = 128;
    ti.krow0 = 0;
    ti.mt = mt;
    return ti;
  }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    tma_load_2d_pair(sA, &a.mapA, kb * 128, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, &a.mapB0, kb * 128, ti.n0 + 128 * rank, bar);
    load_atom_pair(sSF, &a.mapSFA, static_cast<int64_t>(2 * ti.mt + rank) * a.kt_a + kb, bar);
    load_b_atoms_pair(sSF, &a.mapSFB, static_cast<int64_t>(ti.n0 / 128) * a.kt_b + kb, a.kt_b,
                      rank, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue_load(const GemmArgs&, const TileInfo&, uint32_t taddr, int,
                                    int group, Frag& f) {
    tmem_ld128(taddr + 128 * group, f.v);
  }
  MOE_DEV static void epilogue_store(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     const Frag& f, uint8_t*) {
    if (r >= ti.rows) return;
    float* p = static_cast<float*>(a.out0) + (static_cast<int64_t>(ti.m0) + r) * a.ld0 + ti.n0 +
               128 * group;
#pragma unroll
    for (int i = 0; i < 128; i += 4)
      st_global_v4(p + i, __float_as_uint(f.v[i]), __float_as_uint(f.v[i + 1]),
                   __float_as_uint(f.v[i + 2]), __float_as_uint(f.v[i + 3]));
  }
};

}  // namespace moe
