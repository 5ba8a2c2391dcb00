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

// B2-B4 in MXFP8 on CTA pairs with 256 x 192 tiles (N = 192 divides F for
// the Qwen3-shaped layers): two accumulators per CTA fit beside the scale
// slots, so a tile's epilogue overlaps the next tile's MMAs.  Per stage CTA
// `rank` loads its 128 rows of dY (along H), rows n0 + 96 * rank of W_down
// (K-major) and three scale atoms: its own A atom and both atoms of the
// tile's 192 B rows.  W_down's scales come in 192-row blocks of two atoms
// (rows 0..127, then rows 128..191 in the first 64 rows of the second atom):
// atom ((expert * F/192 + n-tile) * 2 + half) * (H/128) + k-tile.
// Epilogue: the SwiGLU backward of DownDgradProblem's staged epilogue (one
// pair of 2 KB buffers per warp, h by TMA, dh and w*a out by TMA stores
// through mapC0 / mapC1), plus dh quantised to E4M3 along F from fp32 (out3
// / out4, as in DownDgradMXProblem); 96 columns per warpgroup and tile, i.e.
// three 32-column steps.
struct DownDgradMXPairProblem {
  static constexpr int BN = 192;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kMX = true;
  static constexpr bool kPair = true;
  static constexpr int kSFAtoms = 3;
  static constexpr size_t kStageBytes = 8 * 2 * kStage64WarpBytes;
  static constexpr size_t kExtraSmem = 1024 + kStageBytes + 8 * sizeof(uint64_t);
  static constexpr int kEpiGroups = 2;
  static constexpr int kSteps = BN / 2 / 32;

  MOE_DEV static uint8_t* stage_base(uint8_t* extra) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(extra) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  }
  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles_pair(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_pair_mx(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t* extra) {
    if (threadIdx.x == 0) {
      uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base(extra) + kStageBytes);
      for (int w = 0; w < 8; ++w) mbar_init(bars + w, 1);
      fence_mbar_init();
    }
  }
  MOE_DEV static void load_mx_pair(const GemmArgs& a, const TileInfo& ti, int kb, int rank,
                                   uint8_t* sA, uint8_t* sB, uint8_t* sSF, uint32_t bar) {
    const int k0 = kb * 128;
    tma_load_2d_pair(sA, &a.mapA, k0, ti.m0 + kBM * rank, bar);
    tma_load_2d_pair(sB, &a.mapB0, k0, ti.e * a.b_group_rows + ti.n0 + (BN / 2) * rank, bar);
    load_atom_pair(sSF, &a.mapSFA, a_atom_row_pair(a, ti, rank) * a.kt_a + kb, bar);
    const int64_t blk = static_cast<int64_t>(ti.e) * a.n_tiles + ti.n0 / BN;
    load_atom_pair(sSF + 512, &a.mapSFB, 2 * blk * a.kt_b + kb, bar);
    load_atom_pair(sSF + 1024, &a.mapSFB, (2 * blk + 1) * a.kt_b + kb, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    constexpr int kHalf = BN / 2;
    const bool valid = r < ti.rows;
    const bool pad = !valid && r < ti.rows_pad;
    const int lane = r & 31;
    const int wslot = group * 4 + (r >> 5);
    uint8_t* buf = stage_base(extra) + wslot * 2 * kStage64WarpBytes;
    uint64_t* hbar = reinterpret_cast<uint64_t*>(stage_base(extra) + kStageBytes) + wslot;
    const int64_t row = static_cast<int64_t>(ti.m0) + ((valid || pad) ? r : 0);
    const int F = a.ld0;
    const int c0 = group * kHalf;
    const int y = ti.m0 + (r & ~31);
    uint8_t* dhq = static_cast<uint8_t*>(a.out3) + row * 2 * F;
    uint8_t* sfq = static_cast<uint8_t*>(a.out4);
    const int64_t atom_row = (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * (2 * F / 128);
    const float w = valid ? __ldg(static_cast<const float*>(a.in1) + row) : 0.f;
    const int never = 0;   // the h waits are cut short only by their time limit
    // h_gate and h_up of step s into the warp's pair; every lane's earlier
    // accesses to the pair are ordered before the asynchronous writes
    auto load_h = [&](int step) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(hbar, 2 * kStage64WarpBytes);
        tma_load_2d(buf, &a.mapB1, ti.n0 + c0 + 32 * step, y, hbar);
        tma_load_2d(buf + kStage64WarpBytes, &a.mapB1, F + ti.n0 + c0 + 32 * step, y, hbar);
      }
    };
    float dw = 0.f;
    load_h(0);
#pragma unroll 1
    for (int step = 0; step < kSteps; ++step) {
      const int c = c0 + 32 * step;
      if (!mbar_wait_bounded(hbar, static_cast<uint32_t>(step) & 1u, &never, a.wait_limit_ns))
        record_timeout(a.status, kWaitEpiLoad);
      uint32_t gw[16], uw[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 ug = *reinterpret_cast<const uint4*>(buf + stage64_off(lane, q));
        const uint4 uu =
            *reinterpret_cast<const uint4*>(buf + kStage64WarpBytes + stage64_off(lane, q));
        gw[4 * q] = ug.x; gw[4 * q + 1] = ug.y; gw[4 * q + 2] = ug.z; gw[4 * q + 3] = ug.w;
        uw[4 * q] = uu.x; uw[4 * q + 1] = uu.y; uw[4 * q + 2] = uu.z; uw[4 * q + 3] = uu.w;
      }
      float g[32];
      tmem_ld32(taddr + c, g);
      float dhg[32], dhu[32];
      uint32_t awp[16];   // w*a of the step's 32 columns, packed bf16
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float awv[16];
        if (valid) {
          DownDgradProblem<256, true>::swiglu_bwd16(g + 16 * half, gw + 8 * half, uw + 8 * half, w,
                                                    dw, dhg + 16 * half, dhu + 16 * half, awv);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) dhg[16 * half + i] = dhu[16 * half + i] = awv[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) awp[8 * half + i] = pack_bf16x2(awv[2 * i], awv[2 * i + 1]);
      }
      stage64_bf16x16(buf, lane, 0, dhg);
      stage64_bf16x16(buf, lane, 1, dhg + 16);
      stage64_bf16x16(buf + kStage64WarpBytes, lane, 0, dhu);
      stage64_bf16x16(buf + kStage64WarpBytes, lane, 1, dhu + 16);
      // dh_gate and dh_up, then w*a, leave by TMA stores (a.mapC0, a.mapC1);
      // the warp's 32 rows lie wholly inside the expert's 64-row aligned
      // padded segment or wholly outside it
      const bool slab_in = (r & ~31) < ti.rows_pad;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && slab_in) {
        tma_store_2d(&a.mapC0, buf, ti.n0 + c, y);
        tma_store_2d(&a.mapC0, buf + kStage64WarpBytes, F + ti.n0 + c, y);
        bulk_commit();
        bulk_wait_read0();
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(buf + stage64_off(lane, q)) =
            make_uint4(awp[4 * q], awp[4 * q + 1], awp[4 * q + 2], awp[4 * q + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && slab_in) {
        tma_store_2d(&a.mapC1, buf, ti.n0 + c, y);
        bulk_commit();
        bulk_wait_read0();
      }
      __syncwarp();
      if (valid) {
        const int cg = ti.n0 + c;           // gate column; up column = F + cg
        mx_block_store(dhg, dhq + cg,
                       sfq + (atom_row + cg / 128) * 512 + sf_atom_offset(r, (cg >> 5) & 3));
        mx_block_store(dhu, dhq + F + cg,
                       sfq + (atom_row + (F + cg) / 128) * 512 + sf_atom_offset(r, ((F + cg) >> 5) & 3));
      }
      if (step + 1 < kSteps) load_h(step + 1);
    }
    if constexpr (kSteps % 2 != 0) {
      // one more (empty) phase, so that every tile starts at parity 0; every
      // lane has passed its last wait
      __syncwarp();
      if (lane == 0) mbar_arrive(hbar);
    }
    // one router-weight partial per (row, n-tile, column half)
    if (valid)
      static_cast<float*>(a.out2)[row * (a.n_tiles * kEpiGroups) + (ti.n0 / BN) * kEpiGroups +
                                  group] = dw;
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
