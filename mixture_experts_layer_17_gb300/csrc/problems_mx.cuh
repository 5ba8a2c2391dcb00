// MXFP8 GEMMs of the MoE layer: E4M3 operands with E8M0 scales per 32
// elements along K, block-scaled tcgen05 MMA, 128 x 128 output tiles, K = 128
// per stage.  Scale atoms (512 bytes: 128 MN-rows x 4 K-blocks) are fetched
// with 1-D bulk copies beside the operand tiles:
//   activations along features (K-major, rows of the permuted layout): atom
//     ((mtile_off[e] + m-tile) * kt_a + k-tile);
//   weights: atom ((expert * n_tiles + n-tile) * kt_b + k-tile);
//   activations along tokens (MN-major, expert segments padded to 128 rows):
//     atom (k-tile * tiles_of_MN + MN-tile), k-tile = mtile_off[e] + local.
// Epilogues match the bf16 problems (problems.cuh, problems_bwd.cuh).
#pragma once

#include "problems_bwd.cuh"

namespace moe {

MOE_DEV const uint8_t* sf_atom(const uint8_t* base, int64_t index) { return base + index * 512; }

// Quantises one 32-element MX block held by this thread (fp32 values) to E4M3
// at dst (32 bytes) and writes its E8M0 scale byte at *scale.
MOE_DEV void mx_block_store(const float (&v)[32], uint8_t* dst, uint8_t* scale) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_exponent(amax);
  const float inv = mx_inv_scale(X);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = to_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
  st_global_v4(dst, w[0], w[1], w[2], w[3]);
  st_global_v4(dst + 16, w[4], w[5], w[6], w[7]);
  *scale = static_cast<uint8_t>(X + 127);
}

MOE_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tmem_ld16(taddr, a);
  tmem_ld16(taddr + 16, b);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}

// Copies 8 x 16 TMEM columns starting at taddr into v (one wait for all).
MOE_DEV void tmem_ld128(uint32_t taddr, float (&v)[128]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) tmem_ld16(taddr + 16 * i, *reinterpret_cast<float(*)[16]>(v + 16 * i));
  tmem_ld_wait();
}

// B operand of a 256-wide MXFP8 tile: two 128-row TMA boxes (K-major: rows
// n0 and n0 + 128 at sB and sB + 16 KB; MN-major: columns n0 and n0 + 128,
// the second chunk at the descriptor's LBO of 16 KB).
MOE_DEV void load_b256_kmajor(const CUtensorMap* map, int k0, int row0, uint8_t* sB, uint64_t* bar) {
  tma_load_2d(sB, map, k0, row0, bar);
  tma_load_2d(sB + 16384, map, k0, row0 + 128, bar);
}
MOE_DEV void load_b256_mnmajor(const CUtensorMap* map, int col0, int krow, uint8_t* sB, uint64_t* bar) {
  tma_load_2d(sB, map, col0, krow, bar);
  tma_load_2d(sB + 16384, map, col0 + 128, krow, bar);
}

// grouped-M tile with 128-element (fp8) K stages
MOE_DEV TileInfo grouped_m_tile_mx(const GemmArgs& a, int t, int nstep) {
  TileInfo ti = grouped_m_tile(a, t, nstep);
  ti.num_kb = a.K / 128;
  return ti;
}

// grouped-K tile over the 128-row padded token layout: expert e's K range is
// k-tiles [mtile_off[e], mtile_off[e+1]) (an expert without tokens has none).
MOE_DEV TileInfo grouped_k_tile_mx(const GemmArgs& a, int t, int BN) {
  const int per = a.m_tiles * a.n_tiles;
  const int gi = t / per;
  const int local = t - gi * per;
  const int mt = local / a.n_tiles;
  const int nt = local - mt * a.n_tiles;
  const int e = a.group_order != nullptr ? __ldg(a.group_order + gi) : gi;
  const int k0 = __ldg(a.mtile_off + e);
  TileInfo ti;
  ti.e = e;
  ti.m0 = mt * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(kBM, a.M - ti.m0);
  ti.rows_pad = ti.rows;
  ti.kb0 = k0;
  ti.num_kb = __ldg(a.mtile_off + e + 1) - k0;
  ti.k_last = 128;
  ti.krow0 = 128 * k0;
  ti.mt = mt;
  return ti;
}

// ------------------------------------------------------------------------
// F7 + F8 in MXFP8: A = x_perm E4M3 [P, H]; B = W_gate|W_up quantised along H
// and interleaved per 128-column block as [64 gate | 64 up] ([E*H, 2F],
// MN-major).  Tile = 128 rows x 256 B columns = two interleaved blocks, i.e.
// 128 F columns; epilogue group g owns block g (64 gate + 64 up columns).
// Outputs: out0 = a as E4M3 [Pa, F] (quantised here from fp32), out1 = h bf16
// [Pa, 2F], out2 = scale atoms of a (((mtile_off[e] + m-tile) * F/128 +
// f/128) * 512).
// ------------------------------------------------------------------------
struct GateUpFwdMXProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = true;
  static constexpr bool kMX = true;
  static constexpr size_t kExtraSmem = kStage64Smem;
  static constexpr int kEpiGroups = 2;
  struct Frag {
    float v[128];   // [0, 64): gate, [64, 128): up
  };

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_mx(a, t, 128); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    const int k0 = kb * 128;
    const int nb = ti.n0 / 64;                // first interleaved 128-column block
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    load_b256_mnmajor(&a.mapB0, nb * 128, ti.e * a.b_group_rows + k0, sB, bar);
    bulk_load(sSF, sf_atom(a.sfA, (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * a.kt_a + kb), 512, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + nb;
    bulk_load(sSF + 512, sf_atom(a.sfB0, wrow * a.kt_b + kb), 512, bar);
    bulk_load(sSF + 1024, sf_atom(a.sfB0, (wrow + 1) * a.kt_b + kb), 512, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue_load(const GemmArgs&, const TileInfo&, uint32_t taddr, int,
                                    int group, Frag& f) {
    tmem_ld128(taddr + 128 * group, f.v);
  }
  MOE_DEV static void epilogue_store(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     Frag& f, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    const int lane = r & 31;
    uint8_t* st = stage64_of(extra, r, group);
    const int F = a.ld0;
    const int f0 = ti.n0 + 64 * group;        // first F column of this group
    __nv_bfloat16* hg = static_cast<__nv_bfloat16*>(a.out1) + row * 2 * F + f0;
    // h_gate then h_up, 32 columns (64 bytes) per staged row
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      stage64_bf16x16(st, lane, 0, f.v + c);
      stage64_bf16x16(st, lane, 1, f.v + c + 16);
      stage64_flush(st, lane, valid ? hg + (c < 64 ? c : F + c - 64) : nullptr, false);
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) f.v[i] = f.v[i] * sigmoidf_fast(f.v[i]) * f.v[64 + i];
    // a: two MX blocks of 32 columns -> 64 E4M3 bytes (staged) and two scale bytes
    uint8_t* sf = static_cast<uint8_t*>(a.out2) +
                  ((static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * (F / 128) + f0 / 128) * 512;
#pragma unroll
    for (int blk2 = 0; blk2 < 2; ++blk2) {
      const float* v = f.v + 32 * blk2;
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const int X = mx_exponent(amax);
      const float inv = mx_inv_scale(X);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = to_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv);
      *reinterpret_cast<uint4*>(st + stage64_off(lane, 2 * blk2)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(st + stage64_off(lane, 2 * blk2 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      if (valid) sf[sf_atom_offset(r, ((f0 >> 5) & 3) + blk2)] = static_cast<uint8_t>(X + 127);
    }
    stage64_flush(st, lane, valid ? static_cast<uint8_t*>(a.out0) + row * F + f0 : nullptr, false);
  }
};


// F9 + F10 in MXFP8: A = a E4M3 [P, F]; B = W_down quantised along F
// ([E*F, H], MN-major); 128 x 256 tiles, weighted scatter epilogue.
struct DownFwdMXProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = true;
  static constexpr bool kMX = true;
  static constexpr size_t kExtraSmem = kStage64Smem;
  static constexpr int kEpiGroups = 2;
  struct Frag {
    float v[128];
  };

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_mx(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    const int k0 = kb * 128;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    load_b256_mnmajor(&a.mapB0, ti.n0, ti.e * a.b_group_rows + k0, sB, bar);
    bulk_load(sSF, sf_atom(a.sfA, (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * a.kt_a + kb), 512, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + ti.n0 / 128;
    bulk_load(sSF + 512, sf_atom(a.sfB0, wrow * a.kt_b + kb), 512, bar);
    bulk_load(sSF + 1024, sf_atom(a.sfB0, (wrow + 1) * a.kt_b + kb), 512, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue_load(const GemmArgs&, const TileInfo&, uint32_t taddr, int,
                                    int group, Frag& f) {
    tmem_ld128(taddr + 128 * group, f.v);
  }
  MOE_DEV static void epilogue_store(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     Frag& f, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    const int lane = r & 31;
    uint8_t* st = stage64_of(extra, r, group);
    float w = 0.f;
    __nv_bfloat16* dst = nullptr;
    if (valid) {
      w = __ldg(static_cast<const float*>(a.in0) + row);
      const int slot = __ldg(static_cast<const int*>(a.in1) + row);
      dst = static_cast<__nv_bfloat16*>(a.out0) + static_cast<int64_t>(slot) * a.ld0 + ti.n0 +
            128 * group;
      MOE_CHECK_INDEX(a.status, kCheckScatterRow, slot, a.T * a.top_k, dst = nullptr);
    }
#pragma unroll
    for (int i = 0; i < 128; ++i) f.v[i] *= w;
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      stage64_bf16x16(st, lane, 0, f.v + c);
      stage64_bf16x16(st, lane, 1, f.v + c + 16);
      stage64_flush(st, lane, valid ? dst + c : nullptr, false);
    }
  }
};


// B2-B4 in MXFP8: A = dY_perm E4M3 [P, H]; B = W_down quantised along H
// ([E*F, H], K-major); the SwiGLU-backward epilogue of DownDgradProblem: dh
// and w*a in bf16 for the weight gradients, the router-weight partials, and
// dh quantised to E4M3 along F straight from fp32 for the gate/up dgrad:
// out3 = dh E4M3 [Pa, 2F], out4 = its scale atoms (((mtile_off[e] +
// m-tile) * 2F/128 + column/128) * 512).  The layer runs BN = 128 with a
// double-buffered accumulator and kStaged (dh_gate, dh_up and w*a through
// three 2 KB shared-memory stages per warp, five stages): the epilogue is
// heavy and overlaps the next tile's MMAs that way (a 256-wide tile with one
// accumulator, whose epilogue runs serially, measured slower).
template <int BN_, bool kStaged = false>
struct DownDgradMXProblem {
  static constexpr int BN = BN_;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kMX = true;
  // kStaged: each epilogue warp owns three 2 KB buffers (1024-byte aligned,
  // hence up to 1 KB of lead-in) and an mbarrier.  Per 32-column step, TMA
  // brings the warp's 32 rows of h_gate and h_up into the first two (64-byte
  // swizzle, the stage64 layout) and the threads read their rows from there;
  // then dh_gate, dh_up and w*a are staged in the three buffers and leave as
  // whole 64-byte row pieces.
  static constexpr size_t kStageBytes = 8 * 3 * kStage64WarpBytes;
  static constexpr size_t kExtraSmem = kStaged ? 1024 + kStageBytes + 8 * sizeof(uint64_t) : 0;
  static constexpr int kEpiGroups = 2;
  // two steps per warp and tile keep the parity of each warp's barrier in
  // step with the step index from one tile to the next
  static_assert(!kStaged || (BN / 2 / 32) % 2 == 0, "an even number of h steps per tile");

  MOE_DEV static uint8_t* stage_base(uint8_t* extra) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(extra) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  }

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_mx(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t* extra) {
    if constexpr (kStaged) {
      if (threadIdx.x == 0) {
        uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base(extra) + kStageBytes);
        for (int w = 0; w < 8; ++w) mbar_init(bars + w, 1);
        fence_mbar_init();
      }
    }
  }
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    const int k0 = kb * 128;
    const int brow = ti.e * a.b_group_rows + ti.n0;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    if constexpr (BN == 256)
      load_b256_kmajor(&a.mapB0, k0, brow, sB, bar);
    else
      tma_load_2d(sB, &a.mapB0, k0, brow, bar);
    bulk_load(sSF, sf_atom(a.sfA, (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * a.kt_a + kb), 512, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (a.b_group_rows / 128) + ti.n0 / 128;
    bulk_load(sSF + 512, sf_atom(a.sfB0, wrow * a.kt_b + kb), 512, bar);
    if constexpr (BN == 256) bulk_load(sSF + 1024, sf_atom(a.sfB0, (wrow + 1) * a.kt_b + kb), 512, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    constexpr int kHalf = BN / 2;
    const bool valid = r < ti.rows;
    const bool pad = !valid && r < ti.rows_pad;
    const int lane = r & 31;
    const int wslot = group * 4 + (r >> 5);
    uint8_t* st = kStaged ? stage_base(extra) + wslot * 3 * kStage64WarpBytes : nullptr;
    uint64_t* hbar = kStaged ? reinterpret_cast<uint64_t*>(stage_base(extra) + kStageBytes) + wslot
                             : nullptr;
    const int64_t row = static_cast<int64_t>(ti.m0) + ((valid || pad) ? r : 0);
    const int F = a.ld0;
    const int c0 = group * kHalf;
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(a.in0) + row * 2 * F + ti.n0;
    __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(a.out0) + row * 2 * F + ti.n0;
    __nv_bfloat16* aw = static_cast<__nv_bfloat16*>(a.out1) + row * F + ti.n0;
    uint8_t* dhq = static_cast<uint8_t*>(a.out3) + row * 2 * F;
    const int64_t atom_row = (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * (2 * F / 128);
    uint8_t* sfq = static_cast<uint8_t*>(a.out4);
    const float w = valid ? __ldg(static_cast<const float*>(a.in1) + row) : 0.f;
    float dw = 0.f;
#pragma unroll 1
    for (int c = c0; c < c0 + kHalf; c += 32) {
      float g[32];
      if constexpr (kStaged) {
        // the warp's 32 rows of h_gate and h_up for columns [c, c + 32) into
        // the first two buffers; every lane's earlier accesses to them are
        // ordered before the asynchronous writes
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = ti.m0 + (r & ~31);
          mbar_arrive_expect_tx(hbar, 2 * kStage64WarpBytes);
          tma_load_2d(st, &a.mapB1, ti.n0 + c, y, hbar);
          tma_load_2d(st + kStage64WarpBytes, &a.mapB1, F + ti.n0 + c, y, hbar);
        }
        tmem_ld32(taddr + c, g);
        const int never = 0;   // this wait is cut short only by its time limit
        if (!mbar_wait_bounded(hbar, static_cast<uint32_t>(((c - c0) >> 5) & 1), &never,
                               a.wait_limit_ns))
          record_timeout(a.status, kWaitEpiLoad);
      } else {
        tmem_ld32(taddr + c, g);
      }
      if (valid) {
        float hg[32], hu[32], dhg[32], dhu[32], awv[32];
        if constexpr (kStaged) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 ug = *reinterpret_cast<const uint4*>(st + stage64_off(lane, q));
            const uint4 uu = *reinterpret_cast<const uint4*>(st + kStage64WarpBytes + stage64_off(lane, q));
            unpack_bf16x2(ug.x, hg[8 * q + 0], hg[8 * q + 1]);
            unpack_bf16x2(ug.y, hg[8 * q + 2], hg[8 * q + 3]);
            unpack_bf16x2(ug.z, hg[8 * q + 4], hg[8 * q + 5]);
            unpack_bf16x2(ug.w, hg[8 * q + 6], hg[8 * q + 7]);
            unpack_bf16x2(uu.x, hu[8 * q + 0], hu[8 * q + 1]);
            unpack_bf16x2(uu.y, hu[8 * q + 2], hu[8 * q + 3]);
            unpack_bf16x2(uu.z, hu[8 * q + 4], hu[8 * q + 5]);
            unpack_bf16x2(uu.w, hu[8 * q + 6], hu[8 * q + 7]);
          }
        } else {
          load_bf16x16(h + c, *reinterpret_cast<float(*)[16]>(hg));
          load_bf16x16(h + c + 16, *reinterpret_cast<float(*)[16]>(hg + 16));
          load_bf16x16(h + F + c, *reinterpret_cast<float(*)[16]>(hu));
          load_bf16x16(h + F + c + 16, *reinterpret_cast<float(*)[16]>(hu + 16));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float s = sigmoidf_fast(hg[i]);
          const float silu = hg[i] * s;
          const float act = silu * hu[i];
          dw = fmaf(g[i], act, dw);
          const float da = w * g[i];
          dhg[i] = da * hu[i] * s * (1.0f + hg[i] * (1.0f - s));
          dhu[i] = da * silu;
          awv[i] = w * act;
        }
        if constexpr (kStaged) {
          stage64_bf16x16(st, lane, 0, dhg);
          stage64_bf16x16(st, lane, 1, dhg + 16);
          stage64_bf16x16(st + kStage64WarpBytes, lane, 0, dhu);
          stage64_bf16x16(st + kStage64WarpBytes, lane, 1, dhu + 16);
          stage64_bf16x16(st + 2 * kStage64WarpBytes, lane, 0, awv);
          stage64_bf16x16(st + 2 * kStage64WarpBytes, lane, 1, awv + 16);
        } else {
          store_bf16x16(dh + c, *reinterpret_cast<float(*)[16]>(dhg));
          store_bf16x16(dh + c + 16, *reinterpret_cast<float(*)[16]>(dhg + 16));
          store_bf16x16(dh + F + c, *reinterpret_cast<float(*)[16]>(dhu));
          store_bf16x16(dh + F + c + 16, *reinterpret_cast<float(*)[16]>(dhu + 16));
          store_bf16x16(aw + c, *reinterpret_cast<float(*)[16]>(awv));
          store_bf16x16(aw + c + 16, *reinterpret_cast<float(*)[16]>(awv + 16));
        }
        const int cg = ti.n0 + c;           // gate column; up column = F + cg
        mx_block_store(dhg, dhq + cg, sfq + (atom_row + cg / 128) * 512 + sf_atom_offset(r, (cg >> 5) & 3));
        mx_block_store(dhu, dhq + F + cg,
                       sfq + (atom_row + (F + cg) / 128) * 512 + sf_atom_offset(r, ((F + cg) >> 5) & 3));
      } else if (kStaged) {
        const float z[16] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f,
                             0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int o = 0; o < 3; ++o) {
          stage64_bf16x16(st + o * kStage64WarpBytes, lane, 0, z);
          stage64_bf16x16(st + o * kStage64WarpBytes, lane, 1, z);
        }
      } else if (pad) {
#pragma unroll
        for (int q = 0; q < 32; q += 8) {
          st_global_v4(dh + c + q, 0u, 0u, 0u, 0u);
          st_global_v4(dh + F + c + q, 0u, 0u, 0u, 0u);
          st_global_v4(aw + c + q, 0u, 0u, 0u, 0u);
        }
      }
      if constexpr (kStaged) {
        const bool w_row = valid || pad;
        stage64_flush(st, lane, w_row ? dh + c : nullptr, false);
        stage64_flush(st + kStage64WarpBytes, lane, w_row ? dh + F + c : nullptr, false);
        stage64_flush(st + 2 * kStage64WarpBytes, lane, w_row ? aw + c : nullptr, false);
      }
    }
    if (valid)
      static_cast<float*>(a.out2)[row * (a.n_tiles * kEpiGroups) + (ti.n0 / BN) * kEpiGroups +
                                  group] = dw;
  }
};


// B6 in MXFP8: A = dh E4M3 [P, 2F] (each half quantised along F); B = W_gate
// then W_up quantised along F ([E*H, F], K-major); 128 x 256 tiles, scatter
// epilogue.
struct GateUpDgradMXProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kMX = true;
  static constexpr size_t kExtraSmem = kStage64Smem;
  static constexpr int kEpiGroups = 2;
  struct Frag {
    float v[128];
  };

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile_mx(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    const int k0 = kb * 128;
    const int brow = ti.e * a.b_group_rows + ti.n0;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    bulk_load(sSF, sf_atom(a.sfA, (static_cast<int64_t>(__ldg(a.mtile_off + ti.e)) + ti.mt) * a.kt_a + kb), 512, bar);
    const int64_t wrow = static_cast<int64_t>(ti.e) * (2 * a.n_tiles) + ti.n0 / 128;
    const bool up = k0 >= a.k_half;
    const uint8_t* sfb = up ? a.sfB1 : a.sfB0;
    const int kbw = up ? kb - a.kt_b : kb;
    load_b256_kmajor(up ? &a.mapB1 : &a.mapB0, up ? k0 - a.k_half : k0, brow, sB, bar);
    bulk_load(sSF + 512, sf_atom(sfb, wrow * a.kt_b + kbw), 512, bar);
    bulk_load(sSF + 1024, sf_atom(sfb, (wrow + 1) * a.kt_b + kbw), 512, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue_load(const GemmArgs&, const TileInfo&, uint32_t taddr, int,
                                    int group, Frag& f) {
    tmem_ld128(taddr + 128 * group, f.v);
  }
  MOE_DEV static void epilogue_store(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     Frag& f, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    const int lane = r & 31;
    uint8_t* st = stage64_of(extra, r, group);
    __nv_bfloat16* dst = nullptr;
    if (valid) {
      const int slot = __ldg(static_cast<const int*>(a.in1) + row);
      dst = static_cast<__nv_bfloat16*>(a.out0) + static_cast<int64_t>(slot) * a.ld0 + ti.n0 +
            128 * group;
      MOE_CHECK_INDEX(a.status, kCheckScatterRow, slot, a.T * a.top_k, dst = nullptr);
    }
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      stage64_bf16x16(st, lane, 0, f.v + c);
      stage64_bf16x16(st, lane, 1, f.v + c + 16);
      stage64_flush(st, lane, valid ? dst + c : nullptr, false);
    }
  }
};


// Weight gradients in MXFP8 over the padded token layout (both operands
// MN-major, quantised along tokens per expert segment); 128 x 256 tiles.
//   Down:    A = w*a [P_pad, F] (M = F), B = dY_perm [P_pad, H] (N = H) -> dW_down [E, F, H]
//   Gate/up: A = x_perm [P_pad, H] (M = H), B = dh [P_pad, 2F] (N = 2F) -> dW_gate, dW_up
// B's two 128-column atoms of a k-tile are adjacent: one 1 KB scale copy.
template <bool kGateUp>
struct WgradMXProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = true;
  static constexpr bool kBMN = true;
  static constexpr bool kMX = true;
  static constexpr size_t kExtraSmem = kStage64Smem;
  static constexpr int kEpiGroups = 2;
  struct Frag {
    float v[128];
  };

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_k_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_k_tile_mx(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    const int kt = ti.kb0 + kb;
    const int krow = 128 * kt;
    tma_load_2d(sA, &a.mapA, ti.m0, krow, bar);
    load_b256_mnmajor(&a.mapB0, ti.n0, krow, sB, bar);
    bulk_load(sSF, sf_atom(a.sfA, static_cast<int64_t>(kt) * a.m_tiles + ti.mt), 512, bar);
    bulk_load(sSF + 512, sf_atom(a.sfB0, static_cast<int64_t>(kt) * (2 * a.n_tiles) + ti.n0 / 128),
              1024, bar);
  }
  // (buffer, element index) of column gc of output row r
  MOE_DEV static void out_loc(const GemmArgs& a, const TileInfo& ti, int r, int gc, void*& base,
                              int64_t& idx) {
    if (kGateUp) {
      const int F = a.ld0;
      base = gc < F ? a.out0 : a.out1;
      idx = (static_cast<int64_t>(ti.e) * a.M + ti.m0 + r) * F + (gc < F ? gc : gc - F);
    } else {
      base = a.out0;
      idx = (static_cast<int64_t>(ti.e) * a.M + ti.m0 + r) * a.ld0 + gc;
    }
  }
  MOE_DEV static void epilogue_empty(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     uint8_t*) {
    if (r >= ti.rows) return;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    void* base;
    int64_t idx;
    out_loc(a, ti, r, ti.n0 + 128 * group, base, idx);   // 128 columns never straddle F
    for (int c = 0; c < 128; c += 16) wgrad_zero16(base, idx + c, acc);
  }
  MOE_DEV static void epilogue_load(const GemmArgs&, const TileInfo&, uint32_t taddr, int,
                                    int group, Frag& f) {
    tmem_ld128(taddr + 128 * group, f.v);
  }
  MOE_DEV static void epilogue_store(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     Frag& f, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    const int lane = r & 31;
    uint8_t* st = stage64_of(extra, r, group);
    void* base;
    int64_t idx;
    out_loc(a, ti, r, ti.n0 + 128 * group, base, idx);   // 128 columns never straddle F
    if (acc) {
      float* dst = static_cast<float*>(base) + idx;
#pragma unroll
      for (int c = 0; c < 128; c += 16) {
        stage64_f32x16(st, lane, f.v + c);
        stage64_flush(st, lane, valid ? dst + c : nullptr, true);
      }
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(base) + idx;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        stage64_bf16x16(st, lane, 0, f.v + c);
        stage64_bf16x16(st, lane, 1, f.v + c + 16);
        stage64_flush(st, lane, valid ? dst + c : nullptr, false);
      }
    }
  }
};


// Dense MXFP8 GEMM for moe_gemm_mxfp8: A [M, K] and B [N, K] E4M3 (K-major),
// atoms (m-tile * kt + k-tile) and (n-tile * kt + k-tile); D fp32 [M, N].
struct DenseMXProblem {
  static constexpr int BN = 128;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kMX = true;
  static constexpr size_t kExtraSmem = 0;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return dense_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) {
    TileInfo ti = dense_tile(a, t, BN);
    ti.num_kb = (a.K + 127) / 128;
    return ti;
  }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load_mx(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                              uint8_t* sB, uint8_t* sSF, uint64_t* bar) {
    tma_load_2d(sA, &a.mapA, kb * 128, ti.m0, bar);
    tma_load_2d(sB, &a.mapB0, kb * 128, ti.n0, bar);
    bulk_load(sSF, sf_atom(a.sfA, static_cast<int64_t>(ti.mt) * a.kt_a + kb), 512, bar);
    bulk_load(sSF + 512, sf_atom(a.sfB0, static_cast<int64_t>(ti.n0 / BN) * a.kt_b + kb), 512, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t*) {
    const bool valid = r < ti.rows;
    float* p = static_cast<float*>(a.out0) + (static_cast<int64_t>(ti.m0) + r) * a.ld0 + ti.n0;
#pragma unroll 1
    for (int c = group * 64; c < group * 64 + 64; c += 16) {
      float v[16];
      tmem_ld16(taddr + c, v);
      tmem_ld_wait();
      if (valid) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          st_global_v4(p + c + i, __float_as_uint(v[i]), __float_as_uint(v[i + 1]),
                       __float_as_uint(v[i + 2]), __float_as_uint(v[i + 3]));
      }
    }
  }
};

}  // namespace moe
