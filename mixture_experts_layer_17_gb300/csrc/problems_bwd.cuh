// Backward-pass GEMMs of the MoE layer and the dense test GEMM, as policies of
// the tcgen05 engine.  Notation as in problems.cuh.
#pragma once

#include "problems.cuh"

namespace moe {

// ------------------------------------------------------------------------
// B2 + B3 + B4: down dgrad g = dY_perm · W_down^T with the fused epilogue
//   a  = silu(h_g) * h_u                 (recomputed from the saved h)
//   dw partial = sum_f g * a             (router-weight gradient, one partial
//                                         per 128/256-column tile)
//   da = w * g;  dh_g = da * h_u * silu'(h_g);  dh_u = da * silu(h_g)
//   aw = w * a                           (A operand of the down wgrad)
//   mapA  = dY_perm [P, H] K-major, box {64, 128}
//   mapB0 = W_down as [E*F, H] K-major, box {64, BN}
//   in0 = h bf16 [P, 2F];  in1 = w_row f32 [P]
//   out0 = dh bf16 [P, 2F];  out1 = aw bf16 [P, F];
//   out2 = dw_part f32 [P, 2 * n_tiles] (one partial per n-tile and column half)
//   ld0 = F;  K = H;  n_tiles = F / BN;  b_group_rows = F
//   mapB1 (kStaged) = h [P, 2F] in 32 x 32 boxes with the 64-byte swizzle
// ------------------------------------------------------------------------
template <int BN_, bool kStaged = false>
struct DownDgradProblem {
  static constexpr int BN = BN_;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  // kStaged (the CTA-pair version): each epilogue warp owns one pair of 2 KB
  // buffers (1024-byte aligned, hence up to 1 KB of lead-in) and an mbarrier.
  // Per 32-column step, TMA brings the warp's 32 rows of h_gate and h_up into
  // the pair (64-byte swizzle, the stage64 layout); every thread keeps its row
  // of both as packed words, then dh_gate and dh_up, and after them w*a, are
  // staged in the same pair and leave by TMA stores (maps mapC0 over dh and
  // mapC1 over w*a, the same 32 x 32 boxes), after which the next step's h
  // is loaded.  One pair per warp (32 KB in all)
  // leaves room for six operand stages; a second pair, to load the next h
  // during the step, would cost a stage, and measured 2% slower at the 235B
  // shape (the h wait is under a sixth of the epilogue's time per tile).
  static constexpr size_t kStageBytes = 8 * 2 * kStage64WarpBytes;
  static constexpr size_t kExtraSmem = kStaged ? 1024 + kStageBytes + 8 * sizeof(uint64_t) : 0;
  static constexpr int kEpiGroups = 2;
  // an even number of steps per warp and tile, so the parity of the warp's
  // barrier follows the step index in every tile
  static_assert(!kStaged || (BN / 2 / 32) % 2 == 0, "an even number of h steps per tile");

  MOE_DEV static uint8_t* stage_base(uint8_t* extra) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(extra) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  }

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t* extra) {
    if constexpr (kStaged) {
      if (threadIdx.x == 0) {
        uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base(extra) + kStageBytes);
        for (int w = 0; w < 8; ++w) mbar_init(bars + w, 1);
        fence_mbar_init();
      }
    }
  }
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = kb * kBK;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    tma_load_2d(sB, &a.mapB0, k0, ti.e * a.b_group_rows + ti.n0, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  // SwiGLU backward of 16 columns: g, the saved h (gate and up, packed) ->
  // dh_gate, dh_up, w*a; dw accumulates sum g * a
  MOE_DEV static void swiglu_bwd16(const float* g, const uint32_t* gw, const uint32_t* uw, float w,
                                   float& dw, float* dhg, float* dhu, float* awv) {
    float hg[16], hu[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      unpack_bf16x2(gw[i], hg[2 * i], hg[2 * i + 1]);
      unpack_bf16x2(uw[i], hu[2 * i], hu[2 * i + 1]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float s = sigmoidf_fast(hg[i]);
      const float silu = hg[i] * s;
      const float act = silu * hu[i];
      dw = fmaf(g[i], act, dw);
      const float da = w * g[i];
      dhg[i] = da * hu[i] * s * (1.0f + hg[i] * (1.0f - s));
      dhu[i] = da * silu;
      awv[i] = w * act;
    }
  }

  // kStaged: one thread = one row, one column half, 32 columns per step
  MOE_DEV static void epilogue_staged(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                      int r, int group, uint8_t* extra) {
    constexpr int kHalf = BN / 2;
    constexpr int kSteps = kHalf / 32;
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
    const float w = valid ? __ldg(static_cast<const float*>(a.in1) + row) : 0.f;
    const int never = 0;   // the h waits are cut short only by their time limit
    // h_gate and h_up of step s (columns c0 + 32 s ..) into the warp's pair;
    // every lane's earlier accesses to the pair are ordered before the writes
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
      uint8_t* st = buf;
      if (!mbar_wait_bounded(hbar, static_cast<uint32_t>(step) & 1u, &never,
                             a.wait_limit_ns))
        record_timeout(a.status, kWaitEpiLoad);
      uint32_t gw[16], uw[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 ug = *reinterpret_cast<const uint4*>(st + stage64_off(lane, q));
        const uint4 uu =
            *reinterpret_cast<const uint4*>(st + kStage64WarpBytes + stage64_off(lane, q));
        gw[4 * q] = ug.x; gw[4 * q + 1] = ug.y; gw[4 * q + 2] = ug.z; gw[4 * q + 3] = ug.w;
        uw[4 * q] = uu.x; uw[4 * q + 1] = uu.y; uw[4 * q + 2] = uu.z; uw[4 * q + 3] = uu.w;
      }
      uint32_t awp[16];   // w*a of the step's 32 columns, packed bf16
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float g[16];
        tmem_ld16(taddr + c + 16 * half, g);
        tmem_ld_wait();
        float dhg[16], dhu[16], awv[16];
        if (valid) {
          swiglu_bwd16(g, gw + 8 * half, uw + 8 * half, w, dw, dhg, dhu, awv);
        } else {
          // zeros for the padded rows (and for rows nobody writes)
#pragma unroll
          for (int i = 0; i < 16; ++i) dhg[i] = dhu[i] = awv[i] = 0.f;
        }
        stage64_bf16x16(st, lane, half, dhg);
        stage64_bf16x16(st + kStage64WarpBytes, lane, half, dhu);
#pragma unroll
        for (int i = 0; i < 8; ++i) awp[8 * half + i] = pack_bf16x2(awv[2 * i], awv[2 * i + 1]);
      }
      // dh_gate and dh_up, then w*a, leave by TMA stores (a.mapC0, a.mapC1: the
      // stage64 layout is the 64-byte swizzle of a 32 x 32 box).  Segments
      // are 64-row aligned, so the warp's 32 rows lie wholly inside the
      // expert's padded segment (valid and padding rows) or wholly outside.
      const bool slab_in = (r & ~31) < ti.rows_pad;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && slab_in) {
        tma_store_2d(&a.mapC0, st, ti.n0 + c, y);
        tma_store_2d(&a.mapC0, st + kStage64WarpBytes, F + ti.n0 + c, y);
        bulk_commit();
        bulk_wait_read0();
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(st + stage64_off(lane, q)) =
            make_uint4(awp[4 * q], awp[4 * q + 1], awp[4 * q + 2], awp[4 * q + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && slab_in) {
        tma_store_2d(&a.mapC1, st, ti.n0 + c, y);
        bulk_commit();
        bulk_wait_read0();
      }
      __syncwarp();
      if (step + 1 < kSteps) load_h(step + 1);
    }
    // one router-weight partial per (row, n-tile, column half)
    if (valid)
      static_cast<float*>(a.out2)[row * (a.n_tiles * kEpiGroups) + (ti.n0 / BN) * kEpiGroups +
                                  group] = dw;
  }

  // Unstaged (single-CTA tiles): one thread = one row, one column half.  The
  // global loads of the saved h for chunk c + 16 are issued before chunk c is
  // computed, so their latency overlaps the arithmetic and stores of chunk c.
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    if constexpr (kStaged) {
      epilogue_staged(a, ti, taddr, r, group, extra);
      return;
    }
    constexpr int kHalf = BN / 2;
    const bool valid = r < ti.rows;
    // rows past the expert's tokens but inside its padded segment: dh and w*a
    // are weight-gradient operands there, so they must read as zero
    const bool pad = !valid && r < ti.rows_pad;
    const int64_t row = static_cast<int64_t>(ti.m0) + ((valid || pad) ? r : 0);
    const int F = a.ld0;
    const int c0 = group * kHalf;
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(a.in0) + row * 2 * F + ti.n0;
    __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(a.out0) + row * 2 * F + ti.n0;
    __nv_bfloat16* aw = static_cast<__nv_bfloat16*>(a.out1) + row * F + ti.n0;
    const float w = valid ? __ldg(static_cast<const float*>(a.in1) + row) : 0.f;
    float dw = 0.f;
    uint4 ng0 = make_uint4(0, 0, 0, 0), ng1 = ng0, nu0 = ng0, nu1 = ng0;
    if (valid) {
      ng0 = ld_global_v4(h + c0);
      ng1 = ld_global_v4(h + c0 + 8);
      nu0 = ld_global_v4(h + F + c0);
      nu1 = ld_global_v4(h + F + c0 + 8);
    }
#pragma unroll 1
    for (int c = c0; c < c0 + kHalf; c += 16) {
      const uint4 g0 = ng0, g1 = ng1, u0 = nu0, u1 = nu1;
      if (valid && c + 16 < c0 + kHalf) {
        ng0 = ld_global_v4(h + c + 16);
        ng1 = ld_global_v4(h + c + 24);
        nu0 = ld_global_v4(h + F + c + 16);
        nu1 = ld_global_v4(h + F + c + 24);
      }
      float g[16];
      tmem_ld16(taddr + c, g);
      tmem_ld_wait();
      if (valid) {
        float dhg[16], dhu[16], awv[16];
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        swiglu_bwd16(g, gw, uw, w, dw, dhg, dhu, awv);
        store_bf16x16(dh + c, dhg);
        store_bf16x16(dh + F + c, dhu);
        store_bf16x16(aw + c, awv);
      } else if (pad) {
        st_global_v4(dh + c, 0u, 0u, 0u, 0u);
        st_global_v4(dh + c + 8, 0u, 0u, 0u, 0u);
        st_global_v4(dh + F + c, 0u, 0u, 0u, 0u);
        st_global_v4(dh + F + c + 8, 0u, 0u, 0u, 0u);
        st_global_v4(aw + c, 0u, 0u, 0u, 0u);
        st_global_v4(aw + c + 8, 0u, 0u, 0u, 0u);
      }
    }
    // one router-weight partial per (row, n-tile, column half)
    if (valid)
      static_cast<float*>(a.out2)[row * (a.n_tiles * kEpiGroups) + (ti.n0 / BN) * kEpiGroups +
                                  group] = dw;
  }
};

// ------------------------------------------------------------------------
// B6 (+ B7 first half): gate/up dgrad dx_perm = dh_g · W_gate^T + dh_u · W_up^T
// over K = 2F; the epilogue scatters rows to the (token, slot)-ordered scratch.
//   mapA  = dh [P, 2F] K-major, box {64, 128}
//   mapB0 = W_gate as [E*H, F] K-major, box {64, 256};  mapB1 = W_up, same
//   in1 = row_slot i32 [P];  out0 = scratch bf16 [P, H]
//   ld0 = H;  K = 2F;  k_half = F;  n_tiles = H / 256;  b_group_rows = H
// ------------------------------------------------------------------------
struct GateUpDgradProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr size_t kExtraSmem = kStageSmem;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_m_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_m_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = kb * kBK;
    const int brow = ti.e * a.b_group_rows + ti.n0;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    if (k0 < a.k_half)
      tma_load_2d(sB, &a.mapB0, k0, brow, bar);
    else
      tma_load_2d(sB, &a.mapB1, k0 - a.k_half, brow, bar);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const int lane = r & 31;
    uint8_t* st = stage_of(extra, r, group);
    const int64_t row = static_cast<int64_t>(ti.m0) + r;
    __nv_bfloat16* dst = nullptr;
    if (valid) {
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
        stage_bf16x16(st, lane, q, v);
      }
      stage_flush(st, lane, valid ? dst + c0 : nullptr);
    }
  }
};

// ------------------------------------------------------------------------
// B5: down wgrad dW_down[e] = (w·a)_e^T · dY_perm_e, K = tokens of expert e.
//   mapA  = aw [P, F] MN-major, box {64, 64}      (M = F)
//   mapB0 = dY_perm [P, H] MN-major, box {64, 64} (N = H)
//   out0 = dW_down bf16 [E, F, H];  M = F;  N = H;  ld0 = H
// ------------------------------------------------------------------------
struct DownWgradProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = true;
  static constexpr bool kBMN = true;
  static constexpr size_t kExtraSmem = kStageSmem;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_k_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_k_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int krow = ti.krow0 + kb * kBK;
#pragma unroll
    for (int c = 0; c < 2; ++c) tma_load_2d(sA + c * kChunkBytes, &a.mapA, ti.m0 + 64 * c, krow, bar);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_2d(sB + c * kChunkBytes, &a.mapB0, ti.n0 + 64 * c, krow, bar);
  }
  MOE_DEV static int64_t out_idx(const GemmArgs& a, const TileInfo& ti, int r) {
    return (static_cast<int64_t>(ti.e) * a.M + ti.m0 + r) * a.ld0 + ti.n0;
  }
  MOE_DEV static void epilogue_empty(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     uint8_t*) {
    if (r >= ti.rows) return;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    for (int c = group * (BN / 2); c < (group + 1) * (BN / 2); c += 16)
      wgrad_zero16(a.out0, out_idx(a, ti, r) + c, acc);
  }
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    const int lane = r & 31;
    uint8_t* st = stage_of(extra, r, group);
    const int64_t idx = valid ? out_idx(a, ti, r) : 0;
    const int step = acc ? 32 : 64;           // columns per 128-byte staged row
#pragma unroll 1
    for (int c0 = group * (BN / 2); c0 < (group + 1) * (BN / 2); c0 += step) {
#pragma unroll 1
      for (int q = 0; q < step / 16; ++q) {
        float v[16];
        tmem_ld16(taddr + c0 + 16 * q, v);
        tmem_ld_wait();
        if (acc)
          stage_f32x16(st, lane, q, v);
        else
          stage_bf16x16(st, lane, q, v);
      }
      if (acc)
        stage_flush_add_f32(st, lane, valid ? static_cast<float*>(a.out0) + idx + c0 : nullptr);
      else
        stage_flush(st, lane, valid ? static_cast<__nv_bfloat16*>(a.out0) + idx + c0 : nullptr);
    }
  }
};

// ------------------------------------------------------------------------
// B8: gate/up wgrad dW_gate[e] = x_perm_e^T · dh_g,e and dW_up[e] = x_perm_e^T ·
// dh_u,e, K = tokens of expert e; N runs over the 2F columns of dh.
//   mapA  = x_perm [P, H] MN-major, box {64, 64}  (M = H)
//   mapB0 = dh [P, 2F] MN-major, box {64, 64}     (N = 2F)
//   out0 = dW_gate, out1 = dW_up bf16 [E, H, F];  M = H;  N = 2F;  ld0 = F
// ------------------------------------------------------------------------
struct GateUpWgradProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = true;
  static constexpr bool kBMN = true;
  static constexpr size_t kExtraSmem = kStageSmem;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return grouped_k_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return grouped_k_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int krow = ti.krow0 + kb * kBK;
#pragma unroll
    for (int c = 0; c < 2; ++c) tma_load_2d(sA + c * kChunkBytes, &a.mapA, ti.m0 + 64 * c, krow, bar);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_2d(sB + c * kChunkBytes, &a.mapB0, ti.n0 + 64 * c, krow, bar);
  }
  // (buffer, element index) of the 16-column chunk at global column gc of the
  // [gate | up] range (F is a multiple of 128, so no chunk straddles the two)
  MOE_DEV static void out_loc(const GemmArgs& a, const TileInfo& ti, int r, int gc, void*& base,
                              int64_t& idx) {
    const int F = a.ld0;
    base = gc < F ? a.out0 : a.out1;
    idx = (static_cast<int64_t>(ti.e) * a.M + ti.m0 + r) * F + (gc < F ? gc : gc - F);
  }
  MOE_DEV static void epilogue_empty(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     uint8_t*) {
    if (r >= ti.rows) return;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    for (int c = group * (BN / 2); c < (group + 1) * (BN / 2); c += 16) {
      void* base;
      int64_t idx;
      out_loc(a, ti, r, ti.n0 + c, base, idx);
      wgrad_zero16(base, idx, acc);
    }
  }
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t* extra) {
    const bool valid = r < ti.rows;
    const bool acc = (a.flags & kGemmAccumF32) != 0;
    const int lane = r & 31;
    uint8_t* st = stage_of(extra, r, group);
    const int step = acc ? 32 : 64;           // columns per 128-byte staged row
#pragma unroll 1
    for (int c0 = group * (BN / 2); c0 < (group + 1) * (BN / 2); c0 += step) {
#pragma unroll 1
      for (int q = 0; q < step / 16; ++q) {
        float v[16];
        tmem_ld16(taddr + c0 + 16 * q, v);
        tmem_ld_wait();
        if (acc)
          stage_f32x16(st, lane, q, v);
        else
          stage_bf16x16(st, lane, q, v);
      }
      void* base;
      int64_t idx;
      out_loc(a, ti, r, ti.n0 + c0, base, idx);   // 64 columns never straddle the gate / up split
      if (acc)
        stage_flush_add_f32(st, lane, valid ? static_cast<float*>(base) + idx : nullptr);
      else
        stage_flush(st, lane, valid ? static_cast<__nv_bfloat16*>(base) + idx : nullptr);
    }
  }
};

// ------------------------------------------------------------------------
// B10 (weight half): dW_r^T = dl^T · x as a split-K GEMM over the tokens;
// each split writes an fp32 partial that a small kernel reduces and transposes.
//   mapA  = dl^T [E, T_pad] K-major bf16, box {64, 128}  (M = E, rows >= E zero)
//   mapB0 = x [T, H] MN-major, box {64, 64}               (N = H)
//   out0 = partials f32 [k_split, E, H];  M = E;  N = H;  K = T;  ld0 = H
// ------------------------------------------------------------------------
struct RouterWgradProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = true;
  static constexpr size_t kExtraSmem = 0;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return split_k_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return split_k_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = (ti.kb0 + kb) * kBK;
    tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_2d(sB + c * kChunkBytes, &a.mapB0, ti.n0 + 64 * c, k0, bar);
  }
  MOE_DEV static float* out_row(const GemmArgs& a, const TileInfo& ti, int r) {
    return static_cast<float*>(a.out0) +
           (static_cast<int64_t>(ti.e) * a.M + ti.m0 + r) * a.ld0 + ti.n0;
  }
  MOE_DEV static void epilogue_empty(const GemmArgs& a, const TileInfo& ti, int r, int group,
                                     uint8_t*) {
    if (r >= ti.rows) return;
    float* p = out_row(a, ti, r);
    for (int c = group * (BN / 2); c < (group + 1) * (BN / 2); c += 4)
      st_global_v4(p + c, 0u, 0u, 0u, 0u);
  }
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t*) {
    const bool valid = r < ti.rows;
    float* p = valid ? out_row(a, ti, r) : nullptr;
#pragma unroll 1
    for (int c = group * (BN / 2); c < (group + 1) * (BN / 2); c += 16) {
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

// ------------------------------------------------------------------------
// Dense GEMM D[M, N] (fp32) = sum_k A(m, k) B(n, k) for moe_gemm_bf16.
//   A K-major: [M, K], box {64, 128};  A MN-major: [K, M], box {64, 64}
//   B K-major: [N, K], box {64, 256};  B MN-major: [K, N], box {64, 64}
//   out0 = D f32 [M, N];  ld0 = N
// ------------------------------------------------------------------------
template <bool A_MN, bool B_MN>
struct DenseProblem {
  static constexpr int BN = 256;
  static constexpr bool kAMN = A_MN;
  static constexpr bool kBMN = B_MN;
  static constexpr size_t kExtraSmem = 0;
  static constexpr int kEpiGroups = 2;

  MOE_DEV static int num_tiles(const GemmArgs& a) { return dense_num_tiles(a); }
  MOE_DEV static TileInfo tile(const GemmArgs& a, int t) { return dense_tile(a, t, BN); }
  MOE_DEV static void init_extra(const GemmArgs&, uint8_t*) {}
  MOE_DEV static void load(const GemmArgs& a, const TileInfo& ti, int kb, uint8_t* sA,
                           uint8_t* sB, uint64_t* bar) {
    const int k0 = kb * kBK;
    if (A_MN) {
      tma_load_2d(sA, &a.mapA, ti.m0, k0, bar);
      tma_load_2d(sA + kChunkBytes, &a.mapA, ti.m0 + 64, k0, bar);
    } else {
      tma_load_2d(sA, &a.mapA, k0, ti.m0, bar);
    }
    if (B_MN) {
#pragma unroll
      for (int c = 0; c < 4; ++c) tma_load_2d(sB + c * kChunkBytes, &a.mapB0, ti.n0 + 64 * c, k0, bar);
    } else {
      tma_load_2d(sB, &a.mapB0, k0, ti.n0, bar);
    }
  }
  MOE_DEV static void epilogue_empty(const GemmArgs&, const TileInfo&, int, int, uint8_t*) {}
  MOE_DEV static void epilogue(const GemmArgs& a, const TileInfo& ti, uint32_t taddr, int r,
                               int group, uint8_t*) {
    const bool valid = r < ti.rows;
    float* p = static_cast<float*>(a.out0) + (static_cast<int64_t>(ti.m0) + r) * a.ld0 + ti.n0;
#pragma unroll 1
    for (int c = group * (BN / 2); c < (group + 1) * (BN / 2); c += 16) {
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
