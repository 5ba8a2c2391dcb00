// Persistent, warp-specialised tcgen05 GEMM engine for the MoE layer.
//
// One CTA per SM walks a static list of 128 x BN output tiles.  Per CTA:
//   warp 0      TMA producer: fills a ring of STAGES shared-memory stages
//               (A: 128 x 64 bf16, B: BN x 64 bf16, 128-byte swizzle);
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//               into a double-buffered TMEM accumulator and commits stage and
//               accumulator barriers;
//   warps 2..   epilogue (one or two warpgroups): tcgen05.ld of the
//               accumulator (thread = output row, warpgroup = column half),
//               the problem's fused element-wise work, and global stores.
// The problem policy (struct P) supplies the tile schedule, the TMA loads and
// the epilogue; the engine is shared by every GEMM of the layer:
//   router logits + top-k, expert gate/up with SwiGLU, expert down with the
//   weighted scatter, their dgrads (SwiGLU backward, router-weight gradient)
//   and their wgrads over ragged per-expert token counts.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace moe {

constexpr int kBM = 128;          // rows of an output tile (TMEM lanes)
constexpr int kBK = 64;           // bf16 elements of K per stage (128 bytes)
// Threads of a CTA: warp 0 (TMA), warp 1 (MMA) and kEpiGroups warpgroups of
// epilogue warps; group g owns columns [g*BN/G, (g+1)*BN/G) of every tile.
template <class P>
constexpr int gemm_threads() { return 64 + 128 * P::kEpiGroups; }
constexpr uint32_t kChunkBytes = 64 * 128;   // one MN-major 64 x 64 bf16 chunk

struct GemmArgs {
  CUtensorMap mapA;
  CUtensorMap mapB0;
  CUtensorMap mapB1;
  // MXFP8 CTA pairs: the scale atoms of A and B as [atoms, 128] u32 tensors
  // (one-atom boxes), loaded by TMA so that the peer's copies complete on the
  // leader's barrier
  CUtensorMap mapSFA;
  CUtensorMap mapSFB;
  CUtensorMap mapSFB1;   // the second B operand's atoms (gate/up dgrad: W_up)
  // staged epilogue outputs leaving by TMA stores (the down dgrads' dh and w*a)
  CUtensorMap mapC0;
  CUtensorMap mapC1;
  int M;               // dense: output rows; grouped-K / split-K: output rows per group
  int N;               // output columns
  int K;               // reduction length (dense, grouped-M, split-K)
  int n_tiles;         // ceil(N / BN)
  int m_tiles;         // grouped-K / split-K: ceil(M / 128)
  int num_groups;      // experts
  int k_split;         // split-K: number of K chunks
  int kb_per_split;    // split-K: k-blocks per chunk
  int b_group_rows;    // rows of one expert in B's 2-D tensor map
  int k_half;          // gate/up dgrad: K index where B switches from W_gate to W_up
  const int* offsets;  // [E + 1] padded segment starts of the internal permuted layout
  const int* counts;   // [E] valid rows of every segment
  const int* mtile_off;     // [E + 1] prefix of ceil(count / 128)
  const int* mtile2_off;    // [E + 1] prefix of ceil(count / 256) (CTA-pair tiles)
  const int* group_order;   // grouped-K: experts in processing order
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  void* out4;
  const void* in0;
  const void* in1;
  const void* in2;
  int64_t T;
  int E;
  int top_k;
  int ld0;
  int ld1;
  const uint8_t* sfA;   // MXFP8: scale atoms of A
  const uint8_t* sfB0;  // MXFP8: scale atoms of B (first map)
  const uint8_t* sfB1;  // MXFP8: scale atoms of B (second map)
  int kt_a;             // MXFP8: K-tiles (of 128) per atom row of A
  int kt_b;             // MXFP8: K-tiles (of 128) per atom row of B
  DeviceStatus* status;
  uint64_t wait_limit_ns;
  uint32_t flags;      // kGemmInjectWait, kGemmAccumF32
};

constexpr uint32_t kGemmInjectWait = 2u;   // wait on a barrier nothing signals (timeout test)
constexpr uint32_t kGemmAccumF32 = 4u;     // weight gradients: out += acc in fp32

struct TileInfo {
  int e;        // expert (group), -1 for dense problems
  int m0;       // first output row (grouped-M: row of the permuted layout)
  int n0;       // first output column
  int rows;     // valid output rows in the tile
  int rows_pad; // rows of the tile inside the expert's padded segment (>= rows)
  int kb0;      // first k-block
  int num_kb;   // k-blocks
  int k_last;   // valid K rows in the last k-block (grouped-K)
  int krow0;    // first K row of the group (grouped-K)
  int mt;       // m-tile index (dense)
};

// ------------------------------------------------------------ schedules

// Grouped-M: expert e's segment starts at the padded offset offsets[e] and
// holds counts[e] rows followed by zero rows up to offsets[e+1]; its m-tiles
// are numbered from mtile_off[e].  Tiles are ordered (expert, n-tile, m-tile)
// so that CTAs running at the same time share the expert's weight panel in L2.
MOE_DEV int grouped_m_num_tiles(const GemmArgs& a) {
  return __ldg(a.mtile_off + a.num_groups) * a.n_tiles;
}

MOE_DEV TileInfo grouped_m_tile(const GemmArgs& a, int t, int BN) {
  const int q = t / a.n_tiles;
  int lo = 0, hi = a.num_groups - 1;   // largest e with mtile_off[e] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.mtile_off + mid) <= q) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mbase = __ldg(a.mtile_off + e);
  const int mt_e = __ldg(a.mtile_off + e + 1) - mbase;
  const int local = t - mbase * a.n_tiles;
  const int nt = local / mt_e;
  const int mt = local - nt * mt_e;
  const int r0 = __ldg(a.offsets + e);
  TileInfo ti;
  ti.e = e;
  ti.m0 = r0 + mt * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(kBM, r0 + __ldg(a.counts + e) - ti.m0);
  ti.rows_pad = min(kBM, __ldg(a.offsets + e + 1) - ti.m0);
  ti.kb0 = 0;
  ti.num_kb = (a.K + kBK - 1) / kBK;
  ti.k_last = kBK;
  ti.krow0 = 0;
  ti.mt = mt;
  return ti;
}

// Grouped-K (weight gradients): every expert owns m_tiles x n_tiles output
// tiles; its K range is its padded segment [offsets[e], offsets[e+1]), whole
// 64-row blocks whose rows past counts[e] are zero.
MOE_DEV int grouped_k_num_tiles(const GemmArgs& a) {
  return a.num_groups * a.m_tiles * a.n_tiles;
}

MOE_DEV TileInfo grouped_k_tile(const GemmArgs& a, int t, int BN) {
  const int per = a.m_tiles * a.n_tiles;
  const int gi = t / per;
  const int local = t - gi * per;
  const int mt = local / a.n_tiles;
  const int nt = local - mt * a.n_tiles;
  const int e = a.group_order != nullptr ? __ldg(a.group_order + gi) : gi;
  const int r0 = __ldg(a.offsets + e);
  TileInfo ti;
  ti.e = e;
  ti.m0 = mt * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(kBM, a.M - ti.m0);
  ti.rows_pad = ti.rows;
  ti.kb0 = 0;
  ti.num_kb = (__ldg(a.offsets + e + 1) - r0) / kBK;
  ti.k_last = kBK;
  ti.krow0 = r0;
  ti.mt = mt;
  return ti;
}

// CTA-pair variants: 256-row tiles.  Grouped-M pair tiles of expert e are
// numbered from mtile2_off[e]; grouped-K uses m_tiles = M / 256.
MOE_DEV int grouped_m_num_tiles_pair(const GemmArgs& a) {
  return __ldg(a.mtile2_off + a.num_groups) * a.n_tiles;
}

MOE_DEV TileInfo grouped_m_tile_pair(const GemmArgs& a, int t, int BN) {
  const int q = t / a.n_tiles;
  int lo = 0, hi = a.num_groups - 1;   // largest e with mtile2_off[e] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.mtile2_off + mid) <= q) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mbase = __ldg(a.mtile2_off + e);
  const int mt_e = __ldg(a.mtile2_off + e + 1) - mbase;
  const int local = t - mbase * a.n_tiles;
  const int nt = local / mt_e;
  const int mt = local - nt * mt_e;
  const int r0 = __ldg(a.offsets + e);
  TileInfo ti;
  ti.e = e;
  ti.m0 = r0 + mt * 2 * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(2 * kBM, r0 + __ldg(a.counts + e) - ti.m0);
  ti.rows_pad = min(2 * kBM, __ldg(a.offsets + e + 1) - ti.m0);
  ti.kb0 = 0;
  ti.num_kb = (a.K + kBK - 1) / kBK;
  ti.k_last = kBK;
  ti.krow0 = 0;
  ti.mt = mt;
  return ti;
}

MOE_DEV TileInfo grouped_k_tile_pair(const GemmArgs& a, int t, int BN) {
  TileInfo ti = grouped_k_tile(a, t, BN);
  ti.m0 = ti.mt * 2 * kBM;
  ti.rows = min(2 * kBM, a.M - ti.m0);
  ti.rows_pad = ti.rows;
  return ti;
}

MOE_DEV int dense_num_tiles(const GemmArgs& a) {
  return ((a.M + kBM - 1) / kBM) * a.n_tiles;
}

MOE_DEV TileInfo dense_tile(const GemmArgs& a, int t, int BN) {
  const int mt = t / a.n_tiles;
  const int nt = t - mt * a.n_tiles;
  TileInfo ti;
  ti.e = -1;
  ti.m0 = mt * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(kBM, a.M - ti.m0);
  ti.rows_pad = ti.rows;
  ti.kb0 = 0;
  ti.num_kb = (a.K + kBK - 1) / kBK;
  ti.k_last = kBK;
  ti.krow0 = 0;
  ti.mt = mt;
  return ti;
}

// Split-K: tiles (split, m-tile, n-tile); each split reduces kb_per_split
// k-blocks and writes an fp32 partial.
MOE_DEV int split_k_num_tiles(const GemmArgs& a) { return a.k_split * a.m_tiles * a.n_tiles; }

MOE_DEV TileInfo split_k_tile(const GemmArgs& a, int t, int BN) {
  const int per = a.m_tiles * a.n_tiles;
  const int ks = t / per;
  const int local = t - ks * per;
  const int mt = local / a.n_tiles;
  const int nt = local - mt * a.n_tiles;
  const int total_kb = (a.K + kBK - 1) / kBK;
  TileInfo ti;
  ti.e = ks;
  ti.m0 = mt * kBM;
  ti.n0 = nt * BN;
  ti.rows = min(kBM, a.M - ti.m0);
  ti.rows_pad = ti.rows;
  ti.kb0 = ks * a.kb_per_split;
  ti.num_kb = max(0, min(total_kb, ti.kb0 + a.kb_per_split) - ti.kb0);
  ti.k_last = kBK;
  ti.krow0 = 0;
  ti.mt = mt;
  return ti;
}

// ------------------------------------------------------------ engine

// Problems with `static constexpr bool kMX = true` run on MXFP8 operands.
template <class P, class = void>
struct IsMX : std::false_type {};
template <class P>
struct IsMX<P, std::void_t<decltype(P::kMX)>> : std::integral_constant<bool, P::kMX> {};

// Problems with `static constexpr bool kPair = true` run as CTA pairs: a
// cluster of two CTAs computes a 256-row tile with M = 256 tcgen05.mma of
// cta_group::2; each CTA stages its own 128 rows of A and half of B.
template <class P, class = void>
struct IsPair : std::false_type {};
template <class P>
struct IsPair<P, std::void_t<decltype(P::kPair)>> : std::integral_constant<bool, P::kPair> {};

// Problems that define `struct Frag` free their TMEM accumulator early: the
// epilogue copies its fragment to registers (P::epilogue_load), releases the
// accumulator to the MMA warp, then computes and stores from registers
// (P::epilogue_store).
template <class P, class = void>
struct HasFrag : std::false_type {};
template <class P>
struct HasFrag<P, std::void_t<typename P::Frag>> : std::true_type {};

// Stage geometry.  bf16: a stage holds K = 64 (128 bytes per row).  MXFP8: a
// stage holds K = 128 E4M3 (128 bytes per row) plus one 512-byte scale atom
// for A and BN/128 for B.  128-wide MXFP8 tiles double-buffer the accumulator
// (TMEM columns [0, 256)) and copy the stage's scales to columns 256 +
// 8*stage (A) and +4 (B); 256-wide tiles have one accumulator (columns
// [0, 256), released early by epilogues with a Frag, else after the
// epilogue) and scales at 256 + 16*stage
// (A), +4 (B rows 0..127) and +8 (B rows 128..255).  kAccBufs: accumulators,
// kAccStride TMEM columns apart; sf_col(stage): the stage's first scale column.
template <class P, bool MX = IsMX<P>::value, bool PAIR = IsPair<P>::value>
struct StageCfg {
  static constexpr int BN = P::BN;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kSFBytes = 0;
  // as many stages as the problem's own shared memory leaves room for
  static constexpr int kFit =
      static_cast<int>((232448 - 1024 - 256 - P::kExtraSmem) / (kABytes + kBBytes));
  static constexpr int kWant = (BN >= 256) ? 4 : (BN >= 128 ? 6 : 8);
  static constexpr int kStages = kWant < kFit ? kWant : kFit;
  static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  static constexpr int kAccBufs = 2;
  static constexpr uint32_t kAccStride = BN;
};

// CTA pair, bf16: per CTA a stage holds its 128 rows of A and BN/2 rows of B
// (32 KB for BN = 256), so six stages fit.
template <class P>
struct StageCfg<P, false, true> {
  static constexpr int BN = P::BN;
  static_assert(BN == 256, "CTA-pair tiles are 256 x 256");
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = (BN / 2) * kBK * 2;
  static constexpr uint32_t kSFBytes = 0;
  static constexpr int kFit =
      static_cast<int>((232448 - 1024 - 256 - P::kExtraSmem) / (kABytes + kBBytes));
  static constexpr int kStages = 6 < kFit ? 6 : kFit;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kAccBufs = 2;
  static constexpr uint32_t kAccStride = BN;
};

template <class P>
struct StageCfg<P, true, false> {
  static constexpr int BN = P::BN;
  static_assert(BN == 128 || BN == 256, "MXFP8 tiles are 128 x 128 or 128 x 256");
  static constexpr uint32_t kABytes = kBM * 128;
  static constexpr uint32_t kBBytes = BN * 128;
  static constexpr uint32_t kSFBytes = 512 + (BN / 128) * 512;
  static constexpr int kFit =
      static_cast<int>((232448 - 1024 - 256 - P::kExtraSmem) / (kABytes + kBBytes + kSFBytes));
  static constexpr int kWant = BN == 256 ? 4 : 6;
  static constexpr int kStages = kWant < kFit ? kWant : kFit;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSFCol0 = 256;
  static constexpr uint32_t kSFStride = BN == 256 ? 16 : 8;   // TMEM columns per stage
  static constexpr int kAccBufs = BN == 256 ? 1 : 2;
  static constexpr uint32_t kAccStride = BN;
  MOE_DEV static uint32_t sf_col(int stage) { return kSFCol0 + kSFStride * stage; }
};

// CTA pair, MXFP8: per CTA a stage holds its 128 rows of A and BN/2 rows of
// B (K = 128 E4M3 each) and the scale atoms the problem loads (P::kSFAtoms
// of 512 bytes: A's first, then B's), copied to 4 * kSFAtoms TMEM columns.
//   BN = 256: one accumulator (columns [0, 256)), the stages' scales from
//             column 256 on;
//   BN = 192: two accumulators (columns [0, 192) and [256, 448)), the stages'
//             scales in the gaps [192, 256) and [448, 512).
template <class P>
struct StageCfg<P, true, true> {
  static constexpr int BN = P::BN;
  static_assert(BN == 256 || BN == 192, "MXFP8 CTA-pair tiles are 256 x 256 or 256 x 192");
  static constexpr uint32_t kABytes = kBM * 128;
  static constexpr uint32_t kBBytes = (BN / 2) * 128;
  static constexpr uint32_t kSFBytes = 512 * P::kSFAtoms;
  static constexpr int kFit =
      static_cast<int>((232448 - 1024 - 256 - P::kExtraSmem) / (kABytes + kBBytes + kSFBytes));
  static constexpr int kStages = 6 < kFit ? 6 : kFit;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSFStride = 4 * P::kSFAtoms;
  static constexpr int kAccBufs = BN == 192 ? 2 : 1;
  static constexpr uint32_t kAccStride = 256;
  // scale slots per gap of the 192-wide layout
  static constexpr int kGapSlots = static_cast<int>((256 - BN) / kSFStride);
  static_assert(BN == 256 ? 256 + kSFStride * kStages <= kTmemCols : kStages <= 2 * kGapSlots,
                "scale slots exceed TMEM");
  MOE_DEV static uint32_t sf_col(int stage) {
    if constexpr (BN == 256) {
      return 256 + kSFStride * stage;
    } else {
      return stage < kGapSlots ? BN + kSFStride * stage : 256 + BN + kSFStride * (stage - kGapSlots);
    }
  }
};

template <class P>
constexpr size_t gemm_smem_bytes() {
  using C = StageCfg<P>;
  return 1024 + static_cast<size_t>(C::kStages) * (C::kABytes + C::kBBytes + C::kSFBytes) + 256 +
         P::kExtraSmem;
}

template <class P>
__global__ void __launch_bounds__(gemm_threads<P>(), 1) gemm_kernel(const __grid_constant__ GemmArgs args) {
  constexpr int BN = P::BN;
  constexpr bool kMX = IsMX<P>::value;
  using C = StageCfg<P>;
  constexpr int S = C::kStages;
  constexpr uint32_t kA = C::kABytes;
  constexpr uint32_t kB = C::kBBytes;
  constexpr uint32_t kSF = C::kSFBytes;
  constexpr bool kPair = IsPair<P>::value;
  constexpr uint32_t kIdesc = kMX ? make_idesc_mxf8(kPair ? 2 * kBM : kBM, BN, P::kAMN, P::kBMN)
                                  : make_idesc_bf16(kPair ? 2 * kBM : kBM, BN, P::kAMN, P::kBMN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kA;
  uint8_t* sSF = sB + S * kB;              // MXFP8 only: [S][kSF] scale atoms
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sSF + S * kSF);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* tfull_bar = empty_bar + S;     // [2]
  uint64_t* tempty_bar = tfull_bar + 2;    // [2]
  uint64_t* drain_bar = tempty_bar + 2;    // [1]
  uint64_t* never_bar = drain_bar + 1;     // [1] nothing ever arrives here
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* zero_flag = abort_flag + 1;   // stays 0: drains are never cut short
  uint8_t* extra = reinterpret_cast<uint8_t*>(full_bar) + 256;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: rank in the cluster (0 issues the MMAs) and the pair's tiles
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int t_first = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int t_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar + s, 1);
      mbar_init(empty_bar + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar + i, 1);
      mbar_init(tempty_bar + i, (kPair ? 2 : 1) * 4 * P::kEpiGroups);
    }
    mbar_init(drain_bar, 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    *zero_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    if constexpr (kPair)
      tmem_alloc_pair(tmem_holder, C::kTmemCols);
    else
      tmem_alloc(tmem_holder, C::kTmemCols);
  }
  P::init_extra(args, extra);
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // the peer's barriers are initialised
  tc_fence_after();
  // the prologue above overlaps the previous kernel's tail; from here on
  // global memory is read and written
  grid_dependency_wait();
  const uint32_t tmem_base = *tmem_holder;
  const int num_tiles = P::num_tiles(args);
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&args.mapA);
      prefetch_tmap(&args.mapB0);
      prefetch_tmap(&args.mapB1);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, parity_mask = 0;
      bool ok = true;
      for (int t = t_first; t < num_tiles && ok; t += t_step) {
        const TileInfo ti = P::tile(args, t);
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait_bounded(empty_bar + stage, phase ^ 1u, abort_flag, limit)) {
            if (!*abort_flag) record_timeout(args.status, kWaitProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if constexpr (kPair && kMX) {
            // both halves and their scale atoms complete on the leader's full barrier
            if (rank == 0) mbar_arrive_expect_tx(full_bar + stage, 2 * (kA + kB + kSF));
            P::load_mx_pair(args, ti, kb, static_cast<int>(rank), sA + stage * kA,
                            sB + stage * kB, sSF + stage * kSF, map_to_rank(full_bar + stage, 0));
          } else if constexpr (kPair) {
            // both halves complete on the leader's full barrier
            if (rank == 0) mbar_arrive_expect_tx(full_bar + stage, 2 * (kA + kB));
            P::load_pair(args, ti, kb, static_cast<int>(rank), sA + stage * kA, sB + stage * kB,
                         map_to_rank(full_bar + stage, 0));
          } else if constexpr (kMX) {
            mbar_arrive_expect_tx(full_bar + stage, kA + kB + kSF);
            P::load_mx(args, ti, kb, sA + stage * kA, sB + stage * kB, sSF + stage * kSF,
                       full_bar + stage);
          } else {
            mbar_arrive_expect_tx(full_bar + stage, kA + kB);
            P::load(args, ti, kb, sA + stage * kA, sB + stage * kB, full_bar + stage);
          }
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let every load already in flight land before the CTA exits (a
        // pair's second CTA cannot observe its loads: it waits 200 us)
        if (!kPair || rank == 0) {
          for (int s = 0; s < S; ++s) {
            if (issued_mask & (1u << s)) {
              mbar_wait_bounded(full_bar + s, (parity_mask >> s) & 1u, zero_flag, 100000000ull);
            }
          }
        } else {
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1 && (!kPair || rank == 0)) {
    // ------------------------------------------------ MMA issuer (pair: leader only)
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool committed_any = false;
    for (int t = t_first; t < num_tiles && ok; t += t_step) {
      const TileInfo ti = P::tile(args, t);
      if (ti.num_kb == 0) continue;
      if (!mbar_wait_bounded(tempty_bar + acc, acc_phase ^ 1u, abort_flag, limit)) {
        if (!*abort_flag) record_timeout(args.status, kWaitMmaTmemEmpty);
        *abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * C::kAccStride;
      for (int kb = 0; kb < ti.num_kb; ++kb) {
        if (!mbar_wait_bounded(full_bar + stage, phase, abort_flag, limit)) {
          if (!*abort_flag) record_timeout(args.status, kWaitMmaFull);
          *abort_flag = 1;
          ok = false;
          break;
        }
        if constexpr (kMX && kPair) {
          if (lane == 0) {
            tc_fence_after();
            // the stage's scale atoms -> the pair's TMEM (the problem's slot
            // layout: A's atom at sf_t, B's from sf_t + 4), then four K = 32
            // block-scaled M = 256 MMAs
            const uint32_t sf_t = tmem_base + C::sf_col(stage);
#pragma unroll
            for (int i = 0; i < P::kSFAtoms; ++i)
              sf_copy_to_tmem_pair(sf_t + 4 * i, sSF + stage * kSF + 512 * i);
            const uint32_t a_base = smem_u32(sA + stage * kA);
            const uint32_t b_base = smem_u32(sB + stage * kB);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t adesc =
                  P::kAMN ? make_smem_desc(a_base + k * 4096, 16384, 1024)
                          : make_smem_desc(a_base + k * 32, 16, 1024);
              const uint64_t bdesc =
                  P::kBMN ? make_smem_desc(b_base + k * 4096, 16384, 1024)
                          : make_smem_desc(b_base + k * 32, 16, 1024);
              mma_mxf8_pair(d_tmem, adesc, bdesc, idesc_with_sf_id(kIdesc, k), sf_t, sf_t + 4,
                            (kb > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit_pair(empty_bar + stage, 0x3);   // frees the stage in both CTAs
            committed_any = true;
          }
        } else if constexpr (kMX) {
          if (lane == 0) {
            tc_fence_after();
            // scales of this stage -> TMEM (4-column aligned slots), then four
            // K = 32 block-scaled MMAs selecting the K-block with sf_id
            const uint32_t sf_t = tmem_base + C::sf_col(stage);
            sf_copy_to_tmem(sf_t, sSF + stage * kSF);
            sf_copy_to_tmem(sf_t + 4, sSF + stage * kSF + 512);
            if constexpr (BN == 256) sf_copy_to_tmem(sf_t + 8, sSF + stage * kSF + 1024);
            const uint32_t a_base = smem_u32(sA + stage * kA);
            const uint32_t b_base = smem_u32(sB + stage * kB);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t adesc =
                  P::kAMN ? make_smem_desc(a_base + k * 4096, 16384, 1024)
                          : make_smem_desc(a_base + k * 32, 16, 1024);
              const uint64_t bdesc =
                  P::kBMN ? make_smem_desc(b_base + k * 4096, 16384, 1024)
                          : make_smem_desc(b_base + k * 32, 16, 1024);
              mma_mxf8(d_tmem, adesc, bdesc, idesc_with_sf_id(kIdesc, k), sf_t, sf_t + 4,
                       (kb > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(empty_bar + stage);
            committed_any = true;
          }
        } else {
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * kA);
            const uint32_t b_base = smem_u32(sB + stage * kB);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint64_t adesc =
                  P::kAMN ? make_smem_desc(a_base + k * 2048, kChunkBytes, 1024)
                          : make_smem_desc(a_base + k * 32, 16, 1024);
              const uint64_t bdesc =
                  P::kBMN ? make_smem_desc(b_base + k * 2048, kChunkBytes, 1024)
                          : make_smem_desc(b_base + k * 32, 16, 1024);
              if constexpr (kPair)
                mma_bf16_pair(d_tmem, adesc, bdesc, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
              else
                mma_bf16(d_tmem, adesc, bdesc, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
            }
            if constexpr (kPair)
              mma_commit_pair(empty_bar + stage, 0x3);   // frees the stage in both CTAs
            else
              mma_commit(empty_bar + stage);
            committed_any = true;
          }
        }
        __syncwarp();
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        const bool inject = (args.flags & kGemmInjectWait) != 0 && t == t_first;
        if (!inject) {
          if constexpr (kPair)
            mma_commit_pair(tfull_bar + acc, 0x3);
          else
            mma_commit(tfull_bar + acc);
        }
      }
      __syncwarp();
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // wait until every MMA this thread issued has completed
    if (lane == 0 && committed_any) {
      if constexpr (kPair)
        mma_commit_pair(drain_bar, 0x1);
      else
        mma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, zero_flag, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (warps 2..)
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int group = (warp - 2) >> 2;       // column group of this warp
    const int r = quarter * 32 + lane;       // row of the tile this thread owns
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool first = true;
    for (int t = t_first; t < num_tiles; t += t_step) {
      TileInfo ti = P::tile(args, t);
      if constexpr (kPair) {
        // this CTA owns rows [128 * rank, 128 * rank + 128) of the pair's tile,
        // its 128-row m-tile within the group being 2 * (pair m-tile) + rank
        ti.m0 += 128 * static_cast<int>(rank);
        ti.mt = 2 * ti.mt + static_cast<int>(rank);
        ti.rows = max(0, min(kBM, ti.rows - 128 * static_cast<int>(rank)));
        ti.rows_pad = max(0, min(kBM, ti.rows_pad - 128 * static_cast<int>(rank)));
      }
      if (ti.num_kb == 0) {
        P::epilogue_empty(args, ti, r, group, extra);
        continue;
      }
      if (first && (args.flags & kGemmInjectWait) != 0) {
        // test hook: a wait on a barrier that nothing signals
        if (!mbar_wait_bounded(never_bar, 0, abort_flag, limit)) {
          record_timeout(args.status, kWaitInjected);
          *abort_flag = 1;
          break;
        }
      }
      first = false;
      if (!mbar_wait_bounded(tfull_bar + acc, acc_phase, abort_flag, limit)) {
        if (!*abort_flag) record_timeout(args.status, kWaitEpiTmemFull);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_off + static_cast<uint32_t>(acc) * C::kAccStride;
      if constexpr (HasFrag<P>::value) {
        // early release: fragment -> registers, accumulator back to the MMA
        // warp, then the element-wise work and the stores
        typename P::Frag f;
        P::epilogue_load(args, ti, taddr, r, group, f);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair && rank != 0)
            mbar_arrive_remote(map_to_rank(tempty_bar + acc, 0));
          else
            mbar_arrive(tempty_bar + acc);
        }
        P::epilogue_store(args, ti, r, group, f, extra);
      } else {
        P::epilogue(args, ti, taddr, r, group, extra);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair && rank != 0)
            mbar_arrive_remote(map_to_rank(tempty_bar + acc, 0));
          else
            mbar_arrive(tempty_bar + acc);
        }
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // the peer is done with this CTA's smem and TMEM
  tc_fence_after();
  if (warp == 0) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace moe
