// C ABI of libmoe (declared in include/moe.h): argument validation, workspace
// layout, TMA descriptor creation and the launch sequences of the routing,
// forward and backward passes.  Host code only; all arithmetic runs in the
// kernels of gemm_*.cu and elementwise.cu.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"
#include "moe.h"

namespace {

using namespace moe;

// ---------------------------------------------------------------- device info

struct DevInfo {
  bool queried = false;
  bool supported = false;
  int sms = 0;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

moe_status_t current_device(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.queried) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    d.queried = true;
  }
  *out = d;
  return d.supported ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

// ---------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major matrix [rows, cols] with the given row
// stride; boxes of box_rows x box_cols (box_cols * 2 = 128 bytes) with the
// 128-byte swizzle.  Reads outside the matrix return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
              uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte (E4M3) tensor map: [rows, cols] bytes, 128 x 128-byte boxes with
// the 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An array of 512-byte MXFP8 scale atoms as a 2-D u32 tensor [atoms, 128]
// with one-atom boxes: CTA pairs load atoms by TMA (the peer's loads complete
// on the leader's barrier).  Atom rows past `atoms` read as zeros.
bool make_map_atoms(CUtensorMap* m, const void* base, uint64_t atoms) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {128, atoms};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- profiling

struct Pending {
  const char* name;
  cudaEvent_t start;
  cudaEvent_t stop;
};
struct Totals {
  int64_t launches = 0;
  double ms = 0.0;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::string g_prof_only;   // when not empty, only launches with this label are timed
std::vector<Pending> g_pending;
std::map<std::string, Totals> g_totals;
std::vector<std::string> g_names;   // storage behind names handed out by moe_profile_read
std::atomic<int64_t> g_launches{0};

// Runs one kernel launch: optional profiling events, launch counting, and
// (with MOE_FLAG_SYNC_CHECK) a synchronising error check.
template <class Fn>
moe_status_t run(const char* name, cudaStream_t s, uint32_t flags, Fn&& fn) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bool prof;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    prof = g_prof_on && (g_prof_only.empty() || g_prof_only == name);
  }
  if (prof) {
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
      return MOE_ERR_CUDA;
    cudaEventRecord(e0, s);
  }
  cudaError_t err = fn();
  g_launches.fetch_add(1);
  if (prof) {
    cudaEventRecord(e1, s);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_pending.push_back({name, e0, e1});
  }
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  if (flags & MOE_FLAG_SYNC_CHECK) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

#define MOE_TRY(expr)                 \
  do {                                \
    moe_status_t _st = (expr);        \
    if (_st != MOE_OK) return _st;    \
  } while (0)

// ---------------------------------------------------------------- layout

constexpr uint64_t kNormalWaitNs = 2000000000ull;   // 2 s: no legitimate wait comes close
constexpr uint64_t kTestWaitNs = 20000000ull;       // 20 ms for MOE_FLAG_TEST_TIMEOUT

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  }
};

int next_pow2_at_least16(int v) {
  int p = 16;
  while (p < v) p <<= 1;
  return p;
}

struct Layout {
  int64_t T, P, T_pad;
  int64_t Pa;        // rows of the padded internal layout: P + 64 * E (64-row aligned segments)
  bool pair_gu_fwd, pair_down_fwd, pair_down_dgrad, pair_gu_dgrad, pair_down_wgrad, pair_gu_wgrad;
  // MXFP8 GEMMs on CTA pairs (block-scaled cta_group::2); the down dgrad,
  // bound by its epilogue, stays on single-CTA tiles
  bool mx_pair_gu_fwd, mx_pair_down_fwd, mx_pair_gu_dgrad, mx_pair_down_wgrad, mx_pair_gu_wgrad;
  // MXFP8 down dgrad on 256 x 192 CTA-pair tiles (two accumulators per CTA)
  bool mx_pair_down_dgrad;
  int H, F, E, k;
  int ntiles;        // router tiles of 128 tokens
  int router_bn;     // N of the router GEMM (power of two >= E, >= 16)
  int dgrad_bn;      // N tile of the bf16 down dgrad (256 if F % 256 == 0, else 128)
  int mx_dgrad_bn;   // N tile of the MXFP8 down dgrad (128: double-buffered, staged outputs)
  int nparts;        // dw partials per row = 2 * F / dgrad_bn
  int wr_split, wr_kbps, wr_mtiles, wr_ntiles;
  // forward / route workspace
  size_t f_status, f_hist, f_base, f_a, f_scratch;
  size_t r_wrt, r_row_slot, r_w_row, r_mtile, r_order, r_poff, r_mtile2, r_slotpad, f_total;
  // context
  size_t c_idx, c_w, c_counts, c_offsets, c_perm, c_slot, c_row_slot, c_w_row, c_mtile,
      c_order, c_wrt, c_xperm, c_h, c_poff, c_mtile2, c_slotpad, c_total;
  size_t c_xt, c_sxt;   // mxfp8: x along the tokens (E4M3, atoms) instead of x_perm
  // backward workspace
  size_t b_status, b_dyp, b_dh, b_aw, b_dwp, b_dl, b_dlt, b_scratch, b_wrp, b_total;
  // MOE_FLAG_RECOMPUTE: x_perm and h live in the forward workspace, and the
  // backward re-dispatches x and recomputes h into its own workspace
  bool recompute;
  size_t f_xperm, f_h, b_xperm, b_h;
  size_t bq_rx, bs_rx, bq_ra, bs_ra, bq_rwgu, bs_rwgu;   // MXFP8 recompute operands
  // MXFP8 buffers (E4M3 data + scale atoms); present only when the precision uses them
  int64_t mt_max;    // upper bound of the 128-row m-tiles (= K-tiles of the padded token layout)
  size_t fq_x, fs_x, fq_a, fs_a, fq_wgu, fs_wgu, fq_wd, fs_wd;
  size_t bq_dy, bs_dy, bq_wdh, bs_wdh, bq_dh, bs_dh, bq_wg, bs_wg, bq_wu, bs_wu;
  size_t bq_awt, bs_awt, bq_dyt, bs_dyt, bq_xt, bs_xt, bq_dht, bs_dht;
  // prepared MXFP8 weights (moe_prepare_weights): every orientation the GEMMs read
  bool prepared;
  size_t q_gu_h, qs_gu_h, q_d_f, qs_d_f, q_g_f, qs_g_f, q_u_f, qs_u_f, q_d_h, qs_d_h, q_total;
  size_t qs_d_h192;   // W_down's scales along H in 192-row blocks (F a multiple of 192)
};

Layout make_layout(const moe_config_t& c, int sms) {
  Layout L{};
  L.T = c.T;
  L.H = c.H;
  L.F = c.F;
  L.E = c.E;
  L.k = c.top_k;
  L.P = L.T * L.k;
  L.Pa = L.P + 64ll * L.E;
  L.T_pad = (L.T + 7) / 8 * 8;
  // CTA pairs (256-row tiles, cta_group::2): each CTA stages half of B, so six
  // stages fit and the operand-latency lookahead grows by half; a pair tile
  // of a grouped-M GEMM wastes more rows at the end of each expert.  Measured
  // on the 235B shape (1024 rows per expert), pairs win for every expert GEMM
  // once the epilogue stores go through shared memory (the down dgrad's by
  // 12%; the gate/up forward's by 4.5%).  With 256 rows per expert (the 30B
  // shape) only the two dgrads still gain (2-4%); the wgrads,
  // whose K is then 4 k-blocks per expert, lose 36%, and the forward GEMMs
  // break even.  MOE_FLAG_CTA_PAIRS_ON / _OFF override.
  const bool pairs_on = (c.flags & MOE_FLAG_CTA_PAIRS_ON) != 0;
  const bool pairs_off = (c.flags & MOE_FLAG_CTA_PAIRS_OFF) != 0;
  const bool bf = c.precision != MOE_MXFP8;        // bf16 forward GEMMs
  const bool bb = c.precision == MOE_BF16;         // bf16 backward GEMMs
  const bool big = L.P >= 512ll * L.E;             // experts average >= 512 rows
  const bool mid = L.P >= 256ll * L.E;             // experts average >= 256 rows
  const bool can_pair = sms >= 2;                    // an SM budget of 1 runs single CTAs
  const bool pp = can_pair && !pairs_off && (pairs_on || big);
  const bool pp_dgrad = can_pair && !pairs_off && (pairs_on || mid);
  L.pair_gu_fwd = bf && pp;
  L.pair_down_fwd = bf && pp;
  L.pair_down_dgrad = bb && pp_dgrad && (L.F % 256 == 0);
  L.pair_gu_dgrad = bb && pp_dgrad;
  L.pair_down_wgrad = bb && pp && (L.F % 256 == 0);
  L.pair_gu_wgrad = bb && pp;
  // MXFP8 GEMMs run as CTA pairs only on request (MOE_FLAG_CTA_PAIRS_ON):
  // their 256-column tiles keep one TMEM accumulator beside the scale
  // factors, and at the 235B shape the pair versions measured 4-9% slower
  // than the single-CTA ones (the accumulator's hand-over waits on both
  // CTAs' epilogues)
  const bool mf = c.precision == MOE_MXFP8;        // MXFP8 forward GEMMs
  const bool mb = c.precision != MOE_BF16;         // MXFP8 backward GEMMs
  const bool mxp = can_pair && pairs_on;
  L.mx_pair_gu_fwd = mf && mxp;
  L.mx_pair_down_fwd = mf && mxp;
  L.mx_pair_gu_dgrad = mb && mxp;
  L.mx_pair_down_wgrad = mb && mxp && (L.F % 256 == 0);
  L.mx_pair_gu_wgrad = mb && mxp;
  // The MXFP8 down dgrad's 256 x 192 pair tiles keep two accumulators per CTA
  // beside the scale slots (128-column single-CTA tiles need 128 B/cycle of
  // operands per SM, these 77); at the 235B shape 1.29 -> 1.09 ms.  Like the
  // bf16 dgrads, they pair once experts average 256 rows.
  L.mx_pair_down_dgrad = mb && can_pair && !pairs_off && (pairs_on || mid) && (L.F % 192 == 0);
  L.recompute = (c.flags & MOE_FLAG_RECOMPUTE) != 0;
  L.prepared = c.precision != MOE_BF16 && c.prepared_weights != nullptr;
  L.ntiles = static_cast<int>((L.T + kBM - 1) / kBM);
  L.router_bn = next_pow2_at_least16(L.E);
  L.dgrad_bn = (L.F % 256 == 0) ? 256 : 128;
  L.mx_dgrad_bn = 128;
  // one router-weight partial per n-tile and epilogue column half (the bf16
  // and MXFP8 down dgrads both use 256-wide tiles when F allows)
  L.nparts = (L.F / (bb ? L.dgrad_bn : (L.mx_pair_down_dgrad ? 192 : L.mx_dgrad_bn))) * 2;
  L.wr_mtiles = (L.E + kBM - 1) / kBM;
  L.wr_ntiles = L.H / 256;
  const int total_kb = static_cast<int>((L.T + kBK - 1) / kBK);
  int split = sms / (L.wr_mtiles * L.wr_ntiles);
  split = split < 1 ? 1 : (split > total_kb ? total_kb : split);
  L.wr_kbps = (total_kb + split - 1) / split;
  L.wr_split = (total_kb + L.wr_kbps - 1) / L.wr_kbps;
  const size_t P = static_cast<size_t>(L.P), T = static_cast<size_t>(L.T);
  const size_t Pa = static_cast<size_t>(L.Pa);
  const size_t H = L.H, F = L.F, E = L.E;

  Carver f;
  L.f_status = f.take(sizeof(DeviceStatus));
  L.f_hist = f.take(sizeof(int) * L.ntiles * E);
  L.f_base = f.take(sizeof(int) * L.ntiles * E);
  L.r_wrt = f.take(2 * E * H);
  L.r_row_slot = f.take(sizeof(int) * Pa);
  L.r_w_row = f.take(sizeof(float) * Pa);
  L.r_mtile = f.take(sizeof(int) * (E + 1));
  L.r_order = f.take(sizeof(int) * E);
  L.r_poff = f.take(sizeof(int) * (E + 1));
  L.r_mtile2 = f.take(sizeof(int) * (E + 1));
  L.r_slotpad = f.take(sizeof(int) * P);
  L.f_a = f.take(2 * Pa * F);
  L.f_scratch = f.take(2 * P * H);
  if (L.recompute) {
    if (c.precision != MOE_MXFP8) L.f_xperm = f.take(2 * Pa * H);   // mxfp8 dispatches to E4M3
    L.f_h = f.take(2 * Pa * 2 * F);
  }
  L.mt_max = (L.P + kBM - 1) / kBM + L.E;
  const size_t mt = static_cast<size_t>(L.mt_max);
  if (c.precision == MOE_MXFP8) {
    L.fq_x = f.take(Pa * H);
    L.fs_x = f.take(mt * (H / 128) * 512);
    L.fq_a = f.take(Pa * F);
    L.fs_a = f.take(mt * (F / 128) * 512);
    if (!L.prepared) {
      L.fq_wgu = f.take(E * H * 2 * F);
      L.fs_wgu = f.take(E * (2 * F / 128) * (H / 128) * 512);
      L.fq_wd = f.take(E * F * H);
      L.fs_wd = f.take(E * (H / 128) * (F / 128) * 512);
    }
  }
  L.f_total = f.off;

  Carver x;
  L.c_idx = x.take(sizeof(int) * P);
  L.c_w = x.take(sizeof(float) * P);
  L.c_counts = x.take(sizeof(int) * E);
  L.c_offsets = x.take(sizeof(int) * (E + 1));
  L.c_perm = x.take(sizeof(int) * P);
  L.c_slot = x.take(sizeof(int) * P);
  L.c_row_slot = x.take(sizeof(int) * Pa);
  L.c_w_row = x.take(sizeof(float) * Pa);
  L.c_mtile = x.take(sizeof(int) * (E + 1));
  L.c_order = x.take(sizeof(int) * E);
  L.c_wrt = x.take(2 * E * H);
  if (!L.recompute) {
    if (c.precision == MOE_MXFP8) {   // what the gate/up wgrad reads of x
      L.c_xt = x.take(128 * mt * H);
      L.c_sxt = x.take(mt * (H / 128) * 512);
    } else {
      L.c_xperm = x.take(2 * Pa * H);
    }
    L.c_h = x.take(2 * Pa * 2 * F);
  }
  L.c_poff = x.take(sizeof(int) * (E + 1));
  L.c_mtile2 = x.take(sizeof(int) * (E + 1));
  L.c_slotpad = x.take(sizeof(int) * P);
  L.c_total = x.off;

  Carver b;
  L.b_status = b.take(sizeof(DeviceStatus));
  if (c.precision == MOE_BF16) L.b_dyp = b.take(2 * Pa * H);   // MXFP8 dispatches dY to E4M3
  L.b_dh = b.take(2 * Pa * 2 * F);
  L.b_aw = b.take(2 * Pa * F);
  L.b_dwp = b.take(sizeof(float) * Pa * L.nparts);
  L.b_dl = b.take(sizeof(float) * P);
  L.b_dlt = b.take(2 * E * static_cast<size_t>(L.T_pad));
  L.b_scratch = b.take(2 * P * H);
  L.b_wrp = b.take(sizeof(float) * L.wr_split * E * H);
  if (L.recompute) {
    if (c.precision != MOE_MXFP8) L.b_xperm = b.take(2 * Pa * H);   // mxfp8 dispatches to E4M3
    L.b_h = b.take(2 * Pa * 2 * F);
    if (c.precision == MOE_MXFP8) {
      L.bq_rx = b.take(Pa * H);
      L.bs_rx = b.take(mt * (H / 128) * 512);
      L.bq_ra = b.take(Pa * F);
      L.bs_ra = b.take(mt * (F / 128) * 512);
      if (!L.prepared) {
        L.bq_rwgu = b.take(E * H * 2 * F);
        L.bs_rwgu = b.take(E * (2 * F / 128) * (H / 128) * 512);
      }
    }
  }
  if (c.precision != MOE_BF16) {
    const size_t Pp = 128 * mt;   // padded token rows
    L.bq_dy = b.take(Pa * H);
    L.bs_dy = b.take(mt * (H / 128) * 512);
    L.bq_dh = b.take(Pa * 2 * F);
    L.bs_dh = b.take(mt * (2 * F / 128) * 512);
    if (!L.prepared) {
      L.bq_wdh = b.take(E * F * H);
      L.bs_wdh = L.mx_pair_down_dgrad ? b.take(E * (F / 192) * 2 * (H / 128) * 512)
                                      : b.take(E * (F / 128) * (H / 128) * 512);
      L.bq_wg = b.take(E * H * F);
      L.bs_wg = b.take(E * (H / 128) * (F / 128) * 512);
      L.bq_wu = b.take(E * H * F);
      L.bs_wu = b.take(E * (H / 128) * (F / 128) * 512);
    }
    L.bq_awt = b.take(Pp * F);
    L.bs_awt = b.take(mt * (F / 128) * 512);
    L.bq_dyt = b.take(Pp * H);
    L.bs_dyt = b.take(mt * (H / 128) * 512);
    if (c.precision == MOE_FP8_BWD || L.recompute) {   // else x along tokens is in ctx
      L.bq_xt = b.take(Pp * H);
      L.bs_xt = b.take(mt * (H / 128) * 512);
    }
    L.bq_dht = b.take(Pp * 2 * F);
    L.bs_dht = b.take(mt * (2 * F / 128) * 512);
  }
  L.b_total = b.off;

  Carver q;   // moe_prepare_weights buffer
  L.q_gu_h = q.take(E * H * 2 * F);
  L.qs_gu_h = q.take(E * (2 * F / 128) * (H / 128) * 512);
  L.q_d_f = q.take(E * F * H);
  L.qs_d_f = q.take(E * (H / 128) * (F / 128) * 512);
  L.q_g_f = q.take(E * H * F);
  L.qs_g_f = q.take(E * (H / 128) * (F / 128) * 512);
  L.q_u_f = q.take(E * H * F);
  L.qs_u_f = q.take(E * (H / 128) * (F / 128) * 512);
  L.q_d_h = q.take(E * F * H);
  L.qs_d_h = q.take(E * (F / 128) * (H / 128) * 512);
  // both layouts of W_down's scales along H, so that the flags of a call may
  // differ from those of the preparation
  L.qs_d_h192 = (F % 192 == 0) ? q.take(E * (F / 192) * 2 * (H / 128) * 512) : 0;
  L.q_total = q.off;
  (void)T;
  return L;
}

moe_status_t validate(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->flags & ~(MOE_FLAG_SYNC_CHECK | MOE_FLAG_TEST_TIMEOUT | MOE_FLAG_CTA_PAIRS_OFF |
                   MOE_FLAG_CTA_PAIRS_ON | MOE_FLAG_RECOMPUTE))
    return MOE_ERR_INVALID_ARG;
  if (c->max_sms < 0) return MOE_ERR_INVALID_ARG;
  if (c->prepared_weights != nullptr &&
      (reinterpret_cast<uintptr_t>(c->prepared_weights) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_CTA_PAIRS_OFF) && (c->flags & MOE_FLAG_CTA_PAIRS_ON))
    return MOE_ERR_INVALID_ARG;
  if (c->precision < MOE_BF16 || c->precision > MOE_FP8_BWD) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->H < 256 || c->H % 256 != 0 || c->H > 65536 || c->F < 128 ||
      c->F % 128 != 0 || c->F > 65536 || c->E < 1 || c->E > 256 || c->top_k < 1 ||
      c->top_k > 16 || c->top_k > c->E)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->T * static_cast<int64_t>(c->top_k) >= (static_cast<int64_t>(1) << 31) - 256)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

GemmArgs base_args(DeviceStatus* st, uint32_t flags) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = st;
  a.wait_limit_ns = kNormalWaitNs;
  a.flags = 0;
  (void)flags;
  return a;
}

int grid_for(int64_t tiles, int sms) {
  if (tiles < 1) return 1;
  return static_cast<int>(tiles < sms ? tiles : sms);
}

// SMs the persistent kernels of a call may use (moe_config_t.max_sms)
int sm_budget(int device_sms, const moe_config_t& c) {
  return (c.max_sms > 0 && c.max_sms < device_sms) ? c.max_sms : device_sms;
}

}  // namespace

namespace {

struct RouteBufs {
  const uint16_t* x;
  const uint16_t* W_r;
  const float* bias;
  float* logits;
  int* idx;
  float* w;
  int* counts;
  int* offsets;
  int* perm;
  int* slot;
  int* row_slot;
  float* w_row;
  int* mtile;
  int* order;
  uint16_t* wrt;
  int* hist;
  int* base;
  DeviceStatus* st;
  int* poff;       // padded segment starts
  int* mtile2;     // pair-tile prefix
  int* slot_pad;   // (t, j) -> row of the padded layout
};

// F1-F5: router GEMM with the fused top-k epilogue, expert scan, permutation.
moe_status_t run_routing(const moe_config_t& c, const Layout& L, const RouteBufs& b, int sms,
                         cudaStream_t s) {
  MOE_TRY(run("transpose_router_weight", s, c.flags,
              [&] { return launch_transpose_bf16(b.W_r, b.wrt, L.H, L.E, s); }));
  GemmArgs a = base_args(b.st, c.flags);
  if (!make_map(&a.mapA, b.x, L.H, L.T, 2ull * L.H, 64, 128) ||
      !make_map(&a.mapB0, b.wrt, L.H, L.E, 2ull * L.H, 64, L.router_bn))
    return MOE_ERR_CUDA;
  a.mapB1 = a.mapB0;
  a.M = static_cast<int>(L.T);
  a.N = L.router_bn;
  a.K = L.H;
  a.n_tiles = 1;
  a.in0 = b.bias;
  a.out0 = b.logits;
  a.out1 = b.idx;
  a.out2 = b.w;
  a.out3 = b.hist;
  a.E = L.E;
  a.top_k = L.k;
  a.T = L.T;
  MOE_TRY(run("router_gemm_topk", s, c.flags, [&] {
    return launch_router_fwd(L.router_bn, a, grid_for(L.ntiles, sms), s);
  }));
  MOE_TRY(run("expert_scan", s, c.flags, [&] {
    return launch_scan(b.hist, L.ntiles, L.E, b.counts, b.offsets, b.poff, b.base, b.mtile,
                       b.mtile2, b.order, s);
  }));
  MOE_TRY(run("permute", s, c.flags, [&] {
    return launch_permute(b.idx, b.w, b.base, b.offsets, b.poff, L.T, L.k, L.E, b.perm, b.slot,
                          b.slot_pad, b.row_slot, b.w_row, b.st, s);
  }));
  return MOE_OK;
}

// The down dgrads' output maps: dh [Pa, 2F] and w*a [Pa, F] bf16 in 32 x 32
// boxes with the 64-byte swizzle, the layout their epilogues stage.
bool make_out_maps(GemmArgs* a, const void* dh, const void* aw, const Layout& L) {
  return make_map(&a->mapC0, dh, 2ull * L.F, L.Pa, 4ull * L.F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) &&
         make_map(&a->mapC1, aw, L.F, L.Pa, 2ull * L.F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

int64_t grouped_m_tile_bound(const Layout& L) { return (L.P + kBM - 1) / kBM + L.E; }
int64_t grouped_m_pair_bound(const Layout& L) { return (L.P + 2 * kBM - 1) / (2 * kBM) + L.E; }

// even grid of at most sms CTAs for `pair_tiles` CTA-pair tiles
int grid_for_pairs(int64_t pair_tiles, int sms) {
  const int64_t cap = sms & ~1;
  const int64_t g = 2 * (pair_tiles < 1 ? 1 : pair_tiles);
  return static_cast<int>(g < cap ? g : cap);
}

bool all_aligned16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr || !aligned(p, 16)) return false;
  return true;
}


// ---------------------------------------------------------------- MXFP8 passes

// F7 + F8 in bf16: the gate/up GEMM with the SwiGLU epilogue, writing a and
// the pre-activations h.  `recompute` names the launch of the backward's
// recomputation (MOE_FLAG_RECOMPUTE).
moe_status_t gate_up_fwd_bf16(const Layout& L, int sms, cudaStream_t s, uint32_t fl,
                              DeviceStatus* st, const uint16_t* xperm, const uint16_t* W_gate,
                              const uint16_t* W_up, const int* poff, const int* counts,
                              const int* mtile, const int* mtile2, uint16_t* act, uint16_t* h,
                              bool recompute) {
  GemmArgs a = base_args(st, fl);
  if (!make_map(&a.mapA, xperm, L.H, L.Pa, 2ull * L.H, 64, 128) ||
      !make_map(&a.mapB0, W_gate, L.F, static_cast<uint64_t>(L.E) * L.H, 2ull * L.F, 64, 64) ||
      !make_map(&a.mapB1, W_up, L.F, static_cast<uint64_t>(L.E) * L.H, 2ull * L.F, 64, 64))
    return MOE_ERR_CUDA;
  a.K = L.H;
  a.N = 2 * L.F;
  a.n_tiles = L.F / 128;
  a.num_groups = L.E;
  a.b_group_rows = L.H;
  a.offsets = poff;
  a.counts = counts;
  a.mtile_off = mtile;
  a.mtile2_off = mtile2;
  a.out0 = act;
  a.out1 = h;
  a.ld0 = L.F;
  if (fl & MOE_FLAG_TEST_TIMEOUT) {
    a.flags = kGemmInjectWait;
    a.wait_limit_ns = kTestWaitNs;
  }
  const char* label = recompute ? "recompute_gate_up_gemm_swiglu" : "gate_up_gemm_swiglu";
  if (L.pair_gu_fwd) {
    const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
    return run(label, s, fl, [&] { return launch_gate_up_fwd_pair(a, grid, s); });
  }
  const int grid = grid_for(grouped_m_tile_bound(L) * a.n_tiles, sms);
  return run(label, s, fl, [&] { return launch_gate_up_fwd(a, grid, s); });
}

// E4M3 operands and scale atoms of the MXFP8 gate/up GEMM
struct MxGateUpBufs {
  uint8_t *xq, *sx, *aq, *sa, *wgu, *swgu;
  bool w_ready = false;   // wgu / swgu prepared by moe_prepare_weights
};

// F7 + F8 in MXFP8: x along H comes quantised from the dispatch (xq / sx);
// W_gate / W_up along H (interleaved per 128 columns) are quantised here
// unless prepared, then the block-scaled gate/up GEMM with SwiGLU whose
// epilogue writes h and quantises a along F from fp32.
moe_status_t gate_up_fwd_mx(const Layout& L, int sms, cudaStream_t s, uint32_t fl,
                            DeviceStatus* st, const uint16_t* W_gate, const uint16_t* W_up,
                            const int* offsets, const int* counts, const int* mtile,
                            const int* mtile2, uint16_t* h, const MxGateUpBufs& q,
                            bool recompute) {
  if (!q.w_ready) {
    MOE_TRY(run(recompute ? "recompute_mx_quant_w_gate_up" : "mx_quant_w_gate_up", s, fl, [&] {
      return launch_quant_cols_gate_up(W_gate, W_up, L.E, L.H, L.F, q.wgu, q.swgu, s);
    }));
  }
  GemmArgs a = base_args(st, fl);
  if (!make_map_u8(&a.mapA, q.xq, L.H, L.Pa, L.H) ||
      !make_map_u8(&a.mapB0, q.wgu, 2ull * L.F, static_cast<uint64_t>(L.E) * L.H, 2ull * L.F))
    return MOE_ERR_CUDA;
  a.mapB1 = a.mapB0;
  a.K = L.H;
  a.N = 2 * L.F;
  a.n_tiles = 2 * L.F / 256;   // 128 x 256 tiles (pairs: 256 x 256)
  a.num_groups = L.E;
  a.b_group_rows = L.H;
  a.offsets = offsets;
  a.counts = counts;
  a.mtile_off = mtile;
  a.mtile2_off = mtile2;
  a.out0 = q.aq;    // a quantised to E4M3 in the epilogue
  a.out1 = h;
  a.out2 = q.sa;    // its scale atoms
  a.ld0 = L.F;
  a.sfA = q.sx;
  a.kt_a = L.H / 128;
  a.sfB0 = q.swgu;
  a.kt_b = L.H / 128;
  if (fl & MOE_FLAG_TEST_TIMEOUT) {
    a.flags = kGemmInjectWait;
    a.wait_limit_ns = kTestWaitNs;
  }
  const char* label = recompute ? "recompute_gate_up_gemm_swiglu_mx" : "gate_up_gemm_swiglu_mx";
  if (L.mx_pair_gu_fwd) {
    if (!make_map_atoms(&a.mapSFA, q.sx, static_cast<uint64_t>(L.mt_max) * (L.H / 128)) ||
        !make_map_atoms(&a.mapSFB, q.swgu,
                        static_cast<uint64_t>(L.E) * (2 * L.F / 128) * (L.H / 128)))
      return MOE_ERR_CUDA;
    const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
    return run(label, s, fl, [&] { return launch_gate_up_fwd_mx_pair(a, grid, s); });
  }
  const int grid = grid_for(((L.P + kBM - 1) / kBM + L.E) * a.n_tiles, sms);
  return run(label, s, fl, [&] { return launch_gate_up_fwd_mx(a, grid, s); });
}

// F7 + F8 and F9 in MXFP8: the gate/up part above, then W_down quantised
// along F and the block-scaled down GEMM with the weighted scatter.
moe_status_t forward_gemms_mx(const Layout& L, int sms, cudaStream_t s, uint32_t fl,
                              DeviceStatus* st, const uint16_t* W_gate, const uint16_t* W_up,
                              const uint16_t* W_down, const int* offsets, const int* counts,
                              const int* mtile, const int* mtile2, const float* w_row,
                              const int* row_slot, uint16_t* h, uint16_t* scratch, void* ws,
                              void* wq) {
  MxGateUpBufs q{at<uint8_t>(ws, L.fq_x), at<uint8_t>(ws, L.fs_x), at<uint8_t>(ws, L.fq_a),
                 at<uint8_t>(ws, L.fs_a), nullptr, nullptr};
  if (wq != nullptr) {
    q.wgu = at<uint8_t>(wq, L.q_gu_h);
    q.swgu = at<uint8_t>(wq, L.qs_gu_h);
    q.w_ready = true;
  } else {
    q.wgu = at<uint8_t>(ws, L.fq_wgu);
    q.swgu = at<uint8_t>(ws, L.fs_wgu);
  }
  uint8_t* aq = q.aq;
  uint8_t* sa = q.sa;
  uint8_t* wd = wq != nullptr ? at<uint8_t>(wq, L.q_d_f) : at<uint8_t>(ws, L.fq_wd);
  uint8_t* swd = wq != nullptr ? at<uint8_t>(wq, L.qs_d_f) : at<uint8_t>(ws, L.fs_wd);
  MOE_TRY(gate_up_fwd_mx(L, sms, s, fl, st, W_gate, W_up, offsets, counts, mtile, mtile2, h, q,
                         false));
  if (wq == nullptr) {
    MOE_TRY(run("mx_quant_w_down_f", s, fl, [&] {
      return launch_quant_cols_weights(W_down, L.E, L.F, L.H, wd, swd, s);
    }));
  }
  {
    GemmArgs a = base_args(st, fl);
    if (!make_map_u8(&a.mapA, aq, L.F, L.Pa, L.F) ||
        !make_map_u8(&a.mapB0, wd, L.H, static_cast<uint64_t>(L.E) * L.F, L.H))
      return MOE_ERR_CUDA;
    a.mapB1 = a.mapB0;
    a.K = L.F;
    a.N = L.H;
    a.n_tiles = L.H / 256;   // 128 x 256 tiles (pairs: 256 x 256)
    a.num_groups = L.E;
    a.b_group_rows = L.F;
    a.offsets = offsets;
    a.counts = counts;
    a.mtile_off = mtile;
    a.mtile2_off = mtile2;
    a.in0 = w_row;
    a.in1 = row_slot;
    a.out0 = scratch;
    a.ld0 = L.H;
    a.T = L.T;           // the scatter's rows are (token, slot) pairs: T * top_k of them
    a.top_k = L.k;
    a.sfA = sa;
    a.kt_a = L.F / 128;
    a.sfB0 = swd;
    a.kt_b = L.F / 128;
    if (L.mx_pair_down_fwd) {
      if (!make_map_atoms(&a.mapSFA, sa, static_cast<uint64_t>(L.mt_max) * (L.F / 128)) ||
          !make_map_atoms(&a.mapSFB, swd, static_cast<uint64_t>(L.E) * (L.H / 128) * (L.F / 128)))
        return MOE_ERR_CUDA;
      const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
      MOE_TRY(run("down_gemm_scatter_mx", s, fl,
                  [&] { return launch_down_fwd_mx_pair(a, grid, s); }));
    } else {
      const int grid = grid_for(((L.P + kBM - 1) / kBM + L.E) * a.n_tiles, sms);
      MOE_TRY(run("down_gemm_scatter_mx", s, fl, [&] { return launch_down_fwd_mx(a, grid, s); }));
    }
  }
  return MOE_OK;
}


struct BwdBufs {
  const uint16_t *W_gate, *W_up, *W_down, *dyp, *xperm, *h;
  const int *offsets, *counts, *mtile, *mtile2, *order, *slot, *row_slot;   // offsets: padded starts
  const float *w_row, *w;
  const int* idx;
  const uint16_t* wrt;
  uint16_t *dh, *aw;
  float *dwp, *dl;
  uint16_t *dlt, *scratch, *dx;
  void *dW_gate, *dW_up, *dW_down;   // bf16, or fp32 accumulation buffers
  void* ws;
  uint32_t wflags;                   // kGemmAccumF32 or 0, for the weight gradients
  void* wq;                          // prepared MXFP8 weights, or nullptr
  const uint8_t *xt, *sxt;           // x along the tokens in E4M3 with its scale atoms
};

// B2-B9 in MXFP8 (precision mxfp8 and fp8_bwd): every expert GEMM of the
// backward runs block-scaled on operands quantised along its K: dY_perm and
// W_down along H (down dgrad), dh along F and W_gate / W_up along F (gate/up
// dgrad), and w*a, dY_perm, x_perm, dh along the tokens of each expert (the
// weight gradients, segments padded to 128 rows).
moe_status_t backward_expert_gemms_mx(const Layout& L, int sms, cudaStream_t s, uint32_t fl,
                                      DeviceStatus* st, const BwdBufs& b) {
  void* ws = b.ws;
  uint8_t* dyq = at<uint8_t>(ws, L.bq_dy);
  uint8_t* sdy = at<uint8_t>(ws, L.bs_dy);
  const bool prep = b.wq != nullptr;
  uint8_t* wdh = prep ? at<uint8_t>(b.wq, L.q_d_h) : at<uint8_t>(ws, L.bq_wdh);
  uint8_t* swdh = prep ? at<uint8_t>(b.wq, L.mx_pair_down_dgrad ? L.qs_d_h192 : L.qs_d_h)
                       : at<uint8_t>(ws, L.bs_wdh);
  uint8_t* dhq = at<uint8_t>(ws, L.bq_dh);
  uint8_t* sdh = at<uint8_t>(ws, L.bs_dh);
  uint8_t* wg = prep ? at<uint8_t>(b.wq, L.q_g_f) : at<uint8_t>(ws, L.bq_wg);
  uint8_t* swg = prep ? at<uint8_t>(b.wq, L.qs_g_f) : at<uint8_t>(ws, L.bs_wg);
  uint8_t* wu = prep ? at<uint8_t>(b.wq, L.q_u_f) : at<uint8_t>(ws, L.bq_wu);
  uint8_t* swu = prep ? at<uint8_t>(b.wq, L.qs_u_f) : at<uint8_t>(ws, L.bs_wu);
  uint8_t* awt = at<uint8_t>(ws, L.bq_awt);
  uint8_t* sawt = at<uint8_t>(ws, L.bs_awt);
  uint8_t* dyt = at<uint8_t>(ws, L.bq_dyt);
  uint8_t* sdyt = at<uint8_t>(ws, L.bs_dyt);
  const uint8_t* xt = b.xt;
  const uint8_t* sxt = b.sxt;
  uint8_t* dht = at<uint8_t>(ws, L.bq_dht);
  uint8_t* sdht = at<uint8_t>(ws, L.bs_dht);
  const uint64_t Pp = 128ull * static_cast<uint64_t>(L.mt_max);
  const int64_t mtiles = (L.P + kBM - 1) / kBM + L.E;

  // B2-B4: down dgrad (dY was dispatched straight into its E4M3 copies)
  if (!prep) {
    MOE_TRY(run("mx_quant_w_down_h", s, fl, [&] {
      return launch_quant_rows_dense(b.W_down, static_cast<int64_t>(L.E) * L.F, L.H, wdh,
                                     L.mx_pair_down_dgrad ? nullptr : swdh, s,
                                     L.mx_pair_down_dgrad ? swdh : nullptr);
    }));
  }
  {
    GemmArgs a = base_args(st, fl);
    if (!make_map_u8(&a.mapA, dyq, L.H, L.Pa, L.H) ||
        !make_map_u8(&a.mapB0, wdh, L.H, static_cast<uint64_t>(L.E) * L.F, L.H,
                     L.mx_pair_down_dgrad ? 96 : 128))
      return MOE_ERR_CUDA;
    // h [Pa, 2F] in 32 x 32 boxes with the 64-byte swizzle: the epilogue's TMA
    // loads of the saved pre-activations into its staging buffers
    if (!make_map(&a.mapB1, b.h, 2ull * L.F, L.Pa, 4ull * L.F, 32, 32,
                  CU_TENSOR_MAP_SWIZZLE_64B))
      return MOE_ERR_CUDA;
    a.K = L.H;
    a.N = L.F;
    a.n_tiles = L.F / (L.mx_pair_down_dgrad ? 192 : L.mx_dgrad_bn);
    a.num_groups = L.E;
    a.b_group_rows = L.F;
    a.offsets = b.offsets;
    a.counts = b.counts;
    a.mtile_off = b.mtile;
    a.in0 = b.h;
    a.in1 = b.w_row;
    a.out0 = b.dh;
    a.out1 = b.aw;
    a.out2 = b.dwp;
    a.out3 = dhq;   // dh quantised to E4M3 along F in the epilogue
    a.out4 = sdh;
    a.ld0 = L.F;
    a.sfA = sdy;
    a.kt_a = L.H / 128;
    a.sfB0 = swdh;
    a.kt_b = L.H / 128;
    if (fl & MOE_FLAG_TEST_TIMEOUT) {
      a.flags = kGemmInjectWait;
      a.wait_limit_ns = kTestWaitNs;
    }
    if (L.mx_pair_down_dgrad) {
      a.mtile2_off = b.mtile2;
      if (!make_out_maps(&a, b.dh, b.aw, L)) return MOE_ERR_CUDA;
      if (!make_map_atoms(&a.mapSFA, sdy, static_cast<uint64_t>(L.mt_max) * (L.H / 128)) ||
          !make_map_atoms(&a.mapSFB, swdh,
                          static_cast<uint64_t>(L.E) * (L.F / 192) * 2 * (L.H / 128)))
        return MOE_ERR_CUDA;
      const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
      MOE_TRY(run("down_dgrad_swiglu_bwd_mx", s, fl,
                  [&] { return launch_down_dgrad_mx_pair(a, grid, s); }));
    } else {
      const int grid = grid_for(mtiles * a.n_tiles, sms);
      MOE_TRY(run("down_dgrad_swiglu_bwd_mx", s, fl,
                  [&] { return launch_down_dgrad_mx(a, grid, s); }));
    }
  }
  // B9: router softmax / top-k backward
  if (cudaMemsetAsync(b.dlt, 0, 2ull * L.E * L.T_pad, s) != cudaSuccess) return MOE_ERR_CUDA;
  MOE_TRY(run("router_bwd", s, fl, [&] {
    return launch_router_bwd(b.dwp, L.nparts, b.slot, b.w, b.idx, L.T, L.k, L.E, L.Pa, b.dl, b.dlt,
                             L.T_pad, st, s);
  }));
  // B5: down wgrad over the padded token layout
  MOE_TRY(run("mx_quant_aw_tokens", s, fl, [&] {
    return launch_quant_cols_tokens(b.aw, L.mt_max, L.F, awt, sawt, b.offsets, b.counts, b.mtile,
                                    L.E, s);
  }));
  // (dY along the tokens came from the dispatch)
  {
    GemmArgs a = base_args(st, fl);
    a.flags = b.wflags;
    if (!make_map_u8(&a.mapA, awt, L.F, Pp, L.F) || !make_map_u8(&a.mapB0, dyt, L.H, Pp, L.H))
      return MOE_ERR_CUDA;
    a.mapB1 = a.mapB0;
    a.M = L.F;
    a.N = L.H;
    a.m_tiles = L.F / 128;
    a.n_tiles = L.H / 256;   // 128 x 256 tiles (pairs: 256 x 256)
    a.num_groups = L.E;
    a.offsets = b.offsets;
    a.counts = b.counts;
    a.mtile_off = b.mtile;
    a.group_order = b.order;
    a.out0 = b.dW_down;
    a.ld0 = L.H;
    a.sfA = sawt;
    a.sfB0 = sdyt;
    if (L.mx_pair_down_wgrad) {
      a.m_tiles = L.F / 256;
      a.kt_a = L.F / 128;     // A's atoms per token k-tile
      if (!make_map_atoms(&a.mapSFA, sawt, static_cast<uint64_t>(L.mt_max) * (L.F / 128)) ||
          !make_map_atoms(&a.mapSFB, sdyt, static_cast<uint64_t>(L.mt_max) * (L.H / 128)))
        return MOE_ERR_CUDA;
      const int grid = grid_for_pairs(static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles, sms);
      MOE_TRY(run("down_wgrad_mx", s, fl, [&] { return launch_down_wgrad_mx_pair(a, grid, s); }));
    } else {
      const int grid = grid_for(static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles, sms);
      MOE_TRY(run("down_wgrad_mx", s, fl, [&] { return launch_down_wgrad_mx(a, grid, s); }));
    }
  }
  // B6 + B7: gate/up dgrad, then the un-permute
  if (!prep) {
    MOE_TRY(run("mx_quant_w_gate_f", s, fl, [&] {
      return launch_quant_rows_dense(b.W_gate, static_cast<int64_t>(L.E) * L.H, L.F, wg, swg, s);
    }));
    MOE_TRY(run("mx_quant_w_up_f", s, fl, [&] {
      return launch_quant_rows_dense(b.W_up, static_cast<int64_t>(L.E) * L.H, L.F, wu, swu, s);
    }));
  }
  {
    GemmArgs a = base_args(st, fl);
    if (!make_map_u8(&a.mapA, dhq, 2ull * L.F, L.Pa, 2ull * L.F) ||
        !make_map_u8(&a.mapB0, wg, L.F, static_cast<uint64_t>(L.E) * L.H, L.F) ||
        !make_map_u8(&a.mapB1, wu, L.F, static_cast<uint64_t>(L.E) * L.H, L.F))
      return MOE_ERR_CUDA;
    a.K = 2 * L.F;
    a.k_half = L.F;
    a.N = L.H;
    a.n_tiles = L.H / 256;   // 128 x 256 tiles
    a.num_groups = L.E;
    a.b_group_rows = L.H;
    a.offsets = b.offsets;
    a.counts = b.counts;
    a.mtile_off = b.mtile;
    a.in1 = b.row_slot;
    a.out0 = b.scratch;
    a.ld0 = L.H;
    a.T = L.T;           // the scatter's rows are (token, slot) pairs: T * top_k of them
    a.top_k = L.k;
    a.sfA = sdh;
    a.kt_a = 2 * L.F / 128;
    a.sfB0 = swg;
    a.sfB1 = swu;
    a.kt_b = L.F / 128;
    a.mtile2_off = b.mtile2;
    if (L.mx_pair_gu_dgrad) {
      const uint64_t w_atoms = static_cast<uint64_t>(L.E) * (L.H / 128) * (L.F / 128);
      if (!make_map_atoms(&a.mapSFA, sdh, static_cast<uint64_t>(L.mt_max) * (2 * L.F / 128)) ||
          !make_map_atoms(&a.mapSFB, swg, w_atoms) || !make_map_atoms(&a.mapSFB1, swu, w_atoms))
        return MOE_ERR_CUDA;
      const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
      MOE_TRY(run("gate_up_dgrad_scatter_mx", s, fl,
                  [&] { return launch_gate_up_dgrad_mx_pair(a, grid, s); }));
    } else {
      const int grid = grid_for(mtiles * a.n_tiles, sms);
      MOE_TRY(run("gate_up_dgrad_scatter_mx", s, fl,
                  [&] { return launch_gate_up_dgrad_mx(a, grid, s); }));
    }
  }
  MOE_TRY(run("unpermute_dx", s, fl, [&] {
    return launch_unpermute(b.scratch, b.dl, b.idx, b.wrt, b.dx, L.T, L.H, L.k, L.E, sms, st, s);
  }));
  // B8: gate/up wgrad over the padded token layout
  MOE_TRY(run("mx_quant_dh_tokens", s, fl, [&] {
    return launch_quant_cols_tokens(b.dh, L.mt_max, 2 * L.F, dht, sdht, b.offsets, b.counts,
                                    b.mtile, L.E, s);
  }));
  {
    GemmArgs a = base_args(st, fl);
    a.flags = b.wflags;
    if (!make_map_u8(&a.mapA, xt, L.H, Pp, L.H) ||
        !make_map_u8(&a.mapB0, dht, 2ull * L.F, Pp, 2ull * L.F))
      return MOE_ERR_CUDA;
    a.mapB1 = a.mapB0;
    a.M = L.H;
    a.N = 2 * L.F;
    a.m_tiles = L.H / 128;
    a.n_tiles = 2 * L.F / 256;   // 128 x 256 tiles (pairs: 256 x 256)
    a.num_groups = L.E;
    a.offsets = b.offsets;
    a.counts = b.counts;
    a.mtile_off = b.mtile;
    a.group_order = b.order;
    a.out0 = b.dW_gate;
    a.out1 = b.dW_up;
    a.ld0 = L.F;
    a.sfA = sxt;
    a.sfB0 = sdht;
    if (L.mx_pair_gu_wgrad) {
      a.m_tiles = L.H / 256;
      a.kt_a = L.H / 128;     // A's atoms per token k-tile
      if (!make_map_atoms(&a.mapSFA, sxt, static_cast<uint64_t>(L.mt_max) * (L.H / 128)) ||
          !make_map_atoms(&a.mapSFB, sdht, static_cast<uint64_t>(L.mt_max) * (2 * L.F / 128)))
        return MOE_ERR_CUDA;
      const int grid = grid_for_pairs(static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles, sms);
      MOE_TRY(run("gate_up_wgrad_mx", s, fl,
                  [&] { return launch_gate_up_wgrad_mx_pair(a, grid, s); }));
    } else {
      const int grid = grid_for(static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles, sms);
      MOE_TRY(run("gate_up_wgrad_mx", s, fl, [&] { return launch_gate_up_wgrad_mx(a, grid, s); }));
    }
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE";
    case MOE_ERR_NOT_IMPLEMENTED: return "MOE_ERR_NOT_IMPLEMENTED";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* fwd_ws, size_t* ctx_bytes,
                                size_t* bwd_ws) {
  MOE_TRY(validate(cfg));
  DevInfo d;
  MOE_TRY(current_device(&d));
  const int sms = sm_budget(d.sms, *cfg);
  const Layout L = make_layout(*cfg, sms);
  if (fwd_ws) *fwd_ws = L.f_total;
  if (ctx_bytes) *ctx_bytes = L.c_total;
  if (bwd_ws) *bwd_ws = L.b_total;
  return MOE_OK;
}

moe_status_t moe_prepared_weights_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (bytes == nullptr || cfg->precision == MOE_BF16) return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  *bytes = make_layout(*cfg, sm_budget(d.sms, *cfg)).q_total;
  return MOE_OK;
}

moe_status_t moe_prepare_weights(const moe_config_t* cfg, const moe_bf16_t* W_gate,
                                 const moe_bf16_t* W_up, const moe_bf16_t* W_down, void* wq,
                                 size_t wq_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  if (cfg->precision == MOE_BF16 || !all_aligned16({W_gate, W_up, W_down}) || wq == nullptr ||
      !aligned(wq, 256))
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  const Layout L = make_layout(*cfg, sm_budget(d.sms, *cfg));
  if (wq_bytes < L.q_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t fl = cfg->flags;
  MOE_TRY(run("prepare_w_gate_up_h", s, fl, [&] {
    return launch_quant_cols_gate_up(W_gate, W_up, L.E, L.H, L.F, at<uint8_t>(wq, L.q_gu_h),
                                     at<uint8_t>(wq, L.qs_gu_h), s);
  }));
  MOE_TRY(run("prepare_w_down_f", s, fl, [&] {
    return launch_quant_cols_weights(W_down, L.E, L.F, L.H, at<uint8_t>(wq, L.q_d_f),
                                     at<uint8_t>(wq, L.qs_d_f), s);
  }));
  MOE_TRY(run("prepare_w_gate_f", s, fl, [&] {
    return launch_quant_rows_dense(W_gate, static_cast<int64_t>(L.E) * L.H, L.F,
                                   at<uint8_t>(wq, L.q_g_f), at<uint8_t>(wq, L.qs_g_f), s);
  }));
  MOE_TRY(run("prepare_w_up_f", s, fl, [&] {
    return launch_quant_rows_dense(W_up, static_cast<int64_t>(L.E) * L.H, L.F,
                                   at<uint8_t>(wq, L.q_u_f), at<uint8_t>(wq, L.qs_u_f), s);
  }));
  return run("prepare_w_down_h", s, fl, [&] {
    return launch_quant_rows_dense(W_down, static_cast<int64_t>(L.E) * L.F, L.H,
                                   at<uint8_t>(wq, L.q_d_h), at<uint8_t>(wq, L.qs_d_h), s,
                                   L.F % 192 == 0 ? at<uint8_t>(wq, L.qs_d_h192) : nullptr);
  });
}

moe_status_t moe_route(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                       const float* logit_bias, float* logits, int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* slot_row,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  if (!all_aligned16({x, W_r}) || topk_idx == nullptr || topk_w == nullptr ||
      counts == nullptr || offsets == nullptr || perm_token == nullptr || slot_row == nullptr ||
      ws == nullptr || !aligned(ws, 256) || !aligned(logit_bias, 4) || !aligned(logits, 4))
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  const int sms = sm_budget(d.sms, *cfg);
  const Layout L = make_layout(*cfg, sms);
  if (ws_bytes < L.f_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(ws, L.f_status);
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  RouteBufs b{x, W_r, logit_bias, logits, topk_idx, topk_w, counts, offsets, perm_token,
              slot_row, at<int>(ws, L.r_row_slot), at<float>(ws, L.r_w_row),
              at<int>(ws, L.r_mtile), at<int>(ws, L.r_order), at<uint16_t>(ws, L.r_wrt),
              at<int>(ws, L.f_hist), at<int>(ws, L.f_base), st, at<int>(ws, L.r_poff),
              at<int>(ws, L.r_mtile2), at<int>(ws, L.r_slotpad)};
  return run_routing(*cfg, L, b, sms, s);
}

moe_status_t moe_forward(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                         const float* logit_bias, const moe_bf16_t* W_gate,
                         const moe_bf16_t* W_up, const moe_bf16_t* W_down, moe_bf16_t* y,
                         void* ctx, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  if (!all_aligned16({x, W_r, W_gate, W_up, W_down, y}) || ctx == nullptr || ws == nullptr ||
      !aligned(ctx, 256) || !aligned(ws, 256) || !aligned(logit_bias, 4))
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  const int sms = sm_budget(d.sms, *cfg);
  const Layout L = make_layout(*cfg, sms);
  if (ws_bytes < L.f_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t fl = cfg->flags;
  DeviceStatus* st = at<DeviceStatus>(ws, L.f_status);
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;

  int* idx = at<int>(ctx, L.c_idx);
  int* offsets = at<int>(ctx, L.c_offsets);
  int* counts = at<int>(ctx, L.c_counts);
  int* poff = at<int>(ctx, L.c_poff);
  int* slot = at<int>(ctx, L.c_slot);
  int* slot_pad = at<int>(ctx, L.c_slotpad);
  int* row_slot = at<int>(ctx, L.c_row_slot);
  float* w_row = at<float>(ctx, L.c_w_row);
  int* mtile = at<int>(ctx, L.c_mtile);
  int* mtile2 = at<int>(ctx, L.c_mtile2);
  // x_perm and h: kept in ctx for the backward, or (recompute) in the workspace
  uint16_t* xperm = L.recompute ? at<uint16_t>(ws, L.f_xperm) : at<uint16_t>(ctx, L.c_xperm);
  uint16_t* h = L.recompute ? at<uint16_t>(ws, L.f_h) : at<uint16_t>(ctx, L.c_h);
  uint16_t* act = at<uint16_t>(ws, L.f_a);
  uint16_t* scratch = at<uint16_t>(ws, L.f_scratch);

  RouteBufs b{x, W_r, logit_bias, nullptr, idx, at<float>(ctx, L.c_w), counts, offsets,
              at<int>(ctx, L.c_perm), slot, row_slot, w_row, mtile, at<int>(ctx, L.c_order),
              at<uint16_t>(ctx, L.c_wrt), at<int>(ws, L.f_hist), at<int>(ws, L.f_base), st,
              poff, mtile2, slot_pad};
  MOE_TRY(run_routing(*cfg, L, b, sms, s));

  // F6: dispatch x to the padded expert-major rows (segment tails zeroed: they
  // are K rows of the gate/up weight gradient)
  if (cfg->precision == MOE_MXFP8) {
    // x dispatched straight into its E4M3 copies: along H for the gate/up GEMM,
    // along the tokens (kept in ctx) for the backward's gate/up wgrad
    xperm = nullptr;
    MOE_TRY(run("dispatch_x_mx", s, fl, [&] {
      return launch_dispatch_quant(x, at<int>(ctx, L.c_perm), offsets, poff, counts, mtile,
                                   L.mt_max, L.E, L.H,
                                   L.recompute ? nullptr : at<uint8_t>(ctx, L.c_xt),
                                   L.recompute ? nullptr : at<uint8_t>(ctx, L.c_sxt),
                                   at<uint8_t>(ws, L.fq_x), at<uint8_t>(ws, L.fs_x), s);
    }));
  } else {
    MOE_TRY(run("gather_x", s, fl, [&] {
      return launch_gather_rows(x, slot_pad, xperm, L.T, L.H, L.k, poff, counts, L.E, L.Pa, st, s);
    }));
  }

  if (cfg->precision == MOE_MXFP8) {
    MOE_TRY(forward_gemms_mx(L, sms, s, fl, st, W_gate, W_up, W_down, poff, counts, mtile, mtile2,
                             w_row, row_slot, h, scratch, ws,
                             const_cast<void*>(cfg->prepared_weights)));
  } else {
    // F7 + F8: gate/up GEMM with SwiGLU
    MOE_TRY(gate_up_fwd_bf16(L, sms, s, fl, st, xperm, W_gate, W_up, poff, counts, mtile, mtile2,
                             act, h, false));
    // F9 + F10: down GEMM with the weighted scatter, then the k-way combine
    {
      GemmArgs a = base_args(st, fl);
      if (!make_map(&a.mapA, act, L.F, L.Pa, 2ull * L.F, 64, 128) ||
          !make_map(&a.mapB0, W_down, L.H, static_cast<uint64_t>(L.E) * L.F, 2ull * L.H, 64, 64))
        return MOE_ERR_CUDA;
      a.mapB1 = a.mapB0;
      a.K = L.F;
      a.N = L.H;
      a.n_tiles = L.H / 256;
      a.num_groups = L.E;
      a.b_group_rows = L.F;
      a.offsets = poff;
      a.counts = counts;
      a.mtile_off = mtile;
      a.mtile2_off = mtile2;
      a.in0 = w_row;
      a.in1 = row_slot;
      a.out0 = scratch;
      a.ld0 = L.H;
      a.T = L.T;           // the scatter's rows are (token, slot) pairs: T * top_k of them
      a.top_k = L.k;
      if (L.pair_down_fwd) {
        const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("down_gemm_scatter", s, fl, [&] { return launch_down_fwd_pair(a, grid, s); }));
      } else {
        const int grid = grid_for(grouped_m_tile_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("down_gemm_scatter", s, fl, [&] { return launch_down_fwd(a, grid, s); }));
      }
    }
  }
  MOE_TRY(run("combine", s, fl, [&] { return launch_combine(scratch, y, L.T, L.H, L.k, s); }));
  return MOE_OK;
}

// moe_backward and moe_backward_accumulate: the weight gradients are bf16
// outputs, or (accum) fp32 buffers the gradients are added into.
static moe_status_t backward_impl(const moe_config_t* cfg, const moe_bf16_t* x,
                                  const moe_bf16_t* W_r, const moe_bf16_t* W_gate,
                                  const moe_bf16_t* W_up, const moe_bf16_t* W_down,
                                  const void* ctx_in, const moe_bf16_t* dY, moe_bf16_t* dx,
                                  void* dW_r, void* dW_gate, void* dW_up, void* dW_down,
                                  bool accum, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  if (!all_aligned16({x, W_r, W_gate, W_up, W_down, dY, dx, dW_r, dW_gate, dW_up, dW_down}) ||
      ctx_in == nullptr || ws == nullptr || !aligned(ctx_in, 256) || !aligned(ws, 256))
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  const int sms = sm_budget(d.sms, *cfg);
  const Layout L = make_layout(*cfg, sms);
  if (ws_bytes < L.b_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t fl = cfg->flags;
  void* ctx = const_cast<void*>(ctx_in);
  DeviceStatus* st = at<DeviceStatus>(ws, L.b_status);
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;

  const int* idx = at<int>(ctx, L.c_idx);
  const float* w = at<float>(ctx, L.c_w);
  const int* counts = at<int>(ctx, L.c_counts);
  const int* poff = at<int>(ctx, L.c_poff);
  const int* slot_pad = at<int>(ctx, L.c_slotpad);
  const int* row_slot = at<int>(ctx, L.c_row_slot);
  const float* w_row = at<float>(ctx, L.c_w_row);
  const int* mtile = at<int>(ctx, L.c_mtile);
  const int* mtile2 = at<int>(ctx, L.c_mtile2);
  const int* order = at<int>(ctx, L.c_order);
  const uint16_t* wrt = at<uint16_t>(ctx, L.c_wrt);
  const uint16_t* xperm = L.recompute ? at<uint16_t>(ws, L.b_xperm) : at<uint16_t>(ctx, L.c_xperm);
  const uint16_t* h = L.recompute ? at<uint16_t>(ws, L.b_h) : at<uint16_t>(ctx, L.c_h);
  // x along the tokens in E4M3 for the gate/up wgrad: mxfp8 has it from the
  // forward's dispatch (ctx) or from the recompute dispatch below (ws);
  // fp8_bwd (bf16 forward) dispatches x into ws with the dY dispatch
  const uint8_t* x_tok = nullptr;
  const uint8_t* x_tok_sf = nullptr;
  if (cfg->precision == MOE_MXFP8 && !L.recompute) {
    x_tok = at<uint8_t>(ctx, L.c_xt);
    x_tok_sf = at<uint8_t>(ctx, L.c_sxt);
  } else if (cfg->precision != MOE_BF16) {
    x_tok = at<uint8_t>(ws, L.bq_xt);
    x_tok_sf = at<uint8_t>(ws, L.bs_xt);
  }
  uint16_t* dyp = at<uint16_t>(ws, L.b_dyp);
  uint16_t* dh = at<uint16_t>(ws, L.b_dh);
  uint16_t* aw = at<uint16_t>(ws, L.b_aw);
  float* dwp = at<float>(ws, L.b_dwp);
  float* dl = at<float>(ws, L.b_dl);
  uint16_t* dlt = at<uint16_t>(ws, L.b_dlt);
  uint16_t* scratch = at<uint16_t>(ws, L.b_scratch);
  float* wrp = at<float>(ws, L.b_wrp);
  (void)W_r;
  const uint32_t wflags = accum ? kGemmAccumF32 : 0u;   // weight-gradient epilogues

  if (L.recompute) {
    // activation checkpointing: dispatch x again and recompute h (and a, which
    // lands in aw and is overwritten by the down dgrad) in the forward's precision
    uint16_t* xp = at<uint16_t>(ws, L.b_xperm);
    uint16_t* hh = at<uint16_t>(ws, L.b_h);
    if (cfg->precision == MOE_MXFP8) {
      MOE_TRY(run("recompute_dispatch_x_mx", s, fl, [&] {
        return launch_dispatch_quant(x, at<int>(ctx, L.c_perm), at<int>(ctx, L.c_offsets), poff,
                                     counts, mtile, L.mt_max, L.E, L.H, at<uint8_t>(ws, L.bq_xt),
                                     at<uint8_t>(ws, L.bs_xt), at<uint8_t>(ws, L.bq_rx),
                                     at<uint8_t>(ws, L.bs_rx), s);
      }));
    } else {
      MOE_TRY(run("recompute_gather_x", s, fl, [&] {
        return launch_gather_rows(x, slot_pad, xp, L.T, L.H, L.k, poff, counts, L.E, L.Pa, st, s);
      }));
    }
    if (cfg->precision == MOE_MXFP8) {
      MxGateUpBufs q{at<uint8_t>(ws, L.bq_rx), at<uint8_t>(ws, L.bs_rx),
                     at<uint8_t>(ws, L.bq_ra), at<uint8_t>(ws, L.bs_ra),
                     at<uint8_t>(ws, L.bq_rwgu), at<uint8_t>(ws, L.bs_rwgu)};
      if (L.prepared) {
        void* wq = const_cast<void*>(cfg->prepared_weights);
        q.wgu = at<uint8_t>(wq, L.q_gu_h);
        q.swgu = at<uint8_t>(wq, L.qs_gu_h);
        q.w_ready = true;
      }
      MOE_TRY(gate_up_fwd_mx(L, sms, s, fl, st, W_gate, W_up, poff, counts, mtile, mtile2, hh, q,
                             true));
    } else {
      MOE_TRY(gate_up_fwd_bf16(L, sms, s, fl, st, xp, W_gate, W_up, poff, counts, mtile, mtile2,
                               at<uint16_t>(ws, L.b_aw), hh, true));
    }
  }

  // B1: dispatch dY to the padded expert-major rows (segment tails zeroed:
  // they are K rows of the down weight gradient)
  if (cfg->precision == MOE_FP8_BWD) {
    // x along the tokens only (the bf16 forward kept x_perm, not this copy)
    MOE_TRY(run("dispatch_x_tokens_mx", s, fl, [&] {
      return launch_dispatch_quant(x, at<int>(ctx, L.c_perm), at<int>(ctx, L.c_offsets), poff,
                                   counts, mtile, L.mt_max, L.E, L.H, at<uint8_t>(ws, L.bq_xt),
                                   at<uint8_t>(ws, L.bs_xt), nullptr, nullptr, s);
    }));
  }
  if (cfg->precision != MOE_BF16) {
    // MXFP8: dY dispatched straight into its two E4M3 copies (along H for the
    // down dgrad, along the tokens for the down wgrad); no bf16 dY_perm
    MOE_TRY(run("dispatch_dy_mx", s, fl, [&] {
      return launch_dispatch_quant(dY, at<int>(ctx, L.c_perm), at<int>(ctx, L.c_offsets), poff,
                                   counts, mtile, L.mt_max, L.E, L.H, at<uint8_t>(ws, L.bq_dyt),
                                   at<uint8_t>(ws, L.bs_dyt), at<uint8_t>(ws, L.bq_dy),
                                   at<uint8_t>(ws, L.bs_dy), s);
    }));
  } else {
    MOE_TRY(run("gather_dy", s, fl, [&] {
      return launch_gather_rows(dY, slot_pad, dyp, L.T, L.H, L.k, poff, counts, L.E, L.Pa, st, s);
    }));
  }

  if (cfg->precision != MOE_BF16) {
    const BwdBufs bb{W_gate, W_up, W_down, dyp, xperm, h, poff, counts, mtile, mtile2, order, slot_pad,
                     row_slot, w_row, w, idx, wrt, dh, aw, dwp, dl, dlt, scratch, dx,
                     dW_gate, dW_up, dW_down, ws, wflags,
                     L.prepared ? const_cast<void*>(cfg->prepared_weights) : nullptr,
                     x_tok, x_tok_sf};
    MOE_TRY(backward_expert_gemms_mx(L, sms, s, fl, st, bb));
  } else {
    // B2-B4: down dgrad with the SwiGLU backward and router-weight partials
    {
      GemmArgs a = base_args(st, fl);
      if (!make_map(&a.mapA, dyp, L.H, L.Pa, 2ull * L.H, 64, 128) ||
          !make_map(&a.mapB0, W_down, L.H, static_cast<uint64_t>(L.E) * L.F, 2ull * L.H, 64,
                    L.pair_down_dgrad ? 128 : L.dgrad_bn))
        return MOE_ERR_CUDA;
      a.mapB1 = a.mapB0;
      // CTA pairs: h [Pa, 2F] in 32 x 32 boxes with the 64-byte swizzle, for the
      // epilogue's TMA loads of the saved pre-activations
      if (L.pair_down_dgrad && !make_map(&a.mapB1, h, 2ull * L.F, L.Pa, 4ull * L.F, 32, 32,
                                         CU_TENSOR_MAP_SWIZZLE_64B))
        return MOE_ERR_CUDA;
      // dh [Pa, 2F] and w*a [Pa, F] in the same boxes: the staged outputs' TMA stores
      if (L.pair_down_dgrad && !make_out_maps(&a, dh, aw, L)) return MOE_ERR_CUDA;
      a.K = L.H;
      a.N = L.F;
      a.n_tiles = L.F / L.dgrad_bn;
      a.num_groups = L.E;
      a.b_group_rows = L.F;
      a.offsets = poff;
      a.counts = counts;
      a.mtile_off = mtile;
      a.mtile2_off = mtile2;
      a.in0 = h;
      a.in1 = w_row;
      a.out0 = dh;
      a.out1 = aw;
      a.out2 = dwp;
      a.ld0 = L.F;
      if (fl & MOE_FLAG_TEST_TIMEOUT) {
        a.flags = kGemmInjectWait;
        a.wait_limit_ns = kTestWaitNs;
      }
      if (L.pair_down_dgrad) {
        const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("down_dgrad_swiglu_bwd", s, fl,
                    [&] { return launch_down_dgrad_pair(a, grid, s); }));
      } else {
        const int grid = grid_for(grouped_m_tile_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("down_dgrad_swiglu_bwd", s, fl,
                    [&] { return launch_down_dgrad(L.dgrad_bn, a, grid, s); }));
      }
    }
    // B9: router softmax / top-k backward
    if (cudaMemsetAsync(dlt, 0, 2ull * L.E * L.T_pad, s) != cudaSuccess) return MOE_ERR_CUDA;
    MOE_TRY(run("router_bwd", s, fl, [&] {
      return launch_router_bwd(dwp, L.nparts, slot_pad, w, idx, L.T, L.k, L.E, L.Pa, dl, dlt,
                               L.T_pad, st, s);
    }));
    // B5: down wgrad over the padded token segments
    {
      GemmArgs a = base_args(st, fl);
      a.flags = wflags;
      if (!make_map(&a.mapA, aw, L.F, L.Pa, 2ull * L.F, 64, 64) ||
          !make_map(&a.mapB0, dyp, L.H, L.Pa, 2ull * L.H, 64, 64))
        return MOE_ERR_CUDA;
      a.mapB1 = a.mapB0;
      a.M = L.F;
      a.N = L.H;
      a.m_tiles = L.F / (L.pair_down_wgrad ? 256 : 128);
      a.n_tiles = L.H / 256;
      a.num_groups = L.E;
      a.offsets = poff;
      a.counts = counts;
      a.group_order = order;
      a.out0 = dW_down;
      a.ld0 = L.H;
      const int64_t tiles = static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles;
      if (L.pair_down_wgrad) {
        const int grid = grid_for_pairs(tiles, sms);
        MOE_TRY(run("down_wgrad", s, fl, [&] { return launch_down_wgrad_pair(a, grid, s); }));
      } else {
        const int grid = grid_for(tiles, sms);
        MOE_TRY(run("down_wgrad", s, fl, [&] { return launch_down_wgrad(a, grid, s); }));
      }
    }
    // B6 + B7: gate/up dgrad with the scatter, then the un-permute (+ router dgrad)
    {
      GemmArgs a = base_args(st, fl);
      const uint32_t brows = L.pair_gu_dgrad ? 128 : 256;
      if (!make_map(&a.mapA, dh, 2ull * L.F, L.Pa, 4ull * L.F, 64, 128) ||
          !make_map(&a.mapB0, W_gate, L.F, static_cast<uint64_t>(L.E) * L.H, 2ull * L.F, 64, brows) ||
          !make_map(&a.mapB1, W_up, L.F, static_cast<uint64_t>(L.E) * L.H, 2ull * L.F, 64, brows))
        return MOE_ERR_CUDA;
      a.K = 2 * L.F;
      a.k_half = L.F;
      a.N = L.H;
      a.n_tiles = L.H / 256;
      a.num_groups = L.E;
      a.b_group_rows = L.H;
      a.offsets = poff;
      a.counts = counts;
      a.mtile_off = mtile;
      a.mtile2_off = mtile2;
      a.in1 = row_slot;
      a.out0 = scratch;
      a.ld0 = L.H;
      a.T = L.T;           // the scatter's rows are (token, slot) pairs: T * top_k of them
      a.top_k = L.k;
      if (L.pair_gu_dgrad) {
        const int grid = grid_for_pairs(grouped_m_pair_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("gate_up_dgrad_scatter", s, fl, [&] { return launch_gate_up_dgrad_pair(a, grid, s); }));
      } else {
        const int grid = grid_for(grouped_m_tile_bound(L) * a.n_tiles, sms);
        MOE_TRY(run("gate_up_dgrad_scatter", s, fl, [&] { return launch_gate_up_dgrad(a, grid, s); }));
      }
    }
    MOE_TRY(run("unpermute_dx", s, fl, [&] {
      return launch_unpermute(scratch, dl, idx, wrt, dx, L.T, L.H, L.k, L.E, sms, st, s);
    }));
    // B8: gate/up wgrad over the padded token segments
    {
      GemmArgs a = base_args(st, fl);
      a.flags = wflags;
      if (!make_map(&a.mapA, xperm, L.H, L.Pa, 2ull * L.H, 64, 64) ||
          !make_map(&a.mapB0, dh, 2ull * L.F, L.Pa, 4ull * L.F, 64, 64))
        return MOE_ERR_CUDA;
      a.mapB1 = a.mapB0;
      a.M = L.H;
      a.N = 2 * L.F;
      a.m_tiles = L.H / (L.pair_gu_wgrad ? 256 : 128);
      a.n_tiles = (2 * L.F) / 256;
      a.num_groups = L.E;
      a.offsets = poff;
      a.counts = counts;
      a.group_order = order;
      a.out0 = dW_gate;
      a.out1 = dW_up;
      a.ld0 = L.F;
      const int64_t tiles = static_cast<int64_t>(L.E) * a.m_tiles * a.n_tiles;
      if (L.pair_gu_wgrad) {
        const int grid = grid_for_pairs(tiles, sms);
        MOE_TRY(run("gate_up_wgrad", s, fl, [&] { return launch_gate_up_wgrad_pair(a, grid, s); }));
      } else {
        const int grid = grid_for(tiles, sms);
        MOE_TRY(run("gate_up_wgrad", s, fl, [&] { return launch_gate_up_wgrad(a, grid, s); }));
      }
    }
  }
  // B10: router weight gradient dW_r = x^T dl (split-K, then reduce + transpose)
  {
    GemmArgs a = base_args(st, fl);
    if (!make_map(&a.mapA, dlt, L.T, L.E, 2ull * L.T_pad, 64, 128) ||
        !make_map(&a.mapB0, x, L.H, L.T, 2ull * L.H, 64, 64))
      return MOE_ERR_CUDA;
    a.mapB1 = a.mapB0;
    a.M = L.E;
    a.N = L.H;
    a.K = static_cast<int>(L.T);
    a.m_tiles = L.wr_mtiles;
    a.n_tiles = L.wr_ntiles;
    a.k_split = L.wr_split;
    a.kb_per_split = L.wr_kbps;
    a.out0 = wrp;
    a.ld0 = L.H;
    const int grid =
        grid_for(static_cast<int64_t>(L.wr_split) * L.wr_mtiles * L.wr_ntiles, sms);
    MOE_TRY(run("router_wgrad", s, fl, [&] { return launch_router_wgrad(a, grid, s); }));
  }
  MOE_TRY(run("router_wgrad_reduce", s, fl,
              [&] { return launch_wr_reduce(wrp, L.wr_split, L.E, L.H, dW_r, accum, s); }));
  return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                          const moe_bf16_t* W_gate, const moe_bf16_t* W_up,
                          const moe_bf16_t* W_down, const void* ctx, const moe_bf16_t* dY,
                          moe_bf16_t* dx, moe_bf16_t* dW_r, moe_bf16_t* dW_gate,
                          moe_bf16_t* dW_up, moe_bf16_t* dW_down, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  return backward_impl(cfg, x, W_r, W_gate, W_up, W_down, ctx, dY, dx, dW_r, dW_gate, dW_up,
                       dW_down, false, ws, ws_bytes, stream);
}

moe_status_t moe_backward_accumulate(const moe_config_t* cfg, const moe_bf16_t* x,
                                     const moe_bf16_t* W_r, const moe_bf16_t* W_gate,
                                     const moe_bf16_t* W_up, const moe_bf16_t* W_down,
                                     const void* ctx, const moe_bf16_t* dY, moe_bf16_t* dx,
                                     float* gW_r, float* gW_gate, float* gW_up,
                                     float* gW_down, void* ws, size_t ws_bytes,
                                     moe_stream_t stream) {
  return backward_impl(cfg, x, W_r, W_gate, W_up, W_down, ctx, dY, dx, gW_r, gW_gate, gW_up,
                       gW_down, true, ws, ws_bytes, stream);
}

moe_status_t moe_gemm_bf16(int64_t M, int64_t N, int64_t K, const moe_bf16_t* A, int a_kmajor,
                           const moe_bf16_t* B, int b_kmajor, float* D, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  if (M < 1 || K < 1 || N < 256 || N % 256 != 0 || M >= (1ll << 31) || N >= (1ll << 31) ||
      K >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int64_t a_row = a_kmajor ? K : M;
  const int64_t b_row = b_kmajor ? K : N;
  if (a_row % 8 != 0 || b_row % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!all_aligned16({A, B, D}) || ws == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(DeviceStatus)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo d;
  MOE_TRY(current_device(&d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceStatus* st = static_cast<DeviceStatus*>(ws);
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  GemmArgs a = base_args(st, 0);
  const bool ok_a = a_kmajor ? make_map(&a.mapA, A, K, M, 2ull * K, 64, 128)
                             : make_map(&a.mapA, A, M, K, 2ull * M, 64, 64);
  const bool ok_b = b_kmajor ? make_map(&a.mapB0, B, K, N, 2ull * K, 64, 256)
                             : make_map(&a.mapB0, B, N, K, 2ull * N, 64, 64);
  if (!ok_a || !ok_b) return MOE_ERR_CUDA;
  a.mapB1 = a.mapB0;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.n_tiles = static_cast<int>(N / 256);
  a.out0 = D;
  a.ld0 = static_cast<int>(N);
  const int64_t tiles = ((M + kBM - 1) / kBM) * a.n_tiles;
  return run("dense_gemm", s, 0, [&] {
    return launch_dense(!a_kmajor, !b_kmajor, a, grid_for(tiles, d.sms), s);
  });
}

moe_status_t moe_gemm_mxfp8(int64_t M, int64_t N, int64_t K, const moe_bf16_t* A,
                            const moe_bf16_t* B, float* D, void* ws, size_t* ws_bytes,
                            moe_stream_t stream) {
  if (ws_bytes == nullptr) return MOE_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || K < 128 || N % 128 != 0 || K % 128 != 0 || M >= (1ll << 31) ||
      N >= (1ll << 31) || K >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const size_t mt = static_cast<size_t>((M + 127) / 128), nt = static_cast<size_t>(N / 128);
  const size_t kt = static_cast<size_t>(K / 128);
  Carver c;
  const size_t o_st = c.take(sizeof(DeviceStatus));
  const size_t o_aq = c.take(static_cast<size_t>(M) * K);
  const size_t o_bq = c.take(static_cast<size_t>(N) * K);
  const size_t o_sa = c.take(mt * kt * 512);
  const size_t o_sb = c.take(nt * kt * 512);
  if (ws == nullptr) {
    *ws_bytes = c.off;
    return MOE_OK;
  }
  if (*ws_bytes < c.off) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!all_aligned16({A, B, D}) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(ws, o_st);
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  uint8_t* aq = at<uint8_t>(ws, o_aq);
  uint8_t* bq = at<uint8_t>(ws, o_bq);
  uint8_t* sa = at<uint8_t>(ws, o_sa);
  uint8_t* sb = at<uint8_t>(ws, o_sb);
  MOE_TRY(run("mx_quant_dense_a", s, 0, [&] { return launch_quant_rows_dense(A, M, static_cast<int>(K), aq, sa, s); }));
  MOE_TRY(run("mx_quant_dense_b", s, 0, [&] { return launch_quant_rows_dense(B, N, static_cast<int>(K), bq, sb, s); }));
  GemmArgs a = base_args(st, 0);
  if (!make_map_u8(&a.mapA, aq, K, M, K) || !make_map_u8(&a.mapB0, bq, K, N, K)) return MOE_ERR_CUDA;
  a.mapB1 = a.mapB0;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.out0 = D;
  a.ld0 = static_cast<int>(N);
  a.sfA = sa;
  a.kt_a = static_cast<int>(kt);
  a.sfB0 = sb;
  a.kt_b = static_cast<int>(kt);
  if (N % 256 == 0 && d.sms >= 2) {   // 256 x 256 CTA-pair tiles
    if (!make_map_atoms(&a.mapSFA, sa, mt * kt) || !make_map_atoms(&a.mapSFB, sb, nt * kt))
      return MOE_ERR_CUDA;
    a.n_tiles = static_cast<int>(N / 256);
    const int64_t tiles = static_cast<int64_t>((M + 255) / 256) * a.n_tiles;
    return run("dense_gemm_mx", s, 0,
               [&] { return launch_dense_mx_pair(a, grid_for_pairs(tiles, d.sms), s); });
  }
  a.n_tiles = static_cast<int>(nt);
  const int64_t tiles = static_cast<int64_t>(mt * nt);
  return run("dense_gemm_mx", s, 0, [&] { return launch_dense_mx(a, grid_for(tiles, d.sms), s); });
}

moe_status_t moe_get_device_status(const void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int code = 0;
  if (cudaMemcpyAsync(&code, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(code);
}

void moe_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
}

void moe_profile_select(const char* name) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_only = name != nullptr ? name : "";
}

int moe_profile_read(const char** names, int64_t* launches, double* total_ms, int cap) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (const Pending& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess) {
      Totals& t = g_totals[p.name];
      t.launches += 1;
      t.ms += ms;
    }
    cudaEventDestroy(p.start);
    cudaEventDestroy(p.stop);
  }
  g_pending.clear();
  g_names.clear();
  for (const auto& kv : g_totals) g_names.push_back(kv.first);
  int n = 0;
  for (const auto& kv : g_totals) {
    if (n < cap) {
      if (names) names[n] = g_names[n].c_str();
      if (launches) launches[n] = kv.second.launches;
      if (total_ms) total_ms[n] = kv.second.ms;
    }
    ++n;
  }
  g_totals.clear();
  return n;
}

int64_t moe_launch_count(void) { return g_launches.load(); }

}  // extern "C"

// ---------------------------------------------------------------- routing without a workspace
//
// moe_route_noalloc: the routing pass with its scratch in a file-scope device
// array instead of a caller workspace, for callers that cannot allocate
// device memory.  Host code must not hand the array's name to a kernel (on
// the host it is only a stand-in symbol); its device address is looked up
// once per device with cudaGetSymbolAddress.

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// The array's device address, cached per device together with the unique id
// of the context it was looked up in: after a device reset (a new primary
// context, the module loaded again) the id differs and the address is looked
// up again instead of being reused.
struct NoallocAddr {
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
std::mutex g_noalloc_mu;
NoallocAddr g_noalloc_addr[64];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if it has none yet).
moe_status_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  return MOE_OK;
}

// Device address of g_noalloc_scratch on the current device: looked up with
// cudaGetSymbolAddress (the array's name is only a host-side stand-in) on the
// first call in a context, with that device current, then reused.
moe_status_t noalloc_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = 0;
  MOE_TRY(current_context_id(&id));
  NoallocAddr& c = g_noalloc_addr[dev];
  if (c.addr == nullptr || id == 0 || c.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    MOE_TRY(current_context_id(&id));   // the lookup has made the context current
    c.ctx_id = id;
    c.addr = p;
  }
  *out = c.addr;
  return MOE_OK;
}

// Scratch of the routing pass alone: status word, per-tile histograms and
// bases, W_r^T, the row -> (token, slot) map, row weights, m-tile prefix and
// expert order.
struct RouteScratch {
  size_t status, hist, base, wrt, row_slot, w_row, mtile, order, poff, mtile2, slot_pad, total;
};

RouteScratch route_scratch_layout(const Layout& L) {
  const size_t P = static_cast<size_t>(L.P), E = L.E, H = L.H;
  Carver c;
  RouteScratch r;
  r.status = c.take(sizeof(DeviceStatus));
  r.hist = c.take(sizeof(int) * L.ntiles * E);
  r.base = c.take(sizeof(int) * L.ntiles * E);
  r.wrt = c.take(2 * E * H);
  r.row_slot = c.take(sizeof(int) * static_cast<size_t>(L.Pa));
  r.w_row = c.take(sizeof(float) * static_cast<size_t>(L.Pa));
  r.mtile = c.take(sizeof(int) * (E + 1));
  r.order = c.take(sizeof(int) * E);
  r.poff = c.take(sizeof(int) * (E + 1));
  r.mtile2 = c.take(sizeof(int) * (E + 1));
  r.slot_pad = c.take(sizeof(int) * P);
  r.total = c.off;
  return r;
}

}  // namespace

extern "C" moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_bf16_t* x,
                                          const moe_bf16_t* W_r, const float* logit_bias,
                                          float* logits, int32_t* topk_idx, float* topk_w,
                                          int32_t* counts, int32_t* offsets,
                                          int32_t* perm_token, int32_t* slot_row,
                                          int32_t* device_status, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  if (!all_aligned16({x, W_r}) || topk_idx == nullptr || topk_w == nullptr ||
      counts == nullptr || offsets == nullptr || perm_token == nullptr || slot_row == nullptr ||
      !aligned(logit_bias, 4) || !aligned(logits, 4) || !aligned(device_status, 4))
    return MOE_ERR_INVALID_ARG;
  DevInfo d;
  MOE_TRY(current_device(&d));
  const int sms = sm_budget(d.sms, *cfg);
  const Layout L = make_layout(*cfg, sms);
  const RouteScratch R = route_scratch_layout(L);
  if (R.total > static_cast<size_t>(MOE_NOALLOC_SCRATCH_BYTES)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* base = nullptr;
  MOE_TRY(noalloc_scratch_address(&base));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(base, R.status);
  // the array keeps the previous call's contents: only the status word has to
  // start at zero (every other scratch value is written before it is read)
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  RouteBufs b{x, W_r, logit_bias, logits, topk_idx, topk_w, counts, offsets, perm_token,
              slot_row, at<int>(base, R.row_slot), at<float>(base, R.w_row),
              at<int>(base, R.mtile), at<int>(base, R.order), at<uint16_t>(base, R.wrt),
              at<int>(base, R.hist), at<int>(base, R.base), st, at<int>(base, R.poff),
              at<int>(base, R.mtile2), at<int>(base, R.slot_pad)};
  MOE_TRY(run_routing(*cfg, L, b, sms, s));
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, &st->code, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
