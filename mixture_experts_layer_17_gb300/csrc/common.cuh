// Device primitives for sm_103a: mbarriers, TMA tile loads, tcgen05 (TMEM
// allocation, MMA issue, commit, TMEM loads) and the shared-memory / instruction
// descriptors of the 5th-generation tensor cores.  Hand-written inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------- status

// Device status word layout (first 256 bytes of every workspace).
struct DeviceStatus {
  int code;        // moe_status_t of the first device-side failure, 0 if none
  int where;       // which wait ran out or which check failed (kWait* / kCheck* below)
  int block;       // blockIdx.x of the CTA that recorded it
  int index;       // failed index checks: the offending value
  int pad[60];
};
static_assert(sizeof(DeviceStatus) == 256, "status block is 256 bytes");

enum : int {
  kWaitProducerEmpty = 1,
  kWaitMmaFull = 2,
  kWaitMmaTmemEmpty = 3,
  kWaitEpiTmemFull = 4,
  kWaitInjected = 5,
  kWaitDrain = 6,
  kWaitEpiLoad = 7,   // an epilogue's own TMA load of an operand it reads
  // index checks: an expert id, row or token outside its array is recorded
  // (and the access skipped) instead of being used
  kCheckRouterExpert = 16,   // router epilogue: selected expert id
  kCheckPermuteExpert = 17,  // permutation: expert id of a (token, slot)
  kCheckGatherRow = 18,      // dispatch: destination row of a token copy
  kCheckRouterRow = 21,      // router backward: permuted row of a (token, slot)
  kCheckScatterRow = 19,     // scatter epilogues: (token, slot) row of a permuted row
  kCheckUnpermuteExpert = 20,// un-permute / router backward: expert id of a (token, slot)
};

constexpr int kStatusInvalidArg = 1;  // == MOE_ERR_INVALID_ARG
constexpr int kStatusTimeout = 5;     // == MOE_ERR_TIMEOUT

MOE_DEV void record_timeout(DeviceStatus* st, int where) {
  if (st != nullptr && atomicCAS(&st->code, 0, kStatusTimeout) == 0) {
    st->where = where;
    st->block = blockIdx.x;
  }
}

// A failed index check: the first one is kept (code MOE_ERR_INVALID_ARG).
MOE_DEV void record_bad_index(DeviceStatus* st, int where, long long value) {
  if (st != nullptr && atomicCAS(&st->code, 0, kStatusInvalidArg) == 0) {
    st->where = where;
    st->block = blockIdx.x;
    st->index = static_cast<int>(value);
  }
}

// v in [0, n): the unsigned compare also rejects negative values
MOE_DEV bool in_range(long long v, long long n) {
  return static_cast<unsigned long long>(v) < static_cast<unsigned long long>(n);
}

// Index checks of the debug build (compiled with -DMOE_DEVICE_CHECKS): a
// value outside [0, n) is recorded in the status word and `on_fail` runs
// (skipping the access) instead of the value being used.  Without the flag
// the check compiles to nothing: the library writes every index it reads.
#ifdef MOE_DEVICE_CHECKS
#define MOE_CHECK_INDEX(st, where, v, n, on_fail)                  \
  do {                                                             \
    if (!::moe::in_range((v), (n))) {                              \
      ::moe::record_bad_index((st), (where), (v));                 \
      on_fail;                                                     \
    }                                                              \
  } while (0)
#else
#define MOE_CHECK_INDEX(st, where, v, n, on_fail) \
  do {                                            \
  } while (0)
#endif

// ---------------------------------------------------------------- misc

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

MOE_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------------- mbarrier

MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

MOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up,
// returning false, when `*abort` becomes non-zero or after `limit_ns`
// nanoseconds; every wait in this library is bounded this way.
MOE_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, const volatile int* abort,
                               uint64_t limit_ns) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// ---------------------------------------------------------------- TMA

MOE_DEV void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` through the transaction count.  c0 is the innermost coordinate (in
// elements; callers keep c0 * element size a multiple of 16 bytes).
MOE_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// TMA tensor store of one box from shared memory (a bulk async-group
// operation of the issuing thread): the box at coordinates (c0, c1) of the
// map's tensor; rows past the tensor's end are not written.
MOE_DEV void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
               : "memory");
}
// Closes the thread's pending bulk stores into one group.
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of the thread has read its shared
// memory source (the source may then be rewritten; the global writes complete
// on their own, at the latest with the kernel).
MOE_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Programmatic dependent launch: the library launches every kernel with
// programmatic stream serialization, so a kernel's CTAs may start while the
// kernel before it in the stream drains.  Each kernel calls this before it
// touches global memory that an earlier kernel writes or reads; it returns
// once those kernels have completed and their writes are visible (at once
// when the launch had no such attribute).
MOE_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor cores / TMA) before they read it.
MOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

MOE_DEV void tmem_alloc(uint32_t* holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

MOE_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
MOE_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulator),
// cta_group::1.  Issued by one thread.
MOE_DEV void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
MOE_DEV void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape: warp w
// of a warpgroup reads lanes 32*(w%4) .. 32*(w%4)+31).
MOE_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (both >> 4), the fixed version field 0b001 at bit
// 46, base offset 0 (tiles are 1024-byte aligned) and the 128-byte swizzle
// mode (value 2 at bits 61-63).
//   K-major operand, 128B swizzle: rows of 64 bf16 (128 B), 8-row groups of
//     1024 B -> SBO = 1024, LBO unused (16).
//   MN-major operand, 128B swizzle: 64-element MN chunks, each [BK rows of
//     128 B]; LBO = distance between MN chunks, SBO = 1024 (8 K-rows).
MOE_DEV uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
// bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
// 15/16 A/B major (1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// ---------------------------------------------------------------- bf16

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

MOE_DEV void unpack_bf16x2(uint32_t u, float& lo, float& hi) {
  lo = __uint_as_float(u << 16);
  hi = __uint_as_float(u & 0xFFFF0000u);
}

MOE_DEV void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

MOE_DEV uint4 ld_global_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

MOE_DEV uint4 ld_global_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16 fp32 values -> 16 bf16 stored as two 16-byte vectors at p (32-byte aligned)
MOE_DEV void store_bf16x16(void* p, const float (&v)[16]) {
  uint32_t u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  st_global_v4(p, u[0], u[1], u[2], u[3]);
  st_global_v4(static_cast<char*>(p) + 16, u[4], u[5], u[6], u[7]);
}

MOE_DEV void load_bf16x16(const void* p, float (&v)[16]) {
  uint4 a = ld_global_v4(p);
  uint4 b = ld_global_v4(static_cast<const char*>(p) + 16);
  unpack_bf16x2(a.x, v[0], v[1]);
  unpack_bf16x2(a.y, v[2], v[3]);
  unpack_bf16x2(a.z, v[4], v[5]);
  unpack_bf16x2(a.w, v[6], v[7]);
  unpack_bf16x2(b.x, v[8], v[9]);
  unpack_bf16x2(b.y, v[10], v[11]);
  unpack_bf16x2(b.z, v[12], v[13]);
  unpack_bf16x2(b.w, v[14], v[15]);
}

// Logistic function for the SwiGLU epilogues: CUDA's fast exponential and
// fast division (a reciprocal approximation, a few ulp; 1 / inf gives 0 and
// the limits at +-inf are exact), ample for bf16 and E4M3 outputs and far
// cheaper than an IEEE division in epilogues that are instruction-bound.
MOE_DEV float sigmoidf_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// p[i] += v[i] for 16 fp32 values at p (16-byte aligned); loads issued first
MOE_DEV void accum_f32x16(void* p, const float (&v)[16]) {
  char* q = static_cast<char*>(p);
  uint4 o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = ld_global_v4(q + 16 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    st_global_v4(q + 16 * i, __float_as_uint(__uint_as_float(o[i].x) + v[4 * i]),
                 __float_as_uint(__uint_as_float(o[i].y) + v[4 * i + 1]),
                 __float_as_uint(__uint_as_float(o[i].z) + v[4 * i + 2]),
                 __float_as_uint(__uint_as_float(o[i].w) + v[4 * i + 3]));
}

// A 16-column chunk of a weight gradient at element idx of base: stored as
// bf16, or (accumulate mode) added into an fp32 buffer.
MOE_DEV void wgrad_store16(void* base, int64_t idx, bool accum, const float (&v)[16]) {
  if (accum)
    accum_f32x16(static_cast<float*>(base) + idx, v);
  else
    store_bf16x16(static_cast<__nv_bfloat16*>(base) + idx, v);
}

// The same chunk of an expert that received no token: bf16 zeros, or nothing
// to add in accumulate mode.
MOE_DEV void wgrad_zero16(void* base, int64_t idx, bool accum) {
  if (accum) return;
  __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + idx;
  st_global_v4(p, 0u, 0u, 0u, 0u);
  st_global_v4(p + 8, 0u, 0u, 0u, 0u);
}

}  // namespace moe

// ---------------------------------------------------------------- MXFP8

#include <cuda_fp8.h>

namespace moe {

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of
// 16), completion through the mbarrier's transaction count.
MOE_DEV void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Copies one 512-byte scale-factor atom (128 MN-rows x 4 K-blocks of 32,
// row r at byte 16*(r%32) + 4*(r/32) + kblock) from shared memory into four
// TMEM columns, replicated to the four lane quarters.  The TMEM column must be
// a multiple of 4.
MOE_DEV void sf_copy_to_tmem(uint32_t tmem_col_addr, const void* smem_atom) {
  const uint64_t desc = static_cast<uint64_t>((smem_u32(smem_atom) & 0x3FFFFu) >> 4) |
                        (static_cast<uint64_t>(128u >> 4) << 16) |
                        (static_cast<uint64_t>(128u >> 4) << 32) | (1ull << 46);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem_col_addr), "l"(desc)
               : "memory");
}

// D[tmem] (+)= (A * 2^sfA) (B * 2^sfB)^T for one K = 32 block of E4M3 operands
// with E8M0 block scales (OCP MX), cta_group::1.  sf_id in the instruction
// descriptor picks the K-block byte inside the 4-block scale column group.
MOE_DEV void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A/B, UE8M0 scales:
// bits 4-5 B scale id, 7-9 A format (0 = E4M3), 10-12 B format, 15/16 majors,
// 17-22 N >> 3, 23 scale format (1 = UE8M0), 24-28 M >> 4, 29-30 A scale id.
__host__ __device__ constexpr uint32_t make_idesc_mxf8(int M, int N, bool a_mn, bool b_mn) {
  return ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((static_cast<uint32_t>(N) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

MOE_DEV uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t sf_id) {
  return idesc | (sf_id << 4) | (sf_id << 29);
}

// OCP MX shared exponent of a block with absolute maximum amax:
// floor(log2(amax)) - 8 (8 = exponent of E4M3's largest power of two),
// clamped to E8M0's [-127, 127]; an all-zero block takes -127.  For a finite
// normal amax, floor(log2(amax)) is its IEEE biased exponent field minus 127;
// a subnormal amax (field 0) lies below 2^-126 and clamps to -127 as well.
MOE_DEV int mx_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  const int x = ((__float_as_int(amax) >> 23) & 0xff) - 127 - 8;
  return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^-X as an fp32 bit pattern, for the X that mx_exponent returns for finite
// blocks (X <= 119, so the biased exponent 127 - X stays in [8, 254])
MOE_DEV float mx_inv_scale(int X) { return __int_as_float((127 - X) << 23); }

// Four fp32 values scaled by 2^-X, rounded to nearest even E4M3 with
// saturation to +-448, packed little-endian into one word.
MOE_DEV uint32_t to_e4m3x4(float a, float b, float c, float d, float inv_scale) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a * inv_scale, b * inv_scale), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c * inv_scale, d * inv_scale), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// byte offset of (MN row r in [0,128), K-block kb in [0,4)) inside an atom
MOE_DEV int sf_atom_offset(int r, int kb) { return 16 * (r & 31) + 4 * (r >> 5) + kb; }

}  // namespace moe

// ---------------------------------------------------------------- CTA pairs (cta_group::2)

namespace moe {

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
  return r;
}

// Address in the shared::cluster window of the same variable in CTA `rank`.
MOE_DEV uint32_t map_to_rank(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// TMEM allocation shared by a CTA pair: one warp of each CTA executes it and
// both get the same columns.
MOE_DEV void tmem_alloc_pair(uint32_t* holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// M = 256 MMA over a CTA pair: A rows 0-127 and B rows (N) 0..N/2-1 come from
// the issuing (even) CTA's shared memory, the other halves from its peer's at
// the same offsets; each CTA's TMEM receives its 128 rows of D.
MOE_DEV void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// sf_copy_to_tmem for a CTA pair, issued by the leader: the atom at this
// shared-memory offset goes to the same TMEM columns of the pair.
MOE_DEV void sf_copy_to_tmem_pair(uint32_t tmem_col_addr, const void* smem_atom) {
  const uint64_t desc = static_cast<uint64_t>((smem_u32(smem_atom) & 0x3FFFFu) >> 4) |
                        (static_cast<uint64_t>(128u >> 4) << 16) |
                        (static_cast<uint64_t>(128u >> 4) << 32) | (1ull << 46);
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(tmem_col_addr), "l"(desc)
               : "memory");
}

// M = 256 block-scaled MMA over a CTA pair (operand halves as in
// mma_bf16_pair; scale factors in TMEM as the problem places them).
MOE_DEV void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this offset in every CTA of `cta_mask` once the
// pair MMAs issued so far by this thread have completed.
MOE_DEV void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA (cluster address).
MOE_DEV void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                              uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster_addr)
      : "memory");
}

MOE_DEV void mbar_arrive_remote(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}

}  // namespace moe
