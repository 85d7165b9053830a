// common.cuh -- device helpers shared by the libmxq kernels (sm_103a).
//
// Conversions use the hardware's own instructions through inline PTX:
//   cvt.rn.satfinite.e4m3x2.f32   two f32 -> two E4M3, nearest-even
//   cvt.rn.satfinite.e2m1x2.f32   two f32 -> two E2M1, nearest-even
//   cvt.rn.f16x2.e4m3x2 / .e2m1x2 exact widening of the 8/4-bit codes
// IEEE binary32 divide / reciprocal / multiply come from CUDA's
// correctly-rounded intrinsics (__fdiv_rn, __frcp_rn, __fmul_rn).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxq {

template <typename T>
__host__ __device__ __forceinline__ T imin(T a, T b) { return a < b ? a : b; }

constexpr float kE4M3Max = 448.0f;
constexpr float kNvfp4ScaleDenom = 2688.0f;   // 6 * 448

// ---------------------------------------------------------------------------
// Packed bf16 helpers (two bf16 in one 32-bit word, element 0 in the low
// half, as they sit in memory).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// Elementwise max of |a| and |b| for two packed bf16 pairs.  For
// non-negative bf16 values the bit patterns order like the values, so the
// max is taken with the packed bf16 max instruction on sign-cleared words.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;"
      : "=r"(r)
      : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Packed max of magnitudes: each half of the result has magnitude
// max(|a|, |b|) (its sign bit is the XOR of the inputs' and must be
// cleared by the caller before the value is used as a magnitude).
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// max of the two halves of a packed word of non-negative bf16 values,
// returned as the 16-bit pattern.
__device__ __forceinline__ uint32_t bf16x2_hmax(uint32_t w) {
  uint32_t lo = w & 0xFFFFu, hi = w >> 16;
  return lo > hi ? lo : hi;
}

// ---------------------------------------------------------------------------
// Format conversions.
// ---------------------------------------------------------------------------
// Two f32 -> two E4M3 bytes; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight f32 -> eight E2M1 nibbles packed in 32 bits; v[0] lands in the
// lowest nibble (the instruction puts its first source in the upper nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
        "f"(v[6]), "f"(v[7]));
  return r;
}

// Packed f16x2 -> two f32 (exact widening); low half -> a.
__device__ __forceinline__ void f16x2_to_f32(uint32_t h2, float& a, float& b) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(h2));
}

// Two E4M3 bytes (low byte = element 0) -> two f32 (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& a,
                                              float& b) {
  uint32_t h2;
  uint16_t c = (uint16_t)(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  f16x2_to_f32(h2, a, b);
}

// One E4M3 byte -> f32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  float a, b;
  e4m3x2_to_f32(code & 0xFFu, a, b);
  return a;
}

// One byte of two E2M1 nibbles (low nibble = element 0) -> two f32.
__device__ __forceinline__ void e2m1x2_to_f32(uint32_t byte, float& a,
                                              float& b) {
  uint32_t h2;
  asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q;\n\t}"
      : "=r"(h2)
      : "r"(byte & 0xFFu));
  f16x2_to_f32(h2, a, b);
}

// Two IEEE binary32 multiplies (round to nearest even, no flush to zero)
// in one packed f32x2 instruction: r0 = a0 * b0, r1 = a1 * b1.
__device__ __forceinline__ void fmul2(float a0, float a1, float b0, float b1,
                                      float& r0, float& r1) {
  asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pb, {%4, %5};\n\tmul.rn.f32x2 pd, pa, pb;\n\t"
      "mov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// A packed bf16 pair scaled by (s_lo, s_hi) and rounded to two E4M3 codes
// (low half -> low byte).
__device__ __forceinline__ uint32_t bf16x2_scale_e4m3x2(uint32_t w, float s_lo,
                                                        float s_hi) {
  float a, b;
  fmul2(bf16lo_to_f32(w), bf16hi_to_f32(w), s_lo, s_hi, a, b);
  return cvt_e4m3x2(a, b);
}

// Two f32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// MXFP8 scale: from the bf16 bit pattern of a block maximum a >= 0, the
// smallest k in [-127, 127] with 448 * 2^k >= a.  For a normal bf16
// a = (1 + m/128) * 2^e: 448 * 2^k = 1.75 * 2^(k+8), so k = e - 8 when
// m <= 96 (1 + m/128 <= 1.75) and k = e - 7 otherwise; zero and subnormal
// maxima clamp to -127.  Returns the E8M0 byte k + 127.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e8m0_from_amax_bits(uint32_t a) {
  int E = (int)(a >> 7) & 0xFF;
  int m = (int)(a & 0x7F);
  if (E == 0) return 0u;
  int k = (E - 127) - 8 + (m > 96 ? 1 : 0);
  k = k < -127 ? -127 : k;
  return (uint32_t)(k + 127);
}

// 2^-k as an f32 for the E8M0 byte s = k + 127, s in [0, 247]:
// 2^-k = 2^(127 - s), a normal f32 whose biased exponent is 254 - s.
__device__ __forceinline__ float e8m0_inv_scale(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}

// 2^(s - 127) for the E8M0 byte s in [0, 254] (2^-127 is the f32
// subnormal 0x00400000); NaN for 0xFF.
__device__ __forceinline__ float e8m0_scale(uint32_t s) {
  return s == 0     ? __uint_as_float(0x00400000u)
         : s == 255 ? __uint_as_float(0x7FC00000u)   // E8M0 NaN
                    : __uint_as_float(s << 23);
}

// ---------------------------------------------------------------------------
// Swizzled scale layout: byte offset of logical (r, c) in a [R x C] scale
// matrix whose tiles are 128 rows x 4 columns (see include/mxq.h).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t swz_offset(int64_t r, int64_t c,
                                              int64_t col_tiles) {
  int64_t tile = (r >> 7) * col_tiles + (c >> 2);
  int rr = (int)(r & 127);
  return tile * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (int)(c & 3);
}

// ---------------------------------------------------------------------------
// Memory access helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 32-byte global store (sm_100 family); p must be 32-byte aligned.  One
// instruction writes a whole 32-byte sector, where two 16-byte stores
// would each write half of it.
__device__ __forceinline__ void st_v8(void* p, uint4 a, uint4 b) {
  asm volatile(
      "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
      "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z),
      "r"(b.w)
      : "memory");
}

// 32 bytes written as one 32-byte store when `wide` (the caller checked
// 32-byte alignment of the buffer), else as two 16-byte stores.
__device__ __forceinline__ void st_32B(void* p, uint4 a, uint4 b, bool wide);

// 32-byte non-allocating load (sm_100 family); p must be 32-byte aligned.
// L2 cache policy that marks the lines an access touches as the first to
// evict (data read for the last time).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  return pol;
}

// 16- and 32-byte streaming loads under an L2 cache policy.
__device__ __forceinline__ uint4 ld_last_v4(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, "
      "[%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void ld_last_v8(const void* p, uint4& a, uint4& b,
                                           uint64_t pol) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y),
        "=r"(b.z), "=r"(b.w)
      : "l"(p), "l"(pol));
}

__device__ __forceinline__ void ld_stream_v8(const void* p, uint4& a,
                                             uint4& b) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, "
      "[%8];"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y),
        "=r"(b.z), "=r"(b.w)
      : "l"(p));
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_32B(void* p, uint4 a, uint4 b, bool wide) {
  if (wide) {
    st_v8(p, a, b);
  } else {
    st_v4(p, a);
    st_v4(static_cast<uint8_t*>(p) + 16, b);
  }
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b)
               : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier / TMA (inline PTX, sm_90+ forms available on sm_103a).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::
          "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  Gives up after limit_ns (~1 s by
// default; or at once if *abort is already set), ORs 1 into the device
// error word *err, sets *abort so that every other wait of the CTA returns
// at once, and returns false.  Callers keep executing their loop (skipping
// work) so that every CTA-wide barrier is still reached by all threads.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort,
                                          unsigned int* err,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  while (true) {
    if (*abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, 1u);
      *abort = 1;
      return false;
    }
  }
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about hint_ns pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar,
                                                   uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// mbar_wait for warps that have nothing else to do meanwhile: the same
// bounds, but the waiting thread sleeps in the barrier (up to 100 us per
// try) instead of spinning, leaving the issue slots to the warps that work.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                volatile int* abort,
                                                unsigned int* err,
                                                uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  while (true) {
    if (*abort) return false;
    if (mbar_try_wait_hint(bar, parity, 100000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, 1u);
      *abort = 1;
      return false;
    }
  }
}

// 2-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map,
                                            int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared of `bytes` bytes (both addresses 16-byte
// aligned, bytes a multiple of 16), completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src,
                                         uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared -> global 2-D tensor store, tracked by the issuing thread's bulk
// groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map,
                                             uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, "
      "%2}], [%3];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until no committed store group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Programmatic dependent launch.  Every kernel calls pdl_wait() before its
// first global-memory access: it returns once the previous kernel on the
// stream has completed and its writes are visible (and at once when the
// kernel was launched without the programmatic-serialization attribute).
// pdl_launch_dependents() lets the next kernel's CTAs be scheduled while
// this grid drains; they still wait in their own pdl_wait().
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace mxq
