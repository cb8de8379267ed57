// gva_device.cuh -- device-side helpers shared by the GVA kernels (sm_103a).
//
// Inline PTX for the Blackwell async-copy machinery (mbarrier transaction counts and the
// bulk-copy engine), bounded waits that report instead of hanging, and the number-format
// conversions the cache needs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gva.h"

namespace gva {

constexpr int kBlockTokens = GVA_BLOCK_TOKENS;
constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMaxDevices = 64;
// A wait on an async copy gives up after this long (the copy engine finishes a tile in
// microseconds; a second means something is wrong) and the kernel reports
// GVA_DEVERR_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (the copy engine) and to the
// other threads of the CTA.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if it did not
// complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---- bulk copy engine -------------------------------------------------------------------

// Contiguous global -> shared copy by the bulk-copy (TMA) engine; completion is counted on
// `bar` as transaction bytes.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before later
// async-proxy (copy engine) accesses, so a buffer can be refilled after it was read.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- number formats ---------------------------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ void bf16x2_to_float2(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// Double -> bf16 with a single round-to-nearest-even.  The double is first narrowed to
// binary32 with round-to-odd (truncate, then force the last bit to 1 if anything was cut
// off); because binary32 keeps at least two more bits than bf16, rounding that value to
// nearest even gives the correctly rounded bf16 (Boldo & Melquiond, "Emulation of FMA and
// correctly rounded sums: proved algorithms using rounding to odd", IEEE TC 2008).
__device__ __forceinline__ __nv_bfloat16 double_to_bf16_rne(double x) {
  float t = __double2float_rz(x);
  if (static_cast<double>(t) != x && isfinite(t)) t = __uint_as_float(__float_as_uint(t) | 1u);
  return __float2bfloat16_rn(t);
}

template <typename T>
struct CacheElem;

template <>
struct CacheElem<float> {
  static __device__ __forceinline__ double to_double(float v) { return static_cast<double>(v); }
  static __device__ __forceinline__ float from_double(double v) { return __double2float_rn(v); }
  static __device__ __forceinline__ float to_float(float v) { return v; }
};

template <>
struct CacheElem<__nv_bfloat16> {
  static __device__ __forceinline__ double to_double(__nv_bfloat16 v) {
    return static_cast<double>(__bfloat162float(v));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_double(double v) {
    return double_to_bf16_rne(v);
  }
  static __device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// ---- fp8 value cache (E4M3 codes with a power-of-two scale per (token, group)) ----------

// Two E4M3 codes (the low 16 bits of x, the first in the low byte) -> two f16 (exact: every
// E4M3 value is an f16 value), the first in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
  uint32_t d;
  const unsigned short h = static_cast<unsigned short>(x & 0xffffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(h));
  return d;
}

// Four E4M3 codes (a 32-bit word, the first in the low byte) -> two f16 pairs: lo holds codes
// 0 and 1, hi codes 2 and 3 (the halves are taken by a register split, not by shifts).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// Two floats -> two E4M3 codes (round to nearest even, magnitudes past 448 clamped to 448),
// the first in the low byte of the result.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(second), "f"(first));
  return d;
}

// 2^e as a float for -126 <= e <= 127 (exact, from the exponent field).
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((e + 127) << 23); }

// Scale exponent of a row of the fp8 value cache whose largest magnitude is amax (a bf16
// value): the smallest e with amax <= 448 * 2^e, clamped to [-126, 120].  From the bits: a
// normal amax = 1.m 2^(E-127) needs e = E - 135, one more when 1.m > 1.75; an amax below
// 2^-126 (or 0) takes the clamp.
__device__ __forceinline__ int fp8_row_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax) & 0x7fffffffu;
  if (u < 0x00800000u) return -126;
  int e = static_cast<int>(u >> 23) - 135 + ((u & 0x7fffffu) > 0x600000u ? 1 : 0);
  return e < -126 ? -126 : (e > 120 ? 120 : e);
}

// RoPE rotation of pair i at position p >= 0: (cos, sin) of p * theta_i, theta_i =
// base^(-2i/d_r).  The context holds, per 8-bit digit of the position, the fp64 cos/sin of
// digit * 256^k * theta_i (computed on the host); the angle of p is the sum of its digits'
// angles, so the rotation is the product of four table rotations (fp64 complex products).
// No transcendental function runs on the device and every int32 position is covered.  The
// four table rows are loaded together (one memory round trip); the digit-0 row is exactly
// (1, 0), so multiplying by it changes nothing.  Table layout: [4 levels][256 digits][pairs]
// of double2 (cos, sin).
constexpr int kRopeLevels = 4;
constexpr int kRopeDigits = 256;

__device__ __forceinline__ void rope_cos_sin(const double2* __restrict__ tab, int pairs,
                                             long long p, int i, double& c, double& s) {
  double2 r[kRopeLevels];
#pragma unroll
  for (int k = 0; k < kRopeLevels; ++k) {
    const int dgt = static_cast<int>((p >> (8 * k)) & (kRopeDigits - 1));
    r[k] = __ldg(&tab[(k * kRopeDigits + dgt) * pairs + i]);
  }
  c = r[0].x;
  s = r[0].y;
#pragma unroll
  for (int k = 1; k < kRopeLevels; ++k) {
    const double c2 = __dsub_rn(__dmul_rn(c, r[k].x), __dmul_rn(s, r[k].y));
    const double s2 = __dadd_rn(__dmul_rn(s, r[k].x), __dmul_rn(c, r[k].y));
    c = c2;
    s = s2;
  }
}

// The same rotation composed in fp32 from the fp32 table (B300's fp64 rate is a small
// fraction of its fp32 rate).  Each table entry is the fp64 value rounded once, so the
// result carries a relative error of a few units of 2^-24: ample for fp32 queries and for
// keys rounded to bf16 afterwards.
__device__ __forceinline__ void rope_cos_sin_f32(const float2* __restrict__ tab, int pairs,
                                                 long long p, int i, float& c, float& s) {
  float2 r[kRopeLevels];
#pragma unroll
  for (int k = 0; k < kRopeLevels; ++k) {
    const int dgt = static_cast<int>((p >> (8 * k)) & (kRopeDigits - 1));
    r[k] = __ldg(&tab[(k * kRopeDigits + dgt) * pairs + i]);
  }
  c = r[0].x;
  s = r[0].y;
#pragma unroll
  for (int k = 1; k < kRopeLevels; ++k) {
    const float c2 = fmaf(c, r[k].x, -s * r[k].y);
    const float s2 = fmaf(s, r[k].x, c * r[k].y);
    c = c2;
    s = s2;
  }
}

// Turns the pair (x0, x1) by the angle whose cosine and sine are (c, s), in fp32.  Every
// fp32 rotation of this library (query and key) goes through this one expression, so a query
// or key rotated by different kernels has the same bits.
__device__ __forceinline__ void rope_rotate_f32(float x0, float x1, float c, float s, float& y0,
                                                float& y1) {
  y0 = fmaf(x0, c, -x1 * s);
  y1 = fmaf(x0, s, x1 * c);
}

// Waits at CTA barrier `id` (1..15; 0 is __syncthreads) for `threads` threads (a multiple of
// 32) and orders their earlier memory accesses before their later ones.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace gva
