// payload_device.cuh -- device-side payload helpers shared by the dispatch
// kernels (dispatch.cu) and the persistent single-launch path (fused.cu):
// streaming loads, bf16 unpacking, the per-128-channel amax and the FP8 e4m3
// quantiser (correctly rounded quotient, satfinite round-to-nearest-even).
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  // x is read exactly once: do not keep it in L1.
  return __ldlu(p);
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// x / s rounded to nearest even, for s = RN(amax / 448) of a block whose amax
// lies in [2^-64, FLT_MAX]: Markstein's FMA-based quotient correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also Muller et al.,
// "Handbook of Floating-Point Arithmetic", section on division with an FMA).
// With yh = RN(1/s) and the float-float reciprocal yh + yl, the first quotient
// q0 = RN(x*yh + x*yl) lies within one ulp of x/s, the residual
// r = x - s*q0 is exact in one FMA, and RN(q0 + r*yh) is the correctly
// rounded quotient. Where x is so small that the residual underflows, the
// result can differ from x/s in its last bits; an exhaustive CPU check over
// every finite bf16 amax >= 2^-64 and every bf16 x with |x| <= amax found such
// differences only for quotients below 2^-40, where every e4m3 code is a
// signed zero (the smallest e4m3 subnormal is 2^-9), and the e4m3 codes
// identical to those of the IEEE quotient everywhere. The sign is carried
// over from x so that -0 stays -0.
__device__ __forceinline__ float div_by_scale(float x, float s, float yh, float yl) {
  const float q0 = __fmaf_rn(x, yh, __fmul_rn(x, yl));
  const float r = __fmaf_rn(-s, q0, x);
  const float q = __fmaf_rn(r, yh, q0);
  return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

// Quantises 8 bf16 values (one 16-byte vector) of a block with amax m and
// scale s = RN(m / 448); returns the 8 codes e4m3_satfinite_rne(x / s), the
// quotient rounded to nearest even in fp32; the codes are converted two per
// instruction (.x in the low byte). Blocks with m in [2^-64, FLT_MAX] take
// the FMA quotient above (one correctly rounded reciprocal per vector instead
// of one division per value); all-zero blocks give zero codes; any other
// block (tiny, infinite or NaN amax) divides value by value.
__device__ __forceinline__ uint2 quant8(const uint4 x, float s, float m) {
  if (m == 0.0f) return make_uint2(0u, 0u);
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2] = {0u, 0u};
  // 0x1F800000 and 0x7F800000 are the bits of 2^-64 and +inf: m in [2^-64, +inf)
  if (__float_as_uint(m) - 0x1F800000u < 0x7F800000u - 0x1F800000u) {
    const float yh = __frcp_rn(s);
    const float yl = __fmul_rn(__fmaf_rn(-s, yh, 1.0f), yh);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 qq = make_float2(div_by_scale(bf16_lo(w[q]), s, yh, yl),
                                    div_by_scale(bf16_hi(w[q]), s, yh, yl));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(qq, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 qq = make_float2(__fdiv_rn(bf16_lo(w[q]), s), __fdiv_rn(bf16_hi(w[q]), s));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(qq, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
  }
  return make_uint2(out[0], out[1]);
}

// 32 bytes (16 bf16 values) in one 256-bit load, last-use hint; p 32-byte aligned.
__device__ __forceinline__ void ld_stream32(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.lu.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

// Asynchronous 16-byte global -> shared copies (cp.async, completion tracked
// per thread in commit groups; the waits are hardware waits, not spins).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most one of this thread's committed groups is still pending.
__device__ __forceinline__ void cp_async_wait_prev() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Two fp32 lanes in one 64-bit register (first value in the low half) and the
// packed round-to-nearest multiply and fused multiply-add, each lane rounded
// exactly as the scalar operation.
__device__ __forceinline__ unsigned long long f32x2(float lo, float hi) {
  return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ unsigned long long mul_f32x2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// quant8 for 16 values (two 16-byte vectors a, b of one block): the same
// quotient and codes, the FMA steps of div_by_scale on two values per
// instruction. Returns the 16 codes in memory order.
__device__ __forceinline__ uint4 quant16(const uint4 a, const uint4 b, float s, float m) {
  if (m == 0.0f) return make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4] = {0u, 0u, 0u, 0u};
  if (__float_as_uint(m) - 0x1F800000u < 0x7F800000u - 0x1F800000u) {
    const float yh = __frcp_rn(s);
    const float yl = __fmul_rn(__fmaf_rn(-s, yh, 1.0f), yh);
    const unsigned long long yh2 = f32x2(yh, yh), yl2 = f32x2(yl, yl), ns2 = f32x2(-s, -s);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned long long x2 = f32x2(bf16_lo(w[q]), bf16_hi(w[q]));
      const unsigned long long q0 = fma_f32x2(x2, yh2, mul_f32x2(x2, yl2));
      const unsigned long long r = fma_f32x2(ns2, q0, x2);
      const unsigned long long qq = fma_f32x2(r, yh2, q0) | (x2 & 0x8000000080000000ull);
      const float2 f = make_float2(__uint_as_float((uint32_t)qq), __uint_as_float((uint32_t)(qq >> 32)));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float2 qq = make_float2(__fdiv_rn(bf16_lo(w[q]), s), __fdiv_rn(bf16_hi(w[q]), s));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(qq, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ float amax8(const uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float m = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    m = fmaxf(m, fabsf(bf16_lo(w[q])));
    m = fmaxf(m, fabsf(bf16_hi(w[q])));
  }
  return m;
}

}  // namespace
}  // namespace moe
