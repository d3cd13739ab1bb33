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

// Quotients x / s rounded to nearest even, for the scale s = RN(amax / 448)
// of a block whose amax lies in [2^-64, FLT_MAX]: one correction step of the
// product by the reciprocal (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990; Muller et al., "Handbook of Floating-Point Arithmetic", division with
// an FMA): with y = RN(1/s), q0 = RN(x*y), the residual r = x - s*q0 is exact
// in one FMA and RN(q0 + r*y) is the correctly rounded quotient. Only where
// the residual underflows (quotients below 2^-40, whose e4m3 code is a
// signed zero since the smallest e4m3 subnormal is 2^-9) can the last bits
// differ; an exhaustive CPU emulation over every bf16 amax >= 2^-64 and every
// bf16 |x| <= amax (tests/fp_emulation.c) finds the codes identical to those
// of the IEEE quotient. The steps run two values per f32x2 instruction.
// The quotient of x = -0 can come out as +0, so the sign of every code is
// taken from x itself (e4m3 codes are sign-magnitude; a nonzero quotient
// already has the sign of x).

// The sign bits of four bf16 values (two 32-bit words, value order) placed
// at the sign bit of four e4m3 codes in one 32-bit word.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t w0, uint32_t w1) {
  return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// Codes of NW = 4 (8 values) or 8 (16 values) bf16 words w of one block with amax m and scale s = RN(m / 448), as e4m3 satfinite RNE of
// the fp32 quotient x / s, packed in value order (.x of each converted pair
// in the low byte). All-zero blocks give zero codes; blocks whose amax lies
// outside [2^-64, FLT_MAX] (tiny, infinite or NaN) divide value by value.
template <int NW>
__device__ __forceinline__ void quant_words(const uint32_t (&w)[NW], float s, float m,
                                            uint32_t (&out)[NW / 2]) {
#pragma unroll
  for (int i = 0; i < NW / 2; ++i) out[i] = 0u;
  if (m == 0.0f) return;
  // 0x1F800000 and 0x7F800000 are the bits of 2^-64 and +inf: m in [2^-64, +inf)
  if (__float_as_uint(m) - 0x1F800000u < 0x7F800000u - 0x1F800000u) {
    const float y = __frcp_rn(s);
    const unsigned long long y2 = f32x2(y, y), ns2 = f32x2(-s, -s);
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const unsigned long long x2 = f32x2(bf16_lo(w[q]), bf16_hi(w[q]));
      const unsigned long long q0 = mul_f32x2(x2, y2);
      const unsigned long long r = fma_f32x2(ns2, q0, x2);
      const unsigned long long qq = fma_f32x2(r, y2, q0);
      const float2 f = make_float2(__uint_as_float((uint32_t)qq), __uint_as_float((uint32_t)(qq >> 32)));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) out[i] |= sign_bytes(w[2 * i], w[2 * i + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const float2 qq = make_float2(__fdiv_rn(bf16_lo(w[q]), s), __fdiv_rn(bf16_hi(w[q]), s));
      const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(qq, __NV_SATFINITE, __NV_E4M3);
      out[q >> 1] |= c << (16 * (q & 1));
    }
  }
}

// Quantises 8 bf16 values (one 16-byte vector) of a block with amax m and
// scale s; returns the 8 codes in value order.
__device__ __forceinline__ uint2 quant8(const uint4 x, float s, float m) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2];
  quant_words<4>(w, s, m, out);
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

// Bulk asynchronous shared -> global copies (the TMA engine, no tensor map):
// both addresses 16-byte aligned, the size a multiple of 16. A thread commits
// its copies in groups and waits for them with hardware waits (no spinning).
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem_src);
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(s), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed group of this thread has read its source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's ordinary shared-memory writes before later bulk
// copies (the async proxy) that read them.
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// quant8 for 16 values (two 16-byte vectors a, b of one block, in order).
__device__ __forceinline__ uint4 quant16(const uint4 a, const uint4 b, float s, float m) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
  quant_words<8>(w, s, m, out);
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Per-lane bf16 maximum of two bf16x2 words (one instruction); a NaN lane
// yields the other operand, as fmaxf does.
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest |x| of a vector's 8 bf16 values, two lanes per word, folded into
// m (a bf16x2 word of non-negative values; start from 0): the sign bits are
// cleared and the bf16 maxima taken, so the result is exact and never NaN.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, const uint4 x) {
  const uint32_t k = 0x7fff7fffu;
  return max_bf16x2(max_bf16x2(m, max_bf16x2(x.x & k, x.y & k)), max_bf16x2(x.z & k, x.w & k));
}

// The block's amax from each lane's packed maxima, over the lanes that hold
// one 128-channel block (xor offsets LANES/2 .. 1). Non-negative bf16 bit
// patterns (no NaN) order like unsigned integers, so the two halves and the
// lanes are combined with integer maxima.
template <int LANES>
__device__ __forceinline__ float block_amax(uint32_t packed) {
  uint32_t m = max(packed & 0xffffu, packed >> 16);
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  return __uint_as_float(m << 16);
}

// amax of a block whose 128 values are 16 per lane over 8 lanes (a, b: a
// lane's two vectors), or 8 per lane over 16 lanes.
__device__ __forceinline__ float block_amax16(const uint4 a, const uint4 b) {
  return block_amax<8>(absmax_bf16x2(absmax_bf16x2(0u, a), b));
}
__device__ __forceinline__ float block_amax8(const uint4 a) {
  return block_amax<16>(absmax_bf16x2(0u, a));
}

}  // namespace
}  // namespace moe
