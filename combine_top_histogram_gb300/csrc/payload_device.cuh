// payload_device.cuh -- device-side payload helpers shared by the dispatch
// kernels (dispatch.cu) and the persistent single-launch path (fused.cu):
// streaming loads, bf16 unpacking, the per-128-channel amax and the FP8 e4m3
// quantiser (IEEE division, satfinite round-to-nearest-even).
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

// Quantises 8 bf16 values (one 16-byte vector) with scale s; returns the 8
// codes e4m3_satfinite_rne(x / s), the quotient an IEEE division; the codes
// are converted two per instruction (.x in the low byte).
__device__ __forceinline__ uint2 quant8(const uint4 x, float s, bool zero_block) {
  if (zero_block) return make_uint2(0u, 0u);
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 qq = make_float2(__fdiv_rn(bf16_lo(w[q]), s), __fdiv_rn(bf16_hi(w[q]), s));
    const uint32_t c = (uint32_t)__nv_cvt_float2_to_fp8x2(qq, __NV_SATFINITE, __NV_E4M3);
    out[q >> 1] |= c << (16 * (q & 1));
  }
  return make_uint2(out[0], out[1]);
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
