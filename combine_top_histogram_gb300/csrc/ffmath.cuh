// ffmath.cuh -- float-float ("double-single") arithmetic on the fp32 pipes,
// used for the router's softmax weights.
//
// Why: the weights are defined as the softmax over the chosen k logits,
// evaluated with ~53-bit precision and rounded once to fp32. GB300 has very
// little FP64 throughput, so evaluating exp/divide in double made the routing
// kernel FP64-bound. A float-float value hi + lo (|lo| <= ulp(hi)/2) carries
// ~48 significant bits using fp32 FMA only, which is enough for the final
// fp32 rounding to agree with a double evaluation except when the exact value
// lies within ~2^-46 (relative) of an fp32 rounding boundary.
//
// Methods (published): error-free sum (Knuth, TAOCP vol. 2, 4.2.2, "TwoSum")
// and fast sum (Dekker 1971), error-free product via FMA; double-length
// multiply / divide after Dekker 1971; exp by the Cody-Waite additive range
// reduction d = n*ln2 + r with ln2 split into two floats, then the Taylor
// series of exp(r) for |r| <= ln2/2: its terms of degree 0..7 in float-float
// by Estrin's scheme (pairs c_i + c_{i+1} r, combined with r^2 and r^4, so the
// dependency chain is three multiply-adds deep instead of thirteen), and the
// terms of degree 8..13, below 2^-27, in plain fp32 by Horner's rule on r.hi,
// added as r^8 * tail. All constants below are values of ln 2 and 1/i!, split
// into hi + lo parts at compile time.
#pragma once

#include <math.h>

namespace moe {
namespace ff {

struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// Requires |a| >= |b| (or a == 0).
__device__ __forceinline__ F2 fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}

__device__ __forceinline__ F2 two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ F2 add(F2 a, F2 b) {
  F2 s = two_sum(a.hi, b.hi);
  F2 t = two_sum(a.lo, b.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = fast_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ F2 mul(F2 a, F2 b) {
  F2 p = two_prod(a.hi, b.hi);
  p.lo = __fmaf_rn(a.hi, b.lo, p.lo);
  p.lo = __fmaf_rn(a.lo, b.hi, p.lo);
  return fast_two_sum(p.hi, p.lo);
}

// a / b: the fp32 quotient q1 (relative error <= 2^-24), the remainder
// a - q1*b of the double-length operands, and one correction q2 = rem / b:
// the error of q1 + q2 is of the order of 2^-47 relative.
__device__ __forceinline__ F2 div(F2 a, F2 b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  const F2 qb = mul(b, F2{q1, 0.0f});
  const F2 r = add(a, F2{-qb.hi, -qb.lo});
  const float q2 = __fdiv_rn(r.hi, b.hi);
  return fast_two_sum(q1, q2);
}

__device__ __forceinline__ F2 scale(F2 a, int n) { return {ldexpf(a.hi, n), ldexpf(a.lo, n)}; }

// ln 2 = 0.693147180559945309417232121458176568..., split hi + lo.
constexpr double kLn2 = 0.693147180559945309417232121458176568;
constexpr float kLn2Hi = (float)kLn2;
constexpr float kLn2Lo = (float)(kLn2 - (double)(float)kLn2);
static_assert(kLn2Hi > 0.0f, "ln 2 split");
constexpr float kInvLn2 = (float)(1.0 / kLn2);

constexpr double inv_fact(int i) { return i <= 1 ? 1.0 : inv_fact(i - 1) / i; }
constexpr float hi_part(double c) { return (float)c; }
constexpr float lo_part(double c) { return (float)(c - (double)(float)c); }
constexpr int kTaylorDegree = 13;  // |r| <= 0.35: the first omitted term is < 2^-52

// 1/i!, i = 0..13, split hi + lo (evaluated by the compiler).
__constant__ float kInvFactHi[kTaylorDegree + 1] = {
    hi_part(inv_fact(0)), hi_part(inv_fact(1)), hi_part(inv_fact(2)), hi_part(inv_fact(3)),
    hi_part(inv_fact(4)), hi_part(inv_fact(5)), hi_part(inv_fact(6)), hi_part(inv_fact(7)),
    hi_part(inv_fact(8)), hi_part(inv_fact(9)), hi_part(inv_fact(10)), hi_part(inv_fact(11)),
    hi_part(inv_fact(12)), hi_part(inv_fact(13))};
__constant__ float kInvFactLo[kTaylorDegree + 1] = {
    lo_part(inv_fact(0)), lo_part(inv_fact(1)), lo_part(inv_fact(2)), lo_part(inv_fact(3)),
    lo_part(inv_fact(4)), lo_part(inv_fact(5)), lo_part(inv_fact(6)), lo_part(inv_fact(7)),
    lo_part(inv_fact(8)), lo_part(inv_fact(9)), lo_part(inv_fact(10)), lo_part(inv_fact(11)),
    lo_part(inv_fact(12)), lo_part(inv_fact(13))};

// exp(d) for a float-float d with -100 < d <= 0: returns m and n with
// exp(d) = 2^n * m, m in [~0.70, ~1.42] as float-float.
__device__ __forceinline__ F2 exp_reduced(F2 d, int& n_out) {
  const float nf = rintf(__fmul_rn(d.hi, kInvLn2));
  // r = d - nf*ln2; nf*ln2 formed as a float-float product
  const F2 t = add(two_prod(nf, kLn2Hi), F2{__fmul_rn(nf, kLn2Lo), 0.0f});
  const F2 r = add(d, F2{-t.hi, -t.lo});
  auto c = [](int i) { return F2{kInvFactHi[i], kInvFactLo[i]}; };
  const F2 p01 = add(F2{1.0f, 0.0f}, r);  // 1/0! + r/1!
  const F2 p23 = add(c(2), mul(c(3), r));
  const F2 p45 = add(c(4), mul(c(5), r));
  const F2 p67 = add(c(6), mul(c(7), r));
  const F2 r2 = mul(r, r);
  const F2 r4 = mul(r2, r2);
  const F2 h = add(add(p01, mul(r2, p23)), mul(r4, add(p45, mul(r2, p67))));
  // degrees 8..13 in fp32: |r^8/8!| < 2^-27, so fp32 rounding stays below 2^-50
  const float x = r.hi, x2 = __fmul_rn(x, x), x4 = __fmul_rn(x2, x2), x8 = __fmul_rn(x4, x4);
  float tail = kInvFactHi[kTaylorDegree];
#pragma unroll
  for (int i = kTaylorDegree - 1; i >= 8; --i) tail = __fmaf_rn(tail, x, kInvFactHi[i]);
  n_out = (int)nf;
  return add(h, F2{__fmul_rn(x8, tail), 0.0f});
}

}  // namespace ff
}  // namespace moe
