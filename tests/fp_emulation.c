/*
 * fp_emulation.c -- CPU emulation, operation for operation, of two
 * floating-point procedures the CUDA kernels use, so that the claims made
 * about them can be checked on the host:
 *
 *   1. the FP8 quantiser's quotient x / s by one Markstein FMA correction of
 *      x * RN(1/s) (payload_device.cuh, quant_words), against the IEEE
 *      quotient RN(x / s);
 *   2. the router's softmax weights in float-float arithmetic (ffmath.cuh and
 *      route_group_warp in layout_device.cuh), against the same softmax
 *      evaluated in double and rounded once to fp32.
 *
 * TEST CODE. It is neither the oracle nor the CUDA path: it restates the
 * kernels' float steps in C so that they can be run exhaustively or on
 * millions of inputs without a GPU. Every fp32 operation here is one IEEE
 * operation with round-to-nearest-even (gcc -O2 -ffp-contract=off, no
 * fast-math; float arithmetic is evaluated in float on x86-64 and AArch64).
 * The fused multiply-add is emulated exactly from doubles by rounding to odd
 * (S. Boldo and G. Melquiond, "Emulation of FMA and correctly rounded sums:
 * proved algorithms using rounding to odd", IEEE Trans. Computers 57(4),
 * 2008), so the results do not depend on the host's fmaf.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float f_of(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}
static uint32_t u_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* RN(a*b + c) for floats: the product of two floats is exact in a double
 * (48 significant bits); the double sum is rounded to odd (made inexact ->
 * odd last bit, from Knuth's exact TwoSum error), and one final rounding to
 * float then equals the correctly rounded fused result, since double carries
 * more than float's 24 + 2 bits. */
float emu_fmaf(float a, float b, float c) {
    const double p = (double)a * (double)b;
    const double dc = (double)c;
    double s = p + dc;
    const double bb = s - p;
    const double e = (p - (s - bb)) + (dc - bb);
    if (e != 0.0) {
        uint64_t bits;
        memcpy(&bits, &s, 8);
        if ((bits & 1u) == 0) s = nextafter(s, e > 0.0 ? INFINITY : -INFINITY);
    }
    return (float)s;
}

/* ---------------------------------------------------------------------- */
/* 1. Markstein quotient                                                   */
/* ---------------------------------------------------------------------- */

/* The kernel's steps for one value: y = RN(1/s), q0 = RN(x*y),
 * r = RN(x - s*q0), q = RN(r*y + q0) (Markstein's single correction). The
 * kernel then takes the sign of the e4m3 code from x itself, so the sign of
 * a zero quotient returned here does not matter. */
float emu_div_by_scale(float x, float s) {
    const float y = 1.0f / s;
    const float q0 = x * y;
    const float r = emu_fmaf(-s, q0, x);
    return emu_fmaf(r, y, q0);
}

/* Every positive finite bf16 amax with encoding in [amax_lo, amax_hi) and
 * amax >= 2^-64 (the range the kernel sends through this quotient), against
 * every non-negative bf16 x <= amax; s = RN(amax / 448) as in the kernel.
 * Counts the pairs, the quotients that differ from RN(x / s) in any bit, and
 * those differences where either quotient is above 2^-10 (a quotient of
 * magnitude at most 2^-10 has the e4m3 code of a signed zero: 2^-10 is half
 * the smallest subnormal step 2^-9 and ties go to the even code 0).
 * *max_ref_at_diff: the largest |RN(x / s)| among differing pairs. */
void markstein_sweep(uint32_t amax_lo, uint32_t amax_hi, int64_t* pairs, int64_t* n_diff,
                     int64_t* n_code_diff, double* max_ref_at_diff) {
    int64_t np_ = 0, nd = 0, ncd = 0;
    double mx = 0.0;
    const float thr = 0x1p-10f;
    for (uint32_t ab = amax_lo; ab < amax_hi; ++ab) {
        const float amax = f_of(ab << 16);
        if (!(amax >= 0x1p-64f) || isinf(amax) || isnan(amax)) continue;
        const float s = amax / 448.0f;
        for (uint32_t xb = 0; xb <= ab; ++xb) {
            const float x = f_of(xb << 16);
            const float q = emu_div_by_scale(x, s);
            const float ref = x / s;
            ++np_;
            if (u_of(q) != u_of(ref)) {
                ++nd;
                if (fabsf(ref) > mx) mx = fabsf(ref);
                if (fabsf(ref) > thr || fabsf(q) > thr) ++ncd;
            }
        }
    }
    *pairs = np_;
    *n_diff = nd;
    *n_code_diff = ncd;
    *max_ref_at_diff = mx;
}

/* The kernel's quotient for given (x, s) pairs (for sampled checks). */
void markstein_many(int64_t n, const float* x, const float* s, float* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = emu_div_by_scale(x[i], s[i]);
}

/* ---------------------------------------------------------------------- */
/* 2. float-float softmax weights                                          */
/* ---------------------------------------------------------------------- */

typedef struct {
    float hi, lo;
} F2;

static F2 two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    const float e = (a - (s - bb)) + (b - bb);
    F2 r = {s, e};
    return r;
}
static F2 fast_two_sum(float a, float b) {
    const float s = a + b;
    F2 r = {s, b - (s - a)};
    return r;
}
static F2 two_prod(float a, float b) {
    const float p = a * b;
    F2 r = {p, emu_fmaf(a, b, -p)};
    return r;
}
static F2 ff_add(F2 a, F2 b) {
    F2 s = two_sum(a.hi, b.hi);
    const F2 t = two_sum(a.lo, b.lo);
    s.lo = s.lo + t.hi;
    s = fast_two_sum(s.hi, s.lo);
    s.lo = s.lo + t.lo;
    return fast_two_sum(s.hi, s.lo);
}
static F2 ff_mul(F2 a, F2 b) {
    F2 p = two_prod(a.hi, b.hi);
    p.lo = emu_fmaf(a.hi, b.lo, p.lo);
    p.lo = emu_fmaf(a.lo, b.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}
static F2 ff_div(F2 a, F2 b) {
    const float q1 = a.hi / b.hi;
    const F2 qb = ff_mul(b, (F2){q1, 0.0f});
    const F2 r = ff_add(a, (F2){-qb.hi, -qb.lo});
    const float q2 = r.hi / b.hi;
    return fast_two_sum(q1, q2);
}

#define TAYLOR_DEGREE 13
static const double kLn2 = 0.693147180559945309417232121458176568;
static float inv_fact_hi[TAYLOR_DEGREE + 1], inv_fact_lo[TAYLOR_DEGREE + 1];
static float ln2_hi, ln2_lo, inv_ln2;
static int tables_ready = 0;

static void init_tables(void) {
    if (tables_ready) return;
    double f = 1.0;
    for (int i = 0; i <= TAYLOR_DEGREE; ++i) {
        if (i >= 2) f = f / i;  /* 1/i! by the same recursion, in double */
        inv_fact_hi[i] = (float)f;
        inv_fact_lo[i] = (float)(f - (double)(float)f);
    }
    ln2_hi = (float)kLn2;
    ln2_lo = (float)(kLn2 - (double)(float)kLn2);
    inv_ln2 = (float)(1.0 / kLn2);
    tables_ready = 1;
}

static F2 cf(int i) {
    F2 r = {inv_fact_hi[i], inv_fact_lo[i]};
    return r;
}

/* exp(d) = 2^n * m for a float-float d in (-100, 0]: Cody-Waite reduction by
 * ln 2 split in two, degrees 0..7 of the Taylor series in float-float by
 * Estrin's scheme, degrees 8..13 in fp32 by Horner's rule. */
static F2 exp_reduced(F2 d, int* n_out) {
    const float nf = rintf(d.hi * inv_ln2);
    const F2 t = ff_add(two_prod(nf, ln2_hi), (F2){nf * ln2_lo, 0.0f});
    const F2 r = ff_add(d, (F2){-t.hi, -t.lo});
    const F2 p01 = ff_add((F2){1.0f, 0.0f}, r);
    const F2 p23 = ff_add(cf(2), ff_mul(cf(3), r));
    const F2 p45 = ff_add(cf(4), ff_mul(cf(5), r));
    const F2 p67 = ff_add(cf(6), ff_mul(cf(7), r));
    const F2 r2 = ff_mul(r, r);
    const F2 r4 = ff_mul(r2, r2);
    const F2 h = ff_add(ff_add(p01, ff_mul(r2, p23)), ff_mul(r4, ff_add(p45, ff_mul(r2, p67))));
    const float x = r.hi, x2 = x * x, x4 = x2 * x2, x8 = x4 * x4;
    float tail = inv_fact_hi[TAYLOR_DEGREE];
    for (int i = TAYLOR_DEGREE - 1; i >= 8; --i) tail = emu_fmaf(tail, x, inv_fact_hi[i]);
    *n_out = (int)nf;
    return ff_add(h, (F2){x8 * tail, 0.0f});
}

static float pow2f(int n) { return f_of((uint32_t)(n + 127) << 23); }

/* exp(d) as evaluated by the kernel, returned as the double (m.hi + m.lo)*2^n,
 * for d in [-80, 0] (an fp32 d, lo part 0). */
void ff_exp_many(int64_t n, const float* d, double* out) {
    init_tables();
    for (int64_t i = 0; i < n; ++i) {
        int e = 0;
        const F2 m = exp_reduced((F2){d[i], 0.0f}, &e);
        out[i] = ldexp((double)m.hi + (double)m.lo, e);
    }
}

/* The softmax weights of T tokens' chosen logits z[T][k] (slot 0 the
 * largest), exactly as one warp evaluates them: slot j on lane j of a group
 * of K2 lanes (k rounded up to a power of two), d_j = z_j - z_0 exactly as a
 * float-float, exp by exp_reduced scaled by 2^n, the group's sum by a
 * butterfly of float-float adds (lanes past k contribute zero), then
 * w_j = RN(RN(q.hi + q.lo) * 2^n) with q = m_j / sum in float-float. A gap
 * above 80 (a weight below 2^-115) is evaluated in double instead. */
void ff_softmax_many(int64_t T, int k, const float* z, float* w) {
    init_tables();
    int K2 = 1;
    while (K2 < k) K2 <<= 1;
    F2 m[64], sum[64], nxt[64];
    float sc[64];
    int tiny[64];
    for (int64_t g = 0; g < T; ++g) {
        const float* zt = z + g * k;
        const float z0 = zt[0];
        for (int j = 0; j < K2; ++j) {
            const int valid = j < k;
            const F2 d = valid ? two_sum(zt[j], -z0) : (F2){0.0f, 0.0f};
            tiny[j] = d.hi < -80.0f;
            int n = 0;
            m[j] = exp_reduced(tiny[j] ? (F2){0.0f, 0.0f} : d, &n);
            sc[j] = pow2f(n);
            sum[j] = (valid && !tiny[j]) ? (F2){m[j].hi * sc[j], m[j].lo * sc[j]}
                                         : (F2){0.0f, 0.0f};
        }
        for (int o = K2 >> 1; o > 0; o >>= 1) {
            for (int j = 0; j < K2; ++j) nxt[j] = ff_add(sum[j], sum[j ^ o]);
            for (int j = 0; j < K2; ++j) sum[j] = nxt[j];
        }
        for (int j = 0; j < k; ++j) {
            if (!tiny[j]) {
                const F2 q = ff_div(m[j], sum[j]);
                w[g * k + j] = (q.hi + q.lo) * sc[j];
            } else {
                w[g * k + j] = (float)(exp((double)zt[j] - (double)z0) /
                                       ((double)sum[j].hi + (double)sum[j].lo));
            }
        }
    }
}
