/*
 * moe_oracle.c -- plain, slow CPU oracle for the MoE expert-parallel
 * token-redistribution path (route -> count -> permute/pack -> dispatch ->
 * expert stand-in -> combine/unpermute).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant generator with the
 * CUDA library; it is written from the pages' definitions:
 *
 *   [p1] "[Infra-10] All-to-All Optimization" (xutianle.me), sections 2, 3.5,
 *        4.1, 4.3, 5.1, 5.2, 8.1.
 *   [p3] "Expert Parallel: MoE Token ..." (charlestar.github.io), sections
 *        "A Top-2 routing example", "Why count and permute before dispatch",
 *        "All-to-All-v", "Combine is not simply sending results back",
 *        "Correctness checks come before tuning".
 *   [p4] "Efficient and portable MoE communication" (perplexity / pplx-kernels
 *        blog), introduction (router top-k, weighted sum) and "Dispatch"
 *        (block scale factors).
 *
 * Every function below is a direct definition: explicit loops, one element at
 * a time, in the order the definition states. Built with -O2 -ffp-contract=off
 * and without fast-math so that float arithmetic is IEEE round-to-nearest.
 *
 * Index conventions (shared with the library only as a documented layout):
 *   P ranks, T_r tokens per rank, T = P*T_r tokens, global token g = s*T_r + t.
 *   E experts, L = E/P local experts per rank, owner(e) = e / L.
 *   k slots per token, assignment a = g*k + j, N_a = T*k.
 *   ids[a] in [0,E) is a valid assignment; -1 (or any other value) is masked.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* fp32 -> bf16, round to nearest, ties to even (IEEE 754 rounding of the
 * 24-bit significand to 8 bits). The result keeps the upper 16 bits of the
 * fp32 encoding; the lower 16 bits decide the rounding. Finite inputs only
 * (the path never produces non-finite values). */
uint16_t oref_bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (upper & 1u)))
        upper += 1u; /* a carry into the exponent is the correct rounding */
    return (uint16_t)upper;
}

float oref_f32_from_bf16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, NaN = S.1111.111, largest finite
 * magnitude 1.75 * 2^8 = 448, exponent field 0 encodes subnormals m * 2^-9. */
double oref_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int ex = (code >> 3) & 0xF;
    int man = code & 7;
    double mag;
    if (ex == 15 && man == 7)
        return NAN;
    if (ex == 0)
        mag = ldexp((double)man, -9);
    else
        mag = ldexp(1.0 + man / 8.0, ex - 7);
    return sign ? -mag : mag;
}

/* fp32 -> e4m3 with round-to-nearest-even on the exact value and saturation
 * to +-448 ("satfinite"); the sign of zero is kept. The non-negative finite
 * codes 0x00..0x7E are monotone in value, so the two neighbours of |v| are
 * found by binary search and the nearer one is taken; an exact tie goes to
 * the code with an even mantissa (even code). Finite inputs only. */
uint8_t oref_e4m3_from_f32(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oref_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - oref_e4m3_value((uint8_t)lo);
    double dhi = oref_e4m3_value((uint8_t)hi) - a;
    int code;
    if (dlo < dhi)
        code = lo;
    else if (dhi < dlo)
        code = hi;
    else
        code = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------ */
/* a1: router top-k ([p4] introduction: the top-k scoring experts are chosen   */
/* from the router's probability distribution and the output is the weighted */
/* sum of their outputs; [p3] router output is [num_tokens, top_k] ids and   */
/* weights).                                                                 */
/* ------------------------------------------------------------------------ */

/* For each token: slot 0 holds the largest logit, slot 1 the next, ...; equal
 * logits are ordered by the lower expert index. Weights are the softmax over
 * the k chosen logits, which equals the full softmax renormalised over the
 * chosen experts; computed in double, rounded once to fp32. */
void oref_route_topk(int64_t T, int E, int k, const float *logits,
                     int32_t *ids, float *w)
{
    char *taken = (char *)malloc((size_t)E);
    double *ex = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t g = 0; g < T; ++g) {
        const float *z = logits + g * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || z[e] > z[best])
                    best = e; /* strict '>' keeps the lower index on ties */
            }
            taken[best] = 1;
            ids[g * k + j] = best;
        }
        double zmax = (double)z[ids[g * k + 0]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)z[ids[g * k + j]] - zmax);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j)
            w[g * k + j] = (float)(ex[j] / sum);
    }
    free(ex);
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* a2..a3: count, prefix sums, capacity, receive-row assignment.             */
/* ------------------------------------------------------------------------ */

/* Output of the layout; every array is caller-allocated.
 *   n_raw[E]        valid assignments per expert before capacity
 *   n_kept[E]       rows per expert after capacity (n_e)
 *   expert_offset[E+1] exclusive prefix sum of n_kept, plus the total
 *   cnt[P*E]        cnt[s][e]: valid assignments from source s to expert e
 *   kept_cnt[P*E]   the same, counting kept assignments only
 *   C[P*P]          C[s][d]: kept assignments from source s to rank d
 *   send_offset[P*P] exclusive prefix of C[s][.] over destinations
 *   recv_offset[P*E] first receive row of source s inside expert e's segment
 *   rank_base[P+1]  first receive row of rank d; rank_base[P] = total kept
 *   inv[N_a]        receive row of each assignment, -1 if masked or dropped
 *   totals[3]       kept, dropped, masked
 * Returns the number of ids outside [-1, E) (they are treated as masked). */
typedef struct {
    int32_t *n_raw, *n_kept, *expert_offset, *cnt, *kept_cnt, *C, *send_offset,
        *recv_offset, *rank_base, *inv, *totals;
} oref_layout_t;

static int cmp_u64(const void *x, const void *y)
{
    uint64_t a = *(const uint64_t *)x, b = *(const uint64_t *)y;
    return (a > b) - (a < b);
}

int64_t oref_layout(int P, int64_t Tr, int E, int k, int64_t cap,
                    const int32_t *ids, oref_layout_t *out)
{
    const int L = E / P;
    const int64_t T = (int64_t)P * Tr;
    const int64_t Na = T * k;
    int64_t bad = 0;

    /* The list of valid assignments, keyed by (expert, flat index). The flat
     * index a = ((s*T_r + t)*k + j) orders assignments by (s, t, j), so
     * sorting by the key is the stable sort by expert of the (s, t, j) list
     * ([p3] worked example: every expert's list is in source order). Keys are
     * unique, so any correct sort yields the one stable order. */
    uint64_t *keys = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(Na > 0 ? Na : 1));
    int64_t nv = 0;
    for (int64_t a = 0; a < Na; ++a) {
        int32_t e = ids[a];
        if (e >= 0 && e < E)
            keys[nv++] = ((uint64_t)e << 40) | (uint64_t)a;
        else if (e != -1)
            ++bad;
        out->inv[a] = -1;
    }
    qsort(keys, (size_t)nv, sizeof(uint64_t), cmp_u64);

    for (int e = 0; e < E; ++e) {
        out->n_raw[e] = 0;
        out->n_kept[e] = 0;
    }
    for (int i = 0; i < P * E; ++i) {
        out->cnt[i] = 0;
        out->kept_cnt[i] = 0;
    }
    for (int i = 0; i < P * P; ++i)
        out->C[i] = 0;

    /* Capacity ([p1] 8.1): an expert takes at most cap rows; the first cap
     * assignments of the stable order are kept, the rest are dropped. The
     * receive row of a kept assignment is its position in the kept list. */
    int64_t row = 0;
    for (int64_t i = 0; i < nv; ++i) {
        int e = (int)(keys[i] >> 40);
        int64_t a = (int64_t)(keys[i] & ((1ull << 40) - 1));
        int64_t g = a / k;
        int s = (int)(g / Tr);
        out->n_raw[e] += 1;
        out->cnt[s * E + e] += 1;
        if (cap > 0 && out->n_kept[e] >= cap)
            continue; /* dropped */
        out->n_kept[e] += 1;
        out->kept_cnt[s * E + e] += 1;
        out->C[s * P + e / L] += 1;
        out->inv[a] = (int32_t)row;
        ++row;
    }
    free(keys);

    /* Exclusive prefix sums ([p3] "Prefix sum computes offsets"). */
    out->expert_offset[0] = 0;
    for (int e = 0; e < E; ++e)
        out->expert_offset[e + 1] = out->expert_offset[e] + out->n_kept[e];
    for (int s = 0; s < P; ++s) {
        int32_t acc = 0;
        for (int d = 0; d < P; ++d) {
            out->send_offset[s * P + d] = acc;
            acc += out->C[s * P + d];
        }
    }
    for (int e = 0; e < E; ++e) {
        int32_t acc = out->expert_offset[e];
        for (int s = 0; s < P; ++s) {
            out->recv_offset[s * E + e] = acc;
            acc += out->kept_cnt[s * E + e];
        }
    }
    for (int d = 0; d < P; ++d)
        out->rank_base[d] = out->expert_offset[d * L];
    out->rank_base[P] = out->expert_offset[E];

    int64_t dropped = 0, sum_raw = 0;
    for (int e = 0; e < E; ++e) {
        dropped += out->n_raw[e] - out->n_kept[e];
        sum_raw += out->n_raw[e];
    }
    out->totals[0] = (int32_t)row;
    out->totals[1] = (int32_t)dropped;
    out->totals[2] = (int32_t)(Na - sum_raw);
    return bad;
}

/* Flat-argument wrapper for ctypes. */
int64_t oref_layout_flat(int P, int64_t Tr, int E, int k, int64_t cap,
                         const int32_t *ids, int32_t *n_raw, int32_t *n_kept,
                         int32_t *expert_offset, int32_t *cnt,
                         int32_t *kept_cnt, int32_t *C, int32_t *send_offset,
                         int32_t *recv_offset, int32_t *rank_base,
                         int32_t *inv, int32_t *totals)
{
    oref_layout_t o = {n_raw, n_kept, expert_offset, cnt, kept_cnt, C,
                       send_offset, recv_offset, rank_base, inv, totals};
    return oref_layout(P, Tr, E, k, cap, ids, &o);
}

/* ------------------------------------------------------------------------ */
/* a4..a5: dispatch payload ([p3] payload schema: hidden state, local expert   */
/* id, source token index, top-k slot / routing weight; [p1] 2.1 and 4.1:     */
/* quantisation scale travels with FP8 payloads; [p4] block scale factors).  */
/* ------------------------------------------------------------------------ */

/* Writes, for every kept assignment a = (s,t,j) with row r = inv[a]:
 *   recv_x[r][:] = x[g][:]           (bf16 bits copied unchanged)
 *   local_expert[r] = e mod L, src_rank[r] = s, src_token[r] = t,
 *   slot[r] = j, weight[r] = w[a]. */
void oref_dispatch_bf16(int P, int64_t Tr, int E, int k, int64_t H,
                        const int32_t *ids, const int32_t *inv,
                        const uint16_t *x, const float *w, uint16_t *recv_x,
                        int32_t *local_expert, int32_t *src_rank,
                        int32_t *src_token, int32_t *slot, float *weight)
{
    const int L = E / P;
    const int64_t T = (int64_t)P * Tr;
    for (int64_t g = 0; g < T; ++g) {
        for (int j = 0; j < k; ++j) {
            int64_t a = g * k + j;
            int32_t r = inv[a];
            if (r < 0)
                continue;
            for (int64_t h = 0; h < H; ++h)
                recv_x[(int64_t)r * H + h] = x[g * H + h];
            local_expert[r] = ids[a] % L;
            src_rank[r] = (int32_t)(g / Tr);
            src_token[r] = (int32_t)(g % Tr);
            slot[r] = j;
            weight[r] = w[a];
        }
    }
}

/* FP8 e4m3 quantisation of one token row, per block of 128 channels:
 *   amax = max |x| over the block (exact in fp32),
 *   s = amax / 448 (fp32 division, round to nearest),
 *   q = e4m3_satfinite_rne(x / s) (fp32 division, then the encoder above);
 *   an all-zero block has s = 0 and codes 0. */
void oref_quantize_row_fp8(int64_t H, const uint16_t *xrow, uint8_t *q,
                           float *scales)
{
    for (int64_t b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(oref_f32_from_bf16(xrow[b * 128 + i]));
            if (v > amax)
                amax = v;
        }
        float s = amax / 448.0f;
        scales[b] = s;
        for (int i = 0; i < 128; ++i) {
            float v = oref_f32_from_bf16(xrow[b * 128 + i]);
            q[b * 128 + i] = (amax == 0.0f) ? 0 : oref_e4m3_from_f32(v / s);
        }
    }
}

void oref_dispatch_fp8(int P, int64_t Tr, int E, int k, int64_t H,
                       const int32_t *ids, const int32_t *inv,
                       const uint16_t *x, const float *w, uint8_t *recv_q,
                       float *recv_scale, int32_t *local_expert,
                       int32_t *src_rank, int32_t *src_token, int32_t *slot,
                       float *weight)
{
    const int L = E / P;
    const int64_t T = (int64_t)P * Tr;
    const int64_t nb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *sc = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
    for (int64_t g = 0; g < T; ++g) {
        int any = 0;
        for (int j = 0; j < k; ++j)
            any |= inv[g * k + j] >= 0;
        if (!any)
            continue;
        oref_quantize_row_fp8(H, x + g * H, q, sc);
        for (int j = 0; j < k; ++j) {
            int64_t a = g * k + j;
            int32_t r = inv[a];
            if (r < 0)
                continue;
            memcpy(recv_q + (int64_t)r * H, q, (size_t)H);
            memcpy(recv_scale + (int64_t)r * nb, sc, sizeof(float) * (size_t)nb);
            local_expert[r] = ids[a] % L;
            src_rank[r] = (int32_t)(g / Tr);
            src_token[r] = (int32_t)(g % Tr);
            slot[r] = j;
            weight[r] = w[a];
        }
    }
    free(sc);
    free(q);
}

/* ------------------------------------------------------------------------ */
/* a6: expert stand-ins (the pages' grouped GEMM is out of scope; these give  */
/* a known per-row function so the round trip can be checked).              */
/* ------------------------------------------------------------------------ */

/* y[r] = bf16(c_e * x[r]) with the fp32 product rounded once to fp32 and then
 * to bf16; e = global expert of row r, found from expert_offset. */
void oref_expert_scale_bf16(int E, int64_t H, const int32_t *expert_offset,
                            const float *c, const uint16_t *recv_x,
                            uint16_t *y)
{
    for (int e = 0; e < E; ++e) {
        for (int64_t r = expert_offset[e]; r < expert_offset[e + 1]; ++r) {
            for (int64_t h = 0; h < H; ++h) {
                float v = c[e] * oref_f32_from_bf16(recv_x[r * H + h]);
                y[r * H + h] = oref_bf16_from_f32(v);
            }
        }
    }
}

/* y[r] = bf16(decode(q) * s_block): dequantising identity expert. */
void oref_expert_dequant_fp8(int64_t rows, int64_t H, const uint8_t *recv_q,
                             const float *recv_scale, uint16_t *y)
{
    const int64_t nb = H / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t h = 0; h < H; ++h) {
            float qv = (float)oref_e4m3_value(recv_q[r * H + h]);
            float v = qv * recv_scale[r * nb + h / 128];
            y[r * H + h] = oref_bf16_from_f32(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* a7: combine ([p3] "Combine is not simply sending results back": restore    */
/* token order and merge with router weights, by stable token index, never in */
/* arrival order; [p4] combine: weighted average of the experts' outputs).    */
/* ------------------------------------------------------------------------ */

/* out[g] = bf16(acc), acc = 0; for j = 0..k-1 with inv >= 0:
 *   acc = fma(w[g,j], y[inv[g,j]], acc)   (fp32, one rounding per step).
 * Masked and dropped slots contribute nothing; weights are not renormalised. */
void oref_combine(int64_t T, int k, int64_t H, const int32_t *inv,
                  const float *w, const uint16_t *y, uint16_t *out)
{
    for (int64_t g = 0; g < T; ++g) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int32_t r = inv[g * k + j];
                if (r < 0)
                    continue;
                acc = fmaf(w[g * k + j], oref_f32_from_bf16(y[(int64_t)r * H + h]), acc);
            }
            out[g * H + h] = oref_bf16_from_f32(acc);
        }
    }
}

/* One output token, for sampled checks at full size. */
void oref_combine_token(int k, int64_t H, const int32_t *inv_g,
                        const float *w_g, const uint16_t *y, uint16_t *out_g)
{
    oref_combine(1, k, H, inv_g, w_g, y, out_g);
}
