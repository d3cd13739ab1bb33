// layout_device.cuh -- device-side pieces of the layout shared by the
// separate layout kernels (layout.cu) and the persistent single-launch path
// (fused.cu): warp top-k routing with float-float softmax weights, ballot peer
// masks, CTA scans, the per-chunk count/rank body and the layout tables.
// Page citations are in layout.cu.
#pragma once

#include <math.h>
#include <stdint.h>

#include "ffmath.cuh"
#include "internal.cuh"
#include "tables_device.cuh"

namespace moe {
namespace {

// Lanes of the warp holding the same expert id as this lane (one
// match.any; a warp multisplit's peer mask, Ashkiani et al., "GPU
// Multisplit", PPoPP 2016). Lanes with e = -1 match one another; callers
// use the mask only for valid ids. (An earlier form built it from one
// ballot per bit of the id: more instructions, and a layout 1-2 us slower.)
__device__ __forceinline__ unsigned peer_mask(int e) { return __match_any_sync(kFull, e); }

// Order-preserving map of a finite float to an unsigned key (larger float ->
// larger key); -0 is mapped like +0 so that equal logits tie. Key 0 is below
// every finite float and marks an empty or already chosen register.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token by one warp: k rounds of a warp-wide arg-max (larger
// logit first, lower expert index on ties), each round one max-reduction of
// the keys and one min-reduction of the tied candidates' expert indices.
// Register i of a lane holds expert i*32 + lane. Lane j < k returns slot j.
template <int EPL>
__device__ __forceinline__ void load_keys(const float* __restrict__ z, int E, int lane,
                                          unsigned (&key)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    key[i] = e < E ? order_key(__ldg(z + e)) : 0u;
  }
}

template <int EPL>
__device__ __forceinline__ void topk_select(unsigned (&key)[EPL], int k, int lane, int& out_id,
                                            float& out_z) {
  out_id = -1;
  out_z = 0.0f;
  for (int j = 0; j < k; ++j) {
    unsigned bk = 0u;
    unsigned bi = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (key[i] > bk) {  // strict: the lowest register (expert) wins a tie in a lane
        bk = key[i];
        bi = (unsigned)(i * 32 + lane);
      }
    }
    const unsigned m = __reduce_max_sync(kFull, bk);
    const unsigned win = __reduce_min_sync(kFull, bk == m ? bi : 0xffffffffu);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (win == (unsigned)(i * 32 + lane)) key[i] = 0u;
    if (lane == j) {
      out_id = (int)win;
      out_z = key_value(m);
    }
  }
}

// topk_select for NT tokens at once, round by round: the NT tokens' local
// scans and warp reductions are independent, so their latencies overlap
// (NT-way instruction-level parallelism). Tokens u >= nu hold zero keys
// (every lane's best is then no expert) and their outputs are unused.
template <int EPL, int NT>
__device__ __forceinline__ void topk_select_multi(unsigned (&key)[NT][EPL], int k, int lane,
                                                  int (&out_id)[NT], float (&out_z)[NT]) {
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    out_id[u] = -1;
    out_z[u] = 0.0f;
  }
  for (int j = 0; j < k; ++j) {
    unsigned bk[NT], bi[NT], mx[NT], wn[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      bk[u] = 0u;
      bi[u] = 0xffffffffu;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (key[u][i] > bk[u]) {  // strict: the lowest register (expert) wins a tie in a lane
          bk[u] = key[u][i];
          bi[u] = (unsigned)(i * 32 + lane);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) mx[u] = __reduce_max_sync(kFull, bk[u]);
#pragma unroll
    for (int u = 0; u < NT; ++u) wn[u] = __reduce_min_sync(kFull, bk[u] == mx[u] ? bi[u] : 0xffffffffu);
#pragma unroll
    for (int u = 0; u < NT; ++u) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (wn[u] == (unsigned)(i * 32 + lane)) key[u][i] = 0u;
      if (lane == j) {
        out_id[u] = (int)wn[u];
        out_z[u] = key_value(mx[u]);
      }
    }
  }
}

// Top-k of one token by one warp through a threshold: tau, the k-th largest
// of the 32 lane maxima (ties counted), is at most the token's k-th largest
// key, since the lanes whose maximum is at least tau hold k such keys. So
// every key of the top k is a candidate key >= tau (for N(0,1) logits, E =
// 256 and k = 8, about a dozen). The candidates are compacted, one per lane,
// through the warp's 32 (key, expert) pairs in cand, and k rounds of the
// warp arg-max (larger key first, lower expert on ties) select them in
// order, so the result is exactly topk_select's. Returns false, with the
// outputs unset, when more than 32 keys are candidates or fewer than k keys
// are non-zero; the caller then runs topk_select. key is left unchanged.
// Lanes hold expert i*32 + lane in register i, as in topk_select.
template <int EPL>
__device__ __forceinline__ bool topk_threshold(const unsigned (&key)[EPL], int k, int lane,
                                               uint2* cand, int& out_id, float& out_z) {
  unsigned rest = key[0];
#pragma unroll
  for (int i = 1; i < EPL; ++i) rest = max(rest, key[i]);
  unsigned tau = 0u;
  int cnt = 0;
  for (int r = 0; r < k; ++r) {  // warp-uniform; m == 0 counts every lane and ends it
    const unsigned m = __reduce_max_sync(kFull, rest);
    cnt += __popc(__ballot_sync(kFull, rest == m));
    if (rest == m) rest = 0u;
    if (cnt >= k) {
      tau = m;
      break;
    }
  }
  if (tau == 0u) return false;
  int n = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) n += key[i] >= tau ? 1 : 0;
  // this lane's first slot in cand: the candidates of the lanes below it
  constexpr int kBits = EPL >= 32 ? 6 : EPL >= 16 ? 5 : EPL >= 8 ? 4 : EPL >= 4 ? 3 : 2;
  const unsigned below = (1u << lane) - 1u;
  int pos = 0, total = 0;
#pragma unroll
  for (int b = 0; b < kBits; ++b) {
    const unsigned bal = __ballot_sync(kFull, (n >> b) & 1);
    pos += __popc(bal & below) << b;
    total += __popc(bal) << b;
  }
  if (total > 32) return false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if (key[i] >= tau) {
      cand[pos] = make_uint2(key[i], (unsigned)(i * 32 + lane));
      ++pos;
    }
  }
  __syncwarp();
  const uint2 c = lane < total ? cand[lane] : make_uint2(0u, 0xffffffffu);
  __syncwarp();  // cand is free for the warp's next token
  unsigned ck = c.x;
  out_id = -1;
  out_z = 0.0f;
  for (int j = 0; j < k; ++j) {
    const unsigned m = __reduce_max_sync(kFull, ck);
    const unsigned win = __reduce_min_sync(kFull, ck == m ? c.y : 0xffffffffu);
    if (c.y == win) ck = 0u;
    if (lane == j) {
      out_id = (int)win;
      out_z = key_value(m);
    }
  }
  return true;
}

__device__ __forceinline__ float pow2f(int n) {  // 2^n for -126 <= n <= 127
  return __uint_as_float((unsigned)(n + 127) << 23);
}

// Routes up to G = 32/K2 consecutive tokens with one warp (K2 = k rounded up
// to a power of two): selects each token's top-k, then evaluates all their
// softmax weights at once, token t's slot j on lane t*K2 + j. Weights are
// w_j = exp(z_j - z_0) / sum_i exp(z_i - z_0) in float-float arithmetic (see
// ffmath.cuh), rounded once to fp32; the sum is a butterfly inside the lane
// group (its order does not matter at this precision).
// Returns, per lane, its token (lane / K2), slot (lane % K2), id and weight;
// valid is false for lanes past the token count or the top-k.
template <int EPL>
__device__ __forceinline__ void route_group_warp(const float* __restrict__ logits, long long g0,
                                                 int ntok, int E, int k, int K2, int lane,
                                                 bool& valid, int& id, float& w) {
  const int grp = lane / K2, slot = lane - grp * K2;
  valid = grp < ntok && slot < k;
  id = -1;
  float my_z = 0.0f;
  // The logits of up to kPre tokens are loaded before any is selected, and
  // their selections run interleaved; one token alone takes the plain path.
  // (two at E <= 512 beyond 256 experts per warp's registers, so that the
  // interleaved keys still fit the kernel's register budget without spills)
  constexpr int kPre = EPL >= 32 ? 1 : EPL >= 8 ? 2 : 4;
  bool done = false;
  if constexpr (EPL >= 4) {
    if (k <= 8) {
      // the threshold top-k (topk_threshold), one token at a time; each warp
      // of the block (at most kLayoutWarps) owns 32 pairs of cand_s
      __shared__ uint2 cand_s[kLayoutWarps][32];
      uint2* cand = cand_s[threadIdx.x >> 5];
      for (int t0 = 0; t0 < ntok; ++t0) {
        unsigned key[EPL];
        load_keys<EPL>(logits + (g0 + t0) * (long long)E, E, lane, key);
        int tid_;
        float tz;
        if (!topk_threshold<EPL>(key, k, lane, cand, tid_, tz))
          topk_select<EPL>(key, k, lane, tid_, tz);
        const int sid = __shfl_sync(kFull, tid_, slot);
        const float sz = __shfl_sync(kFull, tz, slot);
        if (grp == t0) {
          id = sid;
          my_z = sz;
        }
      }
      done = true;
    }
  }
  if (!done) {
    if (ntok == 1 || kPre == 1) {
      for (int t0 = 0; t0 < ntok; ++t0) {
        unsigned key[EPL];
        load_keys<EPL>(logits + (g0 + t0) * (long long)E, E, lane, key);
        int tid_;
        float tz;
        topk_select<EPL>(key, k, lane, tid_, tz);
        const int sid = __shfl_sync(kFull, tid_, slot);
        const float sz = __shfl_sync(kFull, tz, slot);
        if (grp == t0) {
          id = sid;
          my_z = sz;
        }
      }
    } else {
      for (int t0 = 0; t0 < ntok; t0 += kPre) {
        unsigned key[kPre][EPL];
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
          if (t0 + u < ntok) {
            load_keys<EPL>(logits + (g0 + t0 + u) * (long long)E, E, lane, key[u]);
          } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) key[u][i] = 0u;
          }
        }
        int tid_[kPre];
        float tz[kPre];
        topk_select_multi<EPL, kPre>(key, k, lane, tid_, tz);
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
          if (t0 + u < ntok) {
            const int sid = __shfl_sync(kFull, tid_[u], slot);
            const float sz = __shfl_sync(kFull, tz[u], slot);
            if (grp == t0 + u) {
              id = sid;
              my_z = sz;
            }
          }
        }
      }
    }
  }
  const float z0 = __shfl_sync(kFull, my_z, lane & ~(K2 - 1));
  const ff::F2 d = valid ? ff::two_sum(my_z, -z0) : ff::F2{0.0f, 0.0f};  // exact, <= 0
  const bool tiny = d.hi < -80.0f;  // exp(d) < 2^-115: evaluated separately below
  int n = 0;
  const ff::F2 m = ff::exp_reduced(tiny ? ff::F2{0.0f, 0.0f} : d, n);
  const float sc = pow2f(n);
  ff::F2 sum = (valid && !tiny) ? ff::F2{__fmul_rn(m.hi, sc), __fmul_rn(m.lo, sc)}
                                : ff::F2{0.0f, 0.0f};
  for (int o = K2 >> 1; o > 0; o >>= 1) {
    const ff::F2 other{__shfl_xor_sync(kFull, sum.hi, o), __shfl_xor_sync(kFull, sum.lo, o)};
    sum = ff::add(sum, other);
  }
  if (!tiny) {
    const ff::F2 q = ff::div(m, sum);
    w = __fmul_rn(__fadd_rn(q.hi, q.lo), sc);
  } else {
    // logit gap above 80 inside the top-k: a weight below 2^-115, in double
    w = (float)(exp((double)my_z - (double)z0) / ((double)sum.hi + (double)sum.lo));
  }
}

// The layout tables, by the last CTA of the scan kernel: reads n_kept,
// n_raw and the per-(source, expert) prefixes into shared memory, scans the
// kept counts in global expert order (expert offsets) and derives every
// per-(source, expert) and per-(source, rank) table and the totals. With
// p.defer_tables it writes only the expert offsets, rank bases and totals
// (what the dispatch needs), and source_tables builds the rest later.
__device__ void layout_tables(const LayoutArgs& p, int* smem) {
  const int E = p.E, P = p.P, tid = threadIdx.x, NT = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  int* sk = smem;                   // [E]        kept counts -> expert offsets
  int* sraw = sk + E;               // [E]
  int* pre = sraw + E;              // [(P+1)*E]  prefix at each source's first chunk
  int* Cs = pre + (P + 1) * E;      // [P*P]      count matrix
  int* tmp = Cs + P * P;            // [32]
  int* red = tmp + 32;              // [2]        dropped, raw total
  if (tid < 2) red[tid] = 0;
  for (int e = tid; e < E; e += NT) {
    sk[e] = __ldcg(p.n_kept + e);
    sraw[e] = __ldcg(p.n_raw + e);
  }
  if (!p.defer_tables)
    for (int i = tid; i < (P + 1) * E; i += NT) pre[i] = __ldcg(p.src_pre + i);
  __syncthreads();
  {
    int dr = 0, rw = 0;
    for (int e = tid; e < E; e += NT) {
      rw += sraw[e];
      dr += sraw[e] - sk[e];
    }
    if (dr) atomicAdd(&red[0], dr);
    if (rw) atomicAdd(&red[1], rw);
  }
  // Expert offsets: exclusive scan of kept counts in global expert order.
  const int total = cta_exclusive_scan(sk, E, tmp);
  for (int e = tid; e <= E; e += NT) p.expert_offset[e] = e < E ? sk[e] : total;
  for (int d = tid; d <= P; d += NT) p.rank_base[d] = d < P ? sk[d * p.L] : total;
  if (tid == 0) {
    p.totals[0] = total;
    p.totals[1] = red[0];
    p.totals[2] = (int)(p.Na - (long long)red[1]);
    p.totals[3] = 0;
    *p.done = 0u;  // ready for the next layout on this workspace
  }
  if (p.defer_tables) return;
  auto kept_of = [&](int s, int e) {
    const int a = pre[s * E + e];
    const int c = pre[(s + 1) * E + e] - a;
    return p.cap > 0 ? min(max(p.cap - a, 0), c) : c;
  };
  // Per (source, expert): raw and kept counts, receive offsets.
  for (int it = tid; it < P * E; it += NT) {
    const int s = it / E, e = it - s * E;
    const int a = pre[s * E + e];
    p.cnt[it] = pre[(s + 1) * E + e] - a;
    p.kept_cnt[it] = kept_of(s, e);
    p.recv_offset[it] = sk[e] + (p.cap > 0 ? min(a, p.cap) : a);
  }
  // Count matrix C[s][d] = kept assignments of source s to the experts of d:
  // one thread per (s, d) for few local experts, one warp per (s, d) for many.
  if (p.L < 16) {
    for (int it = tid; it < P * P; it += NT) {
      const int s = it / P, d = it - s * P;
      int sum = 0;
      for (int e = d * p.L; e < (d + 1) * p.L; ++e) sum += kept_of(s, e);
      Cs[it] = sum;
      p.C[it] = sum;
    }
  } else {
    for (int it = warp; it < P * P; it += NT / 32) {
      const int s = it / P, d = it - s * P;
      int sum = 0;
      for (int e = d * p.L + lane; e < (d + 1) * p.L; e += 32) sum += kept_of(s, e);
      sum = __reduce_add_sync(kFull, sum);
      if (lane == 0) {
        Cs[it] = sum;
        p.C[it] = sum;
      }
    }
  }
  __syncthreads();
  // Send offsets: exclusive prefix of C[s][.] over destinations, one warp per s.
  for (int s = warp; s < P; s += NT / 32) {
    int carry = 0;
    for (int d0 = 0; d0 < P; d0 += 32) {
      const int d = d0 + lane;
      const int v = d < P ? Cs[s * P + d] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (d < P) p.send_offset[(long long)s * P + d] = carry + x - v;
      carry += __shfl_sync(kFull, x, 31);
    }
  }
}

// One chunk (CTA b): route its tokens or load their ids, count them per warp,
// write the chunk's per-expert counts into the transposed table
// hist[e * nchunks + b], and give every assignment its stable chunk-local rank
// (assignment code). Shared memory: wcnt[kLayoutWarps][E], ids_s[tpc*k].
template <bool ROUTE, int EPL>
__device__ __forceinline__ void layout_chunk(const LayoutArgs& p, int b, int* smem) {
  const int E = p.E;
  int* wcnt = smem;                                         // [warps][E]
  const int wcnt_ints = kLayoutWarps * E;
  int* ids_s = smem + wcnt_ints;                            // [tpc*k]

  const int s = b / p.cps, c = b - s * p.cps;
  const int t0 = c * p.tpc;
  const int nt = min(p.tpc, p.Tr - t0);
  const long long g0 = (long long)s * p.Tr + t0;
  const long long a0 = g0 * p.k;
  const int na = nt * p.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < wcnt_ints; i += kLayoutThreads) wcnt[i] = 0;
  pdl_wait();  // logits / ids may come from the previous kernel

  if (ROUTE) {
    int K2 = 1;
    while (K2 < p.k) K2 <<= 1;
    // tokens routed together by one warp: one when the chunk is small (latency),
    // up to 32/K2 when there are many (fewer instructions per token)
    const int G = min(32 / K2, (nt + kLayoutWarps - 1) / kLayoutWarps);
    for (int tl0 = warp * G; tl0 < nt; tl0 += kLayoutWarps * G) {
      bool valid;
      int id;
      float wt;
      route_group_warp<EPL>(p.logits, g0 + tl0, min(G, nt - tl0), E, p.k, K2, lane, valid, id, wt);
      if (valid) {
        const int tl = tl0 + lane / K2, j = lane % K2;
        ids_s[tl * p.k + j] = id;
        p.ids_out[(g0 + tl) * p.k + j] = id;
        p.w_out[(g0 + tl) * p.k + j] = wt;
      }
    }
  } else {
    for (int i = tid; i < na; i += kLayoutThreads) {
      int e = __ldg(p.ids_in + a0 + i);
      if (e < -1 || e >= E) {
        atomicOr(p.status, MOE_STATUS_BAD_EXPERT_ID);
        e = -1;
      }
      ids_s[i] = e;
    }
  }
  __syncthreads();

  // Pass 1: per-warp expert counts of the warp's contiguous sub-range.
  const int per = (na + kLayoutWarps - 1) / kLayoutWarps;
  const int beg = min(na, warp * per), end = min(na, beg + per);
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids_s[i] : -1;
    const unsigned m = peer_mask(e);
    if (e >= 0 && lane == __ffs(m) - 1) wcnt[warp * E + e] += __popc(m);
  }
  __syncthreads();
  // Per-expert exclusive scan over warps; the chunk's histogram row.
  for (int e = tid; e < E; e += kLayoutThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kLayoutWarps; ++w) {
      const int v = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += v;
    }
    p.hist[(long long)e * p.nchunks + b] = run;  // transposed: [E][nchunks]
    if (p.acc_add && run) atomicAdd(p.acc_add + e, run);  // the expert's total
    if (p.acc_se && run) atomicAdd(p.acc_se + (long long)s * E + e, run);  // its source's
  }
  __syncthreads();
  // Pass 2: stable rank of every assignment within the chunk and expert.
  const unsigned below = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids_s[i] : -1;
    const unsigned m = peer_mask(e);
    int code = -1;
    if (e >= 0) code = (e << 16) | (wcnt[warp * E + e] + __popc(m & below));
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wcnt[warp * E + e] += __popc(m);
    __syncwarp();
    if (i < end) p.acode[a0 + i] = code;
  }
  // The next kernel may launch only now: a dispatch that follows directly
  // (no scan kernel) would otherwise start loading its token rows while the
  // chunks still route, competing with them for the memory system.
  pdl_trigger();
}

}  // namespace
}  // namespace moe
