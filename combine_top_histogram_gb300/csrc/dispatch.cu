// dispatch.cu -- permute + pack + all-to-all-v scatter, with optional fused
// FP8 e4m3 quantisation (per token and 128-channel block, fp32 scale).
//
// Pages: "[Infra-10] All-to-All Optimization", 4.3 (write the permutation
// straight into the destination-contiguous communication buffer, no temporary
// permutation buffer), 5.1 (one pass writes hidden states, token index and
// routing weight), 5.2 (destination segments bucketed by local expert; the
// network output buffer is the expert kernel's input), 4.1 (FP8 on the wire
// with scale metadata); "Expert Parallel: MoE Token ...", payload schema and
// the bijection (every valid assignment sent exactly once);
// "Efficient and portable MoE communication", "Dispatch" (block scale
// factors travel with the tokens).
//
// One GPU: the P virtual ranks' receive segments are ranges of one receive
// buffer, so "sending" an assignment is storing its row at its receive row.
// Each CTA takes one token at a time: reads the bf16 row from HBM once into
// registers (16-byte loads; 32-byte loads for FP8 when x allows), quantises it
// once if FP8, and stores it to each of the token's k receive rows (coalesced
// 16- or 8-byte stores). The receive row of slot j is
//     r = expert_offset[e] + chunk_base[chunk][e] + chunk-local rank
// (the stable (expert, source, token, slot) order) and is kept iff its
// in-expert position is below the capacity. The fixed-slot comparator instead
// uses (e*P + s)*T_r + (rank among source s's assignments to e).
//
// Nothing in the copy needs the per-source tables (cnt, kept counts, receive
// offsets per source, C and the send offsets), so when the layout deferred
// them the first P CTAs of the launch build them, one source rank each, while
// the other CTAs copy tokens; they are complete when the dispatch is.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"
#include "payload_device.cuh"
#include "tables_device.cuh"

namespace moe {
namespace {

constexpr int kDispatchThreads = 128;

// CTA blockIdx.x < p.tab_ctas of a dispatch launch: the tables of source
// rank blockIdx.x (dynamic shared memory: E + 32 ints).
__device__ void tables_cta(const DispatchArgs& p) {
  extern __shared__ int tab_s[];
  pdl_wait();
  pdl_trigger();
  source_tables(p.tab, blockIdx.x, tab_s);
}

__global__ void __launch_bounds__(kDispatchThreads) k_tables(const TablesArgs t) {
  extern __shared__ int tab_s[];
  pdl_wait();
  pdl_trigger();
  source_tables(t, blockIdx.x, tab_s);
}

// The assignment code and weight of slot j = threadIdx.x of token g. With
// the scan kernel between the layout and the dispatch, the codes (and routed
// weights) come from a launch at least two before, so under the launch rule
// above they are complete when the dispatch starts and may be loaded before
// its wait; in direct mode (no scan kernel) they are loaded after it.
struct SlotIn {
  int code;
  float w;
};
__device__ __forceinline__ SlotIn load_slot(const DispatchArgs& p, long long g) {
  const int j = threadIdx.x;
  if (j >= p.k) return SlotIn{-1, 0.0f};
  const long long a = g * p.k + j;
  return SlotIn{__ldg(p.acode + a), __ldg(p.w + a)};
}

// Resolves the k receive rows of token g into rows_s, writes inv and the row
// metadata. Threads 0..k-1 each take one slot (in: load_slot of the token).
__device__ __forceinline__ void resolve_rows(const DispatchArgs& p, long long g, int* rows_s,
                                             SlotIn in, int* owner_s = nullptr) {
  const int j = threadIdx.x;
  if (j >= p.k) return;
  const long long a = g * p.k + j;
  const int code = in.code;
  int r = -1;
  // (debug bounds build: an assignment code naming no expert, or a chunk
  // outside the table, is skipped like a row outside its buffer)
  if (code >= 0 && row_ok(code_expert(code), p.E, p.status) &&
      row_ok((g / p.Tr) * p.cps + (g % p.Tr) / p.tpc, p.nchunks, p.status)) {
    const int e = code_expert(code);
    const int s = (int)(g / p.Tr);
    const int t = (int)(g - (long long)s * p.Tr);
    const int b = s * p.cps + t / p.tpc;
    const int pos = __ldg(p.hist + (long long)e * p.nchunks + b) + code_rank(code);
    // fixed slots: q is the rank among source s's assignments to e; a region
    // has slot_Tr rows, enough unless an id repeats within a token
    const int q = p.slot_Tr > 0 ? pos - __ldg(p.src_pre + (long long)s * p.E + e) : 0;
    if (p.slot_Tr > 0 && q >= p.slot_Tr) atomicOr(p.status, MOE_STATUS_SLOT_OVERFLOW);
    if ((p.cap <= 0 || pos < p.cap) && q < max(p.slot_Tr, 1)) {
      r = p.slot_Tr > 0 ? (e * p.P + s) * p.slot_Tr + q : __ldg(p.expert_offset + e) + pos;
      if (!row_ok(r, p.row_limit, p.status)) r = -1;
      if (r >= 0) {
        p.m_local_expert[r] = e % p.L;
        p.m_src_rank[r] = s;
        p.m_src_token[r] = t;
        p.m_slot[r] = j;
        p.m_weight[r] = in.w;
      }
    }
  }
  p.inv[a] = r;
  if (owner_s) owner_s[j] = code >= 0 ? code_expert(code) / p.L : 0;
  int dst = r;
  if (p.send_pos && r >= 0) {
    const long long se = (long long)code_expert(code) + (long long)(g / p.Tr) * p.E;
    dst = __ldg(p.src_base + g / p.Tr) + __ldg(p.send_pos + se) + (r - __ldg(p.recv_offset + se));
    if (!row_ok(dst, p.row_limit, p.status)) dst = -1;
  }
  rows_s[j] = dst;
}

// ---- direct mode ----------------------------------------------------------
// Small, latency-bound layouts (decode) skip the scan kernel: the dispatch
// follows the layout kernel directly. A slot's receive row is
//   (kept assignments to experts before e) + (assignments to e from earlier
//   sources) + (from the source's earlier chunks) + chunk-local rank,
// from the per-expert totals acc, the per-(source, expert) totals acc_se and
// the raw chunk counts in hist that the layout kernel left: every CTA scans the
// per-expert totals into expert offsets in shared memory, and direct_G lanes
// sum each slot's other terms in one round trip. The launch's first P CTAs
// build the per-source tables the same way (CTA 0 also the per-expert arrays).
//
// Dynamic shared memory of a direct-mode CTA (ints): eoff[E+1] | tmp[32] |
// red[2] | (tables CTAs) sk[E + 32].
__host__ __device__ constexpr int direct_smem_ints(int E) { return (E + 1) + 32 + 2 + (E + 32); }

// The first per-expert totals this thread scans (experts tid and
// tid + blockDim), loaded into registers ahead of the scan; the scan loads
// any further ones (E > 2 * blockDim) itself.
constexpr int kDirectTotalsPerThread = 2;
__device__ __forceinline__ void direct_totals_load(const DispatchArgs& p,
                                                   int (&raw)[kDirectTotalsPerThread]) {
#pragma unroll
  for (int i = 0; i < kDirectTotalsPerThread; ++i) {
    const int e = threadIdx.x + i * blockDim.x;
    raw[i] = e < p.E ? __ldcg(p.acc + e) : 0;
  }
}

// The expert offsets from loaded totals (direct_totals_load), as
// direct_offsets computes them.
__device__ void direct_offsets_scan(const DispatchArgs& p, int* dsm, bool writer,
                                    const int (&raw_in)[kDirectTotalsPerThread]) {
  const int E = p.E, tid = threadIdx.x, NT = blockDim.x;
  int* eoff = dsm;
  int* tmp = eoff + E + 1;
  int* red = tmp + 32;
  if (tid < 2) red[tid] = 0;
  int dr = 0, rw = 0;
  for (int i = 0; tid + i * NT < E; ++i) {
    const int e = tid + i * NT;
    static_assert(kDirectTotalsPerThread == 2, "registers named below");
    const int raw = i == 0 ? raw_in[0] : i == 1 ? raw_in[1] : __ldcg(p.acc + e);
    const int kept = (p.cap > 0 && raw > p.cap) ? p.cap : raw;
    eoff[e] = kept;
    if (writer) {
      p.n_raw[e] = raw;
      p.n_kept[e] = kept;
    }
    rw += raw;
    dr += raw - kept;
  }
  __syncthreads();
  if (writer) {
    if (dr) atomicAdd(&red[0], dr);
    if (rw) atomicAdd(&red[1], rw);
  }
  const int total = cta_exclusive_scan(eoff, E, tmp);
  if (tid == 0) eoff[E] = total;
  if (writer) {
    for (int e = tid; e <= E; e += NT) p.expert_offset_out[e] = e < E ? eoff[e] : total;
    for (int d = tid; d <= p.P; d += NT) p.rank_base[d] = d < p.P ? eoff[d * p.L] : total;
    if (tid == 0) {
      p.totals[0] = total;
      p.totals[1] = red[0];
      p.totals[2] = (int)(p.Na - (long long)red[1]);
      p.totals[3] = 0;
    }
  }
  __syncthreads();
}

// Expert offsets of the layout in eoff[0..E] (kept counts, capacity applied,
// scanned in global expert order); the writer CTA also stores n_raw, n_kept,
// expert_offset, rank_base and the layer totals.
__device__ void direct_offsets(const DispatchArgs& p, int* dsm, bool writer) {
  int raw[kDirectTotalsPerThread];
  direct_totals_load(p, raw);
  direct_offsets_scan(p, dsm, writer, raw);
}

// Every CTA of a direct-mode launch counts itself out on the arrival counter
// once it has read the totals for the last time (thread 0's atomic, whose
// ticket it keeps); the CTA that counted out last clears the totals and the
// counter for the next layout, after its own work.
__device__ __forceinline__ unsigned direct_count_out(const DispatchArgs& p) {
  return threadIdx.x == 0 ? atomicAdd(p.arrive, 1u) : 0u;
}
__device__ void direct_end(const DispatchArgs& p, unsigned ticket) {
  __shared__ unsigned s_ticket;
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = ticket;
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.acc[e] = 0;
  for (int i = threadIdx.x; i < p.P * p.E; i += blockDim.x) p.acc_se[i] = 0;
  if (threadIdx.x == 0) *p.arrive = 0u;
}

// The code of the slot whose terms this thread helps to sum (direct_G lanes
// per slot).
__device__ __forceinline__ int load_group_code(const DispatchArgs& p, long long g) {
  const int jt = threadIdx.x / p.direct_G;
  return jt < p.k ? __ldg(p.acode + g * p.k + jt) : -1;
}

// Slot j's assignments to its expert that precede token g's chunk: those of
// earlier sources (acc_se) and of the source's earlier chunks (raw hist),
// spread over direct_G lanes; this lane's partial sum (its loads issued as
// soon as the code is known), then the sum over the lanes into pre[j].
// Every thread of the CTA takes part in the reduction (warp-wide shuffles).
__device__ __forceinline__ int direct_slot_terms(const DispatchArgs& p, long long g, int code) {
  const int G = p.direct_G, jt = threadIdx.x / G, li = threadIdx.x - jt * G;
  int sp = 0;
  if (jt < p.k && code >= 0 && row_ok(code_expert(code), p.E, p.status)) {
    const int e = code_expert(code);
    const int s = (int)(g / p.Tr);
    const int bs = (int)(g - (long long)s * p.Tr) / p.tpc;  // chunk within the source
    for (int s2 = li; s2 < s; s2 += G) sp += __ldcg(p.acc_se + (long long)s2 * p.E + e);
    const int32_t* col = p.hist + (long long)e * p.nchunks + (long long)s * p.cps;
    for (int c = li; c < bs; c += G) sp += __ldcg(col + c);
  }
  return sp;
}
__device__ __forceinline__ void direct_slot_reduce(const DispatchArgs& p, int sp, int* pre) {
  const int G = p.direct_G, jt = threadIdx.x / G, li = threadIdx.x - jt * G;
  for (int o = G >> 1; o > 0; o >>= 1) sp += __shfl_xor_sync(0xffffffffu, sp, o);
  if (li == 0 && jt < p.k) pre[jt] = sp;
}

// resolve_rows for direct mode: the row of slot j is eoff[e] + pos with
// pos = pre[j] + rank, kept iff pos is below the capacity.
__device__ __forceinline__ void resolve_rows_direct(const DispatchArgs& p, long long g,
                                                    int* rows_s, SlotIn in, const int* eoff,
                                                    const int* pre) {
  const int j = threadIdx.x;
  if (j >= p.k) return;
  const long long a = g * p.k + j;
  const int code = in.code;
  int r = -1;
  if (code >= 0 && row_ok(code_expert(code), p.E, p.status)) {
    const int e = code_expert(code);
    const int pos = pre[j] + code_rank(code);
    if (p.cap <= 0 || pos < p.cap) {
      r = eoff[e] + pos;
      if (!row_ok(r, p.row_limit, p.status)) r = -1;
      if (r >= 0) {
        const int s = (int)(g / p.Tr);
        p.m_local_expert[r] = e % p.L;
        p.m_src_rank[r] = s;
        p.m_src_token[r] = (int)(g - (long long)s * p.Tr);
        p.m_slot[r] = j;
        p.m_weight[r] = in.w;
      }
    }
  }
  p.inv[a] = r;
  rows_s[j] = r;
}

// The k receive rows of token g into rows_s (either mode); the caller ends
// with a barrier before reading rows_s. in: the token's slot codes and
// weights (loaded here in direct mode); dsm: the direct mode's shared memory,
// whose expert offsets the CTA's first token computes (offsets_done).
template <bool DIRECT>
__device__ __forceinline__ void resolve_token(const DispatchArgs& p, long long g, int* rows_s,
                                              SlotIn& in, int* dsm, bool& offsets_done) {
  if (DIRECT) {
    // three round trips overlapped: the codes and (first token) the totals
    // are loaded together, the slot terms as soon as the codes arrive, and
    // those land while the totals are scanned into the expert offsets
    in = load_slot(p, g);
    const int code = load_group_code(p, g);
    int raw[kDirectTotalsPerThread];
    const bool first = !offsets_done;
    if (first) direct_totals_load(p, raw);
    const int sp = direct_slot_terms(p, g, code);
    if (first) direct_offsets_scan(p, dsm, false, raw);
    offsets_done = true;
    __shared__ int pre[MOE_MAX_TOPK];
    direct_slot_reduce(p, sp, pre);
    __syncthreads();
    resolve_rows_direct(p, g, rows_s, in, dsm, pre);
  } else {
    resolve_rows(p, g, rows_s, in);
  }
}

// Direct mode, source s = blockIdx.x < P: the per-source tables from the
// totals (a = assignments to e from earlier sources, c = from s itself), as
// source_tables derives them from the scanned prefixes; CTA 0 writes the
// per-expert arrays too.
__device__ void direct_tables_cta(const DispatchArgs& p, int* dsm) {
  pdl_wait();
  pdl_trigger();
  direct_offsets(p, dsm, blockIdx.x == 0);
  const int E = p.E, s = blockIdx.x;
  const int* eoff = dsm;
  int* sk = dsm + (E + 1) + 32 + 2;
  const long long row = (long long)s * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int a = 0;
    for (int s2 = 0; s2 < s; ++s2) a += __ldcg(p.acc_se + (long long)s2 * E + e);
    const int c = __ldcg(p.acc_se + row + e);
    const int kept = p.cap > 0 ? min(max(p.cap - a, 0), c) : c;
    p.tab.cnt[row + e] = c;
    p.tab.kept_cnt[row + e] = kept;
    p.tab.recv_offset[row + e] = eoff[e] + (p.cap > 0 ? min(a, p.cap) : a);
    sk[e] = kept;
  }
  const int total = cta_exclusive_scan(sk, E, sk + E);  // barriers: all reads above are done
  const unsigned ticket = direct_count_out(p);
  for (int d = threadIdx.x; d < p.P; d += blockDim.x) {
    const int lo = sk[d * p.L];
    const int hi = d + 1 < p.P ? sk[(d + 1) * p.L] : total;
    p.tab.send_offset[(long long)s * p.P + d] = lo;
    p.tab.C[(long long)s * p.P + d] = hi - lo;
  }
  direct_end(p, ticket);
}

template <int VPT, bool DIRECT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_bf16(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  extern __shared__ int dsm[];  // tables CTAs and direct mode
  int par = 0;
  const int nvec = p.H >> 3;  // 16-byte vectors per row
  const int tid = threadIdx.x;
  bool waited = false, offsets_done = false;
  unsigned ticket = 0u;
  if ((int)blockIdx.x < p.tab_ctas) {
    if (DIRECT) direct_tables_cta(p, dsm);
    else tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  // the next token's codes and weights are loaded one token ahead (direct
  // mode: the layout kernel is the launch just before, so its codes are read
  // only after the wait, in resolve_token)
  const long long gfirst = p.g0 + blockIdx.x - p.tab_ctas;
  // regular layout: token n's receive rows are resolved during token n-1
  // (published by token n's barrier), from codes loaded a token before that
  SlotIn si_next = DIRECT ? SlotIn{-1, 0.0f} : load_slot(p, gfirst);
  SlotIn si_next2 = (DIRECT || gfirst + nb >= p.T) ? SlotIn{-1, 0.0f} : load_slot(p, gfirst + nb);
  for (long long g = gfirst; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    SlotIn si = si_next;
    if (!DIRECT) {
      si_next = si_next2;
      if (g + 2 * nb < p.T) si_next2 = load_slot(p, g + 2 * nb);
    }
    const uint4* src = reinterpret_cast<const uint4*>(p.x + g * p.H);
    for (int v0 = 0; v0 < nvec; v0 += VPT * kDispatchThreads) {
      uint4 val[VPT];
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = v0 + i * kDispatchThreads + tid;
        if (v < nvec) val[i] = ld_stream(src + v);
      }
      if (v0 == 0) {
        // x is an input of the path: its first loads overlap the layout's tail
        if (!waited) {
          pdl_wait();
          pdl_trigger();
          waited = true;
          if (!DIRECT) resolve_rows(p, g, rows_s, si);  // the CTA's first token
        }
        if (DIRECT) resolve_token<DIRECT>(p, g, rows_s, si, dsm, offsets_done);
        if (DIRECT && g + nb >= p.T) ticket = direct_count_out(p);  // last read of the totals
        __syncthreads();
        if (!DIRECT && g + nb < p.T) resolve_rows(p, g + nb, rows_buf[par ^ 1], si_next);
      }
      for (int j = 0; j < p.k; ++j) {
        const int r = rows_s[j];
        if (r < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.recv) + (long long)r * p.H);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = v0 + i * kDispatchThreads + tid;
          if (v < nvec) dst[v] = val[i];
        }
      }
    }
    par ^= 1;  // token n+2 rewrites this buffer only after token n+1's barrier
  }
  if (DIRECT) direct_end(p, ticket);
}

// FP8: a 128-channel block is 16 consecutive vectors, held by 16 consecutive
// lanes (blockDim and the vector stride are multiples of 16), so the block's
// amax is a 4-step xor-shuffle reduction inside each half-warp.
template <int VPT, bool DIRECT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_fp8(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  extern __shared__ int dsm[];  // tables CTAs and direct mode
  int par = 0;
  const int nvec = p.H >> 3;
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  bool waited = false, offsets_done = false;
  unsigned ticket = 0u;
  if ((int)blockIdx.x < p.tab_ctas) {
    if (DIRECT) direct_tables_cta(p, dsm);
    else tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  // the next token's codes and weights are loaded one token ahead (direct
  // mode: the layout kernel is the launch just before, so its codes are read
  // only after the wait, in resolve_token)
  SlotIn si_next = DIRECT ? SlotIn{-1, 0.0f} : load_slot(p, p.g0 + blockIdx.x - p.tab_ctas);
  for (long long g = p.g0 + blockIdx.x - p.tab_ctas; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    SlotIn si = si_next;
    if (!DIRECT && g + nb < p.T) si_next = load_slot(p, g + nb);
    const uint4* src = reinterpret_cast<const uint4*>(p.x + g * p.H);
    for (int v0 = 0; v0 < nvec; v0 += VPT * kDispatchThreads) {
      uint4 val[VPT];
      float sc[VPT];
      uint2 code[VPT];
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = v0 + i * kDispatchThreads + tid;
        val[i] = v < nvec ? ld_stream(src + v) : make_uint4(0u, 0u, 0u, 0u);
      }
      if (v0 == 0) {
        if (!waited) {
          pdl_wait();
          pdl_trigger();
          waited = true;
        }
        resolve_token<DIRECT>(p, g, rows_s, si, dsm, offsets_done);
        if (DIRECT && g + nb >= p.T) ticket = direct_count_out(p);
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const float m = block_amax8(val[i]);
        sc[i] = __fdiv_rn(m, 448.0f);
        code[i] = quant8(val[i], sc[i], m);
      }
      for (int j = 0; j < p.k; ++j) {
        const int r = rows_s[j];
        if (r < 0) continue;
        uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.recv) + (long long)r * p.H);
        float* sdst = p.recv_scale + (long long)r * nblk;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = v0 + i * kDispatchThreads + tid;
          if (v < nvec) {
            dst[v] = code[i];
            if ((tid & 15) == 0) sdst[v >> 4] = sc[i];
          }
        }
      }
    }
    par ^= 1;  // token n+2 rewrites this buffer only after token n+1's barrier
  }
  if (DIRECT) direct_end(p, ticket);
}

// FP8 with x 32-byte aligned: each thread takes 16 consecutive values (one
// 256-bit load), so a 128-channel block is 8 consecutive lanes (3-step
// xor-shuffle amax), its scale and reciprocal are computed once per 16 values
// instead of once per 8, and the quotients run two per instruction. Each
// chunk is quantised and stored to the token's k rows (16-byte stores) before
// the next, so only the loaded rows stay in registers.
template <int CPT, bool DIRECT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_fp8w(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  extern __shared__ int dsm[];  // tables CTAs and direct mode
  int par = 0;
  const int nch = p.H >> 4;  // 32-byte chunks (16 values) per row
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  bool waited = false, offsets_done = false;
  unsigned ticket = 0u;
  if ((int)blockIdx.x < p.tab_ctas) {
    if (DIRECT) direct_tables_cta(p, dsm);
    else tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  // the next token's codes and weights are loaded one token ahead (direct
  // mode: the layout kernel is the launch just before, so its codes are read
  // only after the wait, in resolve_token)
  SlotIn si_next = DIRECT ? SlotIn{-1, 0.0f} : load_slot(p, p.g0 + blockIdx.x - p.tab_ctas);
  for (long long g = p.g0 + blockIdx.x - p.tab_ctas; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    SlotIn si = si_next;
    if (!DIRECT && g + nb < p.T) si_next = load_slot(p, g + nb);
    const uint16_t* src = p.x + g * p.H;
    for (int c0 = 0; c0 < nch; c0 += CPT * kDispatchThreads) {
      uint4 va[CPT], vb[CPT];
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = c0 + i * kDispatchThreads + tid;
        if (c < nch) {
          ld_stream32(src + 16 * c, va[i], vb[i]);
        } else {
          va[i] = make_uint4(0u, 0u, 0u, 0u);
          vb[i] = va[i];
        }
      }
      if (c0 == 0) {
        if (!waited) {
          pdl_wait();
          pdl_trigger();
          waited = true;
        }
        resolve_token<DIRECT>(p, g, rows_s, si, dsm, offsets_done);
        if (DIRECT && g + nb >= p.T) ticket = direct_count_out(p);
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const float m = block_amax16(va[i], vb[i]);
        const float sc = __fdiv_rn(m, 448.0f);
        const uint4 code = quant16(va[i], vb[i], sc, m);
        const int c = c0 + i * kDispatchThreads + tid;
        if (c < nch) {
          for (int j = 0; j < p.k; ++j) {
            const int r = rows_s[j];
            if (r < 0) continue;
            reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.recv) + (long long)r * p.H)[c] = code;
            if ((tid & 7) == 0) p.recv_scale[(long long)r * nblk + (c >> 3)] = sc;
          }
        }
      }
    }
    par ^= 1;  // token n+2 rewrites this buffer only after token n+1's barrier
  }
  if (DIRECT) direct_end(p, ticket);
}

// k_dispatch_fp8w for CTAs that take several tokens: while a token is
// quantised and stored, each thread copies its own 32-byte chunks of the
// CTA's next token row into the other half of a two-row shared buffer
// (cp.async), so the row loads of consecutive tokens overlap the stores
// instead of waiting behind them. A thread reads back only the bytes it
// copied, so the staging needs no barrier: cp.async.wait_group orders them.
// Dynamic shared memory: 2 rows of H bf16 values (and E + 32 ints for the
// tables CTAs, if larger).
template <int CPT>
__global__ void __launch_bounds__(kDispatchThreads, 7) k_dispatch_fp8s(const DispatchArgs p) {
  extern __shared__ __align__(16) uint16_t xs[];  // [2][H]
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  const int nch = p.H >> 4;
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  if ((int)blockIdx.x < p.tab_ctas) {
    tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  auto stage = [&](long long tok, int buf) {
    if (tok < p.T) {
      const uint16_t* src = p.x + tok * p.H;
      uint16_t* dst = xs + buf * p.H;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * kDispatchThreads + tid;
        if (c < nch) {
          cp_async16(dst + 16 * c, src + 16 * c);
          cp_async16(dst + 16 * c + 8, src + 16 * c + 8);
        }
      }
    }
    cp_async_commit();
  };
  long long g = p.g0 + blockIdx.x - p.tab_ctas;
  stage(g, 0);
  bool waited = false;
  int par = 0;
  for (; g < p.T; g += nb, par ^= 1) {
    const SlotIn si = load_slot(p, g);
    stage(g + nb, par ^ 1);
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    int* rows_s = rows_buf[par];
    resolve_rows(p, g, rows_s, si);
    __syncthreads();
    cp_async_wait_prev();  // this token's chunks (this thread's own copies) have landed
    const uint16_t* row = xs + par * p.H;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = i * kDispatchThreads + tid;
      uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
      if (c < nch) {
        va = *reinterpret_cast<const uint4*>(row + 16 * c);
        vb = *reinterpret_cast<const uint4*>(row + 16 * c + 8);
      }
      const float m = block_amax16(va, vb);
      const float sc = __fdiv_rn(m, 448.0f);
      const uint4 code = quant16(va, vb, sc, m);
      if (c < nch) {
        for (int j = 0; j < p.k; ++j) {
          const int r = rows_s[j];
          if (r < 0) continue;
          reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.recv) + (long long)r * p.H)[c] = code;
          if ((tid & 7) == 0) p.recv_scale[(long long)r * nblk + (c >> 3)] = sc;
        }
      }
    }
  }
  cp_async_wait_all();  // no copy outlives the CTA
}

// k_dispatch_fp8s with the stores to the k receive rows done by the TMA
// engine: each token's codes and scales are quantised into a shared-memory
// row (two, alternating per token) and one thread of the last warp (the
// issuer) copies them to the token's receive rows with one bulk copy per row
// for the codes and one for the scales. The copy then no longer spends a store
// instruction per 16 bytes and receive row. The stores of token n are issued
// right after the barrier of token n+1, which is also the point where every
// warp has written token n's row, so one barrier per token suffices; before
// that barrier the issuer waits (a hardware wait) until its copies of token
// n-1, the last ones reading the row buffer token n+1 will write, have read
// it. Three receive-row lists rotate, since token n's list is read while
// token n+2's is resolved. Each thread stages (cp.async) and reads the same
// x chunks, so staging the next token's row needs no barrier. Needs H a
// multiple of 512 (16-byte scale rows) and 16-byte aligned receive buffers.
// Dynamic shared memory: x rows [2][H] bf16 | codes [2][H] | scales [2][H/128].
template <int CPT>
__global__ void __launch_bounds__(kDispatchThreads, 5) k_dispatch_fp8b(const DispatchArgs p) {
  extern __shared__ __align__(16) uint16_t xs[];  // [2][H]
  __shared__ int rows_buf[3][MOE_MAX_TOPK];
  const int nch = p.H >> 4;
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  const bool issuer = tid == kDispatchThreads - 32;  // lane 0 of the last warp
  if ((int)blockIdx.x < p.tab_ctas) {
    tables_cta(p);
    return;
  }
  uint8_t* qs = reinterpret_cast<uint8_t*>(xs + 2 * p.H);  // [2][H] codes
  float* scs = reinterpret_cast<float*>(qs + 2 * p.H);     // [2][nblk] scales
  const long long nb = gridDim.x - p.tab_ctas;
  auto stage = [&](long long tok, int buf) {
    if (tok < p.T) {
      const uint16_t* src = p.x + tok * p.H;
      uint16_t* dst = xs + buf * p.H;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * kDispatchThreads + tid;
        if (c < nch) {
          cp_async16(dst + 16 * c, src + 16 * c);
          cp_async16(dst + 16 * c + 8, src + 16 * c + 8);
        }
      }
    }
    cp_async_commit();
  };
  // the issuer's bulk copies of one token (its codes and scales in buffer b)
  auto store_token = [&](const int* rows, int b) {
    const uint8_t* q = qs + b * p.H;
    const float* sq = scs + b * nblk;
    for (int j = 0; j < p.k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      bulk_store(static_cast<uint8_t*>(p.recv) + (long long)r * p.H, q, (uint32_t)p.H);
      bulk_store(p.recv_scale + (long long)r * nblk, sq, (uint32_t)nblk * 4u);
    }
    bulk_commit();
  };
  long long g = p.g0 + blockIdx.x - p.tab_ctas;
  stage(g, 0);
  bool waited = false;
  int n = 0;  // tokens of this CTA so far
  for (; g < p.T; g += nb, ++n) {
    const int par = n & 1;
    const SlotIn si = load_slot(p, g);
    stage(g + nb, par ^ 1);
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    int* rows_s = rows_buf[n % 3];
    resolve_rows(p, g, rows_s, si);
    if (issuer) bulk_wait_read_all();  // token n-2's copies have read buffer par
    __syncthreads();
    // every warp has written token n-1's row (and its fence): store it
    if (issuer && n > 0) store_token(rows_buf[(n + 2) % 3], par ^ 1);
    cp_async_wait_prev();  // this token's chunks (this thread's own copies) have landed
    const uint16_t* row = xs + par * p.H;
    uint8_t* q = qs + par * p.H;
    float* sq = scs + par * nblk;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = i * kDispatchThreads + tid;
      uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
      if (c < nch) {
        va = *reinterpret_cast<const uint4*>(row + 16 * c);
        vb = *reinterpret_cast<const uint4*>(row + 16 * c + 8);
      }
      const float m = block_amax16(va, vb);
      const float sc = __fdiv_rn(m, 448.0f);
      const uint4 code = quant16(va, vb, sc, m);
      if (c < nch) {
        *reinterpret_cast<uint4*>(q + 16 * c) = code;
        if ((tid & 7) == 0) sq[c >> 3] = sc;
      }
    }
    fence_smem_to_async();
  }
  __syncthreads();
  if (issuer) {
    if (n > 0) store_token(rows_buf[(n + 2) % 3], (n - 1) & 1);  // the last token
    bulk_wait_all();
  }
  cp_async_wait_all();  // no copy outlives the CTA
}

// AllGather comparator, stage 1: every token row (quantised once for FP8) is
// written to all P ranks' gathered copies, rows d*T + g.
template <bool FP8, int VPT>
__global__ void __launch_bounds__(kDispatchThreads) k_allgather(const AllGatherArgs a) {
  const DispatchArgs& p = a.dis;
  const int nvec = p.H >> 3, nblk = p.H >> 7, tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  for (long long g = blockIdx.x; g < p.T; g += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + g * p.H);
    for (int v0 = 0; v0 < nvec; v0 += VPT * kDispatchThreads) {
      uint4 val[VPT];
      float sc[VPT];
      uint2 code[VPT];
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = v0 + i * kDispatchThreads + tid;
        val[i] = v < nvec ? ld_stream(src + v) : make_uint4(0u, 0u, 0u, 0u);
        if (FP8) {
          const float m = block_amax8(val[i]);
          sc[i] = __fdiv_rn(m, 448.0f);
          code[i] = quant8(val[i], sc[i], m);
        }
      }
      for (int d = 0; d < a.P; ++d) {
        const long long row = (long long)d * p.T + g;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = v0 + i * kDispatchThreads + tid;
          if (v >= nvec) continue;
          if (FP8) {
            reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.gathered) + row * p.H)[v] = code[i];
            if ((tid & 15) == 0) a.gathered_scale[row * nblk + (v >> 4)] = sc[i];
          } else {
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.gathered) + row * p.H)[v] = val[i];
          }
        }
      }
    }
  }
}

// Stage 2, the local filter: every kept assignment copies its token's row from
// the gathered copy of the rank that owns its expert, into the same receive
// row (with the same metadata and inv) as the fused dispatch.
template <bool FP8>
__global__ void __launch_bounds__(kDispatchThreads) k_allgather_filter(const AllGatherArgs a) {
  __shared__ int rows_s[MOE_MAX_TOPK];
  __shared__ int owner_s[MOE_MAX_TOPK];
  const DispatchArgs& p = a.dis;
  const long long rb = FP8 ? (long long)p.H : 2ll * p.H;  // payload bytes per row
  const int row_vec = (int)(rb >> 4);                     // 16-byte vectors per row
  const int nblk = p.H >> 7;
  pdl_wait();
  pdl_trigger();
  for (long long g = blockIdx.x; g < p.T; g += gridDim.x) {
    resolve_rows(p, g, rows_s, load_slot(p, g), owner_s);
    __syncthreads();
    for (int j = 0; j < p.k; ++j) {
      const int r = rows_s[j];
      if (r < 0) continue;
      const long long srow = (long long)owner_s[j] * p.T + g;
      const uint4* src =
          reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.gathered) + srow * rb);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.recv) + (long long)r * rb);
      for (int v = threadIdx.x; v < row_vec; v += blockDim.x) dst[v] = __ldcs(src + v);
      if (FP8)
        for (int q = threadIdx.x; q < nblk; q += blockDim.x)
          p.recv_scale[(long long)r * nblk + q] = __ldcs(a.gathered_scale + srow * nblk + q);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_allgather(const AllGatherArgs& a, bool fp8, int num_sms, cudaStream_t st) {
  if (a.dis.T <= 0) return cudaSuccess;
  long long blocks = a.dis.T;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  const dim3 grid((int)blocks), block(kDispatchThreads);
  const int nvec = a.dis.H >> 3;
  cudaError_t err;
  if (fp8) {
    err = nvec <= 128   ? launch_pdl(k_allgather<true, 1>, grid, block, 0, st, a)
          : nvec <= 512 ? launch_pdl(k_allgather<true, 4>, grid, block, 0, st, a)
                        : launch_pdl(k_allgather<true, 8>, grid, block, 0, st, a);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_allgather_filter<true>, grid, block, 0, st, a);
  }
  err = nvec <= 128   ? launch_pdl(k_allgather<false, 1>, grid, block, 0, st, a)
        : nvec <= 512 ? launch_pdl(k_allgather<false, 4>, grid, block, 0, st, a)
                      : launch_pdl(k_allgather<false, 8>, grid, block, 0, st, a);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_allgather_filter<false>, grid, block, 0, st, a);
}

template <bool DIRECT>
cudaError_t launch_fp8w(const DispatchArgs& a, dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
  const int nch = a.H >> 4;
  if (nch <= 128) return launch_pdl(k_dispatch_fp8w<1, DIRECT>, grid, block, smem, st, a);
  if (nch <= 256) return launch_pdl(k_dispatch_fp8w<2, DIRECT>, grid, block, smem, st, a);
  return launch_pdl(k_dispatch_fp8w<4, DIRECT>, grid, block, smem, st, a);
}

template <bool FP8, bool DIRECT>
cudaError_t launch_vec(const DispatchArgs& a, dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
  const int nvec = a.H >> 3;
  if (FP8) {
    if (nvec <= 128) return launch_pdl(k_dispatch_fp8<1, DIRECT>, grid, block, smem, st, a);
    if (nvec <= 512) return launch_pdl(k_dispatch_fp8<4, DIRECT>, grid, block, smem, st, a);
    return launch_pdl(k_dispatch_fp8<8, DIRECT>, grid, block, smem, st, a);
  }
  if (nvec <= 128) return launch_pdl(k_dispatch_bf16<1, DIRECT>, grid, block, smem, st, a);
  if (nvec <= 512) return launch_pdl(k_dispatch_bf16<4, DIRECT>, grid, block, smem, st, a);
  return launch_pdl(k_dispatch_bf16<8, DIRECT>, grid, block, smem, st, a);
}

cudaError_t launch_dispatch(const DispatchArgs& a, bool fp8, int num_sms, cudaStream_t st) {
  long long blocks = a.T - a.g0 < 0 ? 0 : a.T - a.g0;
  const long long cap = (long long)num_sms * 16;  // 16 CTAs of 128 threads fill an SM
  if (blocks > cap) blocks = cap;
  if (blocks == 0 && a.tab_ctas == 0) return cudaSuccess;
  if (blocks == 0) return launch_tables(a.tab, st);
  const dim3 grid((int)(blocks + a.tab_ctas)), block(kDispatchThreads);
  const size_t smem = a.direct ? (size_t)direct_smem_ints(a.E) * sizeof(int)
                      : a.tab_ctas > 0 ? (size_t)(a.tab.E + 32) * sizeof(int) : 0;
  if (fp8 && (reinterpret_cast<uintptr_t>(a.x) & 31) == 0) {
    const int nch = a.H >> 4;
    // at least 16 tokens per CTA and two rows fit in shared memory: stage rows
    // ahead (with fewer tokens per CTA the lost CTA per SM costs more); the
    // direct mode (one token per CTA) never has that many
    const size_t stage_smem = (size_t)2 * a.H * sizeof(uint16_t);
    if (!a.direct && a.T - a.g0 >= 16 * blocks && nch <= 4 * kDispatchThreads &&
        stage_smem <= 48 * 1024) {
      // receive rows stored by bulk copies when the scale rows are 16-byte
      // multiples (H a multiple of 512) and the buffers 16-byte aligned
      const size_t bulk_smem = stage_smem + (size_t)2 * a.H + (size_t)2 * (a.H >> 7) * sizeof(float);
      if ((a.H & 511) == 0 && (reinterpret_cast<uintptr_t>(a.recv_scale) & 15) == 0 &&
          bulk_smem <= 48 * 1024 && a.send_pos == nullptr && a.slot_Tr == 0) {
        const size_t sm = bulk_smem > smem ? bulk_smem : smem;
        if (nch <= 128) return launch_pdl(k_dispatch_fp8b<1>, grid, block, sm, st, a);
        else if (nch <= 256) return launch_pdl(k_dispatch_fp8b<2>, grid, block, sm, st, a);
        else return launch_pdl(k_dispatch_fp8b<4>, grid, block, sm, st, a);
      }
      const size_t sm = stage_smem > smem ? stage_smem : smem;
      if (nch <= 128) return launch_pdl(k_dispatch_fp8s<1>, grid, block, sm, st, a);
      else if (nch <= 256) return launch_pdl(k_dispatch_fp8s<2>, grid, block, sm, st, a);
      else return launch_pdl(k_dispatch_fp8s<4>, grid, block, sm, st, a);
    }
    return a.direct ? launch_fp8w<true>(a, grid, block, smem, st)
                    : launch_fp8w<false>(a, grid, block, smem, st);
  }
  if (fp8)  // x only 16-byte aligned
    return a.direct ? launch_vec<true, true>(a, grid, block, smem, st)
                    : launch_vec<true, false>(a, grid, block, smem, st);
  return a.direct ? launch_vec<false, true>(a, grid, block, smem, st)
                  : launch_vec<false, false>(a, grid, block, smem, st);
}

cudaError_t launch_tables(const TablesArgs& t, cudaStream_t st) {
  if (t.P <= 0) return cudaSuccess;
  return launch_pdl(k_tables, dim3(t.P), dim3(kDispatchThreads), (size_t)(t.E + 32) * sizeof(int),
                    st, t);
}

}  // namespace moe
