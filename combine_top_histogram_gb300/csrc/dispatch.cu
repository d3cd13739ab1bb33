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

// The assignment code and weight of slot j = threadIdx.x of token g. The
// codes come from the layout kernel, which is at least two launches before
// any dispatch (the scan sits between them), so under the launch rule above
// they are complete when the dispatch starts; the weights are an input, like
// x. Both may therefore be loaded before the dispatch's wait.
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

template <int VPT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_bf16(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  int par = 0;
  const int nvec = p.H >> 3;  // 16-byte vectors per row
  const int tid = threadIdx.x;
  bool waited = false;
  if ((int)blockIdx.x < p.tab_ctas) {
    tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  for (long long g = p.g0 + blockIdx.x - p.tab_ctas; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    const SlotIn si = load_slot(p, g);
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
        }
        resolve_rows(p, g, rows_s, si);
        __syncthreads();
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
}

// FP8: a 128-channel block is 16 consecutive vectors, held by 16 consecutive
// lanes (blockDim and the vector stride are multiples of 16), so the block's
// amax is a 4-step xor-shuffle reduction inside each half-warp.
template <int VPT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_fp8(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  int par = 0;
  const int nvec = p.H >> 3;
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  bool waited = false;
  if ((int)blockIdx.x < p.tab_ctas) {
    tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  for (long long g = p.g0 + blockIdx.x - p.tab_ctas; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    const SlotIn si = load_slot(p, g);
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
        resolve_rows(p, g, rows_s, si);
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        float m = amax8(val[i]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
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
}

// FP8 with x 32-byte aligned: each thread takes 16 consecutive values (one
// 256-bit load), so a 128-channel block is 8 consecutive lanes (3-step
// xor-shuffle amax), its scale and reciprocal are computed once per 16 values
// instead of once per 8, and the quotients run two per instruction. Each
// chunk is quantised and stored to the token's k rows (16-byte stores) before
// the next, so only the loaded rows stay in registers.
template <int CPT>
__global__ void __launch_bounds__(kDispatchThreads, 8) k_dispatch_fp8w(const DispatchArgs p) {
  // the k receive rows of the current token; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  int par = 0;
  const int nch = p.H >> 4;  // 32-byte chunks (16 values) per row
  const int nblk = p.H >> 7;
  const int tid = threadIdx.x;
  bool waited = false;
  if ((int)blockIdx.x < p.tab_ctas) {
    tables_cta(p);
    return;
  }
  const long long nb = gridDim.x - p.tab_ctas;
  for (long long g = p.g0 + blockIdx.x - p.tab_ctas; g < p.T; g += nb) {
    int* rows_s = rows_buf[par];
    const SlotIn si = load_slot(p, g);
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
        resolve_rows(p, g, rows_s, si);
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        float m = fmaxf(amax8(va[i]), amax8(vb[i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
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
      float m = fmaxf(amax8(va), amax8(vb));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
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
          float m = amax8(val[i]);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
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

cudaError_t launch_dispatch(const DispatchArgs& a, bool fp8, int num_sms, cudaStream_t st) {
  long long blocks = a.T - a.g0 < 0 ? 0 : a.T - a.g0;
  const long long cap = (long long)num_sms * 16;  // 16 CTAs of 128 threads fill an SM
  if (blocks > cap) blocks = cap;
  if (blocks == 0 && a.tab_ctas == 0) return cudaSuccess;
  if (blocks == 0) return launch_tables(a.tab, st);
  const dim3 grid((int)(blocks + a.tab_ctas)), block(kDispatchThreads);
  const size_t smem = a.tab_ctas > 0 ? (size_t)(a.tab.E + 32) * sizeof(int) : 0;
  const int nvec = a.H >> 3;
  if (fp8 && (reinterpret_cast<uintptr_t>(a.x) & 31) == 0) {
    const int nch = a.H >> 4;
    // at least 16 tokens per CTA and two rows fit in shared memory: stage rows
    // ahead (with fewer tokens per CTA the lost CTA per SM costs more)
    const size_t stage_smem = (size_t)2 * a.H * sizeof(uint16_t);
    if (a.T - a.g0 >= 16 * blocks && nch <= 4 * kDispatchThreads && stage_smem <= 48 * 1024) {
      const size_t sm = stage_smem > smem ? stage_smem : smem;
      if (nch <= 128) return launch_pdl(k_dispatch_fp8s<1>, grid, block, sm, st, a);
      else if (nch <= 256) return launch_pdl(k_dispatch_fp8s<2>, grid, block, sm, st, a);
      else return launch_pdl(k_dispatch_fp8s<4>, grid, block, sm, st, a);
    }
    if (nch <= 128) return launch_pdl(k_dispatch_fp8w<1>, grid, block, smem, st, a);
    else if (nch <= 256) return launch_pdl(k_dispatch_fp8w<2>, grid, block, smem, st, a);
    else return launch_pdl(k_dispatch_fp8w<4>, grid, block, smem, st, a);
  }
  if (fp8) {  // x only 16-byte aligned
    if (nvec <= 128) return launch_pdl(k_dispatch_fp8<1>, grid, block, smem, st, a);
    else if (nvec <= 512) return launch_pdl(k_dispatch_fp8<4>, grid, block, smem, st, a);
    else return launch_pdl(k_dispatch_fp8<8>, grid, block, smem, st, a);
  } else {
    if (nvec <= 128) return launch_pdl(k_dispatch_bf16<1>, grid, block, smem, st, a);
    else if (nvec <= 512) return launch_pdl(k_dispatch_bf16<4>, grid, block, smem, st, a);
    else return launch_pdl(k_dispatch_bf16<8>, grid, block, smem, st, a);
  }
}

cudaError_t launch_tables(const TablesArgs& t, cudaStream_t st) {
  if (t.P <= 0) return cudaSuccess;
  return launch_pdl(k_tables, dim3(t.P), dim3(kDispatchThreads), (size_t)(t.E + 32) * sizeof(int),
                    st, t);
}

}  // namespace moe
