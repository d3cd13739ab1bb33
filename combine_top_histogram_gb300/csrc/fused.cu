// fused.cu -- persistent single-launch route/count/scan/dispatch for small,
// latency-bound layers (decode).
//
// Pages: "[Infra-10] All-to-All Optimization", 9 and 10 (a low-latency mode
// with persistent kernels and device-side synchronisation for decode, where
// launches and synchronisation, not bandwidth, dominate) and 5.1 (fuse count,
// offsets and the scatter); "Expert Parallel: MoE Token ...", "Prefill and
// Decode are two EP workloads" (decode wants a latency path).
//
// One cooperative launch, one CTA of 512 threads per SM. CTA b owns layout
// chunk b (whole tokens of one source rank):
//   A  start copying its tokens' x rows into shared memory (cp.async, no
//      registers held), route its tokens (or read their ids), count per warp
//      and rank every assignment -- the same chunk body as the layout kernel;
//   -- grid barrier 1 (bounded spin) --
//   C  every warp of the grid scans expert columns of the chunk table
//      (exclusive chunk bases, per-source prefixes, totals);
//   -- grid barrier 2 --
//   E  every CTA scans the kept counts into expert offsets in shared memory;
//   F  every CTA resolves its assignments' receive rows, writes inv and the row
//      metadata, waits for its x rows, and stores each row (BF16, or FP8 with
//      scales) to its k receive rows;
//   G  the last CTA then writes the layout tables.
// Every wait on another CTA gives up after a bounded number of polls, sets
// MOE_STATUS_TIMEOUT and leaves the kernel; the last CTA to leave resets the
// barrier counters, so a timed-out launch does not poison the next one.
#include <cooperative_groups.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"
#include "layout_device.cuh"
#include "payload_device.cuh"

namespace moe {
namespace {

constexpr int kFusedThreads = kLayoutThreads;  // 512: 16 warps (route, count, scans)

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier: arrive on counter c, wait until every CTA has arrived.
// Returns false (and sets MOE_STATUS_TIMEOUT) after `limit` polls.
__device__ bool grid_barrier(unsigned* c, long long limit, uint32_t* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(c, 1u);
    int ok = 1;
    for (long long it = 0; ld_acquire(c) < gridDim.x; ++it) {
      if (it >= limit) {
        atomicOr(status, MOE_STATUS_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Returns false if a grid barrier timed out.
template <bool ROUTE, bool FP8, int EPL>
__device__ __forceinline__ bool fused_body(const FusedArgs& f, int* smem) {
  const LayoutArgs& p = f.lay;
  const DispatchArgs& d = f.dis;
  const int E = p.E, b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool has_chunk = b < p.nchunks;
  const int s = has_chunk ? b / p.cps : 0, c = has_chunk ? b - s * p.cps : 0;
  const int t0 = c * p.tpc;
  const int nt = has_chunk ? min(p.tpc, p.Tr - t0) : 0;
  const long long g0 = (long long)s * p.Tr + t0;
  const long long a0 = g0 * p.k;
  const int na = nt * p.k;
  const int nvec = d.H >> 3;
  // shared memory: [layout chunk: wcnt, ids] [rows_s: tpc*k] [eoff: E+1]
  //                [tmp: 32] [x rows: tpc * H bf16, 16-byte aligned]
  int* rows_s = smem + kLayoutWarps * E + p.tpc * p.k;
  int* eoff = rows_s + p.tpc * p.k;
  int* tmp = eoff + E + 1;
  uint4* xs = reinterpret_cast<uint4*>(smem + f.xs_offset_ints);

  // A. x rows start streaming into shared memory; route / count / rank.
  if (has_chunk && f.prefetch_x) {
    const uint4* src = reinterpret_cast<const uint4*>(d.x + g0 * d.H);
    for (int i = tid; i < nt * nvec; i += kFusedThreads) cp_async16(xs + i, src + i);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (has_chunk) {
    layout_chunk<ROUTE, EPL>(p, b, smem);
  }
  if (!grid_barrier(f.bar + 0, f.wait_limit, p.status)) return false;

  // C. Column scans of the chunk table, one warp per expert across the grid.
  for (int e = b * (kFusedThreads / 32) + warp; e < E; e += gridDim.x * (kFusedThreads / 32)) {
    int* col = p.hist + (long long)e * p.nchunks;
    int carry = 0;
    for (int c0 = 0; c0 < p.nchunks; c0 += 32) {
      const int bb = c0 + lane;
      const int v = bb < p.nchunks ? __ldcg(col + bb) : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int excl = carry + x - v;
      if (bb < p.nchunks) {
        col[bb] = excl;
        if (bb % p.cps == 0) p.src_pre[(bb / p.cps) * E + e] = excl;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
      p.src_pre[p.P * E + e] = carry;
      p.n_raw[e] = carry;
      p.n_kept[e] = (p.cap > 0 && carry > p.cap) ? p.cap : carry;
    }
  }
  if (!grid_barrier(f.bar + 1, f.wait_limit, p.status)) return false;

  // E. Expert offsets (every CTA, in shared memory).
  for (int e = tid; e < E; e += kFusedThreads) eoff[e] = __ldcg(p.n_kept + e);
  __syncthreads();
  const int total = cta_exclusive_scan(eoff, E, tmp);
  if (tid == 0) eoff[E] = total;

  // F. Receive rows of the chunk's assignments; metadata; payload.
  if (has_chunk) {
    for (int i = tid; i < na; i += kFusedThreads) {
      const long long a = a0 + i;
      const int code = __ldcg(p.acode + a);
      int r = -1;
      if (code >= 0 && row_ok(code_expert(code), p.E, p.status)) {
        const int e = code_expert(code);
        const int pos = __ldcg(p.hist + (long long)e * p.nchunks + b) + code_rank(code);
        if ((p.cap <= 0 || pos < p.cap) && row_ok(eoff[e] + pos, d.row_limit, p.status)) {
          r = eoff[e] + pos;
          const int t = t0 + i / p.k;
          d.m_local_expert[r] = e % p.L;
          d.m_src_rank[r] = s;
          d.m_src_token[r] = t;
          d.m_slot[r] = i % p.k;
          d.m_weight[r] = __ldcg(d.w + a);
        }
      }
      d.inv[a] = r;
      rows_s[i] = r;
    }
    if (f.prefetch_x) cp_async_wait_all();
    __syncthreads();
    const uint4* gsrc = reinterpret_cast<const uint4*>(d.x + g0 * d.H);
    // (token, vector) items; 16 consecutive vectors (one FP8 block) share a
    // half-warp because nvec and the thread stride are multiples of 16.
    for (int it0 = 0; it0 < nt * nvec; it0 += kFusedThreads) {
      const int it = it0 + tid;
      const bool on = it < nt * nvec;
      const int tl = on ? it / nvec : 0, v = on ? it - tl * nvec : 0;
      const uint4 val = on ? (f.prefetch_x ? xs[it] : ld_stream(gsrc + it)) : make_uint4(0u, 0u, 0u, 0u);
      if (FP8) {
        const float m = block_amax8(val);
        const float sc = __fdiv_rn(m, 448.0f);
        const uint2 code = quant8(val, sc, m);
        if (on) {
          for (int j = 0; j < p.k; ++j) {
            const int r = rows_s[tl * p.k + j];
            if (r < 0) continue;
            reinterpret_cast<uint2*>(static_cast<uint8_t*>(d.recv) + (long long)r * d.H)[v] = code;
            if ((tid & 15) == 0) d.recv_scale[(long long)r * (d.H >> 7) + (v >> 4)] = sc;
          }
        }
      } else if (on) {
        for (int j = 0; j < p.k; ++j) {
          const int r = rows_s[tl * p.k + j];
          if (r < 0) continue;
          reinterpret_cast<uint4*>(static_cast<uint16_t*>(d.recv) + (long long)r * d.H)[v] = val;
        }
      }
    }
  }

  // G. The last CTA writes the layout tables (off the other CTAs' paths).
  if (b == gridDim.x - 1) {
    __syncthreads();
    layout_tables(p, smem);
  }
  return true;
}

template <bool ROUTE, bool FP8, int EPL>
__global__ void __launch_bounds__(kFusedThreads) k_fused(const FusedArgs f) {
  extern __shared__ __align__(16) int smem[];
  if (!fused_body<ROUTE, FP8, EPL>(f, smem) && (int)blockIdx.x < f.lay.nchunks) {
    // Timed out: this chunk's slots get no receive row, so a later combine
    // reads nothing out of range. Everything else of the call is undefined.
    const int s = blockIdx.x / f.lay.cps, c = blockIdx.x - s * f.lay.cps;
    const int t0 = c * f.lay.tpc, nt = min(f.lay.tpc, f.lay.Tr - t0);
    const long long a0 = ((long long)s * f.lay.Tr + t0) * f.lay.k;
    for (int i = threadIdx.x; i < nt * f.lay.k; i += blockDim.x) f.dis.inv[a0 + i] = -1;
  }
  // Leave: the last CTA out resets the barrier counters for the next launch
  // (also after a timeout, since every CTA passes here exactly once).
  if (f.prefetch_x) cp_async_wait_all();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(f.bar + 2, 1u) == gridDim.x - 1) {
      f.bar[0] = 0u;
      f.bar[1] = 0u;
      f.bar[2] = 0u;
      __threadfence();
    }
  }
}

template <bool ROUTE, bool FP8>
void* fused_ptr(int epl) {
  switch (epl) {
    case 1: return (void*)k_fused<ROUTE, FP8, 1>;
    case 2: return (void*)k_fused<ROUTE, FP8, 2>;
    case 4: return (void*)k_fused<ROUTE, FP8, 4>;
    case 8: return (void*)k_fused<ROUTE, FP8, 8>;
    case 16: return (void*)k_fused<ROUTE, FP8, 16>;
    default: return (void*)k_fused<ROUTE, FP8, 32>;
  }
}

void* fused_kernel(bool route, bool fp8, int E) {
  int epl = 1;
  while (epl * 32 < E) epl <<= 1;
  if (route) return fp8 ? fused_ptr<true, true>(epl) : fused_ptr<true, false>(epl);
  return fp8 ? fused_ptr<false, true>(epl) : fused_ptr<false, false>(epl);
}

}  // namespace

size_t fused_smem_bytes(int E, int tpc, int k, int H, int P, bool prefetch_x,
                        int* xs_offset_ints) {
  // phases A-F: [wcnt][ids][rows][eoff][tmp]; phase G reuses the front for the
  // layout tables (2E + (P+1)E + P^2 + 34 ints) once the CTA's rows are stored
  size_t ints = (size_t)kLayoutWarps * E + 2 * (size_t)tpc * k + E + 1 + 32;
  const size_t tables = (size_t)2 * E + (size_t)(P + 1) * E + (size_t)P * P + 34;
  if (tables > ints) ints = tables;
  ints = (ints + 3) / 4 * 4;  // 16-byte alignment for the x rows
  *xs_offset_ints = (int)ints;
  return sizeof(int) * ints + (prefetch_x ? (size_t)tpc * H * 2 : 0);
}

cudaError_t fused_prepare(bool route, bool fp8, int E, size_t smem, int* blocks_per_sm) {
  void* fn = fused_kernel(route, fp8, E);
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, fn);
  if (err != cudaSuccess) return err;
  const int dyn_max = optin - (int)fa.sharedSizeBytes;
  if (smem > (size_t)dyn_max) return cudaErrorInvalidValue;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
  if (err != cudaSuccess) return err;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kFusedThreads, smem);
}

cudaError_t launch_fused(const FusedArgs& f, bool route, bool fp8, int grid, size_t smem,
                         cudaStream_t st) {
  void* fn = fused_kernel(route, fp8, f.lay.E);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barriers rely on it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reinterpret_cast<void (*)(const FusedArgs)>(fn), f);
}

}  // namespace moe
