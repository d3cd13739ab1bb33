// layout.cu -- router top-k, per-chunk histograms with stable chunk-local
// ranks, and the device-wide prefix scan that turns them into the count
// matrix and every offset of the dispatch layout.
//
// Pages: "Expert Parallel: MoE Token ...", "Why count and permute before
// dispatch" (owner(e) under uniform contiguous placement, send_count, prefix
// sum -> send_offset, destination-contiguous writes) and "All-to-All-v"
// (count matrix C_ij); "[Infra-10] All-to-All Optimization", 3.5 (count /
// histogram -> prefix sum / offset -> scatter by destination), 5.1 (router
// output produces partial counts in the same pass) and 8.1 (capacity);
// "Efficient and portable MoE communication", introduction (router top-k).
//
// Design (one GPU, P virtual ranks in one HBM):
//   * The assignment list (s, t, j) is cut into chunks of whole tokens that
//     never straddle a source rank. One CTA per chunk.
//   * Route mode: each warp takes one token, holds its E logits in registers
//     (E/32 per lane), and picks the top-k by k warp-wide arg-max reductions
//     (value descending, expert ascending on ties).
//   * Every warp owns a contiguous sub-range of the chunk. Pass 1 counts its
//     experts with __match_any_sync (one shared-memory add per distinct expert
//     per 32 assignments); a per-expert scan over the 16 warps gives each warp
//     its base; pass 2 re-walks the sub-range and gives each assignment its
//     stable rank = warp base + lanes of the same expert below it. No atomics
//     decide any position, so the layout is deterministic.
//   * The chunk histogram goes to global memory; the last CTA to arrive
//     (threadfence + arrival counter, no spinning) scans all chunk histograms
//     and derives n_e, expert_offset, cnt[s][e], C[s][d], send_offset,
//     recv_offset and rank_base, applying the capacity clamp.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Exclusive scan in place of a[0..n) held in shared memory, by the whole CTA.
// tmp: 32 ints of shared scratch. Returns the total. Ends with __syncthreads.
__device__ int cta_exclusive_scan(int* a, int n, int* tmp) {
  const int nt = blockDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (n + nt - 1) / nt;
  const int b0 = min(n, (int)threadIdx.x * per), b1 = min(n, b0 + per);
  int local = 0;
  for (int i = b0; i < b1; ++i) local += a[i];
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = nt >> 5;
    int x = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += u;
    }
    tmp[lane] = x;
  }
  __syncthreads();
  int run = v - local + (warp > 0 ? tmp[warp - 1] : 0);
  const int total = tmp[(nt >> 5) - 1];
  for (int i = b0; i < b1; ++i) {
    int t = a[i];
    a[i] = run;
    run += t;
  }
  __syncthreads();
  return total;
}

// Top-k of one token's logits by one warp. Lane j < k returns slot j's expert
// id and its double-precision softmax weight over the chosen logits.
// Expert index of register i of a lane is i*32 + lane (coalesced loads).
template <int EPL>
__device__ void route_token_warp(const float* __restrict__ z, int E, int k, int lane,
                                 int& out_id, float& out_w) {
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? __ldg(z + e) : -INFINITY;
  }
  unsigned taken = 0;  // bit i: register i already chosen
  int my_id = -1;
  float my_z = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      // total order: larger value first, then smaller expert index; an empty
      // candidate (index INT_MAX) loses to any real one.
      const bool take = (oi != 0x7fffffff) &&
                        (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (take) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_id = bi;
      my_z = bv;
    }
  }
  // Softmax over the chosen logits, in double, summed in slot order.
  const double z0 = (double)__shfl_sync(kFull, my_z, 0);
  const double ex = lane < k ? exp((double)my_z - z0) : 0.0;
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(kFull, ex, j);
  out_id = my_id;
  out_w = (float)(ex / sum);
}

__device__ void layout_scan(const LayoutArgs& p, int* smem) {
  const int E = p.E, P = p.P, NT = blockDim.x, tid = threadIdx.x;
  int ng = NT / E;
  if (ng < 1) ng = 1;
  if (ng > p.nchunks) ng = p.nchunks;
  const int seg = (p.nchunks + ng - 1) / ng;
  int* part = smem;                          // [ng*E] <= max(NT, E)
  int* sk = part + (NT > E ? NT : E);        // [E]  n_kept -> expert_offset
  int* sraw = sk + E;                        // [E]
  int* tmp = sraw + E;                       // [32]
  int* red = tmp + 32;                       // [2]

  // (1) per-expert column scan over chunks, two levels: segment sums ...
  for (int it = tid; it < ng * E; it += NT) {
    const int e = it % E, gi = it / E;
    const int b0 = gi * seg, b1 = min(p.nchunks, b0 + seg);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += __ldcg(p.hist + (long long)b * E + e);
    part[gi * E + e] = sum;
  }
  if (tid < 2) red[tid] = 0;
  __syncthreads();
  // ... exclusive over segments, totals per expert, capacity clamp ...
  for (int e = tid; e < E; e += NT) {
    int run = 0;
    for (int gi = 0; gi < ng; ++gi) {
      const int v = part[gi * E + e];
      part[gi * E + e] = run;
      run += v;
    }
    const int kept = (p.cap > 0 && run > p.cap) ? p.cap : run;
    sraw[e] = run;
    sk[e] = kept;
    p.n_raw[e] = run;
    p.n_kept[e] = kept;
  }
  __syncthreads();
  // ... and the exclusive chunk bases, in place.
  for (int it = tid; it < ng * E; it += NT) {
    const int e = it % E, gi = it / E;
    const int b0 = gi * seg, b1 = min(p.nchunks, b0 + seg);
    int run = part[gi * E + e];
    for (int b = b0; b < b1; ++b) {
      int* h = p.hist + (long long)b * E + e;
      const int v = __ldcg(h);
      *h = run;
      run += v;
    }
  }
  // (2) expert offsets: exclusive scan of kept counts over global expert order.
  const int total = cta_exclusive_scan(sk, E, tmp);
  for (int e = tid; e <= E; e += NT) p.expert_offset[e] = e < E ? sk[e] : total;
  // (3) per (source, expert): raw and kept counts, receive offsets.
  for (int it = tid; it < P * E; it += NT) {
    const int s = it / E, e = it - s * E;
    const int pre = __ldcg(p.hist + (long long)(s * p.cps) * E + e);
    const int nxt = (s + 1 < P) ? __ldcg(p.hist + (long long)((s + 1) * p.cps) * E + e) : sraw[e];
    const int c = nxt - pre;
    int kept = c, start = pre;
    if (p.cap > 0) {
      kept = min(max(p.cap - pre, 0), c);
      start = min(pre, p.cap);
    }
    p.cnt[it] = c;
    p.kept_cnt[it] = kept;
    p.recv_offset[it] = sk[e] + start;
  }
  // dropped and masked totals
  {
    int dr = 0, rw = 0;
    for (int e = tid; e < E; e += NT) {
      rw += sraw[e];
      dr += sraw[e] - ((p.cap > 0 && sraw[e] > p.cap) ? p.cap : sraw[e]);
    }
    if (dr) atomicAdd(&red[0], dr);
    if (rw) atomicAdd(&red[1], rw);
  }
  __syncthreads();
  // (4) count matrix C[s][d] = kept assignments of s to experts owned by d.
  for (int it = tid; it < P * P; it += NT) {
    const int s = it / P, d = it - s * P;
    int sum = 0;
    for (int e = d * p.L; e < (d + 1) * p.L; ++e) sum += __ldcg(p.kept_cnt + (long long)s * E + e);
    p.C[it] = sum;
  }
  for (int d = tid; d <= P; d += NT) p.rank_base[d] = d < P ? sk[d * p.L] : total;
  __syncthreads();
  // (5) send offsets: exclusive prefix of C[s][.] over destinations.
  for (int s = tid; s < P; s += NT) {
    int run = 0;
    for (int d = 0; d < P; ++d) {
      const int v = __ldcg(p.C + (long long)s * P + d);
      p.send_offset[(long long)s * P + d] = run;
      run += v;
    }
  }
  if (tid == 0) {
    p.totals[0] = total;
    p.totals[1] = red[0];
    p.totals[2] = (int)(p.Na - (long long)red[1]);
    p.totals[3] = 0;
    *p.done = 0u;  // ready for the next layout on this workspace
  }
}

template <bool ROUTE, int EPL>
__global__ void __launch_bounds__(kLayoutThreads) k_layout(const LayoutArgs p) {
  extern __shared__ int smem[];
  __shared__ int s_last;
  const int E = p.E;
  int* wcnt = smem;                                         // [warps][E]
  const int wcnt_ints = kLayoutWarps * E;
  const int scan_ints = (kLayoutThreads > E ? kLayoutThreads : E) + 2 * E + 34;
  int* ids_s = smem + (wcnt_ints > scan_ints ? wcnt_ints : scan_ints);  // [tpc*k]

  const int b = blockIdx.x;
  const int s = b / p.cps, c = b - s * p.cps;
  const int t0 = c * p.tpc;
  const int nt = min(p.tpc, p.Tr - t0);
  const long long g0 = (long long)s * p.Tr + t0;
  const long long a0 = g0 * p.k;
  const int na = nt * p.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < wcnt_ints; i += kLayoutThreads) wcnt[i] = 0;

  if (ROUTE) {
    for (int tl = warp; tl < nt; tl += kLayoutWarps) {
      int id;
      float wt;
      route_token_warp<EPL>(p.logits + (g0 + tl) * (long long)E, E, p.k, lane, id, wt);
      if (lane < p.k) {
        ids_s[tl * p.k + lane] = id;
        p.ids_out[(g0 + tl) * p.k + lane] = id;
        p.w_out[(g0 + tl) * p.k + lane] = wt;
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
    const unsigned m = __match_any_sync(kFull, e);
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
    p.hist[(long long)b * E + e] = run;
  }
  __syncthreads();
  // Pass 2: stable rank of every assignment within the chunk and expert.
  const unsigned below = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids_s[i] : -1;
    const unsigned m = __match_any_sync(kFull, e);
    int code = -1;
    if (e >= 0) code = (e << 16) | (wcnt[warp * E + e] + __popc(m & below));
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wcnt[warp * E + e] += __popc(m);
    __syncwarp();
    if (i < end) p.acode[a0 + i] = code;
  }

  // Arrival: the last chunk CTA performs the device-wide scan.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(p.done, 1u) == (unsigned)(p.nchunks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  layout_scan(p, smem);
}

template <int EPL>
__global__ void __launch_bounds__(256) k_route_only(const float* __restrict__ logits,
                                                    int32_t* ids, float* w, long long T, int E,
                                                    int k) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long g = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < T;
       g += warps) {
    int id;
    float wt;
    route_token_warp<EPL>(logits + g * (long long)E, E, k, lane, id, wt);
    if (lane < k) {
      ids[g * k + lane] = id;
      w[g * k + lane] = wt;
    }
  }
}

template <bool ROUTE>
void* layout_kernel_ptr(int epl) {
  switch (epl) {
    case 1: return (void*)k_layout<ROUTE, 1>;
    case 2: return (void*)k_layout<ROUTE, 2>;
    case 4: return (void*)k_layout<ROUTE, 4>;
    case 8: return (void*)k_layout<ROUTE, 8>;
    case 16: return (void*)k_layout<ROUTE, 16>;
    default: return (void*)k_layout<ROUTE, 32>;
  }
}

int experts_per_lane(int E) {
  int epl = 1;
  while (epl * 32 < E) epl <<= 1;
  return epl;
}

}  // namespace

size_t layout_smem_bytes(int E, int tpc, int k) {
  const int wcnt_ints = kLayoutWarps * E;
  const int scan_ints = (kLayoutThreads > E ? kLayoutThreads : E) + 2 * E + 34;
  return sizeof(int) * ((size_t)(wcnt_ints > scan_ints ? wcnt_ints : scan_ints) + (size_t)tpc * k);
}

// The dynamic shared-memory limit is a per-kernel setting shared by every
// handle in the process, so it is raised to the device's opt-in maximum (never
// lowered to one configuration's need); the launch itself asks for what the
// configuration uses.
cudaError_t layout_prepare(int E, int tpc, int k) {
  const size_t smem = layout_smem_bytes(E, tpc, k);
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  const int epl = experts_per_lane(E);
  for (void* fn : {layout_kernel_ptr<true>(epl), layout_kernel_ptr<false>(epl)}) {
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, fn);
    if (err != cudaSuccess) return err;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;  // static shared memory counts too
    if (smem > (size_t)dyn_max) return cudaErrorInvalidValue;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_layout(const LayoutArgs& a, bool route, int /*num_sms*/, cudaStream_t st) {
  const size_t smem = layout_smem_bytes(a.E, a.tpc, a.k);
  const int epl = experts_per_lane(a.E);
  void* fn = route ? layout_kernel_ptr<true>(epl) : layout_kernel_ptr<false>(epl);
  LayoutArgs args = a;
  void* params[] = {&args};
  return cudaLaunchKernel(fn, dim3(a.nchunks), dim3(kLayoutThreads), params, smem, st);
}

cudaError_t launch_route_only(const float* logits, int32_t* ids, float* w, long long T, int E,
                              int k, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  long long blocks = (T + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  switch (experts_per_lane(E)) {
    case 1: k_route_only<1><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
    case 2: k_route_only<2><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
    case 4: k_route_only<4><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
    case 8: k_route_only<8><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
    case 16: k_route_only<16><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
    default: k_route_only<32><<<(int)blocks, 256, 0, st>>>(logits, ids, w, T, E, k); break;
  }
  return cudaGetLastError();
}

}  // namespace moe
