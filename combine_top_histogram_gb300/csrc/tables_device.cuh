// tables_device.cuh -- the CTA-wide exclusive scan and the per-source layout
// tables, shared by the scan kernel's last CTA and the persistent path
// (layout_device.cuh) and by the dispatch kernels, whose first CTAs build the
// per-source tables while the others copy tokens (dispatch.cu).
//
// Pages: "Expert Parallel: MoE Token ...", "All-to-All-v" (count matrix C[s][d])
// and "Why count and permute before dispatch" (send_count -> exclusive prefix
// -> send_offset); "[Infra-10] All-to-All Optimization", 8.1 (capacity: the
// first c assignments of an expert in the stable order are kept).
#pragma once

#include <stdint.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Exclusive scan in place of a[0..n) held in shared memory, by the whole CTA.
// tmp: 32 ints of shared scratch. Returns the total. Starts and ends with
// __syncthreads: a thread scans a run of ceil(n / blockDim) elements that
// other threads may have written just before the call (when n exceeds the
// thread count the runs are not the elements a thread wrote itself).
__device__ int cta_exclusive_scan(int* a, int n, int* tmp) {
  const int nt = blockDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
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

// The tables of source rank s, by one CTA (any blockDim that is a multiple of
// 32, up to 1024): for every expert e, with a = assignments to e from sources
// below s (src_pre[s][e]) and c = those of s itself,
//   cnt[s][e] = c, kept_cnt[s][e] = c clamped to the capacity left after a,
//   recv_offset[s][e] = expert_offset[e] + min(a, cap);
// then the exclusive scan K of kept_cnt[s][.] over experts in global order
// gives, for rank d owning experts [d*L, (d+1)*L),
//   send_offset[s][d] = K[d*L] and C[s][d] = K[(d+1)*L] - K[d*L].
// sk: E + 32 ints of shared memory.
__device__ void source_tables(const TablesArgs& t, int s, int* sk) {
  const int E = t.E;
  const long long row = (long long)s * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int a = __ldcg(t.src_pre + row + e);
    const int c = __ldcg(t.src_pre + row + E + e) - a;
    const int kept = t.cap > 0 ? min(max(t.cap - a, 0), c) : c;
    t.cnt[row + e] = c;
    t.kept_cnt[row + e] = kept;
    t.recv_offset[row + e] = __ldcg(t.expert_offset + e) + (t.cap > 0 ? min(a, t.cap) : a);
    sk[e] = kept;
  }
  __syncthreads();
  const int total = cta_exclusive_scan(sk, E, sk + E);
  for (int d = threadIdx.x; d < t.P; d += blockDim.x) {
    const int lo = sk[d * t.L];
    const int hi = d + 1 < t.P ? sk[(d + 1) * t.L] : total;
    t.send_offset[(long long)s * t.P + d] = lo;
    t.C[(long long)s * t.P + d] = hi - lo;
  }
}

}  // namespace
}  // namespace moe
