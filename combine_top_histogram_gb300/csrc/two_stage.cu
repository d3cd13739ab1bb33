// two_stage.cu -- the "standard" dispatch, kept as a comparator for the fused
// scatter: (1) pack every kept assignment into its source rank's send buffer,
// laid out [to rank 0][to rank 1]... with each destination segment bucketed by
// local expert, then (2) a separate all-to-all-v copy moves each (source,
// expert) segment into the receive regions.
//
// Pages: "[Infra-10] All-to-All Optimization", 5.2 (send buffer
// [to rank 0][to rank 1]..., each segment bucketed [rank r / expert e]) and
// 4.3 (the less efficient form input -> temporary permutation buffer ->
// communication buffer, which the fused path avoids); "Expert Parallel: MoE
// Token ...", "Why count and permute before dispatch" (send_offset).
//
// Send buffer: one pool of rows_max rows; source s owns rows
// [src_base[s], src_base[s+1]); inside it, expert e's rows start at
// send_pos[s][e] = sum of the source's kept counts of experts < e (experts of
// rank d precede those of rank d+1, so send_offset[s][d] is the start of the
// segment for rank d), in (token, slot) order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kPosThreads = 1024;

// send_pos[s][e] (exclusive prefix of kept_cnt[s][.] over e) and src_base
// (exclusive prefix over s of each source's kept total): one CTA, one warp per
// source for the first, warp 0 for the second.
__global__ void __launch_bounds__(kPosThreads) k_send_pos(const int32_t* __restrict__ kept_cnt,
                                                          int32_t* send_pos, int32_t* src_base,
                                                          int P, int E) {
  __shared__ int totals[1024];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = warp; s < P; s += kPosThreads / 32) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? kept_cnt[(long long)s * E + e] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) send_pos[(long long)s * E + e] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) totals[s] = carry;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int s0 = 0; s0 < P; s0 += 32) {
      const int s = s0 + lane;
      const int v = s < P ? totals[s] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (s < P) src_base[s] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) src_base[P] = carry;
  }
}

// Stage 2, the all-to-all-v: every receive row r pulls its row from the send
// pool. Its expert e and source s come from binary searches in expert_offset
// and recv_offset[.][e]; the send row is
//   src_base[s] + send_pos[s][e] + (r - recv_offset[s][e]).
// FP8 rows carry their scale rows along.
__global__ void __launch_bounds__(128) k_a2av(const A2avArgs p) {
  __shared__ long long src_row_s;
  pdl_wait();
  pdl_trigger();
  const int total = __ldg(p.expert_offset + p.E);
  const int nvec = (int)(p.row_bytes >> 4);
  for (long long r = blockIdx.x; r < total; r += gridDim.x) {
    if (threadIdx.x == 0) {
      int lo = 0, hi = p.E - 1;  // largest e with expert_offset[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.expert_offset + mid) <= r) lo = mid;
        else hi = mid - 1;
      }
      const int e = lo;
      int slo = 0, shi = p.P - 1;  // largest s with recv_offset[s][e] <= r
      while (slo < shi) {
        const int mid = (slo + shi + 1) >> 1;
        if (__ldg(p.recv_offset + (long long)mid * p.E + e) <= r) slo = mid;
        else shi = mid - 1;
      }
      const int s = slo;
      src_row_s = (long long)__ldg(p.src_base + s) + __ldg(p.send_pos + (long long)s * p.E + e) +
                  (r - __ldg(p.recv_offset + (long long)s * p.E + e));
    }
    __syncthreads();
    const long long sr = src_row_s;
    if (!row_ok(sr, p.rows_max, p.status) || !row_ok(r, p.rows_max, p.status)) {
      __syncthreads();
      continue;  // debug bounds build only: a send or receive row outside the pool
    }
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.send) +
                                                      sr * p.row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.recv) + r * p.row_bytes);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = __ldcs(src + v);
    if (p.send_scale)
      for (int b = threadIdx.x; b < p.nblk; b += blockDim.x)
        p.recv_scale[r * p.nblk + b] = __ldcs(p.send_scale + sr * p.nblk + b);
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_send_pos(const int32_t* kept_cnt, int32_t* send_pos, int32_t* src_base, int P,
                            int E, cudaStream_t st) {
  return launch_pdl(k_send_pos, dim3(1), dim3(kPosThreads), 0, st, kept_cnt, send_pos, src_base,
                    P, E);
}

cudaError_t launch_a2av(const A2avArgs& a, int num_sms, cudaStream_t st) {
  long long blocks = a.rows_max;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(k_a2av, dim3((int)blocks), dim3(128), 0, st, a);
}

}  // namespace moe
