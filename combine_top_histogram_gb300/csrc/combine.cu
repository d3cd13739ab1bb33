// combine.cu -- combine + unpermute (gather of each token's k expert rows and
// the fp32 weighted sum in slot order, rounded to bf16), and the expert
// stand-in that turns receive rows into expert outputs for tests and
// benchmarks.
//
// Pages: "Expert Parallel: MoE Token ...", "Combine is not simply sending
// results back" (restore the original token order and merge the k outputs
// with the router weights; accumulate by the stable token index, never in
// arrival order, or t3's output silently lands on t4); "Efficient and
// portable MoE communication", "Combine" (weighted average of the experts'
// contributions written to the output tensor); "[Infra-10] All-to-All
// Optimization", 5.1 (fuse the reverse index, the weight multiply and the
// reduction into one pass).
//
// One GPU: the reverse all-to-all is a gather. Each CTA takes one token at a
// time, reads its k receive rows (16-byte loads; all k loads of a vector are
// issued before the first FMA), accumulates acc = fmaf(w_j, y_j, acc) for
// j = 0..k-1 in fp32, and writes one bf16 row (round to nearest even).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ void fma8(float* acc, float w, const uint4 y) {
  const uint32_t u[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = __fmaf_rn(w, bf16_lo(u[q]), acc[2 * q]);
    acc[2 * q + 1] = __fmaf_rn(w, bf16_hi(u[q]), acc[2 * q + 1]);
  }
}

// K > 0: compile-time top-k (all loads of a vector in flight at once);
// K == 0: any k <= MOE_MAX_TOPK, loads issued in groups of 8.
template <int K, int VPT>
__global__ void __launch_bounds__(kCombineThreads) k_combine(const CombineArgs p) {
  // the token's k rows and weights; two buffers, alternating per token
  __shared__ int rows_buf[2][MOE_MAX_TOPK];
  __shared__ float w_buf[2][MOE_MAX_TOPK];
  int par = 0;
  const int nvec = p.H >> 3;
  const int tid = threadIdx.x;
  const int k = K > 0 ? K : p.k;
  pdl_wait();  // y (and inv, when dispatch ran just before) come from earlier kernels
  pdl_trigger();
  for (long long g = p.g0 + blockIdx.x; g < p.T; g += gridDim.x) {
    int* rows_s = rows_buf[par];
    float* w_s = w_buf[par];
    if (tid < k) {
      const int r = __ldg(p.inv + g * k + tid);
      rows_s[tid] = (r >= 0 && row_ok(r, p.row_limit, p.status)) ? r : -1;
      w_s[tid] = __ldg(p.w + g * k + tid);
    }
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(p.out + g * p.H);
    for (int v0 = 0; v0 < nvec; v0 += VPT * kCombineThreads) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = v0 + i * kCombineThreads + tid;
        if (v >= nvec) continue;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        if (K > 0) {
          uint4 yv[K > 0 ? K : 1];
#pragma unroll
          for (int j = 0; j < K; ++j) {
            const int r = rows_s[j];
            yv[j] = r >= 0 ? __ldcs(reinterpret_cast<const uint4*>(p.y + (long long)r * p.H) + v)
                           : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int j = 0; j < K; ++j)
            if (rows_s[j] >= 0) fma8(acc, w_s[j], yv[j]);
        } else {
          for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 yv[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj;
              const int r = j < k ? rows_s[j] : -1;
              yv[jj] = r >= 0 ? __ldcs(reinterpret_cast<const uint4*>(p.y + (long long)r * p.H) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj;
              if (j < k && rows_s[j] >= 0) fma8(acc, w_s[j], yv[jj]);
            }
          }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        dst[v] = o;
      }
    }
    par ^= 1;  // token n+2 rewrites this buffer only after token n+1's barrier
  }
}

template <int K>
cudaError_t launch_combine_k(const CombineArgs& a, int blocks, cudaStream_t st) {
  const int nvec = a.H >> 3;
  if (nvec <= 128) return launch_pdl(k_combine<K, 1>, dim3(blocks), dim3(kCombineThreads), 0, st, a);
  else if (nvec <= 512) return launch_pdl(k_combine<K, 4>, dim3(blocks), dim3(kCombineThreads), 0, st, a);
  else return launch_pdl(k_combine<K, 8>, dim3(blocks), dim3(kCombineThreads), 0, st, a);
  return cudaGetLastError();
}

// Expert stand-in: one CTA per receive row; the row's global expert is found
// by binary search in expert_offset.
__global__ void __launch_bounds__(128) k_standin(const StandinArgs p) {
  __shared__ float c_s;
  const int nvec = p.H >> 3;
  pdl_wait();
  pdl_trigger();
  const int total = __ldg(p.expert_offset + p.E);
  if (total > 0 && blockIdx.x == 0 && threadIdx.x == 0) row_ok(total - 1, p.rows_max, p.status);
  for (long long r = blockIdx.x; r < total && r < p.rows_max; r += gridDim.x) {
    if (threadIdx.x == 0) {
      int lo = 0, hi = p.E - 1;  // largest e with expert_offset[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.expert_offset + mid) <= r) lo = mid;
        else hi = mid - 1;
      }
      c_s = p.expert_scale ? __ldg(p.expert_scale + lo) : 1.0f;
    }
    __syncthreads();
    const float c = c_s;
    uint4* dst = reinterpret_cast<uint4*>(p.y + r * p.H);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float f[8];
      if (p.fp8) {
        const uint2 q = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.recv) + r * p.H)[v];
        const float s = __ldg(p.recv_scale + r * (p.H >> 7) + (v >> 4));
        const uint32_t qq[2] = {q.x, q.y};
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const __nv_fp8_storage_t byte = (__nv_fp8_storage_t)((qq[b >> 2] >> (8 * (b & 3))) & 0xffu);
          const __half_raw hr = __nv_cvt_fp8_to_halfraw(byte, __NV_E4M3);
          f[b] = __fmul_rn(c, __fmul_rn(__half2float(__half(hr)), s));
        }
      } else {
        const uint4 x = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.recv) + r * p.H)[v];
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = __fmul_rn(c, bf16_lo(u[q]));
          f[2 * q + 1] = __fmul_rn(c, bf16_hi(u[q]));
        }
      }
      uint4 o;
      o.x = pack_bf16x2(f[0], f[1]);
      o.y = pack_bf16x2(f[2], f[3]);
      o.z = pack_bf16x2(f[4], f[5]);
      o.w = pack_bf16x2(f[6], f[7]);
      dst[v] = o;
    }
    __syncthreads();
  }
}

// Token-range stand-in: the rows of assignments [a0, a1) (a token chunk's
// slots), found through inv; same per-row function as k_standin.
__global__ void __launch_bounds__(128) k_standin_tokens(const StandinArgs p) {
  __shared__ float c_s;
  __shared__ int r_s;
  const int nvec = p.H >> 3;
  pdl_wait();
  pdl_trigger();
  for (long long a = p.a0 + blockIdx.x; a < p.a1; a += gridDim.x) {
    if (threadIdx.x == 0) {
      int r = __ldg(p.inv + a);
      const long long limit = p.slot_rows > 0 ? p.slot_rows * p.E : p.rows_max;
      if (r >= 0 && !row_ok(r, limit, p.status)) r = -1;
      r_s = r;
      if (r >= 0) {
        int lo = 0, hi = p.E - 1;  // largest e with expert_offset[e] <= r
        if (p.slot_rows > 0) {     // fixed slots: expert regions of slot_rows rows
          lo = (int)(r / p.slot_rows);
        } else {
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.expert_offset + mid) <= r) lo = mid;
            else hi = mid - 1;
          }
        }
        c_s = p.expert_scale ? __ldg(p.expert_scale + lo) : 1.0f;
      }
    }
    __syncthreads();
    const long long r = r_s;
    if (r >= 0) {
      const float c = c_s;
      uint4* dst = reinterpret_cast<uint4*>(p.y + r * p.H);
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float f[8];
        if (p.fp8) {
          const uint2 q = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.recv) + r * p.H)[v];
          const float s = __ldg(p.recv_scale + r * (p.H >> 7) + (v >> 4));
          const uint32_t qq[2] = {q.x, q.y};
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const __nv_fp8_storage_t byte = (__nv_fp8_storage_t)((qq[b >> 2] >> (8 * (b & 3))) & 0xffu);
            const __half_raw hr = __nv_cvt_fp8_to_halfraw(byte, __NV_E4M3);
            f[b] = __fmul_rn(c, __fmul_rn(__half2float(__half(hr)), s));
          }
        } else {
          const uint4 x = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.recv) + r * p.H)[v];
          const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] = __fmul_rn(c, bf16_lo(u[q]));
            f[2 * q + 1] = __fmul_rn(c, bf16_hi(u[q]));
          }
        }
        uint4 o;
        o.x = pack_bf16x2(f[0], f[1]);
        o.y = pack_bf16x2(f[2], f[3]);
        o.z = pack_bf16x2(f[4], f[5]);
        o.w = pack_bf16x2(f[6], f[7]);
        dst[v] = o;
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_standin_tokens(const StandinArgs& a, int num_sms, cudaStream_t st) {
  if (a.a1 - a.a0 <= 0) return cudaSuccess;
  long long blocks = a.a1 - a.a0;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(k_standin_tokens, dim3((int)blocks), dim3(128), 0, st, a);
}

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st) {
  if (a.T - a.g0 <= 0) return cudaSuccess;
  long long blocks = a.T - a.g0;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  switch (a.k) {
    case 1: return launch_combine_k<1>(a, (int)blocks, st);
    case 2: return launch_combine_k<2>(a, (int)blocks, st);
    case 4: return launch_combine_k<4>(a, (int)blocks, st);
    case 8: return launch_combine_k<8>(a, (int)blocks, st);
    default: return launch_combine_k<0>(a, (int)blocks, st);
  }
}

cudaError_t launch_standin(const StandinArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows_max <= 0) return cudaSuccess;
  long long blocks = a.rows_max;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(k_standin, dim3((int)blocks), dim3(128), 0, st, a);
}

}  // namespace moe
