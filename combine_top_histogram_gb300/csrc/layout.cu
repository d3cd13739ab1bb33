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
//   * Route mode: a warp routes one token when chunks are small (latency) and
//     up to 32/k tokens (k rounded up to a power of two) when there are many
//     (fewer instructions per token): for each it holds the E logits as order-preserving keys in
//     registers (E/32 per lane) and picks the top-k by k rounds of a warp
//     max-reduction plus a min-reduction over tied expert indices (value
//     descending, expert ascending on ties); then all their softmax weights
//     are evaluated at once, one lane per (token, slot).
//   * Every warp owns a contiguous sub-range of the chunk. Pass 1 finds, for
//     every 32 assignments, the lanes sharing an expert (one ballot per bit of
//     the expert id) and adds their count once per distinct expert; a
//     per-expert scan over the 16 warps gives each warp its base; pass 2
//     re-walks the sub-range and gives each assignment its stable rank = warp
//     base + lanes of the same expert below it. No atomics decide any
//     position, so the layout is deterministic.
//   * The chunk histogram goes to global memory transposed, [E][nchunks], and
//     each chunk adds its per-expert counts into per-expert totals (integer
//     adds: order-free). A second kernel (k_scan) scans the histogram with one
//     warp per expert column; one extra CTA turns the totals into n_e,
//     expert_offset, rank_base and the layer totals with the capacity clamp.
//     The per-source tables (cnt, kept counts, C, send and receive offsets)
//     are built beside the copy by the dispatch launch (tables_device.cuh).
//     Without the totals (persistent and no-allocation paths) the scan's last
//     CTA to arrive (threadfence + arrival counter, no spinning) derives them.
//     Both kernels use programmatic dependent launch, so the scan's CTAs are
//     resident before the counts land.
//   * The device pieces shared with the persistent path live in
//     layout_device.cuh.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ffmath.cuh"
#include "internal.cuh"
#include "layout_device.cuh"

namespace moe {
namespace {

// Column scan of the chunk histograms, one warp per expert: the table is
// [E][nchunks], so a warp reads its expert's column contiguously and turns it
// into exclusive chunk bases in place. Each lane takes a contiguous run of up
// to kScanRun chunks, issuing all its loads at once, so a column costs one
// L2 round trip and one warp shuffle scan of the lanes' sums; longer columns
// take further passes. The scan also records the prefix at each source
// rank's first chunk and the expert's totals.
//
// With per-expert totals accumulated by the layout kernel (p.acc_add), one
// extra CTA (the last) turns them into the expert offsets, rank bases and
// totals and clears them for the next layout, while the other CTAs scan
// columns: no CTA waits for another. Without them, the last CTA to arrive
// (threadfence + arrival counter) builds the tables.
constexpr int kScanRun = 8;

__device__ void offsets_from_totals(const LayoutArgs& p, int* smem) {
  const int E = p.E, tid = threadIdx.x, NT = blockDim.x;
  int* sk = smem;        // [E] kept counts -> expert offsets
  int* tmp = sk + E;     // [32]
  int* red = tmp + 32;   // [2] dropped, raw total
  if (tid < 2) red[tid] = 0;
  __syncthreads();
  int dr = 0, rw = 0;
  for (int e = tid; e < E; e += NT) {
    const int raw = __ldcg(p.acc_add + e);
    p.acc_add[e] = 0;  // this CTA is the totals' only reader
    const int kept = (p.cap > 0 && raw > p.cap) ? p.cap : raw;
    sk[e] = kept;
    rw += raw;
    dr += raw - kept;
  }
  if (dr) atomicAdd(&red[0], dr);
  if (rw) atomicAdd(&red[1], rw);
  // per-(source, expert) totals of a layout laid out for the direct dispatch
  // are not needed here: clear them too for the next layout
  if (p.acc_se)
    for (int i = tid; i < p.P * E; i += NT) p.acc_se[i] = 0;
  const int total = cta_exclusive_scan(sk, E, tmp);
  for (int e = tid; e <= E; e += NT) p.expert_offset[e] = e < E ? sk[e] : total;
  for (int d = tid; d <= p.P; d += NT) p.rank_base[d] = d < p.P ? sk[d * p.L] : total;
  if (tid == 0) {
    p.totals[0] = total;
    p.totals[1] = red[0];
    p.totals[2] = (int)(p.Na - (long long)red[1]);
    p.totals[3] = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) k_scan(const LayoutArgs p) {
  extern __shared__ int smem[];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * (kScanThreads / 32) + warp;
  pdl_wait();
  if (p.acc_add && blockIdx.x == gridDim.x - 1) {
    offsets_from_totals(p, smem);
    pdl_trigger();
    return;
  }
  if (e < p.E) {
    int* col = p.hist + (long long)e * p.nchunks;
    const int n = p.nchunks;
    const int m = min(kScanRun, (n + 31) / 32);  // chunks per lane and pass
    int carry = 0;
    for (int c0 = 0; c0 < n; c0 += 32 * m) {
      const int b0 = c0 + lane * m;
      int v[kScanRun];
      int sum = 0;
#pragma unroll
      for (int i = 0; i < kScanRun; ++i) {
        v[i] = (i < m && b0 + i < n) ? __ldcg(col + b0 + i) : 0;
        sum += v[i];
      }
      int x = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      int run = carry + x - sum;
      // source rank and offset of chunk b0 (cps chunks per source)
      int s = b0 / p.cps, r = b0 - s * p.cps;
#pragma unroll
      for (int i = 0; i < kScanRun; ++i) {
        if (i < m && b0 + i < n) {
          col[b0 + i] = run;
          if (r == 0) p.src_pre[s * p.E + e] = run;
        }
        run += v[i];
        if (++r == p.cps) {
          r = 0;
          ++s;
        }
      }
      carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) {
      p.src_pre[p.P * p.E + e] = carry;
      p.n_raw[e] = carry;
      p.n_kept[e] = (p.cap > 0 && carry > p.cap) ? p.cap : carry;
    }
  }
  if (p.acc_add) {
    pdl_trigger();
    return;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(p.done, 1u) == gridDim.x - 1);
  __syncthreads();
  // The dependent dispatch launches only now: its row loads, issued before
  // its own wait, would otherwise compete with the column scans and the
  // arrival atomics on the critical path.
  pdl_trigger();
  if (!s_last) return;
  __threadfence();
  layout_tables(p, smem);
}

// Two CTAs per SM (64 registers) where the route fits in them; with 16 or 32
// logits per lane one CTA per SM, so that the keys stay in registers.
template <bool ROUTE, int EPL>
__global__ void __launch_bounds__(kLayoutThreads, EPL >= 16 ? 1 : 2) k_layout(const LayoutArgs p) {
  extern __shared__ int smem[];
  layout_chunk<ROUTE, EPL>(p, blockIdx.x, smem);
}

template <int EPL>
__global__ void __launch_bounds__(256) k_route_only(const float* __restrict__ logits,
                                                    int32_t* ids, float* w, long long T, int E,
                                                    int k) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  int K2 = 1;
  while (K2 < k) K2 <<= 1;
  const int G = 32 / K2;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long g0 = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * G; g0 < T;
       g0 += warps * G) {
    bool valid;
    int id;
    float wt;
    route_group_warp<EPL>(logits, g0, (int)min((long long)G, T - g0), E, k, K2, lane, valid, id,
                          wt);
    if (valid) {
      const long long g = g0 + lane / K2;
      ids[g * k + lane % K2] = id;
      w[g * k + lane % K2] = wt;
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

size_t layout_smem_bytes(int E, int tpc, int k, int /*P*/) {
  return sizeof(int) * ((size_t)kLayoutWarps * E + (size_t)tpc * k);
}

size_t scan_smem_bytes(int E, int P) {
  return sizeof(int) * ((size_t)2 * E + (size_t)(P + 1) * E + (size_t)P * P + 34);
}

// The dynamic shared-memory limit is a per-kernel setting shared by every
// handle in the process, so it is raised to the device's opt-in maximum (never
// lowered to one configuration's need); the launch itself asks for what the
// configuration uses.
cudaError_t layout_prepare(int E, int tpc, int k, int P) {
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  const int epl = experts_per_lane(E);
  struct {
    void* fn;
    size_t need;
  } kernels[] = {{layout_kernel_ptr<true>(epl), layout_smem_bytes(E, tpc, k, P)},
                 {layout_kernel_ptr<false>(epl), layout_smem_bytes(E, tpc, k, P)},
                 {(void*)k_scan, scan_smem_bytes(E, P)}};
  for (auto& kd : kernels) {
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kd.fn);
    if (err != cudaSuccess) return err;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;  // static shared memory counts too
    if (kd.need > (size_t)dyn_max) return cudaErrorInvalidValue;
    err = cudaFuncSetAttribute(kd.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// Raises the dynamic shared-memory limit of every layout kernel variant
// (given ids, any experts-per-lane) and of the scan kernel to the device's
// opt-in maximum, once, and reports how much dynamic shared memory each may
// then take: for callers that set up once and later only launch.
cudaError_t layout_prepare_all(size_t* layout_dyn_max, size_t* scan_dyn_max) {
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  size_t lay_min = (size_t)optin;
  for (int epl = 1; epl <= 32; epl <<= 1) {
    void* fn = layout_kernel_ptr<false>(epl);
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, fn);
    if (err != cudaSuccess) return err;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
    if (err != cudaSuccess) return err;
    if ((size_t)dyn_max < lay_min) lay_min = (size_t)dyn_max;
  }
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, (void*)k_scan);
  if (err != cudaSuccess) return err;
  const int scan_max = optin - (int)fa.sharedSizeBytes;
  err = cudaFuncSetAttribute((void*)k_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, scan_max);
  if (err != cudaSuccess) return err;
  *layout_dyn_max = lay_min;
  *scan_dyn_max = (size_t)scan_max;
  return cudaSuccess;
}

cudaError_t launch_scan(const LayoutArgs& a, cudaStream_t st) {
  const int scan_blocks = (a.E + kScanThreads / 32 - 1) / (kScanThreads / 32) + (a.acc_add ? 1 : 0);
  return launch_pdl(k_scan, dim3(scan_blocks), dim3(kScanThreads), scan_smem_bytes(a.E, a.P), st,
                    a);
}

cudaError_t launch_layout(const LayoutArgs& a, bool route, int /*num_sms*/, cudaStream_t st,
                          bool scan) {
  const size_t smem = layout_smem_bytes(a.E, a.tpc, a.k, a.P);
  const int epl = experts_per_lane(a.E);
  void* fn = route ? layout_kernel_ptr<true>(epl) : layout_kernel_ptr<false>(epl);
  cudaError_t err = launch_pdl(reinterpret_cast<void (*)(const LayoutArgs)>(fn), dim3(a.nchunks),
                               dim3(kLayoutThreads), smem, st, a);
  if (err != cudaSuccess || !scan) return err;
  return launch_scan(a, st);
}

cudaError_t launch_route_only(const float* logits, int32_t* ids, float* w, long long T, int E,
                              int k, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  long long blocks = (T + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  switch (experts_per_lane(E)) {
    case 1: return launch_pdl(k_route_only<1>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
    case 2: return launch_pdl(k_route_only<2>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
    case 4: return launch_pdl(k_route_only<4>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
    case 8: return launch_pdl(k_route_only<8>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
    case 16: return launch_pdl(k_route_only<16>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
    default: return launch_pdl(k_route_only<32>, dim3((int)blocks), dim3(256), 0, st, logits, ids, w, T, E, k);
  }
  return cudaGetLastError();
}

}  // namespace moe
