// layout_noalloc.cu -- moe_dispatch_layout_noalloc: the count + scan layout
// (and the inverse permutation) for callers that cannot allocate device
// memory, with the library's scratch in a fixed file-scope device array.
//
// Who needs this: code that may not call cudaMalloc -- a host framework whose
// plugin interface hands over only inputs and outputs and no workspace, a
// process whose device memory belongs to another allocator (a framework's
// caching allocator, a fixed memory budget) that an extra cudaMalloc would
// overrun or bypass, and code that must not let an allocation or a free
// synchronise the device. Such a caller still provides the ids and every
// output array; the intermediate chunk histograms, per-assignment codes and
// the arrival counter live in g_noalloc_scratch below instead of a caller
// workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.cuh"
#include "moe_ep.h"

namespace {

// Static scratch: every GPU that loads the library holds these bytes until the
// process exits. In host code the symbol names a host-side stand-in, not a
// device address: host code must use the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// What the entry point needs from a device, looked up once per device context:
// the scratch array's device address and the dynamic shared memory the layout
// and scan kernels may take (their limits raised once, here, so that later
// calls only launch).
struct DeviceSetup {
  unsigned long long ctx_id;  // context the entries below belong to
  void* scratch;
  size_t layout_dyn_max, scan_dyn_max;
};
std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices] = {};

typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

// Id of the current device context (the driver's cuCtxGetCurrent and
// cuCtxGetId, reached through the runtime so the library needs no link to the
// driver library). A device reset ends the context, and the next one has a new
// id, so nothing cached for an earlier context is used again.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
      get_cur = reinterpret_cast<CtxGetCurrentFn>(f1);
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    looked_up = true;
  }
  if (!get_cur || !get_id) return false;
  void* ctx = nullptr;
  if (get_cur(&ctx) != 0 || ctx == nullptr) return false;
  return get_id(ctx, id) == 0;
}

// The set-up of the current device, done on the first call in each device
// context: cudaGetSymbolAddress (which also makes the device's primary context
// current) and the kernels' shared-memory limits. Returns nullptr on failure.
const DeviceSetup* device_setup(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSetup& d = g_setup[device];
  unsigned long long id = 0;
  if (d.scratch != nullptr && current_context_id(&id) && id == d.ctx_id) return &d;
  DeviceSetup n{};
  if (cudaGetSymbolAddress(&n.scratch, g_noalloc_scratch) != cudaSuccess) return nullptr;
  if (moe::layout_prepare_all(&n.layout_dyn_max, &n.scan_dyn_max) != cudaSuccess) return nullptr;
  if (!current_context_id(&n.ctx_id)) return nullptr;
  d = n;
  return &d;
}

// Receive row of every assignment from its code, the exclusive chunk bases
// and the expert offsets; -1 for masked or dropped slots.
__global__ void k_inv_from_codes(const int32_t* __restrict__ acode,
                                 const int32_t* __restrict__ hist,
                                 const int32_t* __restrict__ expert_offset, int32_t* inv,
                                 long long Na, int k, int Tr, int E, int tpc, int cps, int cap,
                                 int nchunks) {
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < Na;
       a += (long long)gridDim.x * blockDim.x) {
    const int code = acode[a];
    int r = -1;
    if (code >= 0) {
      const int e = moe::code_expert(code);
      const long long g = a / k;
      const int s = (int)(g / Tr);
      const int t = (int)(g - (long long)s * Tr);
      const int pos = hist[(long long)e * nchunks + (s * cps + t / tpc)] + moe::code_rank(code);
      if (cap <= 0 || pos < cap) r = expert_offset[e] + pos;
    }
    inv[a] = r;
  }
}

// Tokens per layout chunk of this entry point: whole tokens, about 2048
// assignments per chunk, never crossing a source rank.
int chunk_tokens(const moe_config_t* c) {
  int tpc = 2048 / c->top_k;
  if (tpc < 1) tpc = 1;
  if (tpc > moe::kMaxChunkAssign / c->top_k) tpc = moe::kMaxChunkAssign / c->top_k;
  if (tpc > c->tokens_per_rank) tpc = c->tokens_per_rank;
  return tpc;
}

int check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->num_ranks < 1 || c->tokens_per_rank < 1 || c->num_experts < 1 || c->top_k < 1 ||
      c->hidden < 1 || c->expert_capacity < 0 || c->num_experts % c->num_ranks != 0 ||
      c->top_k > c->num_experts)
    return MOE_ERR_INVALID_ARG;
  if (c->num_experts > MOE_MAX_EXPERTS || c->top_k > MOE_MAX_TOPK ||
      c->num_ranks > MOE_MAX_RANKS)
    return MOE_ERR_UNSUPPORTED;
  // The layout kernel keeps per-warp counters and the chunk's ids in shared
  // memory, and the scan's last CTA every per-(source, expert) prefix.
  if (moe::layout_smem_bytes(c->num_experts, chunk_tokens(c), c->top_k, c->num_ranks) >
          moe::kLayoutSmemLimit ||
      moe::scan_smem_bytes(c->num_experts, c->num_ranks) > moe::kLayoutSmemLimit)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_dispatch_layout_noalloc(const moe_config_t* cfg, const int32_t* ids,
                                           const moe_layout_view_t* out, void* stream) {
  int rc = check_config(cfg);
  if (rc != MOE_OK) return rc;
  if (!ids || !out || !out->expert_count || !out->expert_count_raw || !out->expert_offset ||
      !out->src_expert_count || !out->src_expert_kept || !out->count_matrix ||
      !out->send_offset || !out->recv_offset || !out->rank_base || !out->inv || !out->totals)
    return MOE_ERR_INVALID_ARG;
  const int P = cfg->num_ranks, Tr = cfg->tokens_per_rank, E = cfg->num_experts,
            k = cfg->top_k;
  const long long Na = (long long)P * Tr * k;
  const int tpc = chunk_tokens(cfg);
  const int cps = (Tr + tpc - 1) / tpc;
  const int nchunks = P * cps;
  // Scratch map: [control words][chunk histograms][source prefixes][codes].
  const size_t off_hist = 256;
  const size_t off_pre = off_hist + round256((size_t)nchunks * E * 4);
  const size_t off_codes = off_pre + round256((size_t)(P + 1) * E * 4);
  const size_t need = off_codes + round256((size_t)Na * 4);
  if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const DeviceSetup* ds = device_setup(dev);
  if (!ds) return MOE_ERR_CUDA;
  if (moe::layout_smem_bytes(E, tpc, k, P) > ds->layout_dyn_max ||
      moe::scan_smem_bytes(E, P) > ds->scan_dyn_max)
    return MOE_ERR_UNSUPPORTED;
  char* base = static_cast<char*>(ds->scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The scratch keeps the previous call's contents: the control words (status
  // and the chunk arrival counter) must start at zero.
  if (cudaMemsetAsync(base, 0, 256, st) != cudaSuccess) return MOE_ERR_CUDA;

  moe::LayoutArgs a{};
  a.ids_in = ids;
  a.acode = reinterpret_cast<int32_t*>(base + off_codes);
  a.hist = reinterpret_cast<int32_t*>(base + off_hist);
  a.src_pre = reinterpret_cast<int32_t*>(base + off_pre);
  a.n_raw = out->expert_count_raw;
  a.n_kept = out->expert_count;
  a.expert_offset = out->expert_offset;
  a.cnt = out->src_expert_count;
  a.kept_cnt = out->src_expert_kept;
  a.C = out->count_matrix;
  a.send_offset = out->send_offset;
  a.recv_offset = out->recv_offset;
  a.rank_base = out->rank_base;
  a.totals = out->totals;
  a.status = reinterpret_cast<uint32_t*>(base);
  a.done = reinterpret_cast<uint32_t*>(base) + 1;
  a.P = P;
  a.E = E;
  a.k = k;
  a.L = E / P;
  a.Tr = Tr;
  a.tpc = tpc;
  a.cps = cps;
  a.nchunks = nchunks;
  a.cap = cfg->expert_capacity;
  a.Na = Na;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_layout(a, false, sms, st) != cudaSuccess) return MOE_ERR_CUDA;
  long long blocks = (Na + 255) / 256;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (blocks < 1) blocks = 1;
  k_inv_from_codes<<<(int)blocks, 256, 0, st>>>(a.acode, a.hist, out->expert_offset, out->inv,
                                                Na, k, Tr, E, tpc, cps, cfg->expert_capacity,
                                                nchunks);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
