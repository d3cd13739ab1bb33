// api.cu -- the C ABI of libmoe_ep.so: argument checks, workspace carving,
// call-order state, and kernel launches. See include/moe_ep.h for the
// contract of every entry point.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "internal.cuh"
#include "moe_ep.h"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->num_ranks < 1 || c->tokens_per_rank < 1 || c->num_experts < 1 || c->top_k < 1 ||
      c->hidden < 1 || c->expert_capacity < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->num_experts % c->num_ranks != 0) return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->num_experts) return MOE_ERR_INVALID_ARG;
  if (c->dispatch_dtype != MOE_BF16 && c->dispatch_dtype != MOE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
  if (c->combine_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->num_experts > MOE_MAX_EXPERTS || c->top_k > MOE_MAX_TOPK || c->num_ranks > MOE_MAX_RANKS)
    return MOE_ERR_UNSUPPORTED;
  if (c->hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->dispatch_dtype == MOE_FP8_E4M3 && c->hidden % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const long long T = (long long)c->num_ranks * c->tokens_per_rank;
  if (T * c->top_k >= (1ll << 31) - 1) return MOE_ERR_UNSUPPORTED;  // int32 row indices
  // The layout kernels keep their per-warp counters and the per-(source,
  // expert) tables in shared memory.
  if (moe::layout_smem_bytes(c->num_experts, moe::kMaxChunkAssign / c->top_k, c->top_k,
                             c->num_ranks) > moe::kLayoutSmemLimit ||
      moe::scan_smem_bytes(c->num_experts, c->num_ranks) > moe::kLayoutSmemLimit)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

struct Plan {
  int tpc_route, cps_route, tpc_ids, cps_ids, nchunks_max;
  size_t off_ctrl, off_acc, off_acc_se, off_totals, off_n_raw, off_n_kept, off_eoff, off_cnt, off_kept, off_C,
      off_send, off_recv, off_rank, off_hist, off_pre, off_acode, off_inv, off_spos, off_sbase,
      bytes;
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Chunking of the layout kernel. Given ids, a chunk of ~2048 assignments
// keeps the scan short; when routing, chunks are cut smaller (down to one
// token per warp) so the top-k work spreads over about two CTAs per SM.
Plan make_plan(const moe_config_t* c, int num_sms) {
  Plan p{};
  const int P = c->num_ranks, Tr = c->tokens_per_rank, E = c->num_experts, k = c->top_k;
  const long long T = (long long)P * Tr, Na = T * k;
  const int max_tpc = moe::kMaxChunkAssign / k;
  int tpc = 2048 / k;
  if (tpc < 1) tpc = 1;
  if (tpc > max_tpc) tpc = max_tpc;
  if (tpc > Tr) tpc = Tr;
  p.tpc_ids = tpc;
  p.cps_ids = ceil_div(Tr, tpc);
  // Routing chunks: about two per SM, and at least 8 tokens (the 16 warps of
  // a chunk route one token each at most; the route is issue-bound, so fewer
  // routing warps per SM finish sooner, while more chunks lengthen the column
  // scan: 8 measured best at decode).
  int tr = (int)((T + 2ll * num_sms - 1) / (2ll * num_sms));
  if (tr < 8) tr = 8;
  if (tr > 2048 / k) tr = 2048 / k;
  if (tr < 1) tr = 1;
  if (tr > max_tpc) tr = max_tpc;
  if (tr > Tr) tr = Tr;
  // More chunks than the GPU holds at once (two CTAs per SM, one from 512
  // experts up): the layout runs in waves of equal chunks, so take the chunk
  // count per source (up to twice the minimum) with the fewest waves x
  // tokens per chunk, i.e. the shortest last wave (prefill's 32 x 4096
  // tokens: 19 chunks of 216 tokens per source, two full waves on 152 SMs,
  // instead of 16 of 256).
  int cps = ceil_div(Tr, tr);
  const long long slots = (long long)num_sms * (E > 256 ? 1 : 2);
  if ((long long)P * cps > slots) {
    long long best = -1;
    const int c0 = cps;
    for (int c = c0; c <= 2 * c0 && c <= Tr; ++c) {
      const long long cost = ((long long)P * c + slots - 1) / slots * ceil_div(Tr, c);
      if (best < 0 || cost < best) {
        best = cost;
        cps = c;
      }
    }
    tr = ceil_div(Tr, cps);
    cps = ceil_div(Tr, tr);
  }
  p.tpc_route = tr;
  p.cps_route = cps;
  const int n1 = P * p.cps_ids, n2 = P * p.cps_route;
  p.nchunks_max = n1 > n2 ? n1 : n2;
  if (p.nchunks_max < num_sms) p.nchunks_max = num_sms;  // persistent path: one chunk per SM

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  p.off_ctrl = take(64);
  p.off_acc = take((size_t)E * 4);
  p.off_acc_se = take((size_t)P * E * 4);
  p.off_totals = take(4 * sizeof(int32_t));
  p.off_n_raw = take((size_t)E * 4);
  p.off_n_kept = take((size_t)E * 4);
  p.off_eoff = take((size_t)(E + 1) * 4);
  p.off_cnt = take((size_t)P * E * 4);
  p.off_kept = take((size_t)P * E * 4);
  p.off_C = take((size_t)P * P * 4);
  p.off_send = take((size_t)P * P * 4);
  p.off_recv = take((size_t)P * E * 4);
  p.off_rank = take((size_t)(P + 1) * 4);
  p.off_hist = take((size_t)p.nchunks_max * E * 4);
  p.off_pre = take((size_t)(P + 1) * E * 4);
  p.off_acode = take((size_t)Na * 4);
  p.off_inv = take((size_t)Na * 4);
  p.off_spos = take((size_t)P * E * 4);
  p.off_sbase = take((size_t)(P + 1) * 4);
  p.bytes = off;
  return p;
}

int query_sms(int* device, int* sms) {
  if (cudaGetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe::LayoutArgs layout_args(moe_handle_t h, bool route) {
  moe::LayoutArgs a{};
  a.acode = h->acode;
  a.hist = h->hist;
  a.src_pre = h->src_pre;
  a.n_raw = h->n_raw;
  a.n_kept = h->n_kept;
  a.expert_offset = h->expert_offset;
  a.cnt = h->cnt;
  a.kept_cnt = h->kept_cnt;
  a.C = h->C;
  a.send_offset = h->send_offset;
  a.recv_offset = h->recv_offset;
  a.rank_base = h->rank_base;
  a.totals = h->totals;
  a.status = h->status;
  a.done = h->done;
  a.P = h->cfg.num_ranks;
  a.E = h->cfg.num_experts;
  a.k = h->cfg.top_k;
  a.L = h->L;
  a.Tr = h->cfg.tokens_per_rank;
  a.tpc = route ? h->tpc_route : h->tpc_ids;
  a.cps = route ? h->cps_route : h->cps_ids;
  a.nchunks = a.P * a.cps;
  a.cap = h->cfg.expert_capacity;
  a.Na = h->Na;
  a.defer_tables = 1;
  a.acc_add = h->acc;
  return a;
}

moe::TablesArgs tables_args(moe_handle_t h) {
  moe::TablesArgs t{};
  t.src_pre = h->src_pre;
  t.expert_offset = h->expert_offset;
  t.cnt = h->cnt;
  t.kept_cnt = h->kept_cnt;
  t.recv_offset = h->recv_offset;
  t.C = h->C;
  t.send_offset = h->send_offset;
  t.P = h->cfg.num_ranks;
  t.E = h->cfg.num_experts;
  t.L = h->L;
  t.cap = h->cfg.expert_capacity;
  return t;
}

// Builds the per-source tables of the last layout if no launch has yet.
int ensure_tables(moe_handle_t h, cudaStream_t st) {
  if (!h->tables_pending) return MOE_OK;
  const int rc = cuda_rc(moe::launch_tables(tables_args(h), st));
  if (rc == MOE_OK) h->tables_pending = 0;
  return rc;
}

// Rows of the fixed per-(source, expert) slot layout: E regions of P*T_r rows;
// 0 when a capacity is set (the kept set would depend on every source) or the
// rows would not fit int32 indices.
long long fixed_slot_rows(const moe_config_t* c) {
  const long long rows = (long long)c->num_experts * c->num_ranks * c->tokens_per_rank;
  if (c->expert_capacity > 0 || rows >= (1ll << 31)) return 0;
  return rows;
}

// The direct dispatch (no scan kernel between the layout and the dispatch)
// pays off for small, latency-bound layers (decode): per token it sums the
// per-(source, expert) totals of earlier sources and the source's earlier
// chunk counts, and each tables CTA sums the totals of earlier sources, so
// the sources and chunks are bounded; and its token's codes can only be read
// after the wait, which costs a CTA that copies several tokens more than the
// scan kernel saves, so it is used when every dispatch CTA copies one token
// (T <= 16 CTAs per SM).
constexpr int kDirectMaxRanks = 32;
constexpr int kDirectMaxChunks = 256;

// Lanes that sum one slot's earlier counts: a power of two up to 32 such that
// all k slots fit in the dispatch CTA's 128 threads.
int direct_group(int k) {
  int G = 32;
  while (G > 1 && G * k > 128) G >>= 1;
  return G;
}

// Launches the scan kernel for a layout that was laid out for the direct
// dispatch but is needed in scanned form (any other consumer): with the totals
// still pending it consumes and clears them; after a direct dispatch (totals
// already cleared) it rebuilds the per-expert arrays from the chunk counts
// with the arrival counter instead.
int ensure_scanned(moe_handle_t h, cudaStream_t st) {
  if (h->scan_state == 0) return MOE_OK;
  moe::LayoutArgs a = layout_args(h, false);
  a.tpc = h->cur_tpc;
  a.cps = h->cur_cps;
  a.nchunks = h->cfg.num_ranks * h->cur_cps;
  if (h->scan_state == 1) {
    a.acc_se = h->acc_se;  // cleared with the per-expert totals
  } else {
    a.acc_add = nullptr;   // arrival-counter form; the last CTA writes the offsets
  }
  const int rc = cuda_rc(moe::launch_scan(a, st));
  if (rc != MOE_OK) {
    h->acc_dirty = 1;
    return rc;
  }
  h->scan_state = 0;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  int dev = 0, sms = 0;
  if (query_sms(&dev, &sms) != MOE_OK) sms = 152;
  return make_plan(cfg, sms).bytes;
}

int64_t moe_fixed_slot_rows(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  return fixed_slot_rows(cfg);
}

int64_t moe_recv_rows_max(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  const long long Na = (long long)cfg->num_ranks * cfg->tokens_per_rank * cfg->top_k;
  if (cfg->expert_capacity > 0) {
    const long long ec = (long long)cfg->num_experts * cfg->expert_capacity;
    return ec < Na ? ec : Na;
  }
  return Na;
}

int moe_handle_create(const moe_config_t* cfg, void* d_workspace, size_t bytes,
                      moe_handle_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate(cfg);
  if (rc != MOE_OK) return rc;
  if (!d_workspace) return MOE_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  rc = query_sms(&dev, &sms);
  if (rc != MOE_OK) return rc;
  const Plan p = make_plan(cfg, sms);
  if (bytes < p.bytes || !aligned(d_workspace, kAlign)) return MOE_ERR_WORKSPACE;
  // Opt in to the layout kernel's shared memory for the larger chunking.
  const int tpc_max = p.tpc_route > p.tpc_ids ? p.tpc_route : p.tpc_ids;
  if (moe::layout_prepare(cfg->num_experts, tpc_max, cfg->top_k, cfg->num_ranks) != cudaSuccess) return MOE_ERR_CUDA;

  moe_handle* h = static_cast<moe_handle*>(calloc(1, sizeof(moe_handle)));
  if (!h) return MOE_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = sms;
  h->T = (long long)cfg->num_ranks * cfg->tokens_per_rank;
  h->Na = h->T * cfg->top_k;
  h->rows_max = moe_recv_rows_max(cfg);
  h->L = cfg->num_experts / cfg->num_ranks;
  h->tpc_route = p.tpc_route;
  h->cps_route = p.cps_route;
  h->tpc_ids = p.tpc_ids;
  h->cps_ids = p.cps_ids;
  h->nchunks_max = p.nchunks_max;
  char* ws = static_cast<char*>(d_workspace);
  h->ws = ws;
  h->ws_bytes = bytes;
  h->status = reinterpret_cast<uint32_t*>(ws + p.off_ctrl);
  h->done = h->status + 1;
  h->totals = reinterpret_cast<int32_t*>(ws + p.off_totals);
  h->n_raw = reinterpret_cast<int32_t*>(ws + p.off_n_raw);
  h->n_kept = reinterpret_cast<int32_t*>(ws + p.off_n_kept);
  h->expert_offset = reinterpret_cast<int32_t*>(ws + p.off_eoff);
  h->cnt = reinterpret_cast<int32_t*>(ws + p.off_cnt);
  h->kept_cnt = reinterpret_cast<int32_t*>(ws + p.off_kept);
  h->C = reinterpret_cast<int32_t*>(ws + p.off_C);
  h->send_offset = reinterpret_cast<int32_t*>(ws + p.off_send);
  h->recv_offset = reinterpret_cast<int32_t*>(ws + p.off_recv);
  h->rank_base = reinterpret_cast<int32_t*>(ws + p.off_rank);
  h->hist = reinterpret_cast<int32_t*>(ws + p.off_hist);
  h->src_pre = reinterpret_cast<int32_t*>(ws + p.off_pre);
  h->acode = reinterpret_cast<int32_t*>(ws + p.off_acode);
  h->inv = reinterpret_cast<int32_t*>(ws + p.off_inv);
  h->send_pos = reinterpret_cast<int32_t*>(ws + p.off_spos);
  h->src_base = reinterpret_cast<int32_t*>(ws + p.off_sbase);
  h->wait_limit = 1ll << 22;  // ~0.3 s of 64 ns polls
  h->acc = reinterpret_cast<int32_t*>(ws + p.off_acc);
  h->acc_se = reinterpret_cast<int32_t*>(ws + p.off_acc_se);
  h->direct_ok = cfg->num_ranks <= kDirectMaxRanks && h->T <= 16ll * sms;
  if (cudaMemset(ws + p.off_ctrl, 0, 64) != cudaSuccess ||
      cudaMemset(ws + p.off_acc, 0, (size_t)cfg->num_experts * 4) != cudaSuccess ||
      cudaMemset(ws + p.off_acc_se, 0, (size_t)cfg->num_ranks * cfg->num_experts * 4) !=
          cudaSuccess) {
    free(h);
    return MOE_ERR_CUDA;
  }
  *out = h;
  return MOE_OK;
}

int moe_handle_destroy(moe_handle_t h) {
  free(h);
  return MOE_OK;
}

int moe_route_topk(moe_handle_t h, const float* logits, int32_t* ids, float* w, void* stream) {
  if (!h || !logits || !ids || !w) return MOE_ERR_INVALID_ARG;
  return cuda_rc(moe::launch_route_only(logits, ids, w, h->T, h->cfg.num_experts, h->cfg.top_k,
                                        h->num_sms, static_cast<cudaStream_t>(stream)));
}

static int run_layout(moe_handle_t h, bool route, const int32_t* ids_in, const float* logits,
                      int32_t* ids_out, float* w_out, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // A failed launch may have left partial totals, and a layout laid out for
  // the direct dispatch that nothing consumed leaves its totals behind.
  if (h->acc_dirty || h->scan_state == 1) {
    if (cudaMemsetAsync(h->acc, 0, (size_t)h->cfg.num_experts * 4, st) != cudaSuccess ||
        cudaMemsetAsync(h->acc_se, 0, (size_t)h->cfg.num_ranks * h->cfg.num_experts * 4, st) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
    h->acc_dirty = 0;
    h->scan_state = 0;
  }
  moe::LayoutArgs a = layout_args(h, route);
  a.ids_in = ids_in;
  a.logits = logits;
  a.ids_out = ids_out;
  a.w_out = w_out;
  // small layouts: only the layout kernel; the dispatch lays itself out from
  // the totals (direct dispatch), and any other consumer scans first
  const bool direct = h->direct_ok && a.nchunks <= kDirectMaxChunks;
  if (direct) a.acc_se = h->acc_se;
  const int rc = cuda_rc(moe::launch_layout(a, route, h->num_sms, st, !direct));
  if (rc != MOE_OK) {
    h->acc_dirty = 1;
    return rc;
  }
  h->cur_tpc = a.tpc;
  h->cur_cps = a.cps;
  h->layout_gen += 1;
  h->tables_pending = 1;
  h->scan_state = direct ? 1 : 0;
  return MOE_OK;
}

int moe_dispatch_layout(moe_handle_t h, const int32_t* ids, void* stream) {
  if (!h || !ids) return MOE_ERR_INVALID_ARG;
  return run_layout(h, false, ids, nullptr, nullptr, nullptr, stream);
}

int moe_route_dispatch_layout(moe_handle_t h, const float* logits, int32_t* ids, float* w,
                              void* stream) {
  if (!h || !logits || !ids || !w) return MOE_ERR_INVALID_ARG;
  return run_layout(h, true, nullptr, logits, ids, w, stream);
}

int moe_layout_tables(moe_handle_t h, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->layout_gen == 0) return MOE_ERR_STATE;
  const int rc = ensure_scanned(h, static_cast<cudaStream_t>(stream));
  if (rc != MOE_OK) return rc;
  return ensure_tables(h, static_cast<cudaStream_t>(stream));
}

int moe_get_layout(moe_handle_t h, moe_layout_view_t* out) {
  if (!h || !out) return MOE_ERR_INVALID_ARG;
  out->expert_count = h->n_kept;
  out->expert_count_raw = h->n_raw;
  out->expert_offset = h->expert_offset;
  out->src_expert_count = h->cnt;
  out->src_expert_kept = h->kept_cnt;
  out->count_matrix = h->C;
  out->send_offset = h->send_offset;
  out->recv_offset = h->recv_offset;
  out->rank_base = h->rank_base;
  out->inv = h->inv;
  out->totals = h->totals;
  return MOE_OK;
}

static int dispatch_range(moe_handle_t h, long long g0, long long g1, const void* x,
                          const float* w, void* recv_x, float* recv_scale,
                          const moe_recv_meta_t* meta, void* stream, bool fixed = false) {
  if (!h || !x || !w || !recv_x || !meta) return MOE_ERR_INVALID_ARG;
  if (!meta->local_expert || !meta->src_rank || !meta->src_token || !meta->slot || !meta->weight)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  if (fp8 && !recv_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16)) return MOE_ERR_INVALID_ARG;
  if (h->layout_gen == 0) return MOE_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the whole layer into the compact receive rows right after a layout laid
  // out for it: the direct dispatch; anything else needs the scanned layout
  const bool direct = !fixed && g0 == 0 && g1 == h->T && h->scan_state == 1;
  if (!direct) {
    const int rc = ensure_scanned(h, st);
    if (rc != MOE_OK) return rc;
  }
  moe::DispatchArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.w = w;
  a.acode = h->acode;
  a.hist = h->hist;
  a.expert_offset = h->expert_offset;
  a.inv = h->inv;
  a.recv = recv_x;
  a.recv_scale = recv_scale;
  a.m_local_expert = meta->local_expert;
  a.m_src_rank = meta->src_rank;
  a.m_src_token = meta->src_token;
  a.m_slot = meta->slot;
  a.m_weight = meta->weight;
  a.T = g1;
  a.g0 = g0;
  a.Tr = h->cfg.tokens_per_rank;
  a.k = h->cfg.top_k;
  a.E = h->cfg.num_experts;
  a.L = h->L;
  a.H = h->cfg.hidden;
  a.tpc = h->cur_tpc;
  a.cps = h->cur_cps;
  a.nchunks = h->cfg.num_ranks * h->cur_cps;
  a.cap = h->cfg.expert_capacity;
  if (h->tables_pending) {  // built by the launch's first P CTAs
    a.tab = tables_args(h);
    a.tab_ctas = h->cfg.num_ranks;
  }
  a.P = h->cfg.num_ranks;
  a.status = h->status;
  a.row_limit = fixed ? fixed_slot_rows(&h->cfg) : h->rows_max;
  if (fixed) {
    a.src_pre = h->src_pre;
    a.slot_Tr = h->cfg.tokens_per_rank;
  }
  if (direct) {
    a.direct = 1;
    a.direct_G = direct_group(a.k);
    a.acc = h->acc;
    a.acc_se = h->acc_se;
    a.arrive = h->status + 2;
    a.n_raw = h->n_raw;
    a.n_kept = h->n_kept;
    a.expert_offset_out = h->expert_offset;
    a.rank_base = h->rank_base;
    a.totals = h->totals;
    a.Na = h->Na;
    a.tab = tables_args(h);  // the per-source tables, from the totals
    a.tab_ctas = h->cfg.num_ranks;
  }
  const int rc = cuda_rc(moe::launch_dispatch(a, fp8, h->num_sms, st));
  if (rc == MOE_OK) {
    h->dispatch_gen = h->layout_gen;
    h->tables_pending = 0;
    h->fixed_rows = fixed ? 1 : 0;
    if (direct) h->scan_state = 2;
  } else if (direct) {
    h->acc_dirty = 1;
  }
  return rc;
}

int moe_dispatch_fixed_slots(moe_handle_t h, const void* x, const float* w, void* slot_x,
                             float* slot_scale, const moe_recv_meta_t* meta, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (fixed_slot_rows(&h->cfg) == 0) return MOE_ERR_UNSUPPORTED;
  return dispatch_range(h, 0, h->T, x, w, slot_x, slot_scale, meta, stream, true);
}

int moe_dispatch_two_stage(moe_handle_t h, const void* x, const float* w, void* send_x,
                           float* send_scale, void* recv_x, float* recv_scale,
                           const moe_recv_meta_t* meta, void* stream) {
  if (!h || !x || !w || !send_x || !recv_x || !meta) return MOE_ERR_INVALID_ARG;
  if (!meta->local_expert || !meta->src_rank || !meta->src_token || !meta->slot || !meta->weight)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  if (fp8 && (!recv_scale || !send_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(send_x, 16)) return MOE_ERR_INVALID_ARG;
  if (h->layout_gen == 0) return MOE_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = ensure_scanned(h, st);
  if (rc != MOE_OK) return rc;
  rc = ensure_tables(h, st);  // the send positions come from kept_cnt
  if (rc != MOE_OK) return rc;
  rc = cuda_rc(moe::launch_send_pos(h->kept_cnt, h->send_pos, h->src_base,
                                    h->cfg.num_ranks, h->cfg.num_experts, st));
  if (rc != MOE_OK) return rc;
  moe::DispatchArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.w = w;
  a.acode = h->acode;
  a.hist = h->hist;
  a.expert_offset = h->expert_offset;
  a.inv = h->inv;
  a.recv = send_x;
  a.recv_scale = send_scale;
  a.m_local_expert = meta->local_expert;
  a.m_src_rank = meta->src_rank;
  a.m_src_token = meta->src_token;
  a.m_slot = meta->slot;
  a.m_weight = meta->weight;
  a.T = h->T;
  a.Tr = h->cfg.tokens_per_rank;
  a.k = h->cfg.top_k;
  a.E = h->cfg.num_experts;
  a.L = h->L;
  a.H = h->cfg.hidden;
  a.tpc = h->cur_tpc;
  a.cps = h->cur_cps;
  a.nchunks = h->cfg.num_ranks * h->cur_cps;
  a.cap = h->cfg.expert_capacity;
  a.send_pos = h->send_pos;
  a.src_base = h->src_base;
  a.recv_offset = h->recv_offset;
  a.status = h->status;
  a.row_limit = h->rows_max;
  rc = cuda_rc(moe::launch_dispatch(a, fp8, h->num_sms, st));
  if (rc != MOE_OK) return rc;
  moe::A2avArgs c{};
  c.send = send_x;
  c.send_scale = fp8 ? send_scale : nullptr;
  c.recv = recv_x;
  c.recv_scale = recv_scale;
  c.expert_offset = h->expert_offset;
  c.recv_offset = h->recv_offset;
  c.send_pos = h->send_pos;
  c.src_base = h->src_base;
  c.rows_max = h->rows_max;
  c.row_bytes = (long long)h->cfg.hidden * (fp8 ? 1 : 2);
  c.P = h->cfg.num_ranks;
  c.E = h->cfg.num_experts;
  c.nblk = h->cfg.hidden / 128;
  c.status = h->status;
  rc = cuda_rc(moe::launch_a2av(c, h->num_sms, st));
  if (rc == MOE_OK) {
    h->dispatch_gen = h->layout_gen;
    h->fixed_rows = 0;
  }
  return rc;
}

int moe_dispatch(moe_handle_t h, const void* x, const float* w, void* recv_x, float* recv_scale,
                 const moe_recv_meta_t* meta, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  return dispatch_range(h, 0, h->T, x, w, recv_x, recv_scale, meta, stream);
}

int moe_dispatch_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end, const void* x,
                        const float* w, void* recv_x, float* recv_scale,
                        const moe_recv_meta_t* meta, void* stream) {
  if (!h || token_begin < 0 || token_end > h->T || token_begin > token_end)
    return MOE_ERR_INVALID_ARG;
  return dispatch_range(h, token_begin, token_end, x, w, recv_x, recv_scale, meta, stream);
}

int moe_dispatch_allgather(moe_handle_t h, const void* x, const float* w, void* gathered_x,
                           float* gathered_scale, void* recv_x, float* recv_scale,
                           const moe_recv_meta_t* meta, void* stream) {
  if (!h || !x || !w || !gathered_x || !recv_x || !meta) return MOE_ERR_INVALID_ARG;
  if (!meta->local_expert || !meta->src_rank || !meta->src_token || !meta->slot || !meta->weight)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  if (fp8 && (!recv_scale || !gathered_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(gathered_x, 16))
    return MOE_ERR_INVALID_ARG;
  if (h->layout_gen == 0) return MOE_ERR_STATE;
  moe::AllGatherArgs g{};
  moe::DispatchArgs& a = g.dis;
  a.x = static_cast<const uint16_t*>(x);
  a.w = w;
  a.acode = h->acode;
  a.hist = h->hist;
  a.expert_offset = h->expert_offset;
  a.inv = h->inv;
  a.recv = recv_x;
  a.recv_scale = recv_scale;
  a.m_local_expert = meta->local_expert;
  a.m_src_rank = meta->src_rank;
  a.m_src_token = meta->src_token;
  a.m_slot = meta->slot;
  a.m_weight = meta->weight;
  a.T = h->T;
  a.Tr = h->cfg.tokens_per_rank;
  a.k = h->cfg.top_k;
  a.E = h->cfg.num_experts;
  a.L = h->L;
  a.H = h->cfg.hidden;
  a.tpc = h->cur_tpc;
  a.cps = h->cur_cps;
  a.nchunks = h->cfg.num_ranks * h->cur_cps;
  a.cap = h->cfg.expert_capacity;
  a.status = h->status;
  a.row_limit = h->rows_max;
  g.gathered = gathered_x;
  g.gathered_scale = gathered_scale;
  g.P = h->cfg.num_ranks;
  int rc = ensure_scanned(h, static_cast<cudaStream_t>(stream));
  if (rc != MOE_OK) return rc;
  rc = ensure_tables(h, static_cast<cudaStream_t>(stream));
  if (rc != MOE_OK) return rc;
  rc = cuda_rc(moe::launch_allgather(g, fp8, h->num_sms, static_cast<cudaStream_t>(stream)));
  if (rc == MOE_OK) {
    h->dispatch_gen = h->layout_gen;
    h->fixed_rows = 0;
  }
  return rc;
}

int moe_set_wait_limit(moe_handle_t h, int64_t polls) {
  if (!h || polls < 0) return MOE_ERR_INVALID_ARG;
  h->wait_limit = polls;
  return MOE_OK;
}

int moe_layout_dispatch_fused(moe_handle_t h, const float* logits, int32_t* ids, float* w,
                              const void* x, void* recv_x, float* recv_scale,
                              const moe_recv_meta_t* meta, void* stream) {
  if (!h || !ids || !w || !x || !recv_x || !meta) return MOE_ERR_INVALID_ARG;
  if (!meta->local_expert || !meta->src_rank || !meta->src_token || !meta->slot || !meta->weight)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  const bool route = logits != nullptr;
  if (fp8 && !recv_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16)) return MOE_ERR_INVALID_ARG;
  const int P = h->cfg.num_ranks, Tr = h->cfg.tokens_per_rank, E = h->cfg.num_experts,
            k = h->cfg.top_k, H = h->cfg.hidden;
  // One CTA per SM; chunks of whole tokens of one source rank, one per CTA.
  const int grid = h->num_sms;
  int cps = grid / P;
  if (cps < 1) return MOE_ERR_UNSUPPORTED;
  int tpc = ceil_div(Tr, cps);
  cps = ceil_div(Tr, tpc);
  if ((long long)tpc * k > moe::kMaxChunkAssign || P * cps > h->nchunks_max) return MOE_ERR_UNSUPPORTED;
  const bool prefetch = (size_t)tpc * H * 2 <= (size_t)144 * 1024;
  int xs_off = 0;
  const size_t smem = moe::fused_smem_bytes(E, tpc, k, H, P, prefetch, &xs_off);
  int per_sm = 0;
  if (moe::fused_prepare(route, fp8, E, smem, &per_sm) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  moe::FusedArgs f{};
  f.lay = layout_args(h, route);
  f.lay.defer_tables = 0;  // the persistent kernel builds every table itself
  f.lay.acc_add = nullptr;
  f.lay.ids_in = ids;
  f.lay.logits = logits;
  f.lay.ids_out = ids;
  f.lay.w_out = w;
  f.lay.tpc = tpc;
  f.lay.cps = cps;
  f.lay.nchunks = P * cps;
  moe::DispatchArgs& a = f.dis;
  a.x = static_cast<const uint16_t*>(x);
  a.w = w;
  a.acode = h->acode;
  a.hist = h->hist;
  a.expert_offset = h->expert_offset;
  a.inv = h->inv;
  a.recv = recv_x;
  a.recv_scale = recv_scale;
  a.m_local_expert = meta->local_expert;
  a.m_src_rank = meta->src_rank;
  a.m_src_token = meta->src_token;
  a.m_slot = meta->slot;
  a.m_weight = meta->weight;
  a.T = h->T;
  a.Tr = Tr;
  a.k = k;
  a.E = E;
  a.L = h->L;
  a.H = H;
  a.tpc = tpc;
  a.cps = cps;
  a.nchunks = P * cps;
  a.cap = h->cfg.expert_capacity;
  a.status = h->status;
  a.row_limit = h->rows_max;
  f.bar = h->status + 4;
  f.wait_limit = h->wait_limit;
  f.prefetch_x = prefetch ? 1 : 0;
  f.xs_offset_ints = xs_off;
  if (h->scan_state == 1) h->acc_dirty = 1;  // a layout whose totals nothing consumed
  const int rc = cuda_rc(moe::launch_fused(f, route, fp8, grid, smem, static_cast<cudaStream_t>(stream)));
  if (rc != MOE_OK) return rc;
  h->scan_state = 0;
  h->cur_tpc = tpc;
  h->cur_cps = cps;
  h->layout_gen += 1;
  h->dispatch_gen = h->layout_gen;
  h->tables_pending = 0;
  h->fixed_rows = 0;
  return MOE_OK;
}

int moe_expert_standin(moe_handle_t h, const void* recv_x, const float* recv_scale,
                       const float* expert_scale, void* y, void* stream) {
  if (!h || !recv_x || !y) return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  if (fp8 && !recv_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(recv_x, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  if (h->dispatch_gen == 0 || h->dispatch_gen != h->layout_gen) return MOE_ERR_STATE;
  moe::StandinArgs a{};
  a.recv = recv_x;
  a.recv_scale = recv_scale;
  a.expert_scale = expert_scale;
  a.expert_offset = h->expert_offset;
  a.y = static_cast<uint16_t*>(y);
  a.rows_max = h->rows_max;
  a.E = h->cfg.num_experts;
  a.H = h->cfg.hidden;
  a.fp8 = fp8 ? 1 : 0;
  a.status = h->status;
  if (h->fixed_rows) {  // the filled rows of every slot region, found through inv
    a.inv = h->inv;
    a.a0 = 0;
    a.a1 = h->Na;
    a.k = h->cfg.top_k;
    a.slot_rows = (long long)h->cfg.num_ranks * h->cfg.tokens_per_rank;
    return cuda_rc(moe::launch_standin_tokens(a, h->num_sms, static_cast<cudaStream_t>(stream)));
  }
  return cuda_rc(moe::launch_standin(a, h->num_sms, static_cast<cudaStream_t>(stream)));
}

static int combine_range(moe_handle_t h, long long g0, long long g1, const void* y, const float* w,
                         void* out, void* stream) {
  if (!h || !y || !w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  if (h->dispatch_gen == 0 || h->dispatch_gen != h->layout_gen) return MOE_ERR_STATE;
  moe::CombineArgs a{};
  a.y = static_cast<const uint16_t*>(y);
  a.w = w;
  a.inv = h->inv;
  a.out = static_cast<uint16_t*>(out);
  a.T = g1;
  a.g0 = g0;
  a.k = h->cfg.top_k;
  a.H = h->cfg.hidden;
  a.row_limit = h->fixed_rows ? fixed_slot_rows(&h->cfg) : h->rows_max;
  a.status = h->status;
  return cuda_rc(moe::launch_combine(a, h->num_sms, static_cast<cudaStream_t>(stream)));
}

int moe_combine(moe_handle_t h, const void* y, const float* w, void* out, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  return combine_range(h, 0, h->T, y, w, out, stream);
}

int moe_combine_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end, const void* y,
                       const float* w, void* out, void* stream) {
  if (!h || token_begin < 0 || token_end > h->T || token_begin > token_end)
    return MOE_ERR_INVALID_ARG;
  return combine_range(h, token_begin, token_end, y, w, out, stream);
}

int moe_expert_standin_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end,
                              const void* recv_x, const float* recv_scale,
                              const float* expert_scale, void* y, void* stream) {
  if (!h || !recv_x || !y || token_begin < 0 || token_end > h->T || token_begin > token_end)
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = h->cfg.dispatch_dtype == MOE_FP8_E4M3;
  if (fp8 && !recv_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(recv_x, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  if (h->dispatch_gen == 0 || h->dispatch_gen != h->layout_gen) return MOE_ERR_STATE;
  moe::StandinArgs a{};
  a.inv = h->inv;
  a.a0 = token_begin * h->cfg.top_k;
  a.a1 = token_end * h->cfg.top_k;
  a.k = h->cfg.top_k;
  a.recv = recv_x;
  a.recv_scale = recv_scale;
  a.expert_scale = expert_scale;
  a.expert_offset = h->expert_offset;
  a.y = static_cast<uint16_t*>(y);
  a.rows_max = h->rows_max;
  a.E = h->cfg.num_experts;
  a.H = h->cfg.hidden;
  a.fp8 = fp8 ? 1 : 0;
  a.status = h->status;
  if (h->fixed_rows) a.slot_rows = (long long)h->cfg.num_ranks * h->cfg.tokens_per_rank;
  return cuda_rc(moe::launch_standin_tokens(a, h->num_sms, static_cast<cudaStream_t>(stream)));
}

int moe_read_status(moe_handle_t h, uint32_t* flags, void* stream) {
  if (!h || !flags) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(flags, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_copy_h2d_async(void* dst_device, const void* src_host, size_t bytes, void* stream) {
  if ((!dst_device || !src_host) && bytes) return MOE_ERR_INVALID_ARG;
  if (!bytes) return MOE_OK;
  return cuda_rc(cudaMemcpyAsync(dst_device, src_host, bytes, cudaMemcpyHostToDevice,
                                 static_cast<cudaStream_t>(stream)));
}

int moe_copy_d2h_async(void* dst_host, const void* src_device, size_t bytes, void* stream) {
  if ((!dst_host || !src_device) && bytes) return MOE_ERR_INVALID_ARG;
  if (!bytes) return MOE_OK;
  return cuda_rc(cudaMemcpyAsync(dst_host, src_device, bytes, cudaMemcpyDeviceToHost,
                                 static_cast<cudaStream_t>(stream)));
}

int moe_debug_bounds(void) {
#ifdef MOE_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_STATE: return "call order violated";
    default: return "unknown error";
  }
}

}  // extern "C"
