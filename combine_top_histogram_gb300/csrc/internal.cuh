// internal.cuh -- shared declarations of the CUDA side of libmoe_ep.so:
// the handle layout, kernel argument blocks and launcher prototypes.
// Not installed; the public interface is include/moe_ep.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_ep.h"

namespace moe {

// Layout kernel shape: 16 warps per chunk; one warp routes one token at a time.
constexpr int kLayoutThreads = 512;
constexpr int kLayoutWarps = kLayoutThreads / 32;
// Assignments per layout chunk are bounded so that a chunk-local rank fits in
// the low 16 bits of an assignment code (code = expert << 16 | rank).
constexpr int kMaxChunkAssign = 4096;
// Column-scan kernel shape: one warp per expert.
constexpr int kScanThreads = 512;
// Shared memory the layout kernels may use per CTA (GB300: 227 KB opt-in).
constexpr size_t kLayoutSmemLimit = 220 * 1024;

// Per-assignment code written by the layout kernel and read by dispatch:
// (expert << 16) | (stable rank of the assignment among the chunk's
// assignments to that expert), or -1 for a masked slot.
__host__ __device__ inline int code_expert(int c) { return c >> 16; }
__host__ __device__ inline int code_rank(int c) { return c & 0xFFFF; }

struct LayoutArgs {
  const int32_t* ids_in;  // [T*k] given ids (layout-only mode)
  const float* logits;    // [T*E] router logits (route mode)
  int32_t* ids_out;       // [T*k] routed ids (route mode)
  float* w_out;           // [T*k] routed weights (route mode)
  int32_t* acode;         // [T*k] assignment codes
  int32_t* hist;          // [E][nchunks]: chunk counts, then exclusive chunk bases
  int32_t* src_pre;       // [(P+1)*E]: prefix of expert e at source s's first chunk
  int32_t* n_raw;         // [E]
  int32_t* n_kept;        // [E]
  int32_t* expert_offset; // [E+1]
  int32_t* cnt;           // [P*E]
  int32_t* kept_cnt;      // [P*E]
  int32_t* C;             // [P*P]
  int32_t* send_offset;   // [P*P]
  int32_t* recv_offset;   // [P*E]
  int32_t* rank_base;     // [P+1]
  int32_t* totals;        // [4]
  uint32_t* status;
  uint32_t* done;         // chunk arrival counter, reset by the last chunk
  int P, E, k, L, Tr;
  int tpc, cps, nchunks;  // tokens per chunk, chunks per source rank, chunks
  int cap;                // 0 = unlimited
  long long Na;
  // 1: the scan's last CTA writes only n_kept/n_raw-derived outputs (expert
  // offsets, rank bases, totals); the per-source tables are left to
  // source_tables (dispatch CTAs or k_tables). 0: it writes every table.
  int defer_tables;
  // Per-expert totals accumulated by the layout kernel (one integer add per
  // chunk and expert), or null. With them one scan CTA derives the expert
  // offsets while the others scan columns, so the scan needs no arrival
  // counter and no last CTA (requires defer_tables). That CTA is the only
  // reader and clears the totals after reading them, ready for the next
  // layout: no host-side state, so a captured graph replays correctly.
  int32_t* acc_add;
  // Per-(source, expert) totals [P][E] accumulated the same way, or null: with
  // them (and acc_add) the dispatch can lay itself out without the scan
  // kernel (DispatchArgs::direct).
  int32_t* acc_se;
};

// Per-source tables of the layout, one source rank s per CTA (source_tables):
// cnt[s][e], kept_cnt[s][e], recv_offset[s][e], C[s][d], send_offset[s][d].
struct TablesArgs {
  const int32_t* src_pre;        // [(P+1)*E]
  const int32_t* expert_offset;  // [E+1]
  int32_t* cnt;
  int32_t* kept_cnt;
  int32_t* recv_offset;
  int32_t* C;
  int32_t* send_offset;
  int P, E, L, cap;
};

struct DispatchArgs {
  const uint16_t* x;      // bf16 bits [T*H]
  const float* w;         // [T*k]
  const int32_t* acode;   // [T*k]
  const int32_t* hist;    // [E][nchunks] exclusive chunk bases
  const int32_t* expert_offset;
  int32_t* inv;           // [T*k]
  void* recv;             // bf16 [rows*H] or e4m3 [rows*H]
  float* recv_scale;      // [rows*H/128] (FP8)
  int32_t* m_local_expert;
  int32_t* m_src_rank;
  int32_t* m_src_token;
  int32_t* m_slot;
  float* m_weight;
  long long T;            // tokens [g0, T) are dispatched (g0 = 0: all)
  long long g0;
  int Tr, k, E, L, H, tpc, cps, nchunks, cap;
  // Two-stage comparator: when send_pos is set, payload rows go to the send
  // pool row src_base[s] + send_pos[s][e] + (r - recv_offset[s][e]) instead of
  // the receive row r (metadata and inv still describe receive rows).
  const int32_t* send_pos;
  const int32_t* src_base;
  const int32_t* recv_offset;
  // tab_ctas > 0: the first tab_ctas CTAs build the per-source tables (one
  // source each) while the others copy tokens.
  TablesArgs tab;
  int tab_ctas;
  // Fixed per-(source, expert) receive slots when slot_Tr > 0: assignment
  // (s, t, j) -> e goes to row (e*P + s)*slot_Tr + q, q its rank among s's
  // assignments to e; src_pre gives the prefix at s's first chunk.
  const int32_t* src_pre;
  int slot_Tr, P;
  uint32_t* status;       // MOE_STATUS_SLOT_OVERFLOW (fixed slots), MOE_STATUS_BOUNDS
  long long row_limit;    // rows of the destination buffer (debug bounds checks)
  // Direct mode (small layouts, no scan kernel after the layout): the expert
  // offsets come from the per-expert totals acc and a slot's place inside its
  // expert from the per-(source, expert) totals acc_se of earlier sources plus
  // the raw chunk counts in hist of its own source's earlier chunks. CTA 0
  // writes the per-expert arrays; every CTA counts itself out on `arrive`
  // after reading the totals and the last one clears them and the counter.
  // direct_G: lanes that sum one slot's earlier counts (a power of two <= 32,
  // direct_G * k <= the CTA's threads).
  int direct, direct_G;
  int32_t* acc;           // [E]
  int32_t* acc_se;        // [P][E]
  unsigned* arrive;
  int32_t* n_raw;         // [E]  (written by CTA 0)
  int32_t* n_kept;        // [E]
  int32_t* expert_offset_out;  // [E+1]
  int32_t* rank_base;     // [P+1]
  int32_t* totals;        // [4]
  long long Na;
};

// Persistent single-launch route/layout/dispatch (fused.cu).
struct FusedArgs {
  LayoutArgs lay;
  DispatchArgs dis;
  unsigned* bar;          // 3 counters: grid barrier 1, grid barrier 2, exit
  long long wait_limit;   // polls before a grid barrier gives up
  int prefetch_x;         // x rows staged in shared memory during the layout
  int xs_offset_ints;     // where they start in dynamic shared memory
};

// AllGather-style comparator: every virtual rank holds a copy of all tokens
// (gathered rows d*T + g), then keeps the assignments to its own experts.
struct AllGatherArgs {
  DispatchArgs dis;
  void* gathered;         // [P*T] rows (bf16, or e4m3 codes)
  float* gathered_scale;  // [P*T, H/128] (FP8)
  int P;
};

struct A2avArgs {
  const void* send;          // send pool rows
  const float* send_scale;   // FP8 scale rows of the send pool, or null
  void* recv;
  float* recv_scale;
  const int32_t* expert_offset;
  const int32_t* recv_offset;
  const int32_t* send_pos;
  const int32_t* src_base;
  long long rows_max;
  long long row_bytes;       // payload bytes per row (multiple of 16)
  int P, E, nblk;
  uint32_t* status;          // MOE_STATUS_BOUNDS (debug bounds checks)
};

struct CombineArgs {
  const uint16_t* y;      // bf16 [rows*H]
  const float* w;         // [T*k]
  const int32_t* inv;     // [T*k]
  uint16_t* out;          // bf16 [T*H]
  long long T;            // tokens [g0, T) are combined (g0 = 0: all)
  long long g0;
  int k, H;
  long long row_limit;    // rows of y (debug bounds checks)
  uint32_t* status;       // MOE_STATUS_BOUNDS (debug bounds checks)
};

struct StandinArgs {
  const int32_t* inv;      // token-range form: rows of assignments [a0, a1)
  long long a0, a1;
  int k;
  const void* recv;        // bf16 or e4m3 [rows*H]
  const float* recv_scale; // FP8 scales
  const float* expert_scale; // [E] or null
  const int32_t* expert_offset; // [E+1]
  uint16_t* y;
  long long rows_max;
  int E, H, fp8;
  long long slot_rows;     // fixed-slot layout: rows per expert region (P*T_r); 0 = compact
  uint32_t* status;        // MOE_STATUS_BOUNDS (debug bounds checks)
};

// Debug bounds build (compiled with -DMOE_DEBUG_BOUNDS): a row index r that a
// kernel computed is checked against the row count of the buffer it indexes
// before any access through it; outside [0, limit) it sets MOE_STATUS_BOUNDS
// and the caller skips the access. Without the flag this is the constant true
// and the checks compile to nothing. Callers pass only r >= 0 (-1 already
// means "no row").
__device__ __forceinline__ bool row_ok(long long r, long long limit, uint32_t* status) {
#ifdef MOE_DEBUG_BOUNDS
  if (r < 0 || r >= limit) {
    if (status) atomicOr(status, MOE_STATUS_BOUNDS);
    return false;
  }
#else
  (void)r;
  (void)limit;
  (void)status;
#endif
  return true;
}

// Programmatic dependent launch: every kernel of the path is launched with
// programmatic stream serialization, waits for its predecessor grid
// (griddepcontrol.wait) before reading anything the predecessor may write, and
// right after that lets its own dependents launch (their CTAs then wait in
// hardware). Because a kernel triggers only after its own wait, data written
// two or more launches earlier is complete whenever a kernel starts, so it may
// be read before the wait. Without the launch attribute the wait is a no-op.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (return cudaGetLastError() of the launch).
// The layout kernel, then (scan = true) the scan kernel.
cudaError_t launch_layout(const LayoutArgs& a, bool route, int num_sms, cudaStream_t st,
                          bool scan = true);
// The scan kernel alone, for a layout launched with scan = false.
cudaError_t launch_scan(const LayoutArgs& a, cudaStream_t st);
cudaError_t launch_route_only(const float* logits, int32_t* ids, float* w, long long T,
                              int E, int k, int num_sms, cudaStream_t st);
size_t layout_smem_bytes(int E, int tpc, int k, int P);
size_t scan_smem_bytes(int E, int P);
cudaError_t layout_prepare(int E, int tpc, int k, int P);
cudaError_t layout_prepare_all(size_t* layout_dyn_max, size_t* scan_dyn_max);
cudaError_t launch_dispatch(const DispatchArgs& a, bool fp8, int num_sms, cudaStream_t st);
cudaError_t launch_tables(const TablesArgs& t, cudaStream_t st);
cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_standin(const StandinArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_standin_tokens(const StandinArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_send_pos(const int32_t* kept_cnt, int32_t* send_pos, int32_t* src_base, int P,
                            int E, cudaStream_t st);
cudaError_t launch_a2av(const A2avArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_allgather(const AllGatherArgs& a, bool fp8, int num_sms, cudaStream_t st);
size_t fused_smem_bytes(int E, int tpc, int k, int H, int P, bool prefetch_x,
                        int* xs_offset_ints);
cudaError_t fused_prepare(bool route, bool fp8, int E, size_t smem, int* blocks_per_sm);
cudaError_t launch_fused(const FusedArgs& f, bool route, bool fp8, int grid, size_t smem,
                         cudaStream_t st);

}  // namespace moe

// Host-side handle: configuration plus pointers into the caller's workspace.
struct moe_handle {
  moe_config_t cfg;
  int device;
  int num_sms;
  long long T, Na, rows_max;
  int L;
  int tpc_route, cps_route, tpc_ids, cps_ids, nchunks_max;
  int cur_tpc, cur_cps;     // chunking of the most recent layout
  char* ws;
  size_t ws_bytes;
  uint32_t* status;         // ctrl[0]
  uint32_t* done;           // ctrl[1]
  int32_t* totals;          // [4]
  int32_t *n_raw, *n_kept, *expert_offset, *cnt, *kept_cnt, *C, *send_offset,
      *recv_offset, *rank_base, *hist, *src_pre, *acode, *inv, *send_pos, *src_base;
  unsigned long long layout_gen, dispatch_gen;
  int tables_pending;       // per-source tables of the last layout not yet built
  int32_t* acc;             // [E] per-expert totals (zero between layouts)
  int32_t* acc_se;          // [P*E] per-(source, expert) totals (zero between layouts)
  int acc_dirty;            // a failed layout launch may have left partial sums
  // 0: the last layout is scanned (or none ran); 1: laid out for the direct
  // dispatch, not scanned, totals in acc/acc_se; 2: a direct dispatch ran on
  // it (totals consumed and cleared, chunk counts still unscanned)
  int scan_state;
  int direct_ok;            // small enough for the direct dispatch
  int fixed_rows;           // the last dispatch wrote fixed per-(source, expert) slots
  long long wait_limit;     // bounded device waits (persistent path)
};
