/*
 * moe_ep.h -- C ABI of the single-GPU MoE expert-parallel dispatch/combine
 * library (libmoe_ep.so, CUDA, sm_103a).
 *
 * The path: route -> count -> permute/pack -> all-to-all-v dispatch ->
 * (expert) -> combine -> unpermute with the top-k weighted sum.
 * Sources (page title, section):
 *   [A2A]  "[Infra-10] All-to-All Optimization" (xutianle.me):
 *          2 (two all-to-alls per MoE layer), 2.1 (payload carries expert id,
 *          token index, weight, counts, scales), 3.5 (count -> prefix ->
 *          scatter -> pack; unpack -> restore order -> weighted combine),
 *          4.1 (FP8 on the wire), 4.3 (write straight into the
 *          destination-contiguous buffer), 5.2 (segments per destination rank,
 *          bucketed by local expert), 8.1 (capacity and dropping).
 *   [EP]   "Expert Parallel: MoE Token ..." (charlestar.github.io):
 *          "A Top-2 routing example", "Why count and permute before dispatch"
 *          (owner(e), send_count, prefix sum -> send_offset, payload schema,
 *          bijection), "All-to-All-v" (count matrix C_ij), "Combine is not
 *          simply sending results back" (handle contents, stable token order),
 *          "Memory is not only expert weights" (preallocate by the worst case).
 *   [PPLX] "Efficient and portable MoE communication" (pplx-kernels blog):
 *          introduction (router top-k, weighted average), "Dispatch" (block
 *          scale factors), "Combine".
 *
 * One GPU holds P "virtual EP ranks". Rank s owns tokens [s*T_r, (s+1)*T_r)
 * of the input and experts [s*L, (s+1)*L), L = E/P. The all-to-all-v is a
 * device scatter into per-expert contiguous receive segments, driven by the
 * count matrix the library builds on the device: no host sync, no second GPU,
 * no collective.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller
 *     allocates and owns every buffer, including the workspace. The handle
 *     holds only the configuration and pointers into the workspace.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream) and never synchronises the host, except
 *     moe_read_status, which is for tests and debugging.
 *   - Calls on one handle must be ordered on one stream (or ordered by the
 *     caller with events); overlapping calls on one handle race on the
 *     workspace.
 *   - Host-checkable errors return a negative MOE_ERR_* code and enqueue
 *     nothing. Data-dependent problems (for example an expert id outside
 *     [-1, E)) set bits in the device status word and the offending slot is
 *     treated as masked. Capacity drops are counted, not errors.
 *   - Token rows are bf16 [T, H] row-major; T = P*T_r; global token
 *     g = s*T_r + t; assignment a = g*k + j (slot j of token g).
 *   - Kernels are launched with programmatic dependent launch: each waits for
 *     the previous grid on the stream before reading what that grid may have
 *     written, and lets its successor launch right after that wait.
 *     The dispatch entry points start loading x and w before their wait, so
 *     x and w must not be written by the immediately preceding kernel on the
 *     stream if that kernel lets its dependents launch before it finishes
 *     (kernels launched without programmatic dependent launch, and this
 *     library's own kernels, are fine).
 *   - Every call on a handle that launches work is asynchronous and can be
 *     captured in a CUDA graph. Capture a layout call together with the dispatch that
 *     follows it: the layout records on the host that the per-source tables
 *     are pending, and that dispatch's launch builds them.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- limits ------------------------------------------------------------ */
#define MOE_MAX_EXPERTS 1024   /* E */
#define MOE_MAX_TOPK 32        /* k */
#define MOE_MAX_RANKS 1024     /* P */

/* ---- dtypes ------------------------------------------------------------ */
#define MOE_BF16 0
#define MOE_FP8_E4M3 1

/* ---- return codes -------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)  /* null pointer, negative size, E % P != 0, k > E ... */
#define MOE_ERR_UNSUPPORTED (-2)  /* a size beyond the MOE_MAX_* limits, H % 8, FP8 with H % 128,
                                     or layout tables beyond shared memory: about
                                     (P+1)*E + P*P + 2*E > 40000 int32 */
#define MOE_ERR_WORKSPACE (-3)    /* workspace too small or not 256-byte aligned */
#define MOE_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed */
#define MOE_ERR_STATE (-5)        /* call order violated (combine before dispatch ...) */

/* ---- device status bits (sticky until moe_read_status clears them) ------ */
#define MOE_STATUS_BAD_EXPERT_ID 0x1u  /* an id outside [-1, E): slot treated as masked */
#define MOE_STATUS_TIMEOUT 0x2u        /* a bounded device wait gave up */
#define MOE_STATUS_SLOT_OVERFLOW 0x4u  /* fixed slots: more than T_r assignments of one
                                          source to one expert (an id repeated within a
                                          token); the excess is not written, inv = -1 */
#define MOE_STATUS_BOUNDS 0x8u         /* debug bounds build only (moe_debug_bounds()):
                                          a computed row index fell outside its buffer;
                                          that access was skipped (and inv = -1) */

/* Problem description. Passed by pointer; copied into the handle. */
typedef struct {
    int32_t num_ranks;       /* P >= 1 virtual EP ranks */
    int32_t tokens_per_rank; /* T_r >= 1 */
    int32_t num_experts;     /* E, a multiple of P, <= MOE_MAX_EXPERTS */
    int32_t top_k;           /* k, 1 <= k <= min(E, MOE_MAX_TOPK) */
    int32_t hidden;          /* H, a multiple of 8; a multiple of 128 for FP8 */
    int32_t dispatch_dtype;  /* MOE_BF16 or MOE_FP8_E4M3 (per-128-channel fp32 scales) */
    int32_t combine_dtype;   /* MOE_BF16 (the only combine dtype) */
    int32_t expert_capacity; /* per-expert row limit c; 0 = unlimited ([A2A] 8.1) */
} moe_config_t;

/* Opaque handle: configuration + pointers into the caller's workspace. */
typedef struct moe_handle *moe_handle_t;

/* Device pointers to the layout inside the workspace. All int32. When each
 * array is complete, in stream order:
 *   - expert_count, expert_count_raw, expert_offset, rank_base, totals: after
 *     the layout call (moe_dispatch_layout, moe_route_dispatch_layout);
 *     except for small layers (at most 32 ranks and T at most 16 times the
 *     SM count, e.g. decode), whose layout call only counts and whose
 *     following moe_dispatch lays itself out from the counts ("direct
 *     dispatch", one launch boundary less): there these are complete after
 *     that dispatch, or after moe_layout_tables;
 *   - src_expert_count, src_expert_kept, count_matrix, send_offset,
 *     recv_offset (the per-source tables): after the dispatch that follows the
 *     layout. The copy does not need them, so moe_dispatch and
 *     moe_dispatch_tokens build them in the same launch, beside the copy;
 *     moe_dispatch_two_stage and moe_dispatch_allgather build them first. A
 *     caller that wants them without dispatching calls moe_layout_tables;
 *   - inv: after the dispatch;
 *   - everything: after moe_layout_dispatch_fused and
 *     moe_dispatch_layout_noalloc.
 *   expert_count[E]       n_e: receive rows of expert e after capacity
 *   expert_count_raw[E]   valid assignments to e before capacity
 *   expert_offset[E+1]    first receive row of expert e; [E] = total rows.
 *                         Experts are contiguous and in global order, so the
 *                         rows of rank d are [rank_base[d], rank_base[d+1]).
 *   src_expert_count[P*E] cnt[s][e]: valid assignments from source s to e
 *   src_expert_kept[P*E]  the same after capacity
 *   count_matrix[P*P]     C[s][d]: kept assignments from source s to rank d
 *                         ([EP] "All-to-All-v")
 *   send_offset[P*P]      exclusive prefix of C[s][.] over d ([EP] prefix sum)
 *   recv_offset[P*E]      first receive row of source s inside expert e
 *   rank_base[P+1]        first receive row of rank d; [P] = total rows
 *   inv[T*k]              receive row of assignment a, -1 if masked/dropped
 *                         (written by moe_dispatch)
 *   totals[4]             kept rows, dropped (capacity), masked (id -1 or bad),
 *                         reserved
 * Contents are overwritten by the next layout call on the handle. */
typedef struct {
    int32_t *expert_count;
    int32_t *expert_count_raw;
    int32_t *expert_offset;
    int32_t *src_expert_count;
    int32_t *src_expert_kept;
    int32_t *count_matrix;
    int32_t *send_offset;
    int32_t *recv_offset;
    int32_t *rank_base;
    int32_t *inv;
    int32_t *totals;
} moe_layout_view_t;

/* Per-receive-row metadata ([EP] payload schema: local expert id, source
 * token index, top-k slot / routing weight; the source rank travels with it so
 * combine can route the row home). Each array has rows_max entries (see
 * moe_recv_rows_max); rows at or beyond the total kept count are untouched. */
typedef struct {
    int32_t *local_expert; /* e mod L */
    int32_t *src_rank;     /* s */
    int32_t *src_token;    /* t, local to the source rank */
    int32_t *slot;         /* j */
    float *weight;         /* w[g, j] */
} moe_recv_meta_t;

/* Bytes of device workspace a handle for *cfg needs (0 if *cfg is invalid):
 * every count, offset, chunk table and per-assignment array of the layout,
 * sized by the worst case T*k so that no call reads a count back to the host
 * ([EP] "Memory is not only expert weights": preallocate the EP buffers by
 * the maximum token count and reuse them across layers). */
size_t moe_workspace_bytes(const moe_config_t *cfg);

/* Receive rows every recv_* buffer must hold: T*k, or E*c when a capacity c is
 * set and smaller ([EP] "Memory is not only expert weights": preallocate by
 * the worst case). 0 if *cfg is invalid. */
int64_t moe_recv_rows_max(const moe_config_t *cfg);

/* Creates a handle over d_workspace (device, >= moe_workspace_bytes(cfg)
 * bytes, 256-byte aligned, owned by the caller and not freed by the library):
 * the preallocated, reusable EP state of one layer configuration ([EP]
 * "Memory is not only expert weights"; the combine handle of [EP] "Combine is
 * not simply sending results back" lives in it: inv, the per-expert counts
 * and the offsets of the last dispatch).
 * Zeroes the workspace's control words with a synchronous cudaMemset on the
 * current device; call once at set-up, outside stream capture.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
int moe_handle_create(const moe_config_t *cfg, void *d_workspace, size_t bytes,
                      moe_handle_t *out);

/* Housekeeping (no counterpart on the pages): frees the host-side handle
 * only. NULL is accepted. */
int moe_handle_destroy(moe_handle_t h);

/* a1 -- router top-k ([PPLX] introduction; [EP] router output [T, k]).
 * logits: fp32 [T, E]. Writes ids int32 [T, k] (slot 0 = largest logit; equal
 * logits ordered by the lower expert index) and w fp32 [T, k] = softmax over
 * the k chosen logits (= full softmax renormalised over them), evaluated in
 * double and rounded to fp32. Logits must be finite. */
int moe_route_topk(moe_handle_t h, const float *logits, int32_t *ids, float *w,
                   void *stream);

/* a2..a3 -- count + prefix scan + capacity from given ids ([EP] "Why count
 * and permute before dispatch", "All-to-All-v"; [A2A] 3.5, 8.1).
 * ids: int32 [T, k]; -1 marks a padded/invalid slot. Computes every array of
 * moe_layout_view_t except inv. The receive order is the stable order
 * (expert, source rank, token, slot); with a capacity c, the first c
 * assignments of each expert in that order are kept. */
int moe_dispatch_layout(moe_handle_t h, const int32_t *ids, void *stream);

/* a1 + a2..a3 fused in one kernel: routes logits (as moe_route_topk, writing
 * ids and w) and builds the layout from the routed ids. */
int moe_route_dispatch_layout(moe_handle_t h, const float *logits, int32_t *ids,
                              float *w, void *stream);

/* Completes the per-source tables of the last layout on the handle
 * (src_expert_count, src_expert_kept, count_matrix, send_offset, recv_offset;
 * see moe_layout_view_t) without dispatching: one launch of P CTAs if no
 * dispatch has built them yet, nothing otherwise. Their definitions are those
 * of [EP] "All-to-All-v" (C[s][d]) and "Why count and permute before
 * dispatch" (send_offset = exclusive prefix of send_count).
 * Errors: INVALID_ARG, STATE (no layout yet), CUDA. */
int moe_layout_tables(moe_handle_t h, void *stream);

/* Layout pointers (device) of the handle's workspace. Host-only, no launch. */
int moe_get_layout(moe_handle_t h, moe_layout_view_t *out);

/* a4..a5 -- permute + pack + all-to-all-v scatter ([A2A] 4.3, 5.2; [EP]
 * payload schema, bijection). Needs a preceding layout call on the handle.
 * x: bf16 [T, H]; w: fp32 [T, k] (the weights that travel with the rows).
 * recv_x: rows_max rows of H elements: bf16 for MOE_BF16, e4m3 bytes for
 * MOE_FP8_E4M3. recv_scale: fp32 [rows_max, H/128] for FP8 (per token and
 * 128-channel block: s = amax/448 in fp32, codes = e4m3 RNE satfinite of
 * x/s; an all-zero block has s = 0 and zero codes), NULL for BF16.
 * meta: per-row metadata arrays. Also writes the layout's inv[T*k]. */
int moe_dispatch(moe_handle_t h, const void *x, const float *w, void *recv_x,
                 float *recv_scale, const moe_recv_meta_t *meta, void *stream);

/* NEXT-row comparator, pplx-style fixed receive slots ("Efficient and
 * portable MoE communication", "Dispatch" and "Combine": each rank keeps
 * private storage per source, sized by the maximum tokens per rank). The
 * receive buffer has one region of T_r rows per (expert e, source s), at row
 * (e*P + s)*T_r; assignment (s, t, j) -> e lands at row (e*P + s)*T_r + q, q
 * its rank among source s's assignments to e in (t, j) order. No row depends
 * on another source's counts, so no scan across sources is needed, at the
 * price of E*T rows of storage; region (e, s) holds src_expert_count[s][e]
 * filled rows, the rest untouched. A region holds T_r rows, enough when a
 * token's k ids are distinct; an assignment beyond them (an id repeated
 * within a token) is not written, gets inv = -1 and sets
 * MOE_STATUS_SLOT_OVERFLOW. Needs a preceding layout call on a handle
 * without capacity (MOE_ERR_UNSUPPORTED otherwise, or when the rows exceed
 * int32). slot_x: moe_fixed_slot_rows(cfg) rows of H elements (bf16, or e4m3
 * with fp32 slot_scale [rows, H/128]); meta arrays of that many rows. Same
 * payload, scales and metadata per assignment as moe_dispatch; inv holds the
 * slot rows, so moe_combine / moe_expert_standin (which then treats the slot
 * layout) work unchanged on the slot buffers. */
int moe_dispatch_fixed_slots(moe_handle_t h, const void *x, const float *w, void *slot_x,
                             float *slot_scale, const moe_recv_meta_t *meta, void *stream);

/* Rows of the fixed-slot receive buffer: E*P*T_r, 0 if *cfg is invalid, sets a
 * capacity, or the rows exceed int32. */
int64_t moe_fixed_slot_rows(const moe_config_t *cfg);

/* NEXT-row comparator, the AllGather-style dispatcher ([EP] "Why not collect
 * all tokens with AllGather"): every rank first receives every token
 * (gathered_x: P*T rows, rank d's copy of token g at row d*T + g; FP8 rows are
 * quantised once and copied with their scales into gathered_scale
 * [P*T, H/128], NULL for BF16), then keeps the assignments to its own
 * experts. Same receive rows, metadata and inv as moe_dispatch; T*P rows
 * cross the "network" instead of T*k. */
int moe_dispatch_allgather(moe_handle_t h, const void *x, const float *w, void *gathered_x,
                           float *gathered_scale, void *recv_x, float *recv_scale,
                           const moe_recv_meta_t *meta, void *stream);

/* Persistent single-launch path for small, latency-bound layers (decode):
 * route (logits != NULL: ids and w are written, as moe_route_dispatch_layout)
 * or take given ids and w (logits == NULL), build the layout and dispatch the
 * payload -- everything moe_[route_]dispatch_layout + moe_dispatch produce,
 * bit for bit -- in ONE cooperative launch with one CTA per SM ([A2A] 9-10:
 * a low-latency mode with persistent kernels and device-side
 * synchronisation). Each CTA owns a chunk of one source rank's tokens and
 * streams their x rows into shared memory while it routes and counts; two
 * grid barriers separate counting, the column scans and the scatter. Every
 * barrier gives up after the handle's wait limit (moe_set_wait_limit), sets
 * MOE_STATUS_TIMEOUT and leaves the kernel; the outputs of such a call are
 * undefined and the next call works normally.
 * Returns MOE_ERR_UNSUPPORTED (enqueuing nothing) when one chunk per SM would
 * hold more than 4096 assignments, when P exceeds the SM count, or when the
 * cooperative grid cannot be resident; use the separate calls then. */
int moe_layout_dispatch_fused(moe_handle_t h, const float *logits, int32_t *ids, float *w,
                              const void *x, void *recv_x, float *recv_scale,
                              const moe_recv_meta_t *meta, void *stream);

/* Polls a bounded device wait makes before giving up (default 2^22, about
 * 0.3 s). 0 makes every wait give up at once: for testing the timeout path. */
int moe_set_wait_limit(moe_handle_t h, int64_t polls);

/* NEXT-row comparator, the "standard" two-stage dispatch ([A2A] 4.3 and 5.2):
 * stage 1 packs every kept assignment into its source rank's send buffer
 * ([to rank 0][to rank 1]..., each destination segment bucketed by local
 * expert, (token, slot) order inside), stage 2 is a separate all-to-all-v copy
 * of each (source, expert) segment into the receive regions. Produces exactly
 * what moe_dispatch produces (same receive rows, metadata and inv), through one
 * more full write + read of the payload. send_x: rows_max rows like recv_x;
 * send_scale: rows_max x H/128 fp32 for FP8 (NULL for BF16). */
int moe_dispatch_two_stage(moe_handle_t h, const void *x, const float *w, void *send_x,
                           float *send_scale, void *recv_x, float *recv_scale,
                           const moe_recv_meta_t *meta, void *stream);

/* a6 -- expert stand-in (the pages' grouped GEMM is out of scope): for every
 * kept receive row r of expert e, y[r] = bf16(c[e] * x_r), where x_r is the
 * bf16 payload (c = NULL means c[e] = 1) or, for FP8, the dequantised value
 * e4m3(q) * s. y: bf16 [rows_max, H]. Needs a preceding moe_dispatch with the
 * same recv_x / recv_scale. */
int moe_expert_standin(moe_handle_t h, const void *recv_x, const float *recv_scale,
                       const float *expert_scale, void *y, void *stream);

/* a7 -- combine + unpermute ([EP] "Combine is not simply sending results
 * back"; [PPLX] "Combine"): out[g] = bf16_rne(acc), acc = 0.0f and, for
 * j = 0..k-1 in slot order with inv[g*k+j] >= 0,
 * acc = fmaf(w[g,j], y[inv[g*k+j]], acc). Masked and dropped slots add
 * nothing; weights are not renormalised. y: bf16 [rows_max, H] in receive
 * order; w: fp32 [T, k]; out: bf16 [T, H]. Needs a preceding moe_dispatch. */
int moe_combine(moe_handle_t h, const void *y, const float *w, void *out,
                void *stream);

/* ---- layout without any device allocation -------------------------------
 * The pages have no counterpart for this entry point. It serves callers that
 * may not allocate device memory and have no workspace to hand over: host
 * frameworks whose plugin interface passes only inputs and outputs, processes
 * whose device memory belongs to another allocator (a caching allocator or a
 * fixed budget that a cudaMalloc of ours would overrun or bypass), and code
 * that must not let an allocation or a free synchronise the device. It
 * computes what moe_dispatch_layout computes plus the inverse permutation
 * inv[T*k] (which the workspace path writes during moe_dispatch), from ids
 * int32 [T, k], into the caller's arrays named by *out (every pointer of
 * moe_layout_view_t must be a device array of the size given there). No
 * cudaMalloc, cudaFree or allocating library routine is called.
 * Intermediate data lives in one file-scope device array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the library
 * until the process exits; a problem whose scratch (256 + 4*E*P*ceil(T_r/c)
 * + 4*E*(P+1) + 4*T*k bytes, each term rounded up to 256, c = chunk tokens)
 * exceeds it, or whose layout tables exceed the layout kernels' shared
 * memory (as for moe_handle_create), returns MOE_ERR_UNSUPPORTED and
 * enqueues nothing.
 * The first call in each device context (the first call on a device, and the
 * first after that device was reset) does a one-time set-up with that device
 * current: it looks up the array's device address and raises the layout
 * kernels' shared-memory limits (host-side calls, not stream-ordered work).
 * Every call shares the array and finds the previous call's
 * contents: each call clears the control words first, and calls that overlap
 * on the GPU (other streams, other threads) race and must be serialised by
 * the caller. Ids outside [-1, E) are counted as masked; there is no status
 * word. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int moe_dispatch_layout_noalloc(const moe_config_t *cfg, const int32_t *ids,
                                const moe_layout_view_t *out, void *stream);

/* ---- host <-> device staging ---------------------------------------------
 * Asynchronous copies on `stream` with the copy engines (cudaMemcpyAsync),
 * for callers whose tokens live in host memory: copy x / logits / ids / w in
 * before the layer and the restored rows out after it, all stream-ordered.
 * Host buffers should be page-locked for the copies to be asynchronous.
 * The pages have no counterpart for these two utilities. Errors: INVALID_ARG
 * (null pointer), CUDA. */
int moe_copy_h2d_async(void *dst_device, const void *src_host, size_t bytes, void *stream);
int moe_copy_d2h_async(void *dst_host, const void *src_device, size_t bytes, void *stream);

/* ---- token ranges (NEXT-row pipeline) ----------------------------------------
 * The dispatch, expert stand-in and combine of the global tokens
 * [token_begin, token_end) only, after a layout of the whole layer. Each
 * token's k receive rows are written by the dispatch of its own range, so a
 * caller can pipeline chunks: dispatch chunk c+1 on one stream while another
 * stream (ordered after chunk c's dispatch by an event) runs chunk c's expert
 * and combine ([A2A] 7: start the expert as soon as its inputs have arrived;
 * [EP] "How communication and compute overlap"). Results equal the
 * whole-layer calls. Errors: INVALID_ARG (range outside [0, T]), STATE. */
int moe_dispatch_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end, const void *x,
                        const float *w, void *recv_x, float *recv_scale,
                        const moe_recv_meta_t *meta, void *stream);
int moe_expert_standin_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end,
                              const void *recv_x, const float *recv_scale,
                              const float *expert_scale, void *y, void *stream);
int moe_combine_tokens(moe_handle_t h, int64_t token_begin, int64_t token_end, const void *y,
                       const float *w, void *out, void *stream);

/* Housekeeping (no counterpart on the pages): reads and clears the device
 * status word. Synchronises `stream`: tests and debugging only. *flags
 * receives MOE_STATUS_* bits. */
int moe_read_status(moe_handle_t h, uint32_t *flags, void *stream);

/* Housekeeping (no counterpart on the pages): 1 if this library was built
 * with device bounds checks (compiled with MOE_DEBUG_BOUNDS; built beside the
 * release library as libmoe_ep_debug.so). In that build every row index a
 * kernel computes (receive, send-pool, slot, expert-output and restored rows,
 * and the scale and metadata entries of a row) is checked against its
 * buffer's row count before the access; an index outside it sets
 * MOE_STATUS_BOUNDS and the access is skipped. 0 for the release build. */
int moe_debug_bounds(void);

/* Human-readable name of a MOE_ERR_* code (static string). */
const char *moe_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EP_H */
