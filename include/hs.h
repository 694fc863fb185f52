/*
 * hs.h -- C ABI of libhs: the HiSparse decode-step resolver / swap-in on GB300 (sm_103a).
 *
 * Once per decode step, for every request of the batch, the resolver takes the indexer's
 * top-k token positions and gives back the physical device row that sparse attention must
 * read for each of them. A token is found, in this order, in a GPU-resident page, in the
 * request's fixed-size hot buffer (refreshing its LRU stamp), or else it is copied from
 * pinned host memory into the least-recently-used buffer slot that this step does not need.
 * Short sequences that fit the buffer take a no-copy fast path. A second call copies the
 * newest token's row back to host memory (eager backup).
 *
 * Sources, by page title and section:
 *   "HiSparse: Turbocharging Sparse Attention with Hierarchical Memory" (LMSYS blog, as
 *       translated in "vLLM HiSparse local KV offload architecture") - "Efficient swap-in
 *       kernel": one kernel finds the top-k misses in the device buffer, picks LRU
 *       victims, updates the table and fetches the missing rows from host memory.
 *   "HiSparse: moving the long-context decode capacity bottleneck from GPU memory to CPU
 *       memory" - "Per decode step workflow" (swap-in with a fast path when
 *       seq_len <= device_buffer_size; eager backup of the last token), "Core: swap-in
 *       CUDA kernel" (parameters top_k_tokens, seq_lens, host_cache_locs,
 *       device_buffer_locs, lru_slots), "How capacity is computed" (the per-request buffer
 *       carries an extra page for the new token).
 *   "vLLM HiSparse local KV offload architecture" - "Hot-row lookup and LRU" and
 *       "Performance invariants" (resident, then hot, then pinned host; all decisions on
 *       the GPU; no device readback; graph-capturable; layers sharing an indexer share
 *       one miss plan).
 *   "vLLM Hybrid HiSparse source implementation analysis" - 7.1 (per-slot state, one
 *       hot region per request), 7.2 (resident short-circuit, hot hits, miss plan and
 *       victims, corruption tripwires, gather that zeroes a destination whose source row
 *       is out of range), 7.3 (flat physical row IDs), 7.4 (IndexShare replay).
 *   "Hierarchical Sparse Attention" (Alibaba Tair KVCache) - 2.4.3 "LRU Diff Kernel"
 *       (evict only when the buffer is full, coldest first).
 *
 * Policy (fixed; the CPU oracle in the tests implements the same steps):
 *   For request r with S = seq_lens[r] and every top-k entry t = top_k_tokens[r][i]:
 *   - t < 0 is padding: out = -1.  t >= S: out = -1, flag HS_FLAG_TOKEN.  A valid token
 *     repeated in the row: the first occurrence is resolved, later ones get -1 and
 *     HS_FLAG_DUP.
 *   - Resident: if resident_pages[r][t / page_size] = p >= 0, out = p*page_size + t%page_size.
 *   - Fast path (S <= H): out = device_buffer_locs[r][t]; device_buffer_tokens[r][S-1]
 *     is set to S-1; the clock, stamps and pools are untouched.
 *   - Otherwise (slow path): c = ++lru_clock[r].
 *       newest token t = S-1 -> out = device_buffer_locs[r][H] (the reserved row).
 *       Slot state outside (token in [-1, S-2], stamp in [0, c-1]) is reset to
 *       (-1, 0) and flagged HS_FLAG_STATE.
 *       Hit: the lowest slot s holding t; lru_slots[r][s] = c; out = device_buffer_locs[r][s].
 *       (Several slots holding t also flag HS_FLAG_STATE.)
 *       Misses, in top-k order, take victims among the slots not hit in this call:
 *       free slots (token -1) by ascending slot, then occupied slots by ascending
 *       (stamp, slot). Miss j takes victim j: token and stamp c are stored, and for each
 *       layer the row host_pool[l][host_cache_locs[r][t]] is copied to
 *       device_pool[l][device_buffer_locs[r][victim]].
 *   - A host row outside [0, host_rows) zero-fills the destination (HS_FLAG_HOSTROW). A
 *     physical row outside [0, device_rows) gives out = -1 and writes nothing
 *     (HS_FLAG_DEVROW). S outside [0, max_context] leaves the request untouched with
 *     out = -1 (HS_FLAG_SEQLEN).
 *
 * Memory and ownership. The caller owns every buffer; the library allocates no device or
 * pinned memory and never synchronises inside hs_resolve / hs_backup. Device pointers are
 * CUDA device memory of the device current at hs_create. Host pools are pinned and mapped
 * (cudaHostAlloc(..., cudaHostAllocMapped) or hs_host_register); the kernels read and
 * write them directly over the host link. All arrays are dense, row-major, int32:
 *   top_k_tokens         [R, K]            device or pinned host (below), read
 *   seq_lens             [R]               device or pinned host, read
 *   host_cache_locs      [R, max_context]  device, read      token -> host row
 *   device_buffer_locs   [R, H+1]          device, read      slot -> device row; slot H is
 *                                                            the newest-token row
 *   device_buffer_tokens [R, H]            device, read/write slot -> token, -1 = free
 *   lru_slots            [R, H]            device, read/write per-slot LRU stamp
 *   lru_clock            [R]               device, read/write per-request clock
 *   resident_pages       [R, max_pages]    device, read, or NULL   page -> device page
 *   out_rows             [R, K]            device or pinned host, write   physical row per entry
 *   miss_counts          [R]               device or pinned host, write, or NULL
 * Zero-copy step I/O: top_k_tokens, seq_lens, out_rows and miss_counts may instead be pinned,
 * mapped host memory (cudaHostAlloc, or registered, and addressed by its unified pointer) for
 * a scheduler that produces and consumes them on the host. The kernels then read the inputs
 * and write the outputs over the host link themselves, with plain loads and stores, and no
 * separate copies are needed; the caller must not touch those buffers until the stream has
 * passed the call. Every other array stays in device memory.
 * Initial state: long requests tokens = -1, stamps = 0, clock = 0; requests with
 * S <= H hold token s in slot s (rows already written) for s < S.
 * Preconditions not checked on the device: device_buffer_locs rows are distinct and
 * disjoint from resident rows; the forward pass has written the newest token's row to
 * its resident row, or to slot S-1 when S <= H, else to slot H, before hs_resolve.
 * Calls that share state arrays must be ordered on one stream.
 *
 * Errors. Host-side validation returns a status synchronously. A failed launch returns
 * HS_ERR_CUDA. Data anomalies met on the device are OR-ed as HS_FLAG_* bits into the
 * error word in the caller's workspace and never trap; hs_get_error reads them.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HS_API __attribute__((visibility("default")))
#else
#define HS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* hs_stream_t;

typedef enum {
  HS_OK = 0,
  HS_ERR_INVALID_ARG = 1,    /* null pointer, size out of range, wrong memory kind */
  HS_ERR_INVALID_CONFIG = 2, /* configuration the kernels cannot run (limits below) */
  HS_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  HS_ERR_DEVICE_FLAGGED = 4, /* hs_get_error found HS_FLAG_* bits set */
  HS_ERR_TIMEOUT = 5         /* not returned by this version: a bounded device wait that runs out
                                sets HS_FLAG_TIMEOUT in the error word instead (the resolve's copy
                                CTAs waiting for their outcomes, the consumer's role hand-offs) */
} hs_status;

/* Device-side anomaly bits in the workspace error word (sticky until cleared). */
#define HS_FLAG_TOKEN 1u   /* top-k entry >= seq_len */
#define HS_FLAG_DUP 2u     /* repeated valid token in one top-k row */
#define HS_FLAG_STATE 4u   /* corrupt slot token/stamp, or a token held by two slots */
#define HS_FLAG_HOSTROW 8u /* host row out of range: destination zero-filled */
#define HS_FLAG_DEVROW 16u /* device row out of range: output -1, nothing written */
#define HS_FLAG_SEQLEN 32u /* seq_len outside [0, max_context]: request skipped */
#define HS_FLAG_ORDER 64u  /* hs_invalidate_host_rows: rows not ascending, nothing cleared */
#define HS_FLAG_TIMEOUT 128u /* a bounded device wait ran out: that call's outputs are invalid */

/* Limits of this build. */
#define HS_MAX_TOP_K 4096
#define HS_MAX_HOT_SLOTS 16384
#define HS_MAX_LAYERS 8
#define HS_MAX_SPEC_QUERIES 8 /* verify steps of one speculative batch (n_spec + 1) */
#define HS_MAX_MLA_SPLITS 16  /* row splits of hs_sparse_mla_decode */

/* Configuration of one layer group (layers that share one indexer top-k and therefore
 * one slot map; "vLLM Hybrid HiSparse source implementation analysis" 7.4).
 *   max_requests  largest R passed to hs_resolve / hs_backup
 *   top_k         K, 1..HS_MAX_TOP_K
 *   hot_slots     H (device_buffer_size), K..HS_MAX_HOT_SLOTS
 * K and H must also leave the resolve CTA's tables within the device's shared memory per
 * block (227 KB on GB300): about 37 K + 9 H bytes (rounding K up to a power of two for its
 * hash). hs_create rejects a larger pair with HS_ERR_INVALID_CONFIG; e.g. K = 2048 takes any
 * H up to HS_MAX_HOT_SLOTS, K = 4096 H up to ~8,800.
 *   row_bytes     B, bytes of one token's KV row in one layer (656 for fp8 MLA)
 *   num_layers    L, 1..HS_MAX_LAYERS
 *   page_size     residency page size in tokens; 0 disables resident_pages
 *   max_context   row stride of host_cache_locs; seq_len may not exceed it
 *   max_pages     row stride of resident_pages; >= ceil(max_context / page_size)
 *   host_row_stride  bytes from host row h to host row h + 1 inside one layer's host pool;
 *                 0 means row_bytes. Host row h of layer l is read at
 *                 host_pools[l] + h * host_row_stride. With row_bytes (one pool per layer,
 *                 "layer first") each layer's rows are back to back. With
 *                 num_layers * row_bytes and host_pools[l] = base + l * row_bytes ("page
 *                 first") one host row holds every layer's bytes of a token, so a miss reads
 *                 one contiguous span for the whole group. Both are layouts of the host IO
 *                 kernel in "Hierarchical Sparse Attention" (Alibaba Tair KVCache), 2.4.4
 *                 "I/O Transfer Kernel" (layer_first, page_first); "vLLM Hybrid HiSparse
 *                 source implementation analysis", 2.1 and 2.3, likewise packs a hot unit's
 *                 leader and follower layers into one combined page and sizes host blocks by
 *                 one stride. Must be 0 or >= row_bytes. */
typedef struct {
  int32_t max_requests;
  int32_t top_k;
  int32_t hot_slots;
  int32_t row_bytes;
  int32_t num_layers;
  int32_t page_size;
  int32_t max_context;
  int32_t max_pages;
  int32_t host_row_stride;
} hs_config;

typedef struct hs_handle hs_handle;

/* Bytes of device workspace hs_create needs; 0 if the configuration is invalid. The
 * workspace is laid out as:
 *   - 256 bytes: the sticky error word and the per-layer pool table;
 *   - the residency bitmap (the miss "hints"): one bit per (request, token position), set
 *     while the token sits in one of the request's hot slots. Each request's row is
 *     ceil(max_context / 128) x 16 bytes; the whole bitmap is rounded up to 256 bytes. The
 *     kernels keep it current and use it only to start a miss's host transfer before the
 *     exact slot probe finishes (a clear bit predicts a miss). Every result comes from the
 *     probe, so bits left stale by changes the caller makes to the state arrays cost time,
 *     never correctness;
 *   - the follower plans: HS_MAX_SPEC_QUERIES slices, each miss tokens and device rows,
 *     max_requests x top_k int32 each, then max_requests counts, rounded up to 256 bytes. A
 *     plain resolve records its plan in slice 0 (hs_gather replays it), verify step q of a
 *     speculative batch in slice q (hs_gather_spec);
 *   - the same misses grouped by 2 MB region of the host pool: per plan entry its host row
 *     (max_requests x top_k int32), then per plan slice its (host row, device row) pairs
 *     (2 x max_requests x top_k int32), two tables of 16,385 per-region int32 counters and
 *     the pair counts. A copy that takes the rows region by region reuses
 *     the GPU's address translation of each region for several rows; in the order the
 *     resolve finds them, rows spread over several large pools moved at about half the
 *     host link's rate.
 * The caller keeps the workspace for the handle's lifetime and does not write to it.
 * Why the caller allocates it: "vLLM HiSparse local KV offload architecture", "Ownership"
 * -- the allocator provides GPU capacity and holds no KV semantics, while the runtime that
 * resolves hits and picks victims owns the bytes bound to it; here the caller plays the
 * allocator and the library the runtime, so the library never allocates device memory.
 * Host only: no device work, no allocation. */
HS_API size_t hs_workspace_bytes(const hs_config* cfg);

/* Validate the configuration and bind the pools ("vLLM HiSparse local KV offload
 * architecture", "Ownership": the runtime binds host and hot storage that others allocate;
 * "Performance invariants": hot misses copy straight from registered pinned host memory).
 * host_pools / device_pools are arrays of num_layers pointers to pinned+mapped host pools
 * (host_rows rows of row_bytes, host_row_stride apart) and [device_rows, row_bytes] device
 * pools. workspace is caller-owned device memory of hs_workspace_bytes(cfg) bytes, zeroed
 * here (synchronously: set-up, not the decode path). Allocates only the small host-side
 * handle; the pointers must stay valid for its lifetime. Returns HS_ERR_INVALID_ARG (a NULL
 * or misplaced pointer: host pools not pinned and mapped, device pools or workspace not on
 * the current device, workspace not 16-byte aligned), HS_ERR_INVALID_CONFIG (limits above,
 * or tables that do not fit the device's shared memory) or HS_ERR_CUDA, with *out set to
 * NULL. */
HS_API hs_status hs_create(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                    int64_t host_rows, int64_t device_rows, void* workspace, hs_handle** out);

/* One decode step of the resolver for requests 0..num_requests-1 (layout and policy above;
 * "HiSparse: moving the long-context decode capacity bottleneck from GPU memory to CPU
 * memory", "Core: swap-in CUDA kernel" names its arguments; "vLLM HiSparse local KV offload
 * architecture", "Hot-row lookup and LRU" orders resident, hot, host; "Performance
 * invariants": every decision on the GPU, no device scalar readback or CPU round trip,
 * capturable in a CUDA graph). One kernel launch on `stream` -- four when the configuration
 * leaves no room for copy CTAs
 * (more requests than the GPU has SMs, or rows not 16-byte copyable): the resolve then
 * records the miss plan without copying, two small kernels group the misses by host
 * region, and a gather kernel copies every layer's rows, with the same results
 * (hs_launch_shape tells which). No allocation, no synchronisation, capturable in a CUDA
 * graph. num_requests == 0 is a no-op. */
HS_API hs_status hs_resolve(hs_handle* h, int32_t num_requests, const int32_t* top_k_tokens,
                     const int32_t* seq_lens, const int32_t* host_cache_locs,
                     const int32_t* device_buffer_locs, int32_t* device_buffer_tokens,
                     int32_t* lru_slots, int32_t* lru_clock, const int32_t* resident_pages,
                     int32_t* out_rows, int32_t* miss_counts, hs_stream_t stream);

/* hs_resolve for a layer group split into a leader and followers ("vLLM Hybrid HiSparse
 * source implementation analysis", 7.4: layers that share the indexer share the slot plan
 * and copy only their own bytes). The step is resolved exactly as by hs_resolve, but miss
 * rows are copied only for layers [0, copy_layers) (0 <= copy_layers <= num_layers), and
 * the miss plan -- per request, the miss tokens and their device rows in miss order -- is
 * kept in the workspace for hs_gather. When copy_layers < num_layers, or the geometry has
 * no copy CTAs, the call also groups the plan by host region (two more launches), and the
 * gathers that follow copy the rows in that order. hs_resolve is this call with
 * copy_layers = num_layers (it records the plan too). Same rules as hs_resolve. */
HS_API hs_status hs_resolve_layers(hs_handle* h, int32_t num_requests, const int32_t* top_k_tokens,
                                   const int32_t* seq_lens, const int32_t* host_cache_locs,
                                   const int32_t* device_buffer_locs, int32_t* device_buffer_tokens,
                                   int32_t* lru_slots, int32_t* lru_clock, const int32_t* resident_pages,
                                   int32_t* out_rows, int32_t* miss_counts, int32_t copy_layers,
                                   hs_stream_t stream);

/* A speculative batch ("vLLM HiSparse local KV offload architecture", speculative
 * decoding: each verify step is resolved and consumed in order, with its own replayable
 * plan rows and the request's shared hot state; "vLLM Hybrid HiSparse source
 * implementation analysis", 7.4 and 7.1: one resolve per verify step, a buffer of
 * (n_spec + 2) x top_k rows). num_queries = Q = n_spec + 1 (1..HS_MAX_SPEC_QUERIES) verify
 * steps run in order in one kernel launch, each request's cluster looping over its steps
 * (without copy CTAs the launch is followed, step by step, by the grouping of the step's plan
 * by host region and its gather, as in hs_resolve): step q resolves top_k_tokens[q] for
 * committed_lens[r] + q + 1 tokens into out_rows[q] and miss_counts[q]. The batch's
 * positions t >= S0 = committed_lens[r] (the token the last round sampled, then the drafts;
 * the forward pass has written them) resolve to the reserved rows H + (t - S0): with Q
 * queries, device_buffer_locs is [R, H + Q]. The clock advances once per slow-path verify
 * step, so with H >= (Q + 1) * top_k no verify step evicts a row an earlier step of the batch
 * resolved: every step's out_rows stay valid until the batch is consumed. On the fast path a
 * batch records slots S0 - Q .. S0 (committed), never its drafts.
 *   top_k_tokens [Q, R, K], out_rows [Q, R, K], miss_counts [Q, R] or NULL; the rest as in
 *   hs_resolve. Every layer's miss rows are copied, and step q records its miss plan in
 *   plan slice q (hs_gather_spec). */
HS_API hs_status hs_resolve_spec(hs_handle* h, int32_t num_requests, int32_t num_queries,
                                 const int32_t* top_k_tokens, const int32_t* committed_lens,
                                 const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                                 int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                                 const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                                 hs_stream_t stream);

/* hs_resolve_spec for a layer group split into a leader and followers (IndexShare under
 * MTP: "vLLM Hybrid HiSparse source implementation analysis", 7.4, followers replay the
 * leader's plan and every verify step is its own resolve over its own workspace slice).
 * The batch is resolved exactly as by hs_resolve_spec, but each verify step copies miss
 * rows only for layers [0, copy_layers) (0 <= copy_layers <= num_layers); its plan is kept
 * in slice q for hs_gather_spec. When copy_layers < num_layers, or the geometry has no copy
 * CTAs, each step's plan is also grouped by host region (two more launches per step).
 * hs_resolve_spec is this call with copy_layers = num_layers. Same rules as hs_resolve_spec. */
HS_API hs_status hs_resolve_spec_layers(hs_handle* h, int32_t num_requests, int32_t num_queries,
                                        const int32_t* top_k_tokens, const int32_t* committed_lens,
                                        const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                                        int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                                        const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                                        int32_t copy_layers, hs_stream_t stream);

/* Follower gather of one verify step of the last speculative batch: copy step `query`'s
 * miss rows (0 <= query < that batch's num_queries) for layers [first_layer, first_layer +
 * num_layers), as hs_gather does for a plain step: in host-region order when the batch
 * grouped its plans, else in miss order. num_requests must be the batch's. When a slot is reused within the batch (H < (Q + 1) x top_k), replay the steps
 * in step order so that each row ends with the last step's token. HS_ERR_INVALID_ARG when
 * the last resolve was not a speculative batch. One kernel launch, graph-capturable. */
HS_API hs_status hs_gather_spec(hs_handle* h, int32_t num_requests, const int32_t* host_cache_locs,
                                int32_t query, int32_t first_layer, int32_t num_layers, hs_stream_t stream);

/* Eager backup after a speculative batch: the first accepted[r] positions S0 + j of the
 * batch (S0 = committed_lens[r], 0 <= accepted <= num_queries) are now committed, and each
 * one's row -- its resident row, slot S0 + j while the sequence then fit the buffer
 * (S0 + j + 1 <= H), else the reserved row H + j -- goes to its host row, every layer.
 * hs_backup is this call with num_queries = 1, committed_lens = seq_len - 1, accepted = 1.
 * accepted outside [0, num_queries] or past max_context skips the request (HS_FLAG_SEQLEN).
 * One kernel launch; same rules as hs_backup. */
HS_API hs_status hs_backup_spec(hs_handle* h, int32_t num_requests, int32_t num_queries,
                                const int32_t* committed_lens, const int32_t* accepted,
                                const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                                const int32_t* resident_pages, hs_stream_t stream);

/* Follower gather: copy the last resolve's miss rows for layers [first_layer, first_layer +
 * num_layers) -- host_pool[l][host_cache_locs[r][token]] to device_pool[l][row] for every
 * planned miss, zeros (HS_FLAG_HOSTROW) when the host row is out of range -- with no LRU
 * work. host_cache_locs [R, max_context] device, read (the resolve's). It must run after
 * that resolve (same stream, or an event) and before the next one; calls for different
 * layers may run on other streams concurrently. When that resolve grouped its plan by host
 * region (hs_resolve_layers), the rows are copied in that order and num_requests must be
 * the resolve's; otherwise the plan of requests 0..num_requests-1 is replayed in miss order.
 * HS_ERR_INVALID_ARG after a speculative batch (its steps' plans: hs_gather_spec). One
 * kernel launch, layer by layer; no allocation, no synchronisation; graph-capturable.
 * num_layers == 0 is a no-op. */
HS_API hs_status hs_gather(hs_handle* h, int32_t num_requests, const int32_t* host_cache_locs,
                           int32_t first_layer, int32_t num_layers, hs_stream_t stream);

/* Eager backup ("Per decode step workflow", step 5): for every request with seq_len >= 1
 * and every layer, copy the newest token's row -- its resident row, else slot seq_len-1
 * when seq_len <= H, else slot H -- to host_pool[l][host_cache_locs[r][seq_len-1]].
 * One kernel launch on `stream`; same rules as hs_resolve. */
HS_API hs_status hs_backup(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                    const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                    const int32_t* resident_pages, hs_stream_t stream);

/* Hot-slot invalidation by token ("vLLM Hybrid HiSparse source implementation analysis",
 * 6, invalidation propagation: rows rewritten on the host leave the hot set exactly).
 * For each request r, every slot holding one of the tokens
 * tokens[token_offsets[r] .. token_offsets[r+1]) becomes free (token -1, stamp 0) and the
 * token's residency bit is cleared, so the next hs_resolve misses on it and copies its current host
 * row. Only tokens in [0, seq_len - 1) count (no valid slot holds another). Requests with
 * seq_len <= H are on the fast path and are left alone: their device rows are the tokens'
 * own rows, which the forward pass rewrites in place. seq_len outside [0, max_context]
 * skips the request (HS_FLAG_SEQLEN). The clock does not move.
 *   seq_lens      [R]      device, read
 *   token_offsets [R + 1]  device, read, non-decreasing (CSR row pointers; not checked)
 *   tokens        [token_offsets[R]] device, read, any order, repeats and -1 allowed
 * One kernel launch on `stream`; never synchronises or allocates; graph-capturable. */
HS_API hs_status hs_invalidate_tokens(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                                      const int32_t* token_offsets, const int32_t* tokens,
                                      int32_t* device_buffer_tokens, int32_t* lru_slots, hs_stream_t stream);

/* Hot-slot invalidation by host row (same section: host blocks handed to other content).
 * Every slot of every request past the fast path whose token's host row
 * host_cache_locs[r][token] is one of rows[0 .. n) becomes free as above.
 *   rows [n] device, read, ascending, repeats allowed. When n <= 8192 every CTA checks the
 *   order and, if it is broken, clears nothing and sets HS_FLAG_ORDER; a longer list is
 *   binary-searched as given (its order is not checked).
 * One kernel launch on `stream`; same rules as hs_invalidate_tokens. */
HS_API hs_status hs_invalidate_host_rows(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                                         const int32_t* host_cache_locs, const int32_t* rows, int32_t n,
                                         int32_t* device_buffer_tokens, int32_t* lru_slots,
                                         hs_stream_t stream);

/* Synthetic consumer of the row table: sparse-MLA decode attention ("vLLM Hybrid HiSparse
 * source implementation analysis", 7.3: the sparse attention kernel reads the pool's flat view
 * through the resolver's physical rows; 9: an fp8 sparse-MLA row is 656 B -- 512 e4m3 latent
 * codes, 4 fp32 scales (one per 128 codes), 64 bf16 RoPE values). For request r and head h
 * over the rows j = out_rows[r][i] >= 0:
 *   s[h, j] = sm_scale * (q[h, :512] . latent_j + q[h, 512:] . rope_j), latent = e4m3 x scale
 *   o[r, h] = softmax_j(s[h]) . latent,  lse[r, h] = log sum_j exp s[h, j]  (-inf, o = 0 if none)
 * Computed on the tensor cores in fp16 with fp32 accumulation and an online softmax: q and the
 * RoPE values are converted from bf16 to fp16, each latent code times its scale is rounded to
 * fp16, and so is P. The inputs must therefore stay within fp16's range (|value| < 65504;
 * values under 2^-14 lose precision). `splits` (1..HS_MAX_MLA_SPLITS) divides each request's
 * rows over more CTA pairs, whose partial outputs are merged by log-sum-exp: for two splits,
 * when a four-CTA cluster per request fits the device in one wave, inside the kernel (the two
 * pairs of a request share a cluster); otherwise in a second kernel.
 *   q        [R, num_heads, 576] bf16 bits, device, 16-byte aligned (num_heads <= 128)
 *   kv_pool  [pool_rows, 656] bytes, device (a layer's device pool), 16-byte aligned
 *   out_rows [R, top_k] device (hs_resolve's output), top_k <= HS_MAX_TOP_K; rows outside
 *            the pool count as -1
 *   o        [R, num_heads, 512] fp32, device, 16-byte aligned; lse [R, num_heads] fp32, device
 *   workspace: hs_sparse_mla_workspace_bytes(R, num_heads, splits) device bytes (0 for one split)
 *   error_flags: device uint32, HS_FLAG_TIMEOUT OR-ed in if a bounded wait ran out.
 * Two kernel launches at most; no allocation, no synchronisation; graph-capturable. */
HS_API size_t hs_sparse_mla_workspace_bytes(int32_t num_requests, int32_t num_heads, int32_t splits);
/* The kernel launches one hs_sparse_mla_decode call makes for this shape on the current device:
 * 1 (one split, or two splits merged inside the kernel), 2 (the attention kernel and the merge
 * kernel), 0 for a shape hs_sparse_mla_decode refuses (num_requests < 1 here). For two splits
 * the first call on a device asks the runtime how many four-CTA clusters fit at once. */
HS_API int32_t hs_sparse_mla_launches(int32_t num_requests, int32_t num_heads, int32_t splits);
HS_API hs_status hs_sparse_mla_decode(int32_t num_requests, int32_t num_heads, int32_t top_k, int32_t splits,
                                      const uint16_t* q, const uint8_t* kv_pool, int64_t pool_rows,
                                      const int32_t* out_rows, float sm_scale, float* o, float* lse,
                                      void* workspace, size_t workspace_bytes, uint32_t* error_flags,
                                      hs_stream_t stream);

/* Forget the residency bitmap (every bit clear, as hs_create leaves it), in stream order.
 * Call it after changing device_buffer_tokens outside the library -- a request row handed
 * to a new sequence, a restored checkpoint -- so the copy CTAs' miss predictions match the
 * new state again: with every bit clear they first predict every looked-up token to miss,
 * and each hit sets its bit back. Results never depend on it: stale bits cost only speed.
 * One cudaMemsetAsync of about max_requests x max_context / 8 bytes; graph-capturable. */
HS_API hs_status hs_reset_hints(hs_handle* h, hs_stream_t stream);

/* The launch shape hs_create chose for this handle (host only; no device work). copy_ctas:
 * copy CTAs clustered with each request's resolve CTA, 0..3. resolve_launches: kernel launches one hs_resolve makes, 1, or 4 when
 * copy_ctas is 0 (the rows then move in a gather over the plan grouped by host region).
 * Either pointer may be NULL. HS_ERR_INVALID_ARG for a NULL handle. */
HS_API hs_status hs_launch_shape(const hs_handle* h, int32_t* copy_ctas, int32_t* resolve_launches);

/* Read the workspace error word: the HS_FLAG_* bits the kernels OR in when they meet bad
 * data ("vLLM Hybrid HiSparse source implementation analysis", 7.2: corrupt slot state is
 * downgraded to a re-miss rather than trusted, and a source row out of range zero-fills its
 * destination; the kernels never trap). It synchronises the device, so it is kept off the
 * decode path ("vLLM HiSparse local KV offload architecture", "Performance invariants": no
 * device scalar readback per step; 7.1 of the analysis reads its statistics only every 2000
 * calls, outside capture). With clear != 0 the word is reset to zero. Returns
 * HS_ERR_DEVICE_FLAGGED when any bit is set, HS_ERR_INVALID_ARG for a NULL argument,
 * HS_ERR_CUDA when a CUDA call fails. */
HS_API hs_status hs_get_error(hs_handle* h, uint32_t* flags, int clear);

/* Free the host-side handle and nothing else: the pools, tables, state and workspace stay
 * the caller's ("vLLM HiSparse local KV offload architecture", "Ownership": the allocator
 * owns capacity, the runtime binds it). Call it after the last stream work that uses the
 * handle has been issued; work already queued keeps running. NULL is accepted. Always
 * HS_OK. */
HS_API hs_status hs_destroy(hs_handle* h);

/* Static, NUL-terminated description of a status code (never NULL; unknown codes give
 * "unknown status"). The codes follow the error split of this header: host-side validation
 * returns a status at once, device anomalies become HS_FLAG_* bits. */
HS_API const char* hs_status_str(hs_status s);

/* Page-lock an existing host range for the kernels' direct access (cudaHostRegister with
 * the mapped and portable flags) and return the device-side address in *device_ptr. */
HS_API hs_status hs_host_register(void* ptr, size_t bytes, void** device_ptr);

/* Undo hs_host_register. */
HS_API hs_status hs_host_unregister(void* ptr);

/* Host memory placement for the host pools. "Hierarchical Sparse Attention" (Alibaba Tair
 * KVCache), 2.4.4 "I/O Transfer Kernel", reaches its per-GPU copy rate with NUMA binding: the
 * pinned host pool a GPU reads should sit in the host memory nearest that GPU. On a node
 * whose CPUs each serve some of the GPUs, one process per GPU places its own pools.
 *
 * hs_host_numa_node: the host memory node nearest `device` (cudaDevAttrHostNumaId, else the
 * numa_node of the device's PCI function in sysfs), or -1 in *node when the platform does not
 * say. Host only; HS_ERR_INVALID_ARG for a NULL node, HS_ERR_CUDA when the device cannot be
 * queried.
 *
 * hs_host_bind_node: give [ptr, ptr + bytes) a preferred-node memory policy (mbind,
 * MPOL_PREFERRED) for `node`, so the pages it has not touched yet are taken from that node
 * (falling back to others when it is full). Call it on a fresh anonymous mapping before its
 * pages are first touched and before hs_host_register; pages already present do not move.
 * ptr is rounded down and the end up to whole pages. No allocation, no device work.
 * HS_ERR_INVALID_ARG for a NULL range or a negative node, HS_ERR_CUDA (the system error) when
 * the kernel refuses the policy. */
HS_API hs_status hs_host_numa_node(int32_t device, int32_t* node);
HS_API hs_status hs_host_bind_node(void* ptr, size_t bytes, int32_t node);

/* hs_resolve for callers that cannot allocate device memory. The pages have no
 * counterpart for this entry point: it exists for callers with no way to make the
 * workspace allocation hs_create needs -- engines whose device memory is all planned
 * before decoding starts, plugins running inside another framework's allocator, or
 * processes that must not call cudaMalloc on the decode path.
 *
 * It takes the configuration and pools that hs_create takes, plus every argument of
 * hs_resolve, and runs the same resolve kernel with the same results. Instead of a
 * caller workspace it uses a 256-byte file-scope device array inside the library: the
 * error word and the pools table of at most HS_NOALLOC_MAX_LAYERS layers (num_layers
 * above that: HS_ERR_INVALID_CONFIG). Every device that loads the library holds its own
 * copy of that array until the process exits. The call allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *
 * The first call on a device, with that device current, looks up the array's device
 * address (cudaGetSymbolAddress), checks the pools and fits the kernel to the device, and
 * caches all three. A later call with the
 * same configuration and pools reuses them; a changed configuration or pool set redoes the
 * set-up on the host (no allocation). Each call then queues, on `stream`, a one-thread
 * kernel that writes the pools table into the array and clears its error word, the resolve
 * kernel, and, when error_flags is not NULL, a copy of this call's HS_FLAG_* bits into
 * error_flags (one uint32 in device memory). Nothing is copied from host memory.
 * All calls share the array and it keeps the last call's contents, so calls whose work
 * overlaps on the GPU (on streams not ordered against each other) race; order them on
 * one stream. Returns the status codes of hs_create and hs_resolve. */
#define HS_NOALLOC_MAX_LAYERS 8
HS_API hs_status hs_resolve_noalloc(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                                    int64_t host_rows, int64_t device_rows, int32_t num_requests,
                                    const int32_t* top_k_tokens, const int32_t* seq_lens,
                                    const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                                    int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                                    const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                                    uint32_t* error_flags, hs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
