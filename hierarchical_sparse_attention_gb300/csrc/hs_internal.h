// Internal launch interface between the C ABI (hs_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "hs.h"

namespace hs {

constexpr int kResolveThreads = 1024;  // one CTA of 32 warps per request
constexpr int kBackupThreads = 256;    // 8 warps, one (request, layer) row per warp
constexpr int kInvalidateThreads = 1024;  // one CTA per request
constexpr int kGatherThreads = 256;        // one CTA per (request, run of kGatherMisses misses)
constexpr int kGatherMisses = 32;
constexpr int kMaxLayers = HS_MAX_LAYERS;

// Per-layer pool base addresses as the kernels dereference them. hs_create writes this
// table into the caller's workspace at kPoolsOffset, so kernels index it by layer from
// global/shared memory instead of copying a by-value parameter array to local memory.
struct Pools {
  const uint8_t* host[kMaxLayers];  // device-side addresses of the pinned, mapped host pools
  uint8_t* dev[kMaxLayers];
};

// Everything the kernels need to know about one layer group, fixed at hs_create.
struct Geometry {
  int32_t K, H, B, L;
  int32_t page_size, max_context, max_pages;
  int32_t hash_bits;  // top-k hash table holds 1 << hash_bits >= 2K entries
  int32_t sort_cap;   // power of two >= K: capacity of the victim sort buffer
  int32_t vec;        // bytes per copy piece: 16, 4 or 1
  int32_t copy_ctas;  // copy CTAs clustered with each request's resolve CTA (0: it copies alone)
  int32_t copy_cap;   // misses one copy CTA can stage (all layers) in its shared memory
  int32_t dbl_smem;   // 1: the resolve CTA stages the slot -> row table in shared memory; 0: it
                      // reads it from global memory (large H, where the table does not fit)
  int32_t bit_words;  // uint32 words per request in the residency bitmap (a multiple of 4)
  int32_t bits_smem;  // 1: each copy CTA stages its request's bitmap row in shared memory
  int32_t order_shift;    // host rows [b << order_shift, (b + 1) << order_shift) form host region b
  int32_t order_regions;  // regions covering the host pool (<= kOrderRegions); region
                          // order_regions collects misses whose host row is out of range
  int32_t host_interleaved;  // 1: host_pools[l] = host_pools[0] + l * B and host_stride =
                             // L * B ("page first"): one host row holds every layer's
                             // bytes, so a miss of layers [a, b) is one contiguous span
  int32_t sms;               // SMs of the device (grid size of the persistent pair gather)
  int32_t gather_ctas_per_sm;  // pair-gather CTAs resident on one SM at once
  int64_t host_stride;       // bytes from one host row to the next inside a layer's pool
  int64_t host_rows, device_rows;
};

struct ResolveArgs {
  uint32_t* hint;  // [R, bit_words] residency bitmap in the workspace, or NULL
  const int32_t* top_k_tokens;
  const int32_t* seq_lens;
  const int32_t* host_cache_locs;
  const int32_t* device_buffer_locs;
  int32_t* device_buffer_tokens;
  int32_t* lru_slots;
  int32_t* lru_clock;
  const int32_t* resident_pages;
  int32_t* out_rows;
  int32_t* miss_counts;
  int32_t copy_layers;  // layers [0, copy_layers) get their miss rows in this call
  int32_t* plan_tok;    // [R, K] miss tokens in miss order (the follower plan), or NULL
  int32_t* plan_dst;    // [R, K] their device rows (-1: none)
  int32_t* plan_cnt;    // [R] misses per request
  int32_t spec_q;       // -1: a plain step (seq_lens are lengths); q >= 0: verify step q of a
                        // speculative batch (seq_lens are the batch's first positions S0)
  int32_t spec_n;       // reserved rows after the H slots (1, or the batch's Q)
  // One launch for a whole speculative batch: spec_steps > 0 runs verify steps
  // 0..spec_steps - 1 in order inside the kernel (spec_q is then the loop's), step q taking
  // top_k_tokens / out_rows + q * step_rk, miss_counts + q * step_r and plan slice q (the plan
  // pointers + q * step_plan). 0: the one step spec_q.
  int32_t spec_steps = 0;
  int32_t step_r = 0;
  int64_t step_rk = 0;
  int64_t step_plan = 0;
};

struct GatherArgs {
  const int32_t* host_cache_locs;
  const int32_t* plan_tok;
  const int32_t* plan_dst;
  const int32_t* plan_cnt;
  int32_t first_layer, num_layers;
};

// The last resolve's misses as (host row, device row) pairs grouped by host region, built by
// launch_order and copied by launch_gather_pairs. Arrays live in the workspace (order_bytes).
struct OrderArgs {
  const int32_t* host_cache_locs;
  const int32_t* plan_tok;
  const int32_t* plan_dst;
  const int32_t* plan_cnt;
  int32_t* miss_src;   // [R, K] per plan entry: host row, -1 out of range, -2 no device row
  int32_t* pair_src;   // [R * K] host rows (-1: zero-fill), grouped by region (one plan slice's)
  int32_t* pair_dst;   // [R * K] device rows
  int32_t* counts;     // [kOrderRegions + 1] misses per region (zero between steps)
  int32_t* cursors;    // [kOrderRegions + 1] next free position per region
  int32_t* n_pairs;    // pairs in the list
  uint32_t* ticket;    // CTAs of the count kernel done (zero between steps)
  int64_t capacity;    // max_requests * K
};

struct BackupArgs {
  const int32_t* seq_lens;  // lengths, or the batch's first positions S0 with `accepted`
  const int32_t* host_cache_locs;
  const int32_t* device_buffer_locs;
  const int32_t* resident_pages;
  const int32_t* accepted;  // NULL: the newest position; else [R] accepted positions of a batch
  int32_t spec_n;           // reserved rows after the H slots (1, or the batch's Q)
};

struct InvalidateArgs {
  uint32_t* hint;  // [R, bit_words] residency bitmap, or NULL
  const int32_t* seq_lens;
  const int32_t* token_offsets;  // [R + 1]
  const int32_t* tokens;
  int32_t* device_buffer_tokens;
  int32_t* lru_slots;
};

struct InvalidateRowsArgs {
  uint32_t* hint;  // [R, bit_words] residency bitmap, or NULL
  const int32_t* seq_lens;
  const int32_t* host_cache_locs;
  const int32_t* rows;  // ascending
  int32_t n;
  int32_t* device_buffer_tokens;
  int32_t* lru_slots;
};

struct SparseMlaArgs {
  const uint16_t* q;      // [R, num_heads, 576] bf16
  const uint8_t* kv_pool; // [pool_rows, 656] fp8 MLA rows
  int64_t pool_rows;
  const int32_t* out_rows;  // [R, top_k], -1: none
  int32_t top_k, num_heads, splits;
  float sm_scale;
  float* o;    // [R, num_heads, 512]
  float* lse;  // [R, num_heads]
};

// Workspace layout (device memory owned by the caller).
constexpr size_t kErrOffset = 0;     // uint32 sticky HS_FLAG_* word
constexpr size_t kPoolsOffset = 64;  // Pools table
constexpr size_t kWorkspaceBytes = 256;  // header: error word + pools table
static_assert(kPoolsOffset + sizeof(Pools) <= kWorkspaceBytes, "workspace too small for the pools table");
constexpr int kMaxEntriesPerThread = (HS_MAX_TOP_K + kResolveThreads - 1) / kResolveThreads;

// After the header, hs_create's workspace holds the residency bitmap: one bit per (request,
// token position), set while the token sits in one of the request's hot slots. Each request's
// row is hint_words() uint32 words, 16-byte aligned. The kernels keep it current and use it
// only to start miss transfers early (a clear bit predicts a miss); every result still comes
// from the exact slot probe, so a stale bit costs time, never correctness.
inline int32_t hint_words(int64_t max_context) { return (int32_t)(((max_context + 127) / 128) * 4); }
inline size_t hint_bytes(int64_t max_requests, int64_t max_context) {
  return (size_t)(((max_requests * hint_words(max_context) * 4) + 255) & ~(int64_t)255);
}
constexpr int32_t kBitsSmemMax = 64 * 1024;  // largest bitmap row a copy CTA stages

// After the hints: the follower plans, kPlanSlices slices of tokens [R, K], device rows
// [R, K] and counts [R] (int32 each). A plain resolve records its plan in slice 0; verify
// step q of a speculative batch records its own in slice q.
constexpr int kPlanSlices = HS_MAX_SPEC_QUERIES;
inline size_t plan_bytes(int64_t max_requests, int64_t top_k) {
  return (size_t)(((max_requests * top_k * 8 + max_requests * 4) + 255) & ~(int64_t)255);
}

// After the plans: their host-ordered copies (OrderArgs). A gather that takes the misses in
// host-address order, so that neighbouring rows share a 2 MB host region, reuses the GPU's
// translation of each region for several rows; in the order the resolve found them, misses
// spread over several large pools ran at about half the link rate. Layout (int32): per plan
// entry its host row [R, K]; per plan slice its pairs' host rows and device rows [R * K]
// each; the region counters and cursors [kOrderRegions + 1] each; per plan slice its pair
// count; the count kernel's CTA ticket.
constexpr int32_t kOrderRegions = 16384;
constexpr int64_t kOrderRegionBytes = 2 << 20;
inline size_t order_bytes(int64_t max_requests, int64_t top_k) {
  const int64_t rk = max_requests * top_k;
  return (size_t)((((rk * (1 + 2 * kPlanSlices) + 2 * (int64_t)(kOrderRegions + 1) + kPlanSlices + 1) * 4) + 255) &
                  ~(int64_t)255);
}

// The geometry and pools table of one layer group, shared by hs_create and
// hs_resolve_noalloc: validates the configuration, the row counts and the pools (host pools
// pinned and mapped, device pools on `dev`), derives the hash, sort and host-region sizes
// and the copy width, and fits the resolve kernel to the device (resolve_prepare).
// with_hints: the caller's workspace holds the residency bitmap. Returns HS_OK,
// HS_ERR_INVALID_ARG, HS_ERR_INVALID_CONFIG or HS_ERR_CUDA.
hs_status make_geometry(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                        int64_t host_rows, int64_t device_rows, bool with_hints, int dev, Geometry* g,
                        Pools* pools);

// Dynamic shared memory of one resolve-kernel CTA for geometry g.
size_t resolve_smem_bytes(const Geometry& g);
// Fit the resolve CTA's tables to the device's shared memory (sets g.dbl_smem, and for the
// largest top_k a half-full top-k hash), choose the copy CTAs per request (g.copy_ctas /
// g.copy_cap / g.bits_smem from the shared memory, SM count and max_requests) and raise the
// kernel's dynamic shared-memory limit. cudaErrorInvalidValue: g does not fit the device.
cudaError_t resolve_prepare(Geometry& g, int32_t max_requests);
cudaError_t launch_resolve(const Geometry& g, const Pools* pools, const ResolveArgs& a, int32_t num_requests,
                           uint32_t* err_word, cudaStream_t stream);
cudaError_t launch_backup(const Geometry& g, const Pools* pools, const BackupArgs& a, int32_t num_requests,
                          uint32_t* err_word, cudaStream_t stream);
cudaError_t launch_gather(const Geometry& g, const Pools* pools, const GatherArgs& a, int32_t num_requests,
                          uint32_t* err_word, cudaStream_t stream);
// Two launches: count the plan's misses per host region (the last CTA turns the counts into
// region offsets), then place each miss's (host row, device row) pair in its region.
cudaError_t launch_order(const Geometry& g, const OrderArgs& a, int32_t num_requests, uint32_t* err_word,
                         cudaStream_t stream);
// Pair-gather CTAs that fit one SM at once, for the copy width `vec`.
int gather_pairs_ctas_per_sm(int vec);
// Copy the ordered pairs' rows for layers [first_layer, first_layer + num_layers).
cudaError_t launch_gather_pairs(const Geometry& g, const Pools* pools, const OrderArgs& a, int32_t num_requests,
                                int32_t first_layer, int32_t num_layers, cudaStream_t stream);
size_t sparse_mla_smem_bytes();
// Kernel launches launch_sparse_mla makes for this request count and split count on the
// current device (1: one split, or two merged inside the kernel; 2: with the merge kernel).
int sparse_mla_launches(int32_t num_requests, int splits);
cudaError_t launch_sparse_mla(const SparseMlaArgs& a, int32_t num_requests, float* part_o, float* part_lse,
                              uint32_t* err, cudaStream_t stream);
cudaError_t launch_invalidate_tokens(const Geometry& g, const InvalidateArgs& a, int32_t num_requests,
                                     uint32_t* err_word, cudaStream_t stream);
cudaError_t launch_invalidate_host_rows(const Geometry& g, const InvalidateRowsArgs& a, int32_t num_requests,
                                        uint32_t* err_word, cudaStream_t stream);

}  // namespace hs
