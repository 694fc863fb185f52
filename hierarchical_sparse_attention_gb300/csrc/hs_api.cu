// C ABI of libhs (declared in include/hs.h): host-side validation, pool binding and
// the stream-ordered launches. Nothing here allocates device or pinned memory or
// synchronises on the hot path (hs_resolve / hs_backup).
#include <sys/syscall.h>
#include <unistd.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "hs_internal.h"

struct hs_handle {
  hs_config cfg;
  hs::Geometry g;
  const hs::Pools* pools;  // pools table inside the caller's workspace
  uint32_t* err_word;      // error word inside the caller's workspace
  uint32_t* hint;          // residency bitmap inside the caller's workspace
  int32_t* plan_tok;       // follower plan inside the caller's workspace: tokens [R, K],
  int32_t* plan_dst;       //   device rows [R, K],
  int32_t* plan_cnt;       //   counts [R] (slice 0; verify step q of a batch uses slice q)
  size_t plan_slice;       // int32 elements from one plan slice to the next
  hs::OrderArgs order;     // the plans' misses in host-region order (slice 0's pairs; order_slice)
  // What the last resolve left for hs_gather, as the calls were issued (stream order is call
  // order for calls on one stream, and a graph replays its calls in capture order).
  enum { kNoPlan, kPlan, kPairs, kSpec } plan_state;
  int32_t plan_requests;   // num_requests of that resolve
  int32_t spec_queries;    // verify steps of the last speculative batch (its plans: slices 0..Q-1)
  bool spec_ordered;       // that batch's plans were also grouped by host region
  int device;
};

namespace {

constexpr int kNodeMaskWords = 16;  // host memory nodes 0..1023

bool config_ok(const hs_config* c) {
  if (!c) return false;
  if (c->max_requests < 1 || c->top_k < 1 || c->top_k > HS_MAX_TOP_K) return false;
  if (c->hot_slots < c->top_k || c->hot_slots > HS_MAX_HOT_SLOTS) return false;
  if (c->row_bytes < 1 || c->num_layers < 1 || c->num_layers > HS_MAX_LAYERS) return false;
  if (c->max_context < 1 || c->page_size < 0 || c->max_pages < 0) return false;
  if (c->page_size > 0 &&
      (int64_t)c->max_pages * c->page_size < (int64_t)c->max_context)
    return false;
  if (c->host_row_stride != 0 && c->host_row_stride < c->row_bytes) return false;
  return true;
}

int ceil_log2(int64_t x) {
  int b = 0;
  while (((int64_t)1 << b) < x) ++b;
  return b;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The host-ordered arrays of plan slice q (the plain plan is slice 0).
hs::OrderArgs order_slice(const hs_handle* h, int32_t q, const int32_t* host_cache_locs) {
  hs::OrderArgs oa = h->order;
  const size_t RK = (size_t)h->cfg.max_requests * (size_t)h->cfg.top_k;
  oa.host_cache_locs = host_cache_locs;
  oa.plan_tok = h->plan_tok + q * h->plan_slice;
  oa.plan_dst = h->plan_dst + q * h->plan_slice;
  oa.plan_cnt = h->plan_cnt + q * h->plan_slice;
  oa.pair_src = h->order.pair_src + 2 * (size_t)q * RK;
  oa.pair_dst = h->order.pair_dst + 2 * (size_t)q * RK;
  oa.n_pairs = h->order.n_pairs + q;
  return oa;
}

}  // namespace

namespace hs {

hs_status make_geometry(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                        int64_t host_rows, int64_t device_rows, bool with_hints, int dev, Geometry* out,
                        Pools* pools_out) {
  if (!cfg || !host_pools || !device_pools || !out || !pools_out) return HS_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return HS_ERR_INVALID_CONFIG;
  // Row tables are int32: every row index must fit.
  if (host_rows < 1 || device_rows < 1 || host_rows > INT32_MAX || device_rows > INT32_MAX)
    return HS_ERR_INVALID_ARG;
  Geometry g{};
  g.K = cfg->top_k;
  g.H = cfg->hot_slots;
  g.B = cfg->row_bytes;
  g.L = cfg->num_layers;
  g.page_size = cfg->page_size;
  g.max_context = cfg->max_context;
  g.max_pages = cfg->max_pages;
  g.bit_words = with_hints ? hint_words(cfg->max_context) : 0;
  g.hash_bits = ceil_log2(4 * (int64_t)cfg->top_k);  // top-k hash at most a quarter full
  if (g.hash_bits < 5) g.hash_bits = 5;
  g.sort_cap = 1 << ceil_log2(cfg->top_k);
  if (g.hash_bits < ceil_log2(cfg->top_k) + 1) g.hash_bits = ceil_log2(cfg->top_k) + 1;  // room for the aliases
  g.host_rows = host_rows;
  g.device_rows = device_rows;
  g.host_stride = cfg->host_row_stride > 0 ? cfg->host_row_stride : cfg->row_bytes;
  // host regions of at most kOrderRegionBytes of host addresses (at least one row), coarser
  // for pools that would need more than kOrderRegions of them
  g.order_shift = 0;
  while (((int64_t)2 << g.order_shift) * g.host_stride <= kOrderRegionBytes) ++g.order_shift;
  while (((host_rows - 1) >> g.order_shift) + 1 > kOrderRegions) ++g.order_shift;
  g.order_regions = (int32_t)(((host_rows - 1) >> g.order_shift) + 1);

  Pools pools{};
  bool a16 = (g.B % 16) == 0 && (g.host_stride % 16) == 0, a4 = (g.B % 4) == 0 && (g.host_stride % 4) == 0;
  for (int l = 0; l < g.L; ++l) {
    if (!host_pools[l] || !device_pools[l]) return HS_ERR_INVALID_ARG;
    cudaPointerAttributes ha{}, da{};
    if (cudaPointerGetAttributes(&ha, host_pools[l]) != cudaSuccess) {
      cudaGetLastError();
      return HS_ERR_INVALID_ARG;
    }
    if (ha.type != cudaMemoryTypeHost || !ha.devicePointer) return HS_ERR_INVALID_ARG;  // not pinned+mapped
    if (cudaPointerGetAttributes(&da, device_pools[l]) != cudaSuccess) {
      cudaGetLastError();
      return HS_ERR_INVALID_ARG;
    }
    if ((da.type != cudaMemoryTypeDevice && da.type != cudaMemoryTypeManaged) || da.device != dev)
      return HS_ERR_INVALID_ARG;
    pools.host[l] = static_cast<const uint8_t*>(ha.devicePointer);
    pools.dev[l] = static_cast<uint8_t*>(device_pools[l]);
    a16 = a16 && aligned(pools.host[l], 16) && aligned(pools.dev[l], 16);
    a4 = a4 && aligned(pools.host[l], 4) && aligned(pools.dev[l], 4);
  }
  g.vec = a16 ? 16 : (a4 ? 4 : 1);
  // "page first": layer l's rows start l * B into one pool whose rows are L * B apart
  g.host_interleaved = g.L > 1 && g.host_stride == (int64_t)g.L * g.B;
  for (int l = 1; l < g.L && g.host_interleaved; ++l)
    g.host_interleaved = pools.host[l] == pools.host[0] + (size_t)l * g.B;

  if (const cudaError_t e = resolve_prepare(g, cfg->max_requests); e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? HS_ERR_INVALID_CONFIG : HS_ERR_CUDA;
  }
  g.gather_ctas_per_sm = gather_pairs_ctas_per_sm(g.vec);
  *out = g;
  *pools_out = pools;
  return HS_OK;
}

}  // namespace hs

extern "C" {

size_t hs_workspace_bytes(const hs_config* cfg) {
  return config_ok(cfg) ? hs::kWorkspaceBytes + hs::hint_bytes(cfg->max_requests, cfg->max_context) +
                              hs::kPlanSlices * hs::plan_bytes(cfg->max_requests, cfg->top_k) +
                              hs::order_bytes(cfg->max_requests, cfg->top_k)
                        : 0;
}

hs_status hs_create(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                    int64_t host_rows, int64_t device_rows, void* workspace, hs_handle** out) {
  if (!out) return HS_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !host_pools || !device_pools || !workspace) return HS_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return HS_ERR_INVALID_CONFIG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  hs::Geometry g{};
  hs::Pools pools{};
  if (const hs_status st = hs::make_geometry(cfg, host_pools, device_pools, host_rows, device_rows, true, dev, &g,
                                             &pools);
      st != HS_OK)
    return st;

  cudaPointerAttributes wa{};
  if (cudaPointerGetAttributes(&wa, workspace) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_INVALID_ARG;
  }
  if ((wa.type != cudaMemoryTypeDevice && wa.type != cudaMemoryTypeManaged) || wa.device != dev ||
      !aligned(workspace, 16))
    return HS_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (cudaMemset(ws, 0, hs::kWorkspaceBytes) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemset(ws + hs::kWorkspaceBytes, 0, hs::hint_bytes(cfg->max_requests, cfg->max_context)) !=
      cudaSuccess)
    return HS_ERR_CUDA;  // no token is known to be resident yet
  uint8_t* plan = ws + hs::kWorkspaceBytes + hs::hint_bytes(cfg->max_requests, cfg->max_context);
  if (cudaMemset(plan, 0, hs::kPlanSlices * hs::plan_bytes(cfg->max_requests, cfg->top_k)) != cudaSuccess)
    return HS_ERR_CUDA;  // no plan yet: a gather before the first resolve copies nothing
  uint8_t* order = plan + hs::kPlanSlices * hs::plan_bytes(cfg->max_requests, cfg->top_k);
  if (cudaMemset(order, 0, hs::order_bytes(cfg->max_requests, cfg->top_k)) != cudaSuccess)
    return HS_ERR_CUDA;  // region counts and the count kernel's ticket start at zero
  if (cudaMemcpy(ws + hs::kPoolsOffset, &pools, sizeof(pools), cudaMemcpyHostToDevice) != cudaSuccess)
    return HS_ERR_CUDA;

  hs_handle* h = static_cast<hs_handle*>(std::calloc(1, sizeof(hs_handle)));
  if (!h) return HS_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->g = g;
  h->pools = reinterpret_cast<const hs::Pools*>(ws + hs::kPoolsOffset);
  h->err_word = reinterpret_cast<uint32_t*>(ws + hs::kErrOffset);
  h->hint = reinterpret_cast<uint32_t*>(ws + hs::kWorkspaceBytes);
  const size_t RK = (size_t)cfg->max_requests * (size_t)cfg->top_k;
  h->plan_tok = reinterpret_cast<int32_t*>(plan);
  h->plan_dst = h->plan_tok + RK;
  h->plan_cnt = h->plan_dst + RK;
  h->plan_slice = hs::plan_bytes(cfg->max_requests, cfg->top_k) / sizeof(int32_t);
  hs::OrderArgs& oa = h->order;  // the region laid out as hs::order_bytes counts it
  oa = hs::OrderArgs{};
  oa.plan_tok = h->plan_tok;
  oa.plan_dst = h->plan_dst;
  oa.plan_cnt = h->plan_cnt;
  oa.miss_src = reinterpret_cast<int32_t*>(order);
  oa.pair_src = oa.miss_src + RK;                    // slice q: + 2 q RK
  oa.pair_dst = oa.pair_src + RK;                    // slice q: + 2 q RK
  oa.counts = oa.pair_src + 2 * hs::kPlanSlices * RK;
  oa.cursors = oa.counts + (hs::kOrderRegions + 1);
  oa.n_pairs = oa.cursors + (hs::kOrderRegions + 1);  // slice q: + q
  oa.ticket = reinterpret_cast<uint32_t*>(oa.n_pairs + hs::kPlanSlices);
  oa.capacity = (int64_t)RK;
  h->plan_state = hs_handle::kNoPlan;
  h->device = dev;
  *out = h;
  return HS_OK;
}

hs_status hs_resolve_layers(hs_handle* h, int32_t num_requests, const int32_t* top_k_tokens,
                            const int32_t* seq_lens, const int32_t* host_cache_locs,
                            const int32_t* device_buffer_locs, int32_t* device_buffer_tokens, int32_t* lru_slots,
                            int32_t* lru_clock, const int32_t* resident_pages, int32_t* out_rows,
                            int32_t* miss_counts, int32_t copy_layers, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (copy_layers < 0 || copy_layers > h->cfg.num_layers) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!top_k_tokens || !seq_lens || !host_cache_locs || !device_buffer_locs || !device_buffer_tokens ||
      !lru_slots || !lru_clock || !out_rows)
    return HS_ERR_INVALID_ARG;
  if (resident_pages && h->cfg.page_size <= 0) return HS_ERR_INVALID_ARG;
  // Without copy CTAs (more requests than the SMs give clusters to), each resolve CTA would
  // copy its own miss rows, in miss order, once its exact pass is done. The resolve then
  // copies nothing; its plan is put in host-region order and one gather over a wide grid
  // copies every layer's rows, in stream order, with the same results. The ordered plan is
  // also built whenever follower layers are left for hs_gather.
  const bool gather_after = h->g.copy_ctas == 0 && copy_layers > 0;
  const bool order = h->g.copy_ctas == 0 || copy_layers < h->cfg.num_layers;
  hs::ResolveArgs a{h->hint,   top_k_tokens, seq_lens,   host_cache_locs, device_buffer_locs, device_buffer_tokens,
                    lru_slots, lru_clock,    resident_pages, out_rows,   miss_counts,        gather_after ? 0 : copy_layers,
                    h->plan_tok, h->plan_dst, h->plan_cnt, -1, 1};
  if (hs::launch_resolve(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  h->plan_state = order ? hs_handle::kPairs : hs_handle::kPlan;
  h->plan_requests = num_requests;
  if (order) {
    const hs::OrderArgs oa = order_slice(h, 0, host_cache_locs);
    if (hs::launch_order(h->g, oa, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
      return HS_ERR_CUDA;
    if (gather_after &&
        hs::launch_gather_pairs(h->g, h->pools, oa, num_requests, 0, copy_layers, (cudaStream_t)stream) != cudaSuccess)
      return HS_ERR_CUDA;
  }
  return HS_OK;
}

hs_status hs_resolve(hs_handle* h, int32_t num_requests, const int32_t* top_k_tokens,
                     const int32_t* seq_lens, const int32_t* host_cache_locs,
                     const int32_t* device_buffer_locs, int32_t* device_buffer_tokens, int32_t* lru_slots,
                     int32_t* lru_clock, const int32_t* resident_pages, int32_t* out_rows,
                     int32_t* miss_counts, hs_stream_t stream) {
  if (!h) return HS_ERR_INVALID_ARG;
  return hs_resolve_layers(h, num_requests, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs,
                           device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows, miss_counts,
                           h->cfg.num_layers, stream);
}

hs_status hs_resolve_spec_layers(hs_handle* h, int32_t num_requests, int32_t num_queries,
                                 const int32_t* top_k_tokens, const int32_t* committed_lens,
                                 const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                                 int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                                 const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                                 int32_t copy_layers, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (num_queries < 1 || num_queries > HS_MAX_SPEC_QUERIES) return HS_ERR_INVALID_ARG;
  if (copy_layers < 0 || copy_layers > h->cfg.num_layers) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!top_k_tokens || !committed_lens || !host_cache_locs || !device_buffer_locs || !device_buffer_tokens ||
      !lru_slots || !lru_clock || !out_rows)
    return HS_ERR_INVALID_ARG;
  if (resident_pages && h->cfg.page_size <= 0) return HS_ERR_INVALID_ARG;
  const size_t RK = (size_t)num_requests * (size_t)h->cfg.top_k;
  // Without copy CTAs, each verify step is resolved without copies, its plan is grouped by
  // host region and the leader layers' rows are gathered, as for a plain step; each step's
  // plan is also grouped whenever follower layers are left for hs_gather_spec.
  const bool gather_after = h->g.copy_ctas == 0 && copy_layers > 0;
  const bool order = h->g.copy_ctas == 0 || copy_layers < h->cfg.num_layers;
  h->plan_state = hs_handle::kSpec;
  h->plan_requests = num_requests;
  h->spec_queries = num_queries;
  h->spec_ordered = order;
  // One launch runs the verify steps in order over the shared state (each cluster loops over
  // its request's steps); step q records its miss plan in plan slice q.
  hs::ResolveArgs a{h->hint,   top_k_tokens, committed_lens, host_cache_locs, device_buffer_locs,
                    device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows, miss_counts,
                    gather_after ? 0 : copy_layers, h->plan_tok, h->plan_dst, h->plan_cnt, 0, num_queries};
  a.spec_steps = num_queries;
  a.step_r = num_requests;
  a.step_rk = (int64_t)RK;
  a.step_plan = (int64_t)h->plan_slice;
  if (hs::launch_resolve(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  // Without copy CTAs, or with follower layers left, each step's plan is then grouped by host
  // region (and its leader rows gathered), step by step in step order: the rows a later step
  // places in a slot an earlier step filled are the last written, as in the steps themselves.
  if (order)
    for (int32_t q = 0; q < num_queries; ++q) {
      const hs::OrderArgs oa = order_slice(h, q, host_cache_locs);
      if (hs::launch_order(h->g, oa, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
        return HS_ERR_CUDA;
      if (gather_after &&
          hs::launch_gather_pairs(h->g, h->pools, oa, num_requests, 0, copy_layers, (cudaStream_t)stream) !=
              cudaSuccess)
        return HS_ERR_CUDA;
    }
  return HS_OK;
}

hs_status hs_resolve_spec(hs_handle* h, int32_t num_requests, int32_t num_queries, const int32_t* top_k_tokens,
                          const int32_t* committed_lens, const int32_t* host_cache_locs,
                          const int32_t* device_buffer_locs, int32_t* device_buffer_tokens, int32_t* lru_slots,
                          int32_t* lru_clock, const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                          hs_stream_t stream) {
  if (!h) return HS_ERR_INVALID_ARG;
  return hs_resolve_spec_layers(h, num_requests, num_queries, top_k_tokens, committed_lens, host_cache_locs,
                                device_buffer_locs, device_buffer_tokens, lru_slots, lru_clock, resident_pages,
                                out_rows, miss_counts, h->cfg.num_layers, stream);
}

hs_status hs_gather_spec(hs_handle* h, int32_t num_requests, const int32_t* host_cache_locs, int32_t query,
                         int32_t first_layer, int32_t num_layers, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (first_layer < 0 || num_layers < 0 || first_layer + num_layers > h->cfg.num_layers) return HS_ERR_INVALID_ARG;
  if (h->plan_state != hs_handle::kSpec || query < 0 || query >= h->spec_queries) return HS_ERR_INVALID_ARG;
  if (num_requests != h->plan_requests) return HS_ERR_INVALID_ARG;
  if (num_requests == 0 || num_layers == 0) return HS_OK;
  if (!host_cache_locs) return HS_ERR_INVALID_ARG;
  if (h->spec_ordered) {
    if (hs::launch_gather_pairs(h->g, h->pools, order_slice(h, query, host_cache_locs), num_requests, first_layer,
                                num_layers, (cudaStream_t)stream) != cudaSuccess)
      return HS_ERR_CUDA;
    return HS_OK;
  }
  hs::GatherArgs a{host_cache_locs, h->plan_tok + query * h->plan_slice, h->plan_dst + query * h->plan_slice,
                   h->plan_cnt + query * h->plan_slice, first_layer, num_layers};
  if (hs::launch_gather(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_backup_spec(hs_handle* h, int32_t num_requests, int32_t num_queries, const int32_t* committed_lens,
                         const int32_t* accepted, const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                         const int32_t* resident_pages, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (num_queries < 1 || num_queries > HS_MAX_SPEC_QUERIES) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!committed_lens || !accepted || !host_cache_locs || !device_buffer_locs) return HS_ERR_INVALID_ARG;
  if (resident_pages && h->cfg.page_size <= 0) return HS_ERR_INVALID_ARG;
  hs::BackupArgs a{committed_lens, host_cache_locs, device_buffer_locs, resident_pages, accepted, num_queries};
  if (hs::launch_backup(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_gather(hs_handle* h, int32_t num_requests, const int32_t* host_cache_locs, int32_t first_layer,
                    int32_t num_layers, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (first_layer < 0 || num_layers < 0 || first_layer + num_layers > h->cfg.num_layers) return HS_ERR_INVALID_ARG;
  if (num_requests == 0 || num_layers == 0) return HS_OK;
  if (!host_cache_locs) return HS_ERR_INVALID_ARG;
  if (h->plan_state == hs_handle::kSpec) return HS_ERR_INVALID_ARG;  // a batch's plans: hs_gather_spec
  if (h->plan_state == hs_handle::kPairs) {
    // the ordered plan covers the resolve's requests, all of them
    if (num_requests != h->plan_requests) return HS_ERR_INVALID_ARG;
    if (hs::launch_gather_pairs(h->g, h->pools, h->order, num_requests, first_layer, num_layers,
                                (cudaStream_t)stream) != cudaSuccess)
      return HS_ERR_CUDA;
    return HS_OK;
  }
  hs::GatherArgs a{host_cache_locs, h->plan_tok, h->plan_dst, h->plan_cnt, first_layer, num_layers};
  if (hs::launch_gather(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_backup(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                    const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                    const int32_t* resident_pages, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!seq_lens || !host_cache_locs || !device_buffer_locs) return HS_ERR_INVALID_ARG;
  if (resident_pages && h->cfg.page_size <= 0) return HS_ERR_INVALID_ARG;
  hs::BackupArgs a{seq_lens, host_cache_locs, device_buffer_locs, resident_pages, nullptr, 1};
  if (hs::launch_backup(h->g, h->pools, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_invalidate_tokens(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                               const int32_t* token_offsets, const int32_t* tokens, int32_t* device_buffer_tokens,
                               int32_t* lru_slots, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!seq_lens || !token_offsets || !tokens || !device_buffer_tokens || !lru_slots) return HS_ERR_INVALID_ARG;
  hs::InvalidateArgs a{h->hint, seq_lens, token_offsets, tokens, device_buffer_tokens, lru_slots};
  if (hs::launch_invalidate_tokens(h->g, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_invalidate_host_rows(hs_handle* h, int32_t num_requests, const int32_t* seq_lens,
                                  const int32_t* host_cache_locs, const int32_t* rows, int32_t n,
                                  int32_t* device_buffer_tokens, int32_t* lru_slots, hs_stream_t stream) {
  if (!h || num_requests < 0 || num_requests > h->cfg.max_requests || n < 0) return HS_ERR_INVALID_ARG;
  if (num_requests == 0 || n == 0) return HS_OK;
  if (!seq_lens || !host_cache_locs || !rows || !device_buffer_tokens || !lru_slots) return HS_ERR_INVALID_ARG;
  hs::InvalidateRowsArgs a{h->hint, seq_lens, host_cache_locs, rows, n, device_buffer_tokens, lru_slots};
  if (hs::launch_invalidate_host_rows(h->g, a, num_requests, h->err_word, (cudaStream_t)stream) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

size_t hs_sparse_mla_workspace_bytes(int32_t num_requests, int32_t num_heads, int32_t splits) {
  if (num_requests < 1 || num_heads < 1 || num_heads > 128 || splits < 1 || splits > HS_MAX_MLA_SPLITS) return 0;
  if (splits == 1) return 0;
  const size_t rows = (size_t)splits * num_requests * num_heads;
  return rows * 512 * sizeof(float) + rows * sizeof(float);
}

int32_t hs_sparse_mla_launches(int32_t num_requests, int32_t num_heads, int32_t splits) {
  if (num_requests < 1 || num_heads < 1 || num_heads > 128 || splits < 1 || splits > HS_MAX_MLA_SPLITS) return 0;
  if (splits == 1) return 1;  // no device query needed
  return hs::sparse_mla_launches(num_requests, splits);
}

hs_status hs_sparse_mla_decode(int32_t num_requests, int32_t num_heads, int32_t top_k, int32_t splits,
                               const uint16_t* q, const uint8_t* kv_pool, int64_t pool_rows,
                               const int32_t* out_rows, float sm_scale, float* o, float* lse, void* workspace,
                               size_t workspace_bytes, uint32_t* error_flags, hs_stream_t stream) {
  if (num_requests < 0 || num_heads < 1 || num_heads > 128 || top_k < 1 || top_k > HS_MAX_TOP_K || splits < 1 ||
      splits > HS_MAX_MLA_SPLITS || pool_rows < 1)
    return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!q || !kv_pool || !out_rows || !o || !lse || !error_flags) return HS_ERR_INVALID_ARG;
  if (((uintptr_t)q % 16) || ((uintptr_t)kv_pool % 16) || ((uintptr_t)o % 16)) return HS_ERR_INVALID_ARG;
  const size_t need = hs_sparse_mla_workspace_bytes(num_requests, num_heads, splits);
  if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace % 16))) return HS_ERR_INVALID_ARG;
  const size_t rows = (size_t)splits * num_requests * num_heads;
  float* part_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  float* part_lse = splits > 1 ? part_o + rows * 512 : nullptr;
  hs::SparseMlaArgs a{q, kv_pool, pool_rows, out_rows, top_k, num_heads, splits, sm_scale, o, lse};
  if (hs::launch_sparse_mla(a, num_requests, part_o, part_lse, error_flags, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

hs_status hs_reset_hints(hs_handle* h, hs_stream_t stream) {
  if (!h) return HS_ERR_INVALID_ARG;
  if (cudaMemsetAsync(h->hint, 0, hs::hint_bytes(h->cfg.max_requests, h->cfg.max_context),
                      (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

hs_status hs_launch_shape(const hs_handle* h, int32_t* copy_ctas, int32_t* resolve_launches) {
  if (!h) return HS_ERR_INVALID_ARG;
  if (copy_ctas) *copy_ctas = h->g.copy_ctas;
  if (resolve_launches) *resolve_launches = h->g.copy_ctas == 0 ? 4 : 1;
  return HS_OK;
}

hs_status hs_get_error(hs_handle* h, uint32_t* flags, int clear) {
  if (!h || !flags) return HS_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemcpy(flags, h->err_word, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return HS_ERR_CUDA;
  if (clear && cudaMemset(h->err_word, 0, sizeof(uint32_t)) != cudaSuccess) return HS_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  return *flags ? HS_ERR_DEVICE_FLAGGED : HS_OK;
}

hs_status hs_destroy(hs_handle* h) {
  std::free(h);
  return HS_OK;
}

const char* hs_status_str(hs_status s) {
  switch (s) {
    case HS_OK: return "ok";
    case HS_ERR_INVALID_ARG: return "invalid argument";
    case HS_ERR_INVALID_CONFIG: return "invalid configuration";
    case HS_ERR_CUDA: return "CUDA error";
    case HS_ERR_DEVICE_FLAGGED: return "device flagged anomalies in the inputs";
    case HS_ERR_TIMEOUT: return "timed out";
  }
  return "unknown status";
}

hs_status hs_host_register(void* ptr, size_t bytes, void** device_ptr) {
  if (!ptr || !bytes || !device_ptr) return HS_ERR_INVALID_ARG;
  *device_ptr = nullptr;
  if (cudaHostRegister(ptr, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  if (cudaHostGetDevicePointer(device_ptr, ptr, 0) != cudaSuccess) {
    cudaGetLastError();
    cudaHostUnregister(ptr);
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

hs_status hs_host_numa_node(int32_t device, int32_t* node) {
  if (!node) return HS_ERR_INVALID_ARG;
  *node = -1;
  int v = -1;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrHostNumaId, device) == cudaSuccess && v >= 0) {
    *node = v;
    return HS_OK;
  }
  cudaGetLastError();
  char bus[32] = {};
  if (cudaDeviceGetPCIBusId(bus, (int)sizeof(bus), device) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  for (char* c = bus; *c; ++c)
    if (*c >= 'A' && *c <= 'F') *c = (char)(*c - 'A' + 'a');  // sysfs spells the address in lower case
  char path[96];
  std::snprintf(path, sizeof(path), "/sys/bus/pci/devices/%s/numa_node", bus);
  if (FILE* f = std::fopen(path, "r")) {
    int n = -1;
    if (std::fscanf(f, "%d", &n) == 1 && n >= 0) *node = n;
    std::fclose(f);
  }
  return HS_OK;
}

hs_status hs_host_bind_node(void* ptr, size_t bytes, int32_t node) {
  if (!ptr || !bytes || node < 0 || node >= 64 * kNodeMaskWords) return HS_ERR_INVALID_ARG;
  const uintptr_t page = (uintptr_t)sysconf(_SC_PAGESIZE);
  const uintptr_t lo = (uintptr_t)ptr & ~(page - 1);
  const uintptr_t hi = ((uintptr_t)ptr + bytes + page - 1) & ~(page - 1);
  unsigned long mask[kNodeMaskWords] = {};
  mask[node / 64] = 1ul << (node % 64);
  constexpr int kMpolPreferred = 1;  // <linux/mempolicy.h> MPOL_PREFERRED
  // the kernel reads maxnode - 1 bits of the mask
  if (syscall(SYS_mbind, (void*)lo, (unsigned long)(hi - lo), kMpolPreferred, mask,
              (unsigned long)(64 * kNodeMaskWords + 1), 0u) != 0)
    return HS_ERR_CUDA;
  return HS_OK;
}

hs_status hs_host_unregister(void* ptr) {
  if (!ptr) return HS_ERR_INVALID_ARG;
  if (cudaHostUnregister(ptr) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

}  // extern "C"
