// hs_resolve_noalloc: the resolve step for callers that cannot allocate device memory.
//
// hs_create needs a caller-allocated device workspace (the per-handle pools table that the
// kernel indexes by layer, and the sticky error word). Some callers have no way to make
// that allocation: code that runs where the device memory is all planned up front (a
// serving engine's fixed memory budget, a plugin inside another framework's allocator, a
// process that must not call cudaMalloc once decoding has started). This entry point
// keeps that scratch in a file-scope device array instead, so one call does everything
// with memory the caller already owns: no cudaMalloc, no cudaFree, no library allocation.
//
// The array is shared by every call in the process, on every device that loads the library
// (each device holds its own copy until the process exits), and it keeps the last call's
// contents. Each call rewrites the pools table and zeroes the error word before the kernel
// runs, so results never depend on an earlier call; but two calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on the array.
#include <mutex>

#include "hs_internal.h"

namespace {

// Scratch of one call: the error word at kErrOffset and the pools table at kPoolsOffset,
// the same layout as the workspace hs_create binds. kWorkspaceBytes = 256 bytes.
static __device__ __align__(256) unsigned char g_noalloc_scratch[hs::kWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_addr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// Device-side address of the scratch array for the current device. In host code the
// symbol names only a host-side stand-in, so the address is looked up once per device
// (with that device current) and cached.
hs_status scratch_for(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_addr[dev];
  return HS_OK;
}

int ceil_log2_i64(int64_t x) {
  int b = 0;
  while (((int64_t)1 << b) < x) ++b;
  return b;
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" {

hs_status hs_resolve_noalloc(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                             int64_t host_rows, int64_t device_rows, int32_t num_requests,
                             const int32_t* top_k_tokens, const int32_t* seq_lens, const int32_t* host_cache_locs,
                             const int32_t* device_buffer_locs, int32_t* device_buffer_tokens, int32_t* lru_slots,
                             int32_t* lru_clock, const int32_t* resident_pages, int32_t* out_rows,
                             int32_t* miss_counts, uint32_t* error_flags, hs_stream_t stream) {
  if (!cfg || !host_pools || !device_pools) return HS_ERR_INVALID_ARG;
  // Configuration limits are those of hs_create; the scratch array holds the pools table
  // of at most HS_NOALLOC_MAX_LAYERS layers, and anything larger is refused here.
  if (cfg->num_layers < 1 || cfg->num_layers > HS_NOALLOC_MAX_LAYERS) return HS_ERR_INVALID_CONFIG;
  if (cfg->max_requests < 1 || cfg->top_k < 1 || cfg->top_k > HS_MAX_TOP_K || cfg->hot_slots < cfg->top_k ||
      cfg->hot_slots > HS_MAX_HOT_SLOTS || cfg->row_bytes < 1 || cfg->max_context < 1 || cfg->page_size < 0 ||
      cfg->max_pages < 0 ||
      (cfg->page_size > 0 && (int64_t)cfg->max_pages * cfg->page_size < (int64_t)cfg->max_context))
    return HS_ERR_INVALID_CONFIG;
  if (host_rows < 1 || device_rows < 1 || host_rows > INT32_MAX || device_rows > INT32_MAX)
    return HS_ERR_INVALID_ARG;
  if (num_requests < 0 || num_requests > cfg->max_requests) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!top_k_tokens || !seq_lens || !host_cache_locs || !device_buffer_locs || !device_buffer_tokens ||
      !lru_slots || !lru_clock || !out_rows)
    return HS_ERR_INVALID_ARG;
  if (resident_pages && cfg->page_size <= 0) return HS_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  unsigned char* scratch = nullptr;
  const hs_status st = scratch_for(dev, &scratch);
  if (st != HS_OK) return st;

  hs::Geometry g{};
  g.K = cfg->top_k;
  g.H = cfg->hot_slots;
  g.B = cfg->row_bytes;
  g.L = cfg->num_layers;
  g.page_size = cfg->page_size;
  g.max_context = cfg->max_context;
  g.max_pages = cfg->max_pages;
  g.hash_bits = ceil_log2_i64(4 * (int64_t)cfg->top_k);  // top-k hash at most a quarter full
  if (g.hash_bits < 5) g.hash_bits = 5;
  g.sort_cap = 1 << ceil_log2_i64(cfg->top_k);
  if (g.hash_bits < ceil_log2_i64(cfg->top_k) + 1) g.hash_bits = ceil_log2_i64(cfg->top_k) + 1;
  g.host_rows = host_rows;
  g.device_rows = device_rows;

  hs::Pools pools{};
  bool a16 = (g.B % 16) == 0, a4 = (g.B % 4) == 0;
  for (int l = 0; l < g.L; ++l) {
    if (!host_pools[l] || !device_pools[l]) return HS_ERR_INVALID_ARG;
    cudaPointerAttributes ha{}, da{};
    if (cudaPointerGetAttributes(&ha, host_pools[l]) != cudaSuccess ||
        cudaPointerGetAttributes(&da, device_pools[l]) != cudaSuccess) {
      cudaGetLastError();
      return HS_ERR_INVALID_ARG;
    }
    if (ha.type != cudaMemoryTypeHost || !ha.devicePointer) return HS_ERR_INVALID_ARG;
    if ((da.type != cudaMemoryTypeDevice && da.type != cudaMemoryTypeManaged) || da.device != dev)
      return HS_ERR_INVALID_ARG;
    pools.host[l] = static_cast<const uint8_t*>(ha.devicePointer);
    pools.dev[l] = static_cast<uint8_t*>(device_pools[l]);
    a16 = a16 && aligned_to(pools.host[l], 16) && aligned_to(pools.dev[l], 16);
    a4 = a4 && aligned_to(pools.host[l], 4) && aligned_to(pools.dev[l], 4);
  }
  g.vec = a16 ? 16 : (a4 ? 4 : 1);
  if (hs::resolve_prepare(g, cfg->max_requests) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_INVALID_CONFIG;  // shared memory does not fit this device
  }

  cudaStream_t s = (cudaStream_t)stream;
  // The pools table comes from a stack copy: cudaMemcpyAsync from pageable memory has
  // taken the bytes by the time it returns. The error word must start each call at zero.
  if (cudaMemcpyAsync(scratch + hs::kPoolsOffset, &pools, sizeof(pools), cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(scratch + hs::kErrOffset, 0, sizeof(uint32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  // no hint table here (misses start their transfer after the exact probe) and no plan
  hs::ResolveArgs a{nullptr,   top_k_tokens, seq_lens,       host_cache_locs, device_buffer_locs, device_buffer_tokens,
                    lru_slots, lru_clock,    resident_pages, out_rows,        miss_counts,        g.L,
                    nullptr,   nullptr,      nullptr,        -1,              1};  // every layer; no plan
  uint32_t* err_word = reinterpret_cast<uint32_t*>(scratch + hs::kErrOffset);
  if (hs::launch_resolve(g, reinterpret_cast<const hs::Pools*>(scratch + hs::kPoolsOffset), a, num_requests,
                         err_word, s) != cudaSuccess)
    return HS_ERR_CUDA;
  if (error_flags &&
      cudaMemcpyAsync(error_flags, err_word, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

}  // extern "C"
