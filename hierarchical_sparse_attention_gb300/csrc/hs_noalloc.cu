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
#include <cstring>
#include <mutex>

#include "hs_internal.h"

namespace {

// Scratch of one call: the error word at kErrOffset and the pools table at kPoolsOffset,
// the same layout as the workspace hs_create binds. kWorkspaceBytes = 256 bytes.
static __device__ __align__(256) unsigned char g_noalloc_scratch[hs::kWorkspaceBytes];

// Writes one call's pools table into the scratch array and clears its error word, in stream
// order before the resolve. A kernel argument carries the table, so nothing is copied from
// host memory (a copy from a stack variable would be pageable and could block the host).
__global__ void noalloc_setup_kernel(const hs::Pools pools, unsigned char* scratch) {
  *reinterpret_cast<hs::Pools*>(scratch + hs::kPoolsOffset) = pools;
  *reinterpret_cast<uint32_t*>(scratch + hs::kErrOffset) = 0u;
}

constexpr int kMaxDevices = 64;

// Per-device set-up, kept so that later calls with the same configuration and pools skip
// the host-side checks and kernel fitting (pointer queries, function attributes).
struct DeviceSetup {
  unsigned char* scratch;  // device address of g_noalloc_scratch on this device
  bool valid;              // cfg / pools below describe geom / pools_table
  hs_config cfg;
  const void* host_pools[hs::kMaxLayers];
  const void* device_pools[hs::kMaxLayers];
  int64_t host_rows, device_rows;
  hs::Geometry geom;
  hs::Pools pools_table;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices] = {};

bool same_call(const DeviceSetup& s, const hs_config* cfg, void* const* host_pools, void* const* device_pools,
               int64_t host_rows, int64_t device_rows) {
  if (!s.valid || std::memcmp(&s.cfg, cfg, sizeof(hs_config)) != 0 || s.host_rows != host_rows ||
      s.device_rows != device_rows)
    return false;
  for (int l = 0; l < cfg->num_layers; ++l)
    if (s.host_pools[l] != host_pools[l] || s.device_pools[l] != device_pools[l]) return false;
  return true;
}

// The device address of the scratch array and the geometry for this call, on device `dev`
// (current). In host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device, with that device current, and cached.
hs_status setup_for(int dev, const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                    int64_t host_rows, int64_t device_rows, unsigned char** scratch, hs::Geometry* g,
                    hs::Pools* pools) {
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.scratch) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    s.scratch = static_cast<unsigned char*>(p);
  }
  if (!same_call(s, cfg, host_pools, device_pools, host_rows, device_rows)) {
    s.valid = false;
    // no hint table here (misses start their transfer after the exact probe)
    const hs_status st =
        hs::make_geometry(cfg, host_pools, device_pools, host_rows, device_rows, false, dev, &s.geom, &s.pools_table);
    if (st != HS_OK) return st;
    s.cfg = *cfg;
    for (int l = 0; l < cfg->num_layers; ++l) {
      s.host_pools[l] = host_pools[l];
      s.device_pools[l] = device_pools[l];
    }
    s.host_rows = host_rows;
    s.device_rows = device_rows;
    s.valid = true;
  }
  *scratch = s.scratch;
  *g = s.geom;
  *pools = s.pools_table;
  return HS_OK;
}

}  // namespace

extern "C" {

hs_status hs_resolve_noalloc(const hs_config* cfg, void* const* host_pools, void* const* device_pools,
                             int64_t host_rows, int64_t device_rows, int32_t num_requests,
                             const int32_t* top_k_tokens, const int32_t* seq_lens, const int32_t* host_cache_locs,
                             const int32_t* device_buffer_locs, int32_t* device_buffer_tokens, int32_t* lru_slots,
                             int32_t* lru_clock, const int32_t* resident_pages, int32_t* out_rows,
                             int32_t* miss_counts, uint32_t* error_flags, hs_stream_t stream) {
  if (!cfg || !host_pools || !device_pools) return HS_ERR_INVALID_ARG;
  // The scratch array holds the pools table of at most HS_NOALLOC_MAX_LAYERS layers; a
  // larger group is refused here. Every other limit is hs_create's (make_geometry).
  if (cfg->num_layers < 1 || cfg->num_layers > HS_NOALLOC_MAX_LAYERS) return HS_ERR_INVALID_CONFIG;
  if (num_requests < 0 || num_requests > cfg->max_requests) return HS_ERR_INVALID_ARG;
  if (num_requests == 0) return HS_OK;
  if (!top_k_tokens || !seq_lens || !host_cache_locs || !device_buffer_locs || !device_buffer_tokens ||
      !lru_slots || !lru_clock || !out_rows)
    return HS_ERR_INVALID_ARG;
  if (resident_pages && cfg->page_size <= 0) return HS_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  unsigned char* scratch = nullptr;
  hs::Geometry g{};
  hs::Pools pools{};
  if (const hs_status st = setup_for(dev, cfg, host_pools, device_pools, host_rows, device_rows, &scratch, &g, &pools);
      st != HS_OK)
    return st;

  cudaStream_t s = (cudaStream_t)stream;
  noalloc_setup_kernel<<<1, 1, 0, s>>>(pools, scratch);
  if (cudaGetLastError() != cudaSuccess) return HS_ERR_CUDA;
  // no hint table and no plan: every layer's rows are copied by the resolve kernel itself
  hs::ResolveArgs a{nullptr,   top_k_tokens, seq_lens,       host_cache_locs, device_buffer_locs, device_buffer_tokens,
                    lru_slots, lru_clock,    resident_pages, out_rows,        miss_counts,        g.L,
                    nullptr,   nullptr,      nullptr,        -1,              1};
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
