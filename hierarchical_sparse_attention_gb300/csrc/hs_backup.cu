// Eager backup: the newest token's KV row, device -> pinned host, one warp per
// (request, layer).
//
// Source: "HiSparse: moving the long-context decode capacity bottleneck from GPU memory to
// CPU memory", "Per decode step workflow", step 5 (after attention, the last token's KV is
// copied back from device to host so the host pool stays complete). The row sits in its
// resident page when that page is GPU-resident ("vLLM HiSparse local KV offload
// architecture", "Hot-row lookup and LRU"), in buffer slot seq_len-1 while the sequence
// fits the buffer, else in the reserved slot H ("How capacity is computed": the buffer
// carries an extra page for the new token).
#include "hs_internal.h"

namespace hs {
namespace {

__device__ __forceinline__ void copy_row(const Geometry& g, const Pools* __restrict__ pools, int l, int64_t row,
                                         int64_t host, int lane) {
  const uint8_t* src = pools->dev[l] + (size_t)row * g.B;
  uint8_t* dst = const_cast<uint8_t*>(pools->host[l]) + (size_t)host * g.B;
  if (g.vec == 16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int q = lane; q < (g.B >> 4); q += 32) d4[q] = s4[q];
  } else if (g.vec == 4) {
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d4 = reinterpret_cast<uint32_t*>(dst);
    for (int q = lane; q < (g.B >> 2); q += 32) d4[q] = s4[q];
  } else {
    for (int q = lane; q < g.B; q += 32) dst[q] = src[q];
  }
}

__global__ void __launch_bounds__(kBackupThreads)
    backup_kernel(const Geometry g, const Pools* __restrict__ pools, const BackupArgs a, int32_t num_requests,
                  uint32_t* __restrict__ err_word) {
  const int lane = threadIdx.x & 31;
  const int w = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const bool active = w < num_requests * g.L;  // whole warps
  const int r = active ? w / g.L : 0, l = active ? w - r * g.L : 0;
  const int32_t S = active ? a.seq_lens[r] : 0;
  uint32_t flag = 0;
  int64_t row = -1, host = -1;
  if (!active) {
    // spare warp of the last block: nothing to copy
  } else if (S < 0 || S > g.max_context) {
    flag = HS_FLAG_SEQLEN;
  } else if (S >= 1) {
    const int32_t t = S - 1;
    int32_t page = -1;
    if (a.resident_pages) page = a.resident_pages[(size_t)r * g.max_pages + t / g.page_size];
    if (page >= 0) row = (int64_t)page * g.page_size + t % g.page_size;
    else row = a.device_buffer_locs[(size_t)r * (g.H + 1) + (S <= g.H ? t : g.H)];
    host = a.host_cache_locs[(size_t)r * g.max_context + t];
    if (row < 0 || row >= g.device_rows) flag = HS_FLAG_DEVROW;
    else if (host < 0 || host >= g.host_rows) flag = HS_FLAG_HOSTROW;
  }
  if (flag) {
    if (lane == 0) atomicOr(err_word, flag);
  } else if (row >= 0) {  // row < 0: empty sequence, nothing to back up
    copy_row(g, pools, l, row, host, lane);
  }
  // Launched as a programmatic dependent of the resolve, this kernel may run beside it
  // (the two touch disjoint rows); it completes only after the resolve has, so work
  // queued after it on the stream still sees both finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_backup(const Geometry& g, const Pools* pools, const BackupArgs& a, int32_t num_requests,
                          uint32_t* err_word, cudaStream_t stream) {
  const long long warps = (long long)num_requests * g.L;
  const int per_block = kBackupThreads / 32;
  const unsigned blocks = (unsigned)((warps + per_block - 1) / per_block);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kBackupThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, backup_kernel, g, pools, a, num_requests, err_word);
}

}  // namespace hs
