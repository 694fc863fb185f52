// Eager backup: the newest token's KV row -- or, after a speculative batch, the rows of its
// accepted positions -- device -> pinned host, one warp per (request, layer, position).
//
// Source: "HiSparse: moving the long-context decode capacity bottleneck from GPU memory to
// CPU memory", "Per decode step workflow", step 5 (after attention, the last token's KV is
// copied back from device to host so the host pool stays complete). The row sits in its
// resident page when that page is GPU-resident ("vLLM HiSparse local KV offload
// architecture", "Hot-row lookup and LRU"), in buffer slot seq_len-1 while the sequence
// fits the buffer, else in the reserved slot H ("How capacity is computed": the buffer
// carries an extra page for the new token). A speculative batch's positions S0 + j sit in
// their resident rows, in slot S0 + j while the sequence then fit the buffer, else in the
// reserved row H + j ("vLLM Hybrid HiSparse source implementation analysis", 7.1: the buffer
// holds (n_spec + 2) x top_k rows).
#include "hs_internal.h"

namespace hs {
namespace {

__device__ __forceinline__ void copy_row(const Geometry& g, const Pools* __restrict__ pools, int l, int64_t row,
                                         int64_t host, int lane) {
  const uint8_t* src = pools->dev[l] + (size_t)row * g.B;
  uint8_t* dst = const_cast<uint8_t*>(pools->host[l]) + (size_t)host * g.host_stride;
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
  const int per_req = g.L * a.spec_n;
  const bool active = w < num_requests * per_req;  // whole warps
  const int r = active ? w / per_req : 0, rem = active ? w - r * per_req : 0;
  const int l = rem / a.spec_n, j = rem - l * a.spec_n;
  uint32_t flag = 0;
  int64_t row = -1, host = -1;
  if (active) {
    // position base + j for j < n: the newest token (base = S - 1, n = 1 unless empty), or a
    // speculative batch's accepted positions (base = S0, n = accepted)
    const int32_t in = a.seq_lens[r];
    const int32_t n = a.accepted ? a.accepted[r] : (in >= 1 ? 1 : 0);
    const int32_t base = a.accepted ? in : in - 1;
    const bool bad = a.accepted ? (in < 0 || n < 0 || n > a.spec_n || (int64_t)in + n > g.max_context)
                                : (in < 0 || in > g.max_context);
    if (bad) {
      if (j == 0) flag = HS_FLAG_SEQLEN;
    } else if (j < n) {
      const int32_t t = base + j;
      int32_t page = -1;
      if (a.resident_pages) page = a.resident_pages[(size_t)r * g.max_pages + t / g.page_size];
      if (page >= 0) row = (int64_t)page * g.page_size + t % g.page_size;
      else row = a.device_buffer_locs[(size_t)r * (g.H + a.spec_n) + (t + 1 <= g.H ? t : g.H + j)];
      host = a.host_cache_locs[(size_t)r * g.max_context + t];
      if (row < 0 || row >= g.device_rows) flag = HS_FLAG_DEVROW;
      else if (host < 0 || host >= g.host_rows) flag = HS_FLAG_HOSTROW;
    }
  }
  if (flag) {
    if (lane == 0) atomicOr(err_word, flag);
  } else if (row >= 0) {  // row < 0: nothing to back up here
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
  const long long warps = (long long)num_requests * g.L * a.spec_n;
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
