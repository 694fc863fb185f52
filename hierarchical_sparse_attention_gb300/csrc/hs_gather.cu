// Miss-row copies that run apart from the resolve kernel: follower gathers and the copies of
// a step without copy CTAs.
//
// Sources (page title, section): "vLLM Hybrid HiSparse source implementation analysis", 7.4
// (layers that share the indexer see the same indices and the same slot plan; only their
// bytes differ, so each follower copies its own rows following the leader's plan, with no
// LRU work) and "vLLM HiSparse local KV offload architecture", "Performance invariants"
// (compatible layers still share one miss plan).
//
// The plan is what the last resolve recorded in the workspace: per request, the miss tokens
// and their device rows in miss order. Two forms copy it:
//   - gather_kernel replays it as recorded: a CTA takes a run of kGatherMisses misses of one
//     request and one layer, looks up their host rows and streams the rows;
//   - order_count_kernel and order_scatter_kernel first regroup it as (host row, device row)
//     pairs by 2 MB region of the host pool, and gather_pairs_kernel copies those. Rows that
//     share a region are then requested together and share the GPU's translation of it; in
//     miss order, rows spread over several large pools moved at about half the link's rate.
// Both copy with 16-byte (else 4- or 1-byte) loads streamed past the caches, several in
// flight per thread, and both grids are layer-major: one layer's rows move before the next
// layer's start, so the host pages read at any moment span one layer's pool. Called on a copy
// stream, one call per layer with an event after each, layer l + 1's rows move while layer
// l's attention runs. Bound: the host link.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int T = kGatherThreads;
constexpr int M = kGatherMisses;
constexpr int kUnroll = 4;

template <int V>
struct Piece;
template <>
struct Piece<16> {
  using type = uint4;
  __device__ static type load(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ static type zero() { return make_uint4(0u, 0u, 0u, 0u); }
};
template <>
struct Piece<4> {
  using type = uint32_t;
  __device__ static type load(const void* p) { return __ldcs(reinterpret_cast<const unsigned int*>(p)); }
  __device__ static type zero() { return 0u; }
};
template <>
struct Piece<1> {
  using type = uint8_t;
  __device__ static type load(const void* p) { return *reinterpret_cast<const uint8_t*>(p); }
  __device__ static type zero() { return 0; }
};

template <int V>
__global__ void __launch_bounds__(T) gather_kernel(const Geometry g, const Pools* __restrict__ pools,
                                                   const GatherArgs a, uint32_t* __restrict__ err_word) {
  __shared__ int32_t s_src[M], s_dst[M];
  using P = Piece<V>;
  const int r = blockIdx.x;
  const int j0 = (int)blockIdx.y * M;
  const int layer = a.first_layer + (int)blockIdx.z;
  const int m = a.plan_cnt[r];
  if (j0 >= m) return;
  const int nm = min(M, m - j0);
  uint32_t flags = 0;
  const uint8_t* host = pools->host[layer];
  uint8_t* dev = pools->dev[layer];
  if ((int)threadIdx.x < nm) {
    const size_t at = (size_t)r * g.K + j0 + threadIdx.x;
    const int32_t d = a.plan_dst[at];
    int32_t src = -1;
    if (d >= 0) {
      const int32_t t = a.plan_tok[at];
      const int32_t hr = (t >= 0 && t < g.max_context) ? a.host_cache_locs[(size_t)r * g.max_context + t] : -1;
      if (hr >= 0 && (int64_t)hr < g.host_rows) src = hr;
      else flags |= HS_FLAG_HOSTROW;  // the destination is zero-filled, as the leader's was
    }
    s_src[threadIdx.x] = src;
    s_dst[threadIdx.x] = d;
  }
  __syncthreads();
  const int per_row = g.B / V;
  const int total = nm * per_row;
  for (int base = threadIdx.x; base < total; base += T * kUnroll) {
    typename P::type v[kUnroll];
    uint8_t* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = base + u * T;
      dst[u] = nullptr;
      if (c < total) {
        const int j = c / per_row, q = c - j * per_row;
        const int32_t d = s_dst[j];
        if (d >= 0) {
          const int32_t sr = s_src[j];
          dst[u] = dev + (size_t)d * g.B + (size_t)q * V;
          v[u] = sr >= 0 ? P::load(host + (size_t)sr * g.B + (size_t)q * V) : P::zero();
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u]) *reinterpret_cast<typename P::type*>(dst[u]) = v[u];
  }
  if (flags) atomicOr(err_word, flags);
}

constexpr int kOrderThreads = 1024;  // one CTA per request; its threads stride over the plan
constexpr int32_t kNoRow = -2;      // plan entry without a device row: nothing to copy
constexpr int kScanBatch = 8;       // counters loaded together in the region scan

__device__ __forceinline__ int32_t region_of(const Geometry& g, int32_t src) {
  return src >= 0 ? (src >> g.order_shift) : g.order_regions;
}

// Count the plan's misses per host region. One CTA per request walks its plan; the last CTA
// to finish (a ticket taken after a fence, so every count is in L2) turns the counts into
// exclusive offsets, zeroes them for the next step and stores the total. (CTAs per run of
// entries, most of them empty, spent more time taking the one ticket in turn than counting.)
__global__ void __launch_bounds__(kOrderThreads) order_count_kernel(const Geometry g, const OrderArgs a,
                                                                    uint32_t* __restrict__ err_word) {
  __shared__ int32_t s_warp[kOrderThreads / 32];
  __shared__ int s_last;
  const int r = blockIdx.x;
  const int m = min(a.plan_cnt[r], g.K);
  for (int j = threadIdx.x; j < m; j += kOrderThreads) {
    const size_t at = (size_t)r * g.K + j;
    const int32_t d = a.plan_dst[at], t = a.plan_tok[at];
    int32_t src = kNoRow;
    if (d >= 0) {
      const int32_t hr = (t >= 0 && t < g.max_context) ? a.host_cache_locs[(size_t)r * g.max_context + t] : -1;
      src = (hr >= 0 && (int64_t)hr < g.host_rows) ? hr : -1;
      if (src < 0) atomicOr(err_word, HS_FLAG_HOSTROW);  // its rows are zero-filled, as the resolve's are
      atomicAdd(a.counts + region_of(g, src), 1);
    }
    a.miss_src[at] = src;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // each thread scans a contiguous run of counters, eight loads in flight at a time (the
  // counters sit in L2; one dependent load per counter made this the kernel's longest part)
  const int n = g.order_regions + 1;
  const int per = (n + kOrderThreads - 1) / kOrderThreads;
  const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
  int sum = 0;
  for (int i0 = lo; i0 < hi; i0 += kScanBatch) {
    int v[kScanBatch];
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) v[u] = i0 + u < hi ? __ldcg(a.counts + i0 + u) : 0;
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) sum += v[u];
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += s_warp[w];
  for (int i0 = lo; i0 < hi; i0 += kScanBatch) {
    int v[kScanBatch];
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) v[u] = i0 + u < hi ? __ldcg(a.counts + i0 + u) : 0;
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u)
      if (i0 + u < hi) {
        a.cursors[i0 + u] = run;
        run += v[u];
        a.counts[i0 + u] = 0;
      }
  }
  if (threadIdx.x == kOrderThreads - 1) {
    *a.n_pairs = run;  // the last thread's range ends the array: run is the total
    *a.ticket = 0u;
  }
}

// Place each counted miss at its region's next position (one CTA per request).
__global__ void __launch_bounds__(kOrderThreads) order_scatter_kernel(const Geometry g, const OrderArgs a) {
  const int r = blockIdx.x;
  const int m = min(a.plan_cnt[r], g.K);
  for (int j = threadIdx.x; j < m; j += kOrderThreads) {
    const size_t at = (size_t)r * g.K + j;
    const int32_t src = a.miss_src[at], d = a.plan_dst[at];
    if (src == kNoRow) continue;
    const int pos = atomicAdd(a.cursors + region_of(g, src), 1);
    if (pos < 0 || pos >= a.capacity) continue;  // only a workspace the caller overwrote gets here
    a.pair_src[pos] = src;
    a.pair_dst[pos] = d;
  }
}

// Copy rows of the ordered pairs: a CTA takes M consecutive pairs of one layer; blocks are
// dispatched layer-major (blockIdx.y slowest).
template <int V>
__global__ void __launch_bounds__(T) gather_pairs_kernel(const Geometry g, const Pools* __restrict__ pools,
                                                         const OrderArgs a, int first_layer) {
  __shared__ int32_t s_src[M], s_dst[M];
  using P = Piece<V>;
  const int64_t n = min((int64_t)*a.n_pairs, a.capacity);
  const int64_t j0 = (int64_t)blockIdx.x * M;
  if (j0 >= n) return;
  const int nm = (int)min((int64_t)M, n - j0);
  const int layer = first_layer + (int)blockIdx.y;
  const uint8_t* host = pools->host[layer];
  uint8_t* dev = pools->dev[layer];
  if ((int)threadIdx.x < nm) {
    s_src[threadIdx.x] = a.pair_src[j0 + threadIdx.x];
    s_dst[threadIdx.x] = a.pair_dst[j0 + threadIdx.x];
  }
  __syncthreads();
  const int per_row = g.B / V;
  const int total = nm * per_row;
  for (int base = threadIdx.x; base < total; base += T * kUnroll) {
    typename P::type v[kUnroll];
    uint8_t* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = base + u * T;
      dst[u] = nullptr;
      if (c < total) {
        const int j = c / per_row, q = c - j * per_row;
        const int32_t d = s_dst[j], sr = s_src[j];
        if (d >= 0) {
          dst[u] = dev + (size_t)d * g.B + (size_t)q * V;
          v[u] = sr >= 0 ? P::load(host + (size_t)sr * g.B + (size_t)q * V) : P::zero();
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u]) *reinterpret_cast<typename P::type*>(dst[u]) = v[u];
  }
}

}  // namespace

cudaError_t launch_gather(const Geometry& g, const Pools* pools, const GatherArgs& a, int32_t num_requests,
                          uint32_t* err_word, cudaStream_t stream) {
  // layer-major: blocks are dispatched z-slowest
  const dim3 grid(num_requests, (g.K + kGatherMisses - 1) / kGatherMisses, a.num_layers);
  if (g.vec == 16) gather_kernel<16><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  else if (g.vec == 4) gather_kernel<4><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  else gather_kernel<1><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  return cudaGetLastError();
}

cudaError_t launch_order(const Geometry& g, const OrderArgs& a, int32_t num_requests, uint32_t* err_word,
                         cudaStream_t stream) {
  order_count_kernel<<<num_requests, kOrderThreads, 0, stream>>>(g, a, err_word);
  order_scatter_kernel<<<num_requests, kOrderThreads, 0, stream>>>(g, a);
  return cudaGetLastError();
}

cudaError_t launch_gather_pairs(const Geometry& g, const Pools* pools, const OrderArgs& a, int32_t num_requests,
                                int32_t first_layer, int32_t num_layers, cudaStream_t stream) {
  const int64_t most = (int64_t)num_requests * g.K;  // the pair count is known only on the device
  const dim3 grid((unsigned)((most + M - 1) / M), num_layers);
  if (g.vec == 16) gather_pairs_kernel<16><<<grid, T, 0, stream>>>(g, pools, a, first_layer);
  else if (g.vec == 4) gather_pairs_kernel<4><<<grid, T, 0, stream>>>(g, pools, a, first_layer);
  else gather_pairs_kernel<1><<<grid, T, 0, stream>>>(g, pools, a, first_layer);
  return cudaGetLastError();
}

}  // namespace hs
