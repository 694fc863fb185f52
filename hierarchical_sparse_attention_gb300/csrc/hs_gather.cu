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
// flight per thread. With one host pool per layer both go layer-major: one layer's rows move
// before the next layer's start, so the host pages read at any moment span one layer's pool.
// With every layer's bytes of a token in one host row ("page first", the other host layout of
// "Hierarchical Sparse Attention" (Alibaba Tair KVCache), 2.4.4 "I/O Transfer Kernel"), the
// pair gather reads each miss's layers as one contiguous span instead. Called on a copy
// stream, one call per layer with an event after each, layer l + 1's rows move while layer
// l's attention runs. Bound: the host link.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int T = kGatherThreads;
constexpr int M = kGatherMisses;
constexpr int kUnroll = 4;
constexpr int kGatherCtasPerSm = 2048 / T;  // a full SM's threads, when the occupancy is not known

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
          v[u] = sr >= 0 ? P::load(host + (size_t)sr * g.host_stride + (size_t)q * V) : P::zero();
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

// Copy rows of the ordered pairs for layers [first_layer, first_layer + num_layers). The grid
// is persistent (a few CTAs per SM, as many as one wave holds): the pair count is known only
// on the device, and a grid sized for the largest count spent a wave's worth of time per
// layer on CTAs with nothing to copy. The work is a list of items, each M consecutive pairs;
// CTA b takes items b, b + gridDim.x, ... so the CTAs move through the list together.
//   - Layers in one pool each ("layer first"): an item is (layer, M pairs), layer-major, so
//     the host rows read at any moment lie in one layer's pool.
//   - Interleaved host rows ("page first", g.host_interleaved): an item is M pairs of every
//     requested layer. Host row h of layers [first_layer, first_layer + num_layers) is then
//     one contiguous span of num_layers * B bytes, read front to back; only the device side
//     splits it by layer.
template <int V>
__global__ void __launch_bounds__(T) gather_pairs_kernel(const Geometry g, const Pools* __restrict__ pools,
                                                         const OrderArgs a, int first_layer, int num_layers) {
  __shared__ int32_t s_src[M], s_dst[M];
  using P = Piece<V>;
  const int64_t n = min((int64_t)*a.n_pairs, a.capacity);
  const int64_t chunks = (n + M - 1) / M;
  const bool span = g.host_interleaved != 0;
  const int per_row = g.B / V;
  const int64_t items = span ? chunks : chunks * num_layers;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int layer0 = span ? first_layer : first_layer + (int)(item / chunks);
    const int64_t j0 = (span ? item : item % chunks) * M;
    const int nm = (int)min((int64_t)M, n - j0);
    const int nl = span ? num_layers : 1;  // layers this item copies, from layer0 on
    __syncthreads();  // the previous item is done with the pair table
    if ((int)threadIdx.x < nm) {
      s_src[threadIdx.x] = a.pair_src[j0 + threadIdx.x];
      s_dst[threadIdx.x] = a.pair_dst[j0 + threadIdx.x];
    }
    __syncthreads();
    const uint8_t* host = pools->host[layer0];
    const int per_pair = per_row * nl;
    const int total = nm * per_pair;
    for (int base = threadIdx.x; base < total; base += T * kUnroll) {
      typename P::type v[kUnroll];
      uint8_t* dst[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = base + u * T;
        dst[u] = nullptr;
        if (c < total) {
          const int j = c / per_pair, qs = c - j * per_pair;  // piece qs of the pair's span
          const int l = qs / per_row, q = qs - l * per_row;
          const int32_t d = s_dst[j], sr = s_src[j];
          if (d >= 0) {
            dst[u] = pools->dev[layer0 + l] + (size_t)d * g.B + (size_t)q * V;
            v[u] = sr >= 0 ? P::load(host + (size_t)sr * g.host_stride + (size_t)qs * V) : P::zero();
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (dst[u]) *reinterpret_cast<typename P::type*>(dst[u]) = v[u];
    }
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

int gather_pairs_ctas_per_sm(int vec) {
  int n = 0;
  const cudaError_t e =
      vec == 16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gather_pairs_kernel<16>, T, 0)
      : vec == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gather_pairs_kernel<4>, T, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gather_pairs_kernel<1>, T, 0);
  if (e != cudaSuccess || n < 1) {
    cudaGetLastError();
    return kGatherCtasPerSm;
  }
  return n;
}

cudaError_t launch_gather_pairs(const Geometry& g, const Pools* pools, const OrderArgs& a, int32_t num_requests,
                                int32_t first_layer, int32_t num_layers, cudaStream_t stream) {
  // the pair count is known only on the device: at most num_requests * K pairs, so no more
  // CTAs than items, and no more than one wave (the CTAs that fit an SM at once, times the
  // SMs): a CTA of a second wave would start its items only when one of the first finished
  const int64_t most = (int64_t)num_requests * g.K;
  const int64_t items = ((most + M - 1) / M) * (g.host_interleaved ? 1 : num_layers);
  int64_t ctas = (int64_t)(g.sms > 0 ? g.sms : 1) * (g.gather_ctas_per_sm > 0 ? g.gather_ctas_per_sm : kGatherCtasPerSm);
  if (ctas > items) ctas = items;
  if (ctas < 1) ctas = 1;
  const dim3 grid((unsigned)ctas);
  if (g.vec == 16) gather_pairs_kernel<16><<<grid, T, 0, stream>>>(g, pools, a, first_layer, num_layers);
  else if (g.vec == 4) gather_pairs_kernel<4><<<grid, T, 0, stream>>>(g, pools, a, first_layer, num_layers);
  else gather_pairs_kernel<1><<<grid, T, 0, stream>>>(g, pools, a, first_layer, num_layers);
  return cudaGetLastError();
}

}  // namespace hs
