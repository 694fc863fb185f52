// Follower gather: replay the leader's miss plan for other layers of the group.
//
// Sources (page title, section): "vLLM Hybrid HiSparse source implementation analysis", 7.4
// (layers that share the indexer see the same indices and the same slot plan; only their
// bytes differ, so each follower copies its own rows following the leader's plan, with no
// LRU work) and "vLLM HiSparse local KV offload architecture", "Performance invariants"
// (compatible layers still share one miss plan).
//
// The plan is what the last hs_resolve / hs_resolve_layers recorded in the workspace: per
// request, the miss tokens and their device rows in miss order. A CTA takes a run of
// kGatherMisses misses of one request, looks up their host rows once, and copies their
// rows for the requested layers with 16-byte (else 4- or 1-byte) loads streamed past the
// caches, several in flight per thread. Run on a copy stream, one call per layer (or per
// few layers) with an event after each, layer l + 1's rows move while layer l's attention
// runs. Bound: the host link (miss rows), like the resolve's own copies.
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
  __shared__ const uint8_t* s_host[kMaxLayers];
  __shared__ uint8_t* s_dev[kMaxLayers];
  using P = Piece<V>;
  const int r = blockIdx.x;
  const int j0 = (int)blockIdx.y * M;
  const int m = a.plan_cnt[r];
  if (j0 >= m) return;
  const int nm = min(M, m - j0);
  uint32_t flags = 0;
  if (threadIdx.x < (unsigned)a.num_layers) {
    s_host[threadIdx.x] = pools->host[a.first_layer + threadIdx.x];
    s_dev[threadIdx.x] = pools->dev[a.first_layer + threadIdx.x];
  }
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
  const int per_miss = per_row * a.num_layers;
  const int total = nm * per_miss;
  for (int base = threadIdx.x; base < total; base += T * kUnroll) {
    typename P::type v[kUnroll];
    uint8_t* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = base + u * T;
      dst[u] = nullptr;
      if (c < total) {
        const int j = c / per_miss, rem = c - j * per_miss, l = rem / per_row, q = rem - l * per_row;
        const int32_t d = s_dst[j];
        if (d >= 0) {
          const int32_t sr = s_src[j];
          dst[u] = s_dev[l] + (size_t)d * g.B + (size_t)q * V;
          v[u] = sr >= 0 ? P::load(s_host[l] + (size_t)sr * g.B + (size_t)q * V) : P::zero();
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u]) *reinterpret_cast<typename P::type*>(dst[u]) = v[u];
  }
  if (flags) atomicOr(err_word, flags);
}

}  // namespace

cudaError_t launch_gather(const Geometry& g, const Pools* pools, const GatherArgs& a, int32_t num_requests,
                          uint32_t* err_word, cudaStream_t stream) {
  const dim3 grid(num_requests, (g.K + kGatherMisses - 1) / kGatherMisses);
  if (g.vec == 16) gather_kernel<16><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  else if (g.vec == 4) gather_kernel<4><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  else gather_kernel<1><<<grid, kGatherThreads, 0, stream>>>(g, pools, a, err_word);
  return cudaGetLastError();
}

}  // namespace hs
