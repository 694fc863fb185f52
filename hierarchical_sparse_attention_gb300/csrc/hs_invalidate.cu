// Hot-slot invalidation: drop cached rows whose host content changed.
//
// Source (page title, section): "vLLM Hybrid HiSparse source implementation analysis", 6
// (worker data plane, invalidation propagation: hot entries pointing at rows of host blocks
// handed to other content must go, and rows prefill rewrote in this step are cleared
// exactly; the worker matches a sorted list of the affected rows against the hot entries).
//
// A cleared slot becomes free (token -1, stamp 0), so the next resolve misses on its token
// and copies the current row. The clock does not move; the token's residency bit is cleared. Slots
// are keyed by token, so the exact form names tokens per request; the host-row form names
// host rows and reaches each held token's row through host_cache_locs. Only tokens in
// [0, seq_len - 1) count (no valid slot holds another), and requests on the fast path
// (seq_len <= H) are left alone: their device rows are the tokens' own rows, which the
// forward pass rewrites in place.
//
// The grid is (request, block of T slots): each thread owns one slot and looks it up once per
// chunk of the clear list. The work is a few KB of state per request, so the kernel is
// bound by launch and load latency, not bandwidth: spreading a request over several CTAs
// puts every slot's dependent loads in flight at once.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int T = kInvalidateThreads;
constexpr int kHashBits = 13;
constexpr int kClearHash = 1 << kHashBits;   // open-addressing table of tokens in shared memory
constexpr int kClearChunk = kClearHash / 2;  // tokens hashed per pass: the table stays half empty
constexpr int kRowStage = 8192;              // sorted host rows staged in shared memory

__device__ __forceinline__ uint32_t token_bucket(int32_t t) {
  return ((uint32_t)t * 2654435761u) >> (32 - kHashBits);  // Knuth multiplicative
}

// Clear slot s of a request: free, stamp 0, the token's residency bit cleared.
__device__ __forceinline__ void clear_slot(int32_t* tok, int32_t* st, uint32_t* bits, int s, int32_t t) {
  tok[s] = -1;
  st[s] = 0;
  if (bits) atomicAnd(&bits[t >> 5], ~(1u << (t & 31)));  // the token is no longer resident
}

// Whether request r's slots are subject to invalidation; flags a bad seq_len.
__device__ __forceinline__ bool applies(const Geometry& g, int32_t S, uint32_t* err_word) {
  if (S < 0 || S > g.max_context) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err_word, HS_FLAG_SEQLEN);
    return false;
  }
  return S > g.H;
}

__global__ void __launch_bounds__(T) invalidate_tokens_kernel(const Geometry g, const InvalidateArgs a,
                                                              uint32_t* __restrict__ err_word) {
  __shared__ int32_t s_tab[kClearHash];
  const int r = blockIdx.x;
  const int s = (int)blockIdx.y * T + (int)threadIdx.x;  // this thread's slot
  int32_t* tok = a.device_buffer_tokens + (size_t)r * g.H;
  int32_t t = s < g.H ? tok[s] : -1;  // issued with seq_len and the list bounds: one round trip
  const int32_t S = a.seq_lens[r];
  if (!applies(g, S, err_word)) return;
  const int32_t k0 = a.token_offsets[r], k1 = a.token_offsets[r + 1];
  int32_t* st = a.lru_slots + (size_t)r * g.H;
  uint32_t* hint = a.hint ? a.hint + (size_t)r * g.bit_words : nullptr;
  for (int32_t c0 = k0; c0 < k1; c0 += kClearChunk) {
    const int32_t c1 = min(k1, c0 + kClearChunk);
    for (int i = threadIdx.x; i < kClearHash; i += T) s_tab[i] = -1;
    __syncthreads();
    for (int32_t k = c0 + (int32_t)threadIdx.x; k < c1; k += T) {
      const int32_t c = a.tokens[k];
      if (c < 0 || c >= S - 1) continue;
      uint32_t h = token_bucket(c);
      for (;;) {  // at most kClearChunk keys in 2 * kClearChunk buckets: ends
        const int32_t prev = atomicCAS(&s_tab[h], -1, c);
        if (prev == -1 || prev == c) break;
        h = (h + 1) & (kClearHash - 1);
      }
    }
    __syncthreads();
    if (t >= 0 && t < S - 1) {
      uint32_t h = token_bucket(t);
      for (;;) {
        const int32_t v = s_tab[h];
        if (v == -1) break;
        if (v == t) {
          clear_slot(tok, st, hint, s, t);
          t = -1;  // a later chunk finds the slot free
          break;
        }
        h = (h + 1) & (kClearHash - 1);
      }
    }
    __syncthreads();  // the table is rebuilt for the next chunk; this CTA's slot writes are seen
  }
}

__global__ void __launch_bounds__(T) invalidate_host_rows_kernel(const Geometry g, const InvalidateRowsArgs a,
                                                                 uint32_t* __restrict__ err_word) {
  __shared__ int32_t s_rows[kRowStage];
  __shared__ int s_unsorted;
  const int r = blockIdx.x;
  const int s = (int)blockIdx.y * T + (int)threadIdx.x;  // this thread's slot
  int32_t* tok = a.device_buffer_tokens + (size_t)r * g.H;
  const int32_t* hcl = a.host_cache_locs + (size_t)r * g.max_context;
  // the slot's token and its host row go out first, beside seq_len and the row list
  const int32_t t = s < g.H ? tok[s] : -1;
  const int32_t hr = (t >= 0 && t < g.max_context) ? hcl[t] : -1;
  const int32_t S = a.seq_lens[r];
  if (!applies(g, S, err_word)) return;
  const int32_t n = a.n;
  const bool staged = n <= kRowStage;
  if (threadIdx.x == 0) s_unsorted = 0;
  __syncthreads();
  if (staged) {  // stage the list and check its order
    for (int i = threadIdx.x; i < n; i += T) {
      const int32_t v = a.rows[i];
      s_rows[i] = v;
      if (i + 1 < n && a.rows[i + 1] < v) s_unsorted = 1;
    }
    __syncthreads();
    if (s_unsorted) {
      if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err_word, HS_FLAG_ORDER);
      return;
    }
  }
  const int32_t* rows = staged ? s_rows : a.rows;
  int32_t* st = a.lru_slots + (size_t)r * g.H;
  uint32_t* hint = a.hint ? a.hint + (size_t)r * g.bit_words : nullptr;
  if (t < 0 || t >= S - 1) return;
  int lo = 0, hi = n;  // first index with rows[i] >= hr
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (rows[mid] < hr) lo = mid + 1;
    else hi = mid;
  }
  if (lo < n && rows[lo] == hr) clear_slot(tok, st, hint, s, t);
}

}  // namespace

cudaError_t launch_invalidate_tokens(const Geometry& g, const InvalidateArgs& a, int32_t num_requests,
                                     uint32_t* err_word, cudaStream_t stream) {
  invalidate_tokens_kernel<<<dim3(num_requests, (g.H + T - 1) / T), T, 0, stream>>>(g, a, err_word);
  return cudaGetLastError();
}

cudaError_t launch_invalidate_host_rows(const Geometry& g, const InvalidateRowsArgs& a, int32_t num_requests,
                                        uint32_t* err_word, cudaStream_t stream) {
  invalidate_host_rows_kernel<<<dim3(num_requests, (g.H + T - 1) / T), T, 0, stream>>>(g, a, err_word);
  return cudaGetLastError();
}

}  // namespace hs
