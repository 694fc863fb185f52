// Fused decode-step resolver / swap-in: one CTA of 1024 threads per request.
//
// Sources (page title, section):
//   "HiSparse: Turbocharging Sparse Attention with Hierarchical Memory" (LMSYS), "Efficient
//     swap-in kernel": one kernel finds the top-k misses in the device buffer, picks LRU
//     victims, updates the table and fetches the missing rows from host memory.
//   "HiSparse: moving the long-context decode capacity bottleneck from GPU memory to CPU
//     memory", "Per decode step workflow" step 3 (fast path for seq_len <= buffer size)
//     and "How capacity is computed" (one reserved row for the newest token).
//   "vLLM HiSparse local KV offload architecture", "Hot-row lookup and LRU" (resident page,
//     then hot row with LRU refresh, then a victim filled from pinned host memory).
//   "vLLM Hybrid HiSparse source implementation analysis", 7.2 (resident short-circuit;
//     a shared-memory hash of the top-k; ballot/scan compaction of the misses; victims
//     from the cold end; out-of-range state downgraded to a re-miss; warp-wide 16-byte
//     copies that zero the destination when the source row is out of range), 7.3 (flat
//     physical row IDs) and 7.4 (layers sharing the indexer reuse the same slot plan).
//   "Hierarchical Sparse Attention" (Alibaba Tair), 2.4.3 "LRU Diff Kernel" (evict only
//     when the buffer is full, coldest first).
//
// Phases of one CTA (request r), all state in shared memory:
//   1  load the top-k row, reject padding / out-of-range tokens, build an open-addressing
//      hash (Knuth multiplicative) of the valid tokens; repeated tokens keep the first index
//   2  classify: resident row, fast-path identity, reserved newest row, or hot lookup
//   3  load slot tokens and stamps, reset corrupt entries, probe each slot's token in the
//      hash; the lowest slot holding a looked-up token claims it (atomicMin)
//   4  hits: stamp = clock, output the slot's row
//   5  one packed block scan compacts the misses (top-k order) and the free slots (slot order);
//      each miss's host row is looked up and a bulk L2 prefetch of it is issued right away
//   6  if misses outnumber free slots: radix-select the stamp threshold over the occupied,
//      un-hit slots, gather exactly the needed victims, bitonic-sort them by (stamp, slot)
//   7  pair miss j with victim j, update the map, build the copy plan
//   8  write back the changed slots, the output row table and the clock
//   9  copy every miss row of every layer (now mostly in L2) to its victim's device row
//      (16-byte pieces spread over all 1024 threads, several loads in flight per thread)
#include <climits>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int T = kResolveThreads;
constexpr int NW = T / 32;
constexpr unsigned FULL = 0xffffffffu;
constexpr int32_t INF = 0x7fffffff;
constexpr int kCopyUnroll = 4;

enum : uint8_t { C_PAD = 0, C_BAD, C_DUP, C_VALID, C_RES, C_FAST, C_NEWEST, C_LOOKUP };
enum : uint8_t { SF_USED = 1, SF_DIRTY = 2 };
enum { SC_LO = 0, SC_HI, SC_DIGIT, SC_RANK, SC_COUNT };

// Shared-memory carve-up; identical arithmetic on host (size) and device (pointers).
// The top-k hash (1 << hash_bits = 2 * sort_cap int32 keys and values) is dead after
// phase 3, so the victim sort keys (phase 6) and the copy plan (phases 7-9) reuse it:
// 8*sort_cap bytes of keys, then K source rows and K destination rows (K <= sort_cap).
struct Layout {
  size_t hkey, hval, keys, psrc, pdst, tk, out, claim, miss, vict, tok, stamp, sent, cls, sflag, wsum, hist,
      sc, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline Layout make_layout(const Geometry& g) {
  Layout l;
  size_t o = 0;
  const size_t K = (size_t)g.K, H = (size_t)g.H, HS = (size_t)1 << g.hash_bits;
  l.hkey = o; o = align16(o + 4 * HS);
  l.hval = o; o = align16(o + 4 * HS);
  l.keys = l.hkey;
  l.psrc = l.hkey + sizeof(uint64_t) * (size_t)g.sort_cap;
  l.pdst = l.psrc + 4 * K;
  l.tk = o; o = align16(o + 4 * K);
  l.out = o; o = align16(o + 4 * K);
  l.claim = o; o = align16(o + 4 * K);
  l.miss = o; o = align16(o + 4 * K);
  l.vict = o; o = align16(o + 4 * K);
  l.tok = o; o = align16(o + 4 * H);
  l.stamp = o; o = align16(o + 4 * H);
  l.sent = o; o = align16(o + 2 * H);
  l.cls = o; o = align16(o + K);
  l.sflag = o; o = align16(o + H);
  l.wsum = o; o = align16(o + 4 * (NW + 1));
  l.hist = o; o = align16(o + 4 * 256);
  l.sc = o; o = align16(o + 4 * SC_COUNT);
  l.total = o;
  return l;
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix sum of v over the CTA, in thread order. Ends synchronised, so wsum
// can be reused by the next call.
__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int s = wsum[lane];
    const int si = warp_incl_scan(s);
    wsum[lane] = si - s;
    if (lane == 31) wsum[NW] = si;
  }
  __syncthreads();
  const int res = incl - v + wsum[w];
  *total = wsum[NW];
  __syncthreads();
  return res;
}

__device__ __forceinline__ uint32_t hash_slot(int32_t t, int bits) {
  return ((uint32_t)t * 2654435761u) >> (32 - bits);
}

// Insert token t for top-k index i; a repeated token keeps the smallest index.
__device__ __forceinline__ void hash_insert(int32_t* hkey, int32_t* hval, int bits, int32_t t, int32_t i) {
  const uint32_t mask = (1u << bits) - 1;
  uint32_t h = hash_slot(t, bits);
  for (;;) {  // ends: the table is at most half full
    const int32_t prev = atomicCAS(&hkey[h], -1, t);
    if (prev == -1 || prev == t) {
      atomicMin(&hval[h], i);
      return;
    }
    h = (h + 1) & mask;
  }
}

__device__ __forceinline__ int hash_find(const int32_t* hkey, int bits, int32_t t) {
  const uint32_t mask = (1u << bits) - 1;
  uint32_t h = hash_slot(t, bits);
  for (;;) {  // ends: at least half the table is empty
    const int32_t k = hkey[h];
    if (k == t) return (int)h;
    if (k == -1) return -1;
    h = (h + 1) & mask;
  }
}

__device__ __forceinline__ int32_t checked_row(int64_t row, int64_t rows, uint32_t& flags) {
  if (row < 0 || row >= rows) {
    flags |= HS_FLAG_DEVROW;
    return -1;
  }
  return (int32_t)row;
}

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory.
__device__ void bitonic_sort(uint64_t* keys, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int idx = threadIdx.x; idx < (n >> 1); idx += T) {
        const int i = ((idx & ~(j - 1)) << 1) | (idx & (j - 1));
        const int pi = i + j;
        const uint64_t x = keys[i], y = keys[pi];
        const bool up = (i & k) == 0;
        if ((x > y) == up) {
          keys[i] = y;
          keys[pi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Miss rows are read once: stream them past the caches.
__device__ __forceinline__ uint4 load_host16(const uint4* p) { return __ldcs(p); }

// Start pulling a host row into L2 as soon as the miss is known, so the link transfer
// overlaps victim selection; the copy in phase 9 then reads it from L2.
__device__ __forceinline__ void prefetch_row_l2(const uint8_t* p, int bytes, int vec) {
  if (vec == 16) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
  } else {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    for (uintptr_t line = a & ~uintptr_t(127); line < a + (uintptr_t)bytes; line += 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
  }
}

// Copy the m planned rows of every layer: host pool -> device pool (phase 9).
__device__ void copy_rows(const Geometry& g, const Pools& p, const int32_t* psrc, const int32_t* pdst, int m) {
  // p lives in shared memory: the per-layer bases are indexed without a local copy.
  if (g.vec == 16) {
    const int per_row = g.B >> 4;
    const int per_miss = per_row * g.L;
    const int total = m * per_miss;
    for (int base = threadIdx.x; base < total; base += T * kCopyUnroll) {
      uint4 v[kCopyUnroll];
      uint4* dst[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int c = base + u * T;
        dst[u] = nullptr;
        if (c < total) {
          const int j = c / per_miss;
          const int rem = c - j * per_miss;
          const int l = rem / per_row;
          const int q = rem - l * per_row;
          const int32_t d = pdst[j];
          if (d >= 0) {
            dst[u] = reinterpret_cast<uint4*>(p.dev[l] + (size_t)d * g.B) + q;
            const int32_t s = psrc[j];
            v[u] = s >= 0 ? load_host16(reinterpret_cast<const uint4*>(p.host[l] + (size_t)s * g.B) + q)
                          : make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (dst[u]) *dst[u] = v[u];
    }
  } else if (g.vec == 4) {
    const int per_row = g.B >> 2;
    const int per_miss = per_row * g.L;
    const int total = m * per_miss;
    for (int c = threadIdx.x; c < total; c += T) {
      const int j = c / per_miss, rem = c - j * per_miss, l = rem / per_row, q = rem - l * per_row;
      const int32_t d = pdst[j], s = psrc[j];
      if (d < 0) continue;
      uint32_t v = s >= 0 ? reinterpret_cast<const uint32_t*>(p.host[l] + (size_t)s * g.B)[q] : 0u;
      reinterpret_cast<uint32_t*>(p.dev[l] + (size_t)d * g.B)[q] = v;
    }
  } else {
    const int per_miss = g.B * g.L;
    const int total = m * per_miss;
    for (int c = threadIdx.x; c < total; c += T) {
      const int j = c / per_miss, rem = c - j * per_miss, l = rem / g.B, q = rem - l * g.B;
      const int32_t d = pdst[j], s = psrc[j];
      if (d < 0) continue;
      p.dev[l][(size_t)d * g.B + q] = s >= 0 ? p.host[l][(size_t)s * g.B + q] : (uint8_t)0;
    }
  }
}

__device__ __forceinline__ void flush_flags(uint32_t flags, uint32_t* err_word) {
  const uint32_t f = __reduce_or_sync(FULL, flags);
  if ((threadIdx.x & 31) == 0 && f) atomicOr(err_word, f);
}

__global__ void __launch_bounds__(T, 1)
    resolve_kernel(const Geometry g, const Pools* __restrict__ pools, const ResolveArgs a,
                   uint32_t* __restrict__ err_word) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Pools s_pools;
  const Layout lay = make_layout(g);
  uint64_t* s_keys = reinterpret_cast<uint64_t*>(smem + lay.keys);
  int32_t* s_tk = reinterpret_cast<int32_t*>(smem + lay.tk);
  int32_t* s_out = reinterpret_cast<int32_t*>(smem + lay.out);
  int32_t* s_claim = reinterpret_cast<int32_t*>(smem + lay.claim);
  int32_t* s_miss = reinterpret_cast<int32_t*>(smem + lay.miss);
  int32_t* s_vict = reinterpret_cast<int32_t*>(smem + lay.vict);
  int32_t* s_psrc = reinterpret_cast<int32_t*>(smem + lay.psrc);
  int32_t* s_pdst = reinterpret_cast<int32_t*>(smem + lay.pdst);
  int32_t* s_hkey = reinterpret_cast<int32_t*>(smem + lay.hkey);
  int32_t* s_hval = reinterpret_cast<int32_t*>(smem + lay.hval);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem + lay.tok);
  int32_t* s_stamp = reinterpret_cast<int32_t*>(smem + lay.stamp);
  int16_t* s_sent = reinterpret_cast<int16_t*>(smem + lay.sent);
  uint8_t* s_cls = smem + lay.cls;
  uint8_t* s_sflag = smem + lay.sflag;
  int32_t* s_wsum = reinterpret_cast<int32_t*>(smem + lay.wsum);
  int32_t* s_hist = reinterpret_cast<int32_t*>(smem + lay.hist);
  uint32_t* s_sc = reinterpret_cast<uint32_t*>(smem + lay.sc);

  // The eager backup touches only the newest token's rows, which this kernel never reads
  // or writes: let it launch now and run beside the resolve (it orders its own exit).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x;
  const int r = blockIdx.x;
  const int K = g.K, H = g.H;
  const int HS = 1 << g.hash_bits;
  const int32_t S = a.seq_lens[r];
  const int32_t* tk_g = a.top_k_tokens + (size_t)r * K;
  int32_t* out_g = a.out_rows + (size_t)r * K;
  const int32_t* dbl = a.device_buffer_locs + (size_t)r * (H + 1);
  uint32_t flags = 0;

  if (S < 0 || S > g.max_context) {
    for (int i = tid; i < K; i += T) out_g[i] = -1;
    if (tid == 0) {
      if (a.miss_counts) a.miss_counts[r] = 0;
      atomicOr(err_word, HS_FLAG_SEQLEN);
    }
    return;
  }

  // ---- phase 1: top-k row, validity, hash of the valid tokens
  for (int h = tid; h < HS; h += T) {
    s_hkey[h] = -1;
    s_hval[h] = INF;
  }
  if (tid == 0) {
    s_sc[SC_LO] = 0xffffffffu;
    s_sc[SC_HI] = 0u;
  }
  if (tid < (int)(sizeof(Pools) / sizeof(uint64_t)))
    reinterpret_cast<uint64_t*>(&s_pools)[tid] = reinterpret_cast<const uint64_t*>(pools)[tid];
  __syncthreads();
  for (int i = tid; i < K; i += T) {
    const int32_t t = tk_g[i];
    uint8_t c;
    if (t < 0) {
      c = C_PAD;
    } else if (t >= S) {
      c = C_BAD;
      flags |= HS_FLAG_TOKEN;
    } else {
      c = C_VALID;
      hash_insert(s_hkey, s_hval, g.hash_bits, t, i);
    }
    s_tk[i] = t;
    s_cls[i] = c;
    s_out[i] = -1;
    s_claim[i] = INF;
  }
  __syncthreads();

  // ---- phase 2: classify (resident, fast path, newest, hot lookup)
  const bool fast = S <= H;
  for (int i = tid; i < K; i += T) {
    if (s_cls[i] != C_VALID) continue;
    const int32_t t = s_tk[i];
    const int h = hash_find(s_hkey, g.hash_bits, t);
    if (s_hval[h] != i) {
      s_cls[i] = C_DUP;
      flags |= HS_FLAG_DUP;
      continue;
    }
    int32_t page = -1;
    if (a.resident_pages) page = a.resident_pages[(size_t)r * g.max_pages + t / g.page_size];
    if (page >= 0) {
      s_out[i] = checked_row((int64_t)page * g.page_size + t % g.page_size, g.device_rows, flags);
      s_cls[i] = C_RES;
    } else if (fast) {
      s_out[i] = checked_row(dbl[t], g.device_rows, flags);
      s_cls[i] = C_FAST;
    } else if (t == S - 1) {
      s_out[i] = checked_row(dbl[H], g.device_rows, flags);
      s_cls[i] = C_NEWEST;
    } else {
      s_cls[i] = C_LOOKUP;
    }
  }
  __syncthreads();

  if (fast) {
    for (int i = tid; i < K; i += T) out_g[i] = s_out[i];
    if (tid == 0) {
      if (S >= 1) a.device_buffer_tokens[(size_t)r * H + (S - 1)] = S - 1;
      if (a.miss_counts) a.miss_counts[r] = 0;
    }
    flush_flags(flags, err_word);
    return;
  }

  // ---- phase 3: slot state, tripwires, membership probe
  const int32_t clock = a.lru_clock[r] + 1;
  int32_t* tok_g = a.device_buffer_tokens + (size_t)r * H;
  int32_t* st_g = a.lru_slots + (size_t)r * H;
  for (int s = tid; s < H; s += T) {
    int32_t tkn = tok_g[s];
    int32_t st = st_g[s];
    uint8_t f = 0;
    if (st < 0 || st > clock - 1 || tkn < -1 || tkn >= S - 1) {
      tkn = -1;
      st = 0;
      f = SF_DIRTY;
      flags |= HS_FLAG_STATE;
    }
    int32_t ent = -1;
    if (tkn >= 0) {
      const int h = hash_find(s_hkey, g.hash_bits, tkn);
      if (h >= 0) {
        const int32_t i = s_hval[h];
        if (s_cls[i] == C_LOOKUP) {
          ent = i;
          atomicMin(&s_claim[i], s);
        }
      }
    }
    s_tok[s] = tkn;
    s_stamp[s] = st;
    s_sflag[s] = f;
    s_sent[s] = (int16_t)ent;
  }
  __syncthreads();

  // ---- phase 4: hits refresh their stamp
  for (int s = tid; s < H; s += T) {
    const int32_t i = s_sent[s];
    if (i < 0) continue;
    if (s_claim[i] == s) {
      s_stamp[s] = clock;
      s_sflag[s] |= SF_USED | SF_DIRTY;
      s_out[i] = checked_row(dbl[s], g.device_rows, flags);
    } else {
      flags |= HS_FLAG_STATE;  // a second slot holds the same token
    }
  }
  __syncthreads();

  // ---- phase 5: compact misses (top-k order) and free slots (slot order) in one scan
  const int ept = (K + T - 1) / T;
  const int spt = (H + T - 1) / T;
  const int i0 = min(K, tid * ept), i1 = min(K, i0 + ept);
  const int s0 = min(H, tid * spt), s1 = min(H, s0 + spt);
  int nmiss = 0, nfree = 0;
  for (int i = i0; i < i1; ++i) nmiss += (s_cls[i] == C_LOOKUP && s_claim[i] == INF);
  for (int s = s0; s < s1; ++s) nfree += (s_tok[s] == -1);
  int packed_total;
  const int packed = block_excl_scan((nmiss << 16) | nfree, s_wsum, &packed_total);
  const int m = packed_total >> 16;
  const int F = packed_total & 0xffff;
  {
    int pos = packed >> 16;
    for (int i = i0; i < i1; ++i)
      if (s_cls[i] == C_LOOKUP && s_claim[i] == INF) {
        const int32_t hr = a.host_cache_locs[(size_t)r * g.max_context + s_tk[i]];
        const bool ok = hr >= 0 && (int64_t)hr < g.host_rows;
        s_psrc[pos] = ok ? hr : -1;
        if (ok)
          for (int l = 0; l < g.L; ++l) prefetch_row_l2(s_pools.host[l] + (size_t)hr * g.B, g.B, g.vec);
        s_miss[pos++] = i;
      }
    pos = packed & 0xffff;
    for (int s = s0; s < s1; ++s)
      if (s_tok[s] == -1) {
        if (pos < m) s_vict[pos] = s;
        ++pos;
      }
  }
  const int take_free = min(m, F);
  const int m2 = m - take_free;

  // ---- phase 6: the m2 oldest occupied, un-hit slots, ordered by (stamp, slot)
  if (m2 > 0) {
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int s = tid; s < H; s += T)
      if (s_tok[s] >= 0 && !(s_sflag[s] & SF_USED)) {
        lo = min(lo, (uint32_t)s_stamp[s]);
        hi = max(hi, (uint32_t)s_stamp[s]);
      }
    lo = __reduce_min_sync(FULL, lo);
    hi = __reduce_max_sync(FULL, hi);
    if ((tid & 31) == 0) {
      atomicMin(&s_sc[SC_LO], lo);
      atomicMax(&s_sc[SC_HI], hi);
    }
    __syncthreads();
    const uint32_t base = s_sc[SC_LO];
    const uint32_t maxd = s_sc[SC_HI] - base;
    const int nbits = maxd ? 32 - __clz(maxd) : 0;
    const int passes = (nbits + 7) >> 3;
    uint32_t prefix = 0;
    int rank = m2;  // 1-based rank of the last victim among the candidates
    for (int pz = passes - 1; pz >= 0; --pz) {
      const int shift = pz * 8;
      if (tid < 256) s_hist[tid] = 0;
      __syncthreads();
      for (int s = tid; s < H; s += T) {
        if (s_tok[s] < 0 || (s_sflag[s] & SF_USED)) continue;
        const uint32_t d = (uint32_t)s_stamp[s] - base;
        const bool match = (shift + 8 >= 32) || ((d >> (shift + 8)) == (prefix >> (shift + 8)));
        if (match) atomicAdd(&s_hist[(d >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid < 32) {
        int loc[8];
        int sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          loc[b] = s_hist[tid * 8 + b];
          sum += loc[b];
        }
        const int incl = warp_incl_scan(sum);
        const unsigned ball = __ballot_sync(FULL, incl >= rank);
        const int first = __ffs(ball) - 1;
        if (tid == first) {
          int cum = incl - sum;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (cum + loc[b] >= rank) {
              s_sc[SC_DIGIT] = (uint32_t)(tid * 8 + b);
              s_sc[SC_RANK] = (uint32_t)(rank - cum);
              break;
            }
            cum += loc[b];
          }
        }
      }
      __syncthreads();
      prefix |= s_sc[SC_DIGIT] << shift;
      rank = (int)s_sc[SC_RANK];
      __syncthreads();
    }
    const uint32_t thr = prefix;    // stamp - base of the last victim
    const int need_eq = rank;       // victims taken among the candidates at the threshold
    const int n_lt = m2 - need_eq;  // candidates strictly below the threshold
    int c_lt = 0, c_eq = 0;
    for (int s = s0; s < s1; ++s) {
      if (s_tok[s] < 0 || (s_sflag[s] & SF_USED)) continue;
      const uint32_t d = (uint32_t)s_stamp[s] - base;
      c_lt += d < thr;
      c_eq += d == thr;
    }
    int tot2;
    const int pk = block_excl_scan((c_lt << 16) | c_eq, s_wsum, &tot2);
    int p_lt = pk >> 16, p_eq = pk & 0xffff;
    for (int s = s0; s < s1; ++s) {
      if (s_tok[s] < 0 || (s_sflag[s] & SF_USED)) continue;
      const uint32_t d = (uint32_t)s_stamp[s] - base;
      if (d < thr) {
        s_keys[p_lt++] = ((uint64_t)d << 32) | (uint32_t)s;
      } else if (d == thr) {
        if (p_eq < need_eq) s_keys[n_lt + p_eq] = ((uint64_t)d << 32) | (uint32_t)s;
        ++p_eq;
      }
    }
    int n = 1;
    while (n < m2) n <<= 1;
    for (int i = m2 + tid; i < n; i += T) s_keys[i] = ~0ull;
    __syncthreads();
    bitonic_sort(s_keys, n);
    for (int j = tid; j < m2; j += T) s_vict[take_free + j] = (int32_t)(s_keys[j] & 0xffffffffu);
  }
  __syncthreads();

  // ---- phase 7: miss j takes victim j
  for (int j = tid; j < m; j += T) {
    const int32_t v = s_vict[j];
    const int32_t i = s_miss[j];
    const int32_t t = s_tk[i];
    if ((uint32_t)v >= (uint32_t)H) {  // unreachable by construction; never index with it
      flags |= HS_FLAG_STATE;
      s_pdst[j] = -1;
      continue;
    }
    s_tok[v] = t;
    s_stamp[v] = clock;
    s_sflag[v] |= SF_DIRTY;
    const int32_t d = checked_row(dbl[v], g.device_rows, flags);
    s_out[i] = d;
    if (d >= 0 && s_psrc[j] < 0) flags |= HS_FLAG_HOSTROW;  // destination is zero-filled
    s_pdst[j] = d;
  }
  __syncthreads();

  // ---- phase 8: write back changed slots, the row table and the clock
  for (int s = tid; s < H; s += T)
    if (s_sflag[s] & SF_DIRTY) {
      tok_g[s] = s_tok[s];
      st_g[s] = s_stamp[s];
    }
  for (int i = tid; i < K; i += T) out_g[i] = s_out[i];
  if (tid == 0) {
    a.lru_clock[r] = clock;
    if (a.miss_counts) a.miss_counts[r] = m;
  }

  // ---- phase 9: miss rows, all layers, from pinned host memory
  copy_rows(g, s_pools, s_psrc, s_pdst, m);
  flush_flags(flags, err_word);
}

}  // namespace

size_t resolve_smem_bytes(const Geometry& g) { return make_layout(g).total; }

// Raise the kernel's dynamic shared-memory ceiling to the most the device allows beside
// the kernel's static shared memory (not to this geometry's size): the attribute is per
// function and device, so a smaller value set for one handle would make launches of a
// larger, earlier handle fail.
cudaError_t resolve_prepare(const Geometry& g) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, resolve_kernel);
  if (e != cudaSuccess) return e;
  const int max_dynamic = optin - (int)fa.sharedSizeBytes;
  if (resolve_smem_bytes(g) > (size_t)max_dynamic) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic);
}

cudaError_t launch_resolve(const Geometry& g, const Pools* pools, const ResolveArgs& a, int32_t num_requests,
                           uint32_t* err_word, cudaStream_t stream) {
  resolve_kernel<<<num_requests, T, resolve_smem_bytes(g), stream>>>(g, pools, a, err_word);
  return cudaGetLastError();
}

}  // namespace hs
