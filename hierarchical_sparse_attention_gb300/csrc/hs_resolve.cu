// Fused decode-step resolver / swap-in: one thread block cluster per request.
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
//     from the cold end; out-of-range state downgraded to a re-miss; wide vector copies
//     that zero the destination when the source row is out of range), 7.3 (flat physical
//     row IDs) and 7.4 (layers sharing the indexer reuse the same slot plan).
//   "Hierarchical Sparse Attention" (Alibaba Tair), 2.4.3 "LRU Diff Kernel" (evict only
//     when the buffer is full, coldest first).
//
// The step is latency-bound (a few MB over the host link, a few tens of KB of state per
// request), so the kernel is arranged to start the host-link transfer as early as
// possible and to hide the rest of the bookkeeping behind it. Each request gets a thread
// block cluster of 1024-thread CTAs: CTA 0 resolves, and up to three copy CTAs on other
// SMs move the miss rows.
// Phases of the resolve CTA (request r):
//   0  cp.async the top-k row, the slot map, the stamps and the slot->row table into
//      shared memory while the hash table is cleared
//   1  reject padding / out-of-range tokens; hash the valid ones (open addressing,
//      Knuth multiplicative; a repeated token keeps its first index) and classify each
//      entry: resident row, fast-path identity, reserved newest row, or hot lookup
//   3  reset corrupt slots; probe each slot's token; the first slot to claim a looked-up
//      token takes the hit (stamp = clock) and the other candidates enter an age
//      histogram. Two holders of one token (corrupt state only) are settled afterwards in
//      favour of the lowest slot
//   4  hits output their slot's row and tell the entry's copy CTA the slot
//   5  one packed block scan orders the misses (top-k order) and the free slots (slot order)
//   6  if misses outnumber free slots: the stamp threshold among occupied, un-hit slots
//      comes from the age histogram (exact radix select when the histogram cannot decide);
//      exactly the needed victims are gathered and ordered by (stamp, slot)
//   7  pair miss j with victim j: update the map and the residency bitmap; publish each
//      miss's device row to its copy CTA (distributed shared memory, then a release-arrive
//      on that copy CTA's publication mbarrier)
//   8  write back the changed slots, the row table and the clock
//   9  copy the misses no copy CTA took (only when the geometry runs without copy CTAs)
//      straight from host memory
// A copy CTA owns a slice of the top-k row. At kernel start it predicts its slice's
// misses from the residency bitmap (a looked-up token whose bit is clear), looks
// up their host rows and pulls them into shared memory while the resolve CTA does the
// exact work; once the resolve CTA has published the outcomes (its own mbarrier, so it does
// not wait for the other copy CTAs) it stores the staged rows of exact misses to their device
// rows and copies any unpredicted miss straight from host memory.
#include <climits>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int T = kResolveThreads;
constexpr int NW = T / 32;
constexpr unsigned FULL = 0xffffffffu;
constexpr int32_t INF = 0x7fffffff;
constexpr int kCopyUnroll = 4;

enum : uint8_t { C_PAD = 0, C_BAD, C_DUP, C_RES, C_FAST, C_NEWEST, C_LOOKUP };
constexpr uint8_t C_BADROW = 0x80;  // with C_RES / C_FAST / C_NEWEST: its row is out of range
enum : uint8_t { SF_USED = 1, SF_DIRTY = 2 };
enum { SC_LO = 0, SC_HI, SC_DIGIT, SC_RANK, SC_CONFLICT, SC_DIRECT, SC_GATHER, SC_COUNT };
// Victim phase: gathering every candidate at or below the threshold stamp in one pass saves
// a counting pass (about a slot pass of work) but ranks n_le keys instead of m2; ranking is
// n^2 / T compares per thread, so the one pass is taken while n_le^2 - m2^2 stays below this.
constexpr int kOnePassSlack = 64 * 1024;

// Shared-memory carve-up of the resolve CTA; identical arithmetic on host (size) and device
// (pointers). The top-k hash (1 << hash_bits buckets of one 64-bit word: token << 32 |
// top-k index; at least 2 * sort_cap of them) is dead after phase 3, so it holds the
// victim keys of phase 6 and the copy plan of phases 7-9. The slot->row table gets three
// spare words so it can start at its global row's 16-byte phase (whole-vector loads).
struct Layout {
  size_t hash, keys, psrc, pdst, tk, out, claim, miss, vict, tok, stamp, dbl, cls, sflag, wsum, hist, sc, total;
};

// Shared-memory carve-up of a copy CTA q (rank 1..C). It owns top-k entries
// [(q-1) * per, q * per) with per = ceil(K / C): their outcomes, published by the resolve CTA
// (res: device row of a miss, -2 - slot for a hit, -1 otherwise), its slice of the top-k row,
// per entry the staging index and host row, the lists of staged and of directly copied
// entries, two counters, the request's residency bitmap row (when it is staged), and the
// staging area (copy_cap entries x L rows of B bytes).
struct CopyLayout {
  size_t res, tk, stg, hrow, list, dlist, cnt, bits, stage, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline Layout make_layout(const Geometry& g) {
  Layout l;
  size_t o = 0;
  const size_t K = (size_t)g.K, H = (size_t)g.H, HS = (size_t)1 << g.hash_bits;
  l.hash = o; o = align16(o + 8 * HS);
  l.keys = l.hash;
  l.psrc = l.hash + sizeof(uint64_t) * (size_t)g.sort_cap;
  l.pdst = l.psrc + 4 * K;
  l.tk = o; o = align16(o + 4 * K);
  l.out = o; o = align16(o + 4 * K);
  l.claim = o; o = align16(o + 4 * K);
  l.miss = o; o = align16(o + 4 * K);
  l.vict = o; o = align16(o + 4 * K);
  l.tok = o; o = align16(o + 4 * H);
  l.stamp = o; o = align16(o + 4 * H);
  l.dbl = o; o = align16(o + (g.dbl_smem ? 4 * (H + 1 + 3) : 0));
  l.cls = o; o = align16(o + K);
  l.sflag = o; o = align16(o + H);
  l.wsum = o; o = align16(o + 4 * (NW + 1));
  l.hist = o; o = align16(o + 4 * 256);
  l.sc = o; o = align16(o + 4 * SC_COUNT);
  l.total = o;
  return l;
}

__host__ __device__ inline int copy_slice(const Geometry& g) {
  return g.copy_ctas > 0 ? (g.K + g.copy_ctas - 1) / g.copy_ctas : 0;
}

__host__ __device__ inline CopyLayout make_copy_layout(const Geometry& g) {
  CopyLayout l;
  size_t o = 0;
  const size_t per = (size_t)copy_slice(g), cap = (size_t)g.copy_cap;
  l.res = o; o = align16(o + 4 * per);
  l.tk = o; o = align16(o + 4 * per);
  l.stg = o; o = align16(o + 2 * per);
  l.hrow = o; o = align16(o + 4 * per);
  l.list = o; o = align16(o + 2 * cap);
  l.dlist = o; o = align16(o + 2 * per);
  l.cnt = o; o = align16(o + 16);
  l.bits = o; o = align16(o + (g.bits_smem ? 4 * (size_t)g.bit_words : 0));
  l.stage = o; o = align16(o + cap * (size_t)g.L * (size_t)g.B);
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

__device__ __forceinline__ uint32_t hash_slot(int32_t t, int bits) {
  return ((uint32_t)t * 2654435761u) >> (32 - bits);
}

constexpr uint64_t kEmpty = ~0ull;  // bucket never written (tokens are < 2^31)

// Insert token t for top-k index i; a repeated token keeps the smallest index (same key
// bits, so the 64-bit minimum picks the smaller index).
__device__ __forceinline__ void hash_insert(unsigned long long* tab, int bits, int32_t t, int32_t i) {
  const uint32_t mask = (1u << bits) - 1;
  const unsigned long long w = ((unsigned long long)(uint32_t)t << 32) | (uint32_t)i;
  uint32_t h = hash_slot(t, bits);
  for (;;) {  // ends: the table is at most a quarter full
    const unsigned long long prev = atomicCAS(&tab[h], kEmpty, w);
    if (prev == kEmpty) return;
    if ((uint32_t)(prev >> 32) == (uint32_t)t) {
      atomicMin(&tab[h], w);
      return;
    }
    h = (h + 1) & mask;
  }
}

// Top-k index recorded for token t, or -1.
__device__ __forceinline__ int32_t hash_find(const unsigned long long* tab, int bits, int32_t t) {
  const uint32_t mask = (1u << bits) - 1;
  uint32_t h = hash_slot(t, bits);
  for (;;) {  // ends: at least three quarters of the table are empty
    const unsigned long long w = tab[h];
    if (w == kEmpty) return -1;
    if ((uint32_t)(w >> 32) == (uint32_t)t) return (int32_t)(uint32_t)w;
    h = (h + 1) & mask;
  }
}

// Top-k index whose token a slot holds, if that entry is a hot lookup; else -1.
__device__ __forceinline__ int32_t lookup_entry(const unsigned long long* tab, const uint8_t* cls, int bits,
                                                int32_t tkn) {
  if (tkn < 0) return -1;
  const int32_t i = hash_find(tab, bits, tkn);
  return (i >= 0 && cls[i] == C_LOOKUP) ? i : -1;
}

__device__ __forceinline__ int32_t checked_row(int64_t row, int64_t rows, uint32_t& flags) {
  if (row < 0 || row >= rows) {
    flags |= HS_FLAG_DEVROW;
    return -1;
  }
  return (int32_t)row;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Asynchronous copies global -> shared (completed by cp_async_wait_all + a barrier).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// Queue an asynchronous copy of n int32 from global src to shared dst: 16-byte pieces over
// the part where both addresses are 16-byte aligned (same phase), 4-byte pieces elsewhere.
__device__ __forceinline__ void cp_async_words(int32_t* dst, const int32_t* src, int n) {
  const int head = ((uintptr_t)src & 15) == ((uintptr_t)smem_addr(dst) & 15)
                       ? min(n, (int)((16 - ((uintptr_t)src & 15)) & 15) / 4)
                       : n;
  const int body = (n - head) & ~3;
  for (int i = threadIdx.x; i < head; i += T) cp_async4(dst + i, src + i);
  for (int i = threadIdx.x; i < body / 4; i += T) cp_async16(dst + head + 4 * i, src + head + 4 * i);
  for (int i = head + body + threadIdx.x; i < n; i += T) cp_async4(dst + i, src + i);
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Thread block cluster primitives: this CTA's rank, a store into another CTA's shared
// memory (distributed shared memory), and the split cluster barrier. A release-arrive
// publishes this thread's earlier stores (local or remote) to threads that acquire-wait.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void st_remote(const void* local_addr, uint32_t rank, int32_t v) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_addr(local_addr)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(raddr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

constexpr int kPublishTryNs = 20000, kPublishTries = 10000;  // about 200 ms of tries at most

// The resolve CTA tells copy CTA `rank` that this step's outcomes are in its shared memory:
// an arrival (release, cluster scope) on the copy CTA's `pub` mbarrier. The calling thread
// comes after a CTA barrier that follows every outcome store of the CTA.
__device__ __forceinline__ void publish_to(uint64_t* pub, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_addr(pub)), "r"(rank));
  asm volatile("fence.acq_rel.cluster;\n\tmbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr)
               : "memory");
}
// A copy CTA's wait for phase `parity` of its `pub` mbarrier, by one thread (the others wait at
// a CTA barrier). Each try sleeps until the phase completes or kPublishTryNs pass; the bound is
// a count of tries, not a clock, because the waiting thread's own host loads may still be in
// flight (a first access to host pages can stall far longer than the resolve CTA's work).
// False if the bound ran out.
__device__ __forceinline__ bool publish_wait(uint64_t* pub, uint32_t parity) {
  for (int tries = 0; tries < kPublishTries; ++tries) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(pub)), "r"(parity), "n"(kPublishTryNs)
        : "memory");
    if (done) return true;
  }
  return false;
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

// The arguments that differ between the verify steps one launch runs (ResolveArgs.spec_steps).
struct StepArgs {
  int32_t spec_q;
  const int32_t* top_k_tokens;
  int32_t* out_rows;
  int32_t* miss_counts;
  int32_t* plan_tok;
  int32_t* plan_dst;
  int32_t* plan_cnt;
};
__device__ __forceinline__ StepArgs step_args(const ResolveArgs& a, int step) {
  if (step < 0)
    return StepArgs{a.spec_q, a.top_k_tokens, a.out_rows, a.miss_counts, a.plan_tok, a.plan_dst, a.plan_cnt};
  const size_t q = (size_t)step;
  return StepArgs{step,
                  a.top_k_tokens + q * a.step_rk,
                  a.out_rows + q * a.step_rk,
                  a.miss_counts ? a.miss_counts + q * a.step_r : nullptr,
                  a.plan_tok ? a.plan_tok + q * a.step_plan : nullptr,
                  a.plan_dst ? a.plan_dst + q * a.step_plan : nullptr,
                  a.plan_cnt ? a.plan_cnt + q * a.step_plan : nullptr};
}

// Miss rows are read once: stream them past the caches.
__device__ __forceinline__ uint4 load_host16(const uint4* p) { return __ldcs(p); }

// Phase 9 of the resolve CTA: copy every planned miss row of layers [0, L) straight from
// host memory to its victim's device row (psrc < 0: zero-fill; pdst < 0: nothing to do,
// e.g. a row a copy CTA moves).
__device__ void copy_rows(const Geometry& g, const Pools& p, const int32_t* psrc, const int32_t* pdst, int m,
                          int L) {
  if (g.vec == 16) {
    const int per_row = g.B >> 4;
    const int per_miss = per_row * L;
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
            v[u] = s >= 0 ? load_host16(reinterpret_cast<const uint4*>(p.host[l] + (size_t)s * g.host_stride) + q)
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
    const int per_miss = per_row * L;
    const int total = m * per_miss;
    for (int c = threadIdx.x; c < total; c += T) {
      const int j = c / per_miss, rem = c - j * per_miss, l = rem / per_row, q = rem - l * per_row;
      const int32_t d = pdst[j], s = psrc[j];
      if (d < 0) continue;
      uint32_t v = s >= 0 ? reinterpret_cast<const uint32_t*>(p.host[l] + (size_t)s * g.host_stride)[q] : 0u;
      reinterpret_cast<uint32_t*>(p.dev[l] + (size_t)d * g.B)[q] = v;
    }
  } else {
    const int per_miss = g.B * L;
    const int total = m * per_miss;
    for (int c = threadIdx.x; c < total; c += T) {
      const int j = c / per_miss, rem = c - j * per_miss, l = rem / g.B, q = rem - l * g.B;
      const int32_t d = pdst[j], s = psrc[j];
      if (d < 0) continue;
      p.dev[l][(size_t)d * g.B + q] = s >= 0 ? p.host[l][(size_t)s * g.host_stride + q] : (uint8_t)0;
    }
  }
}

// Copy CTA q of request r (cluster rank q >= 1; its shared outcome table was cleared to -1
// and its counters to 0 before the cluster's first barrier).
// With a residency bitmap and a request past the fast path, it first predicts which of its
// entries miss: a hot lookup whose bit is clear (the bits are exact while the caller leaves
// the state to the kernels; a stale set bit only turns a miss into an unpredicted one, and
// the miss's new slot rewrites it). The bitmap row comes into shared memory with the top-k
// slice when it is small enough, so the prediction costs no memory round trip of its own.
// It looks up the predicted
// misses' host rows and reads those rows into shared memory right away (16-byte loads,
// kCopyUnroll in flight per thread), so the host-link transfer runs while the resolve CTA
// does the exact work. The resolve CTA then publishes the exact outcome of every entry.
// Exact misses store their staged row; misses that were not staged (a stale bit, no
// room) are copied straight from host memory. A predicted miss that was a hit sets the
// token's bit again.
__device__ void copy_cta(const Geometry& g, const Pools& p, const ResolveArgs& a, const StepArgs& sa, int r, int q,
                         int32_t seq_r, unsigned char* smem, uint64_t* pub, uint32_t pub_parity, uint32_t* err_word) {
  const CopyLayout cl = make_copy_layout(g);
  const int32_t* c_res = reinterpret_cast<const int32_t*>(smem + cl.res);
  int32_t* c_tk = reinterpret_cast<int32_t*>(smem + cl.tk);
  int16_t* c_stg = reinterpret_cast<int16_t*>(smem + cl.stg);
  int32_t* c_hrow = reinterpret_cast<int32_t*>(smem + cl.hrow);
  int16_t* c_list = reinterpret_cast<int16_t*>(smem + cl.list);
  int16_t* c_dlist = reinterpret_cast<int16_t*>(smem + cl.dlist);
  uint32_t* c_cnt = reinterpret_cast<uint32_t*>(smem + cl.cnt);
  uint8_t* c_stage = smem + cl.stage;
  const int tid = threadIdx.x;
  const int per = copy_slice(g);
  const int e0 = (q - 1) * per;
  const int ne = max(0, min(g.K, e0 + per) - e0);
  const bool may_predict = a.hint != nullptr && a.copy_layers > 0;
  uint32_t* bits_g = a.hint ? a.hint + (size_t)r * g.bit_words : nullptr;  // residency bitmap row
  const uint32_t* bits = g.bits_smem ? reinterpret_cast<const uint32_t*>(smem + cl.bits) : bits_g;
  const int32_t* hcl_row = a.host_cache_locs + (size_t)r * g.max_context;
  const int32_t* tk_g = sa.top_k_tokens + (size_t)r * g.K + e0;
  const int per_row = g.B >> 4;
  const int per_miss = per_row * a.copy_layers;  // the leader layers this call copies
  uint32_t flags = 0;
  int staged = 0;

  // The prediction's inputs (the bitmap row, the top-k slice) are requested before the
  // request's length is known, so their latency overlaps that of seq_lens.
  if (may_predict) {
    if (g.bits_smem)
      cp_async_words(reinterpret_cast<int32_t*>(smem + cl.bits), reinterpret_cast<const int32_t*>(bits_g),
                     g.bit_words);
    cp_async_commit();
    for (int e = tid; e < ne; e += T) c_tk[e] = tk_g[e];  // plain loads: the row may be host memory
  }
  const int32_t S = sa.spec_q < 0 ? seq_r : seq_r + sa.spec_q + 1;
  const int32_t base = sa.spec_q < 0 ? S - 1 : seq_r;  // first position new to the cache
  const bool predict = may_predict && S > g.H && S <= g.max_context;
  if (predict) {
    cp_async_wait_all();
    __syncthreads();
    for (int e = tid; e < ne; e += T) {
      const int32_t t = c_tk[e];
      int16_t st = -1;  // -1: not predicted to miss; -2: predicted, no staging room
      // The host-row lookup waits for the prediction: issuing it for every entry up front
      // saves a round trip but adds one HBM request per top-k entry at kernel start, which
      // delays the whole cluster's loads more than it saves (measured).
      if (t >= 0 && t < base &&
          !(a.resident_pages && a.resident_pages[(size_t)r * g.max_pages + t / g.page_size] >= 0)) {
        if (!((bits[t >> 5] >> (t & 31)) & 1u)) {
          const uint32_t k = atomicAdd(&c_cnt[0], 1u);
          if ((int)k < g.copy_cap) {
            st = (int16_t)k;
            c_list[k] = (int16_t)e;
            const int32_t hr = hcl_row[t];
            c_hrow[e] = (hr >= 0 && (int64_t)hr < g.host_rows) ? hr : -1;
          } else {
            st = -2;
          }
        }
      }
      c_stg[e] = st;
    }
    __syncthreads();
    staged = min((int)c_cnt[0], g.copy_cap);
    const int total = staged * per_miss;
    for (int base = tid; base < total; base += T * kCopyUnroll) {
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int c = base + u * T;
        if (c < total) {
          const int k = c / per_miss, rem = c - k * per_miss, l = rem / per_row, qq = rem - l * per_row;
          const int32_t hr = c_hrow[c_list[k]];
          v[u] = hr >= 0 ? load_host16(reinterpret_cast<const uint4*>(p.host[l] + (size_t)hr * g.host_stride) + qq)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int c = base + u * T;
        if (c < total) reinterpret_cast<uint4*>(c_stage)[c] = v[u];  // entry k, layer l at (k*L + l)*B
      }
    }
  }
  cluster_wait();  // phase A (arrived at kernel start)
  cp_async_wait_all();  // the pools table, when no prediction waited for it
  // The resolve CTA's outcomes for this step: each copy CTA goes on as soon as they are in and
  // its own staged rows have landed, not when its sibling copy CTAs are done too.
  if (!__syncthreads_and(tid != 0 || publish_wait(pub, pub_parity))) {
    if (tid == 0) atomicOr(err_word, HS_FLAG_TIMEOUT);  // no outcomes: this CTA copies nothing
    return;
  }

  // staged entries that are exact misses
  for (int c = tid; c < staged * per_miss; c += T) {
    const int k = c / per_miss, rem = c - k * per_miss, l = rem / per_row, qq = rem - l * per_row;
    const int e = c_list[k];
    const int32_t d = c_res[e];
    if (d >= 0)
      reinterpret_cast<uint4*>(p.dev[l] + (size_t)d * g.B)[qq] =
          c_hrow[e] >= 0 ? reinterpret_cast<const uint4*>(c_stage)[c] : make_uint4(0u, 0u, 0u, 0u);
  }
  // the rest: bitmap repairs, and the list of exact misses to copy straight from host
  for (int e = tid; e < ne; e += T) {
    const int32_t d = c_res[e];
    const int st = predict ? c_stg[e] : -1;
    if (d >= 0) {
      if (st >= 0) {
        if (c_hrow[e] < 0) flags |= HS_FLAG_HOSTROW;  // destination was zero-filled
      } else {
        const int32_t t = predict ? c_tk[e] : tk_g[e];
        const int32_t hr = hcl_row[t];
        const bool ok = hr >= 0 && (int64_t)hr < g.host_rows;
        if (!ok) flags |= HS_FLAG_HOSTROW;
        c_hrow[e] = ok ? hr : -1;
        c_dlist[atomicAdd(&c_cnt[1], 1u)] = (int16_t)e;
      }
    } else if (d <= -2 && st != -1) {
      const int32_t t = c_tk[e];  // predicted a miss, was a hit: the token is resident
      atomicOr(&bits_g[t >> 5], 1u << (t & 31));
    }
  }
  __syncthreads();
  const int nd = (int)c_cnt[1];
  const int dtotal = nd * per_miss;
  for (int base = tid; base < dtotal; base += T * kCopyUnroll) {
    uint4 v[kCopyUnroll];
    uint4* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int c = base + u * T;
      dst[u] = nullptr;
      if (c < dtotal) {
        const int j = c / per_miss, rem = c - j * per_miss, l = rem / per_row, qq = rem - l * per_row;
        const int e = c_dlist[j];
        const int32_t hr = c_hrow[e];
        dst[u] = reinterpret_cast<uint4*>(p.dev[l] + (size_t)c_res[e] * g.B) + qq;
        v[u] = hr >= 0 ? load_host16(reinterpret_cast<const uint4*>(p.host[l] + (size_t)hr * g.host_stride) + qq)
                       : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
  const uint32_t f = __reduce_or_sync(FULL, flags);
  if ((threadIdx.x & 31) == 0 && f) atomicOr(err_word, f);
}

// Rank n <= T distinct keys (stamp << 32 | slot) and write the slot of each key whose rank
// (number of smaller keys) is below m to out[rank]. P threads share a key (P a power of two
// with n * P <= T, at most a warp), each counting over every P-th key; the group sums with
// shuffles. Lanes of one warp read the same few keys, so the loads are broadcasts.
__device__ __forceinline__ void rank_keys(const uint64_t* keys, int n, int m, int32_t* out) {
  int P = 1;
  while (P < 32 && n * (P * 2) <= T) P <<= 1;
  const int key = threadIdx.x / P, part = threadIdx.x & (P - 1);
  const uint64_t kj = key < n ? keys[key] : 0ull;
  int rk = 0;
#pragma unroll 4
  for (int u = part; u < n; u += P) rk += (int)(keys[u] < kj);
  for (int o = P >> 1; o > 0; o >>= 1) rk += __shfl_xor_sync(FULL, rk, o);
  if (key < n && part == 0 && rk < m) out[rk] = (int32_t)(kj & 0xffffffffu);
}

__device__ __forceinline__ void flush_flags(uint32_t flags, uint32_t* err_word) {
  const uint32_t f = __reduce_or_sync(FULL, flags);
  if ((threadIdx.x & 31) == 0 && f) atomicOr(err_word, f);
}

// What a resolve CTA that leaves a step early (a skipped request, the fast path) still owes
// its copy CTAs: cluster barrier phase A, and the (empty) publication of the outcomes.
__device__ __forceinline__ void finish_phases(int C, uint64_t* pub) {
  if (C > 0) {
    cluster_wait();  // phase A: the copy CTAs' publication barriers are initialised
    if (threadIdx.x < C) publish_to(pub, threadIdx.x + 1);
  }
}

// The resolve CTA of request r for one step (phases 0-9 below). Every exit completes cluster
// barrier phase A and publishes the outcomes (none on an early exit) to each copy CTA.
__device__ __forceinline__ void resolve_cta(const Geometry& g, const Pools& s_pools, const ResolveArgs& a,
                                            const StepArgs& sa, uint32_t* __restrict__ err_word, unsigned char* smem,
                                            uint64_t* pub, int r, int32_t seq_r) {
  const int tid = threadIdx.x;
  const int C = g.copy_ctas;
  const Layout lay = make_layout(g);
  uint64_t* s_keys = reinterpret_cast<uint64_t*>(smem + lay.keys);
  int32_t* s_tk = reinterpret_cast<int32_t*>(smem + lay.tk);
  int32_t* s_out = reinterpret_cast<int32_t*>(smem + lay.out);
  int32_t* s_claim = reinterpret_cast<int32_t*>(smem + lay.claim);
  int32_t* s_miss = reinterpret_cast<int32_t*>(smem + lay.miss);
  int32_t* s_vict = reinterpret_cast<int32_t*>(smem + lay.vict);
  int32_t* s_psrc = reinterpret_cast<int32_t*>(smem + lay.psrc);
  int32_t* s_pdst = reinterpret_cast<int32_t*>(smem + lay.pdst);
  unsigned long long* s_hash = reinterpret_cast<unsigned long long*>(smem + lay.hash);
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem + lay.tok);
  int32_t* s_stamp = reinterpret_cast<int32_t*>(smem + lay.stamp);
  // the table starts at the same 16-byte phase as its global row
  int32_t* s_dbl_staged = reinterpret_cast<int32_t*>(smem + lay.dbl) +
                          ((((uintptr_t)(a.device_buffer_locs + (size_t)r * (g.H + a.spec_n))) & 15) >> 2);
  uint8_t* s_cls = smem + lay.cls;
  uint8_t* s_sflag = smem + lay.sflag;
  int32_t* s_wsum = reinterpret_cast<int32_t*>(smem + lay.wsum);
  int32_t* s_hist = reinterpret_cast<int32_t*>(smem + lay.hist);
  uint32_t* s_sc = reinterpret_cast<uint32_t*>(smem + lay.sc);

  const int K = g.K, H = g.H;
  const int HS = 1 << g.hash_bits;
  // A plain step's one new position is the newest token, S - 1. Verify step q of a
  // speculative batch attends over S0 + q + 1 tokens, and the batch's positions t >= S0 (the
  // token the last round sampled, then the drafts) sit in the reserved rows H + (t - S0).
  const int32_t S = sa.spec_q < 0 ? seq_r : seq_r + sa.spec_q + 1;
  const int32_t base = sa.spec_q < 0 ? S - 1 : seq_r;
  const int32_t* tk_g = sa.top_k_tokens + (size_t)r * K;
  int32_t* out_g = sa.out_rows + (size_t)r * K;
  const int32_t* dbl_g = a.device_buffer_locs + (size_t)r * (H + a.spec_n);
  const int32_t* s_dbl = g.dbl_smem ? s_dbl_staged : dbl_g;  // slot -> row table
  int32_t* tok_g = a.device_buffer_tokens + (size_t)r * H;
  int32_t* st_g = a.lru_slots + (size_t)r * H;
  uint32_t flags = 0;

  // ---- phase 0: state into shared memory: the slot state asynchronously, the top-k row by
  // plain loads (top_k_tokens may be pinned host memory, which cp.async is not used on). It is
  // requested before the request's length is known (the slot state even if the request turns
  // out to be on the fast path), so its latency overlaps that of seq_lens.
  if (g.dbl_smem) cp_async_words(s_dbl_staged, dbl_g, H + 1);
  cp_async_words(s_tok, tok_g, H);
  cp_async_words(s_stamp, st_g, H);
  cp_async_commit();
  for (int i = tid; i < K; i += T) s_tk[i] = tk_g[i];
  for (int h = tid; h < HS; h += T) s_hash[h] = kEmpty;
  for (int i = tid; i < K; i += T) s_claim[i] = INF;
  if (tid < SC_COUNT) s_sc[tid] = tid == SC_LO ? 0xffffffffu : 0u;
  if (tid < 256) s_hist[tid] = 0;
  if (S < 0 || S > g.max_context) {
    for (int i = tid; i < K; i += T) out_g[i] = -1;
    if (tid == 0) {
      if (sa.miss_counts) sa.miss_counts[r] = 0;
      if (sa.plan_cnt) sa.plan_cnt[r] = 0;
      atomicOr(err_word, HS_FLAG_SEQLEN);
    }
    cp_async_wait_all();  // the copies issued above and at kernel start
    finish_phases(C, pub);
    return;
  }
  const bool fast = S <= H;
  cp_async_wait_all();
  __syncthreads();

  // ---- phase 1: validity, class and the hash of the valid tokens. A repeated token is
  // only known once every insert is done, so classes and rows here are provisional for
  // repeats (settled in phase 4, or right below on the fast path).
  uint32_t* hint_row = a.hint ? a.hint + (size_t)r * g.bit_words : nullptr;  // residency bitmap
  for (int i = tid; i < K; i += T) {
    const int32_t t = s_tk[i];
    uint8_t c;
    int64_t row = -1;
    if (t < 0) {
      c = C_PAD;
    } else if (t >= S) {
      c = C_BAD;
      flags |= HS_FLAG_TOKEN;
    } else {
      hash_insert(s_hash, g.hash_bits, t, i);
      int32_t page = -1;
      if (a.resident_pages) page = a.resident_pages[(size_t)r * g.max_pages + t / g.page_size];
      if (page >= 0) {
        c = C_RES;
        row = (int64_t)page * g.page_size + t % g.page_size;
      } else if (fast) {
        c = C_FAST;
        row = s_dbl[t];
      } else if (t >= base) {
        c = C_NEWEST;
        row = t == base ? s_dbl[H] : dbl_g[H + (t - base)];
      } else {
        c = C_LOOKUP;
      }
      if (c != C_LOOKUP && (row < 0 || row >= g.device_rows)) {
        c |= C_BADROW;
        row = -1;
      }
    }
    s_cls[i] = c;
    s_out[i] = (int32_t)row;
  }
  __syncthreads();

  if (fast) {
    for (int i = tid; i < K; i += T) {
      const uint8_t c = s_cls[i];
      int32_t o = s_out[i];
      if (c != C_PAD && c != C_BAD) {
        if (hash_find(s_hash, g.hash_bits, s_tk[i]) != i) {
          flags |= HS_FLAG_DUP;
          o = -1;
        } else if (c & C_BADROW) {
          flags |= HS_FLAG_DEVROW;
        }
      }
      out_g[i] = o;
    }
    if (sa.spec_q < 0) {
      if (tid == 0 && S >= 1) tok_g[S - 1] = S - 1;
    } else {  // committed positions only: S0 and the ones before it the last batch accepted
      const int32_t t = max(0, base - a.spec_n) + tid;  // spec_n + 1 <= T threads
      if (t <= base) tok_g[t] = t;
    }
    if (tid == 0) {
      if (sa.miss_counts) sa.miss_counts[r] = 0;
      if (sa.plan_cnt) sa.plan_cnt[r] = 0;
    }
    if (hint_row) {  // slot t holds token t for every committed t: exact once the sequence outgrows the buffer
      const int nb = min(S, base + 1);
      for (int w = tid; w < (nb + 31) / 32; w += T)
        hint_row[w] = nb - 32 * w >= 32 ? ~0u : (1u << (nb - 32 * w)) - 1u;
    }
    flush_flags(flags, err_word);
    finish_phases(C, pub);
    return;
  }

  // ---- phase 3: tripwires, membership probe, hits. From here on warp w walks its own run
  // of slots [sw0, sw1) and of top-k entries [ew0, ew1), 32 consecutive ones at a time, so
  // shared loads are conflict-free and ballots count in slot / entry order.
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int SW = (H + T - 1) / T * 32, EW = (K + T - 1) / T * 32;
  const int sw0 = min(H, warp * SW), sw1 = min(H, sw0 + SW);
  const int ew0 = min(K, warp * EW), ew1 = min(K, ew0 + EW);
  const int32_t clock = a.lru_clock[r] + 1;
  int wfree = 0;  // free slots in this warp's run
  for (int b = sw0; b < sw1; b += 32) {
    const int s = b + lane;
    bool is_free = false;
    if (s < sw1) {
      int32_t tkn = s_tok[s];
      const int32_t st = s_stamp[s];
      uint8_t f = 0;
      if (st < 0 || st > clock - 1 || tkn < -1 || tkn >= base) {
        tkn = -1;
        s_tok[s] = -1;
        s_stamp[s] = 0;
        f = SF_DIRTY;
        flags |= HS_FLAG_STATE;
      }
      const int32_t i = lookup_entry(s_hash, s_cls, g.hash_bits, tkn);
      bool used = false;
      if (i >= 0) {
        if (atomicCAS(&s_claim[i], INF, s) == INF) {
          s_stamp[s] = clock;
          f |= SF_USED | SF_DIRTY;
          used = true;
        } else {
          s_sc[SC_CONFLICT] = 1u;  // a second slot holds the token: settled below
        }
      }
      if (tkn >= 0 && !used)  // an eviction candidate: count it by age, oldest bin = 255 and up
        atomicAdd(&s_hist[min(clock - 1 - st, 255)], 1);
      s_sflag[s] = f;
      is_free = tkn == -1;
    }
    wfree += __popc(__ballot_sync(FULL, is_free));
  }
  __syncthreads();

  if (s_sc[SC_CONFLICT]) {
    // Corrupt state only: several slots hold one looked-up token. The lowest slot is the
    // hit; an earlier claim by another slot is undone (its stamp is still in global memory,
    // untouched, since a corrupt stamp would have freed the slot).
    for (int i = tid; i < K; i += T) s_vict[i] = INF;
    __syncthreads();
    for (int s = tid; s < H; s += T) {
      const int32_t i = lookup_entry(s_hash, s_cls, g.hash_bits, s_tok[s]);
      if (i >= 0) atomicMin(&s_vict[i], s);
    }
    __syncthreads();
    for (int s = tid; s < H; s += T) {
      const int32_t i = lookup_entry(s_hash, s_cls, g.hash_bits, s_tok[s]);
      if (i < 0) continue;
      const int32_t w = s_vict[i];
      if (s != w) flags |= HS_FLAG_STATE;
      if (s_claim[i] == w) continue;
      if (s == s_claim[i]) {
        s_stamp[s] = st_g[s];
        s_sflag[s] &= (uint8_t)~SF_USED;
      } else if (s == w) {
        s_stamp[s] = clock;
        s_sflag[s] |= SF_USED | SF_DIRTY;
      }
    }
    __syncthreads();
    for (int i = tid; i < K; i += T)
      if (s_vict[i] != INF) s_claim[i] = s_vict[i];
    __syncthreads();
  }

  // ---- phase 4: repeats settle; hits output their slot's row (and tell the entry's copy
  // CTA which slot, so a wrong miss prediction can repair the token's bit)
  const int per = copy_slice(g);
  const CopyLayout cl = make_copy_layout(g);
  if (C > 0) cluster_wait();  // phase A: the copy CTAs run and their tables are cleared
  int wmiss = 0;  // misses in this warp's run of entries
  for (int b = ew0; b < ew1; b += 32) {
    const int i = b + lane;
    bool is_miss = false;
    if (i < ew1) {
      const uint8_t cls = s_cls[i];
      if (cls != C_PAD && cls != C_BAD && hash_find(s_hash, g.hash_bits, s_tk[i]) != i) {
        s_cls[i] = C_DUP;  // a later repeat of a valid token
        s_out[i] = -1;
        flags |= HS_FLAG_DUP;
      } else if (cls & C_BADROW) {
        flags |= HS_FLAG_DEVROW;
      } else if (cls == C_LOOKUP) {
        const int32_t c = s_claim[i];
        if (c != INF) {
          s_out[i] = checked_row(s_dbl[c], g.device_rows, flags);
          if (C > 0) st_remote(smem + cl.res + 4 * (size_t)(i % per), 1 + i / per, -2 - c);
        } else {
          is_miss = true;
        }
      }
    }
    wmiss += __popc(__ballot_sync(FULL, is_miss));
  }
  if (lane == 0) s_wsum[warp] = (wmiss << 16) | wfree;
  __syncthreads();

  // ---- phase 5: order the misses (top-k order) and the free slots (slot order): each
  // warp's base is the sum of the earlier warps' counts (16-bit fields: m <= K, F <= H)
  int m, F;
  {
    const int v = lane < NW ? s_wsum[lane] : 0;
    const int tot = __reduce_add_sync(FULL, v);
    const int before = __reduce_add_sync(FULL, lane < warp ? v : 0);
    m = tot >> 16;
    F = tot & 0xffff;
    int pos = before >> 16;
    for (int b = ew0; b < ew1; b += 32) {
      const int i = b + lane;
      const bool p = i < ew1 && s_cls[i] == C_LOOKUP && s_claim[i] == INF;
      const unsigned bal = __ballot_sync(FULL, p);
      if (p) s_miss[pos + __popc(bal & lt_mask)] = i;
      pos += __popc(bal);
    }
    pos = before & 0xffff;
    for (int b = sw0; b < sw1 && pos < m; b += 32) {
      const int s = b + lane;
      const bool p = s < sw1 && s_tok[s] == -1;
      const unsigned bal = __ballot_sync(FULL, p);
      const int at = pos + __popc(bal & lt_mask);
      if (p && at < m) s_vict[at] = s;
      pos += __popc(bal);
    }
  }
  const int take_free = min(m, F);
  const int m2 = m - take_free;

  // ---- phase 6: the m2 oldest occupied, un-hit slots, ordered by (stamp, slot)
  if (m2 > 0) {
    // The threshold stamp thr_st: every candidate with an older stamp is a victim, and so
    // are the need_eq lowest-numbered candidates stamped thr_st. It comes from the age
    // histogram phase 3 built (age = clock - 1 - stamp, ages of 255 and more share the last
    // bin) when phase 3's claims stood and the threshold age is below 255; otherwise from an
    // exact radix select over the stamps.
    int32_t thr_st = 0;
    int need_eq = 0;
    bool by_age = s_sc[SC_CONFLICT] == 0u;
    if (by_age) {
      if (tid < 32) {  // lane l holds bins 255-8l .. 248-8l: the oldest first
        int loc[8];
        int sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          loc[b] = s_hist[255 - (tid * 8 + b)];
          sum += loc[b];
        }
        const int incl = warp_incl_scan(sum);
        const unsigned ball = __ballot_sync(FULL, incl >= m2);
        const int first = __ffs(ball) - 1;
        if (tid == first) {
          int cum = incl - sum;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (cum + loc[b] >= m2) {
              s_sc[SC_DIGIT] = (uint32_t)(255 - (tid * 8 + b));
              s_sc[SC_RANK] = (uint32_t)(m2 - cum);
              break;
            }
            cum += loc[b];
          }
        }
      }
      __syncthreads();
      by_age = s_sc[SC_DIGIT] < 255u;
      thr_st = clock - 1 - (int32_t)s_sc[SC_DIGIT];
      need_eq = (int)s_sc[SC_RANK];
    }
    if (!by_age) {
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
      thr_st = (int32_t)(base + prefix);  // the last victim's stamp
      need_eq = rank;                     // victims taken among the candidates stamped thr_st
    }
    const int n_lt = m2 - need_eq;
    // From the histogram, n_le = the candidates stamped thr_st or older (exact: the bins below
    // 255 hold one age each). When they are few, one pass gathers them all, in any order, and
    // ranking keeps the m2 smallest (stamp, slot) keys.
    const int n_le = by_age ? n_lt + s_hist[s_sc[SC_DIGIT]] : INT_MAX;
    if (n_le <= T && n_le <= g.sort_cap && n_le * n_le <= m2 * m2 + kOnePassSlack) {
      for (int b = sw0; b < sw1; b += 32) {
        const int s = b + lane;
        const bool cand = s < sw1 && s_tok[s] >= 0 && !(s_sflag[s] & SF_USED);
        const int32_t st = cand ? s_stamp[s] : 0;
        const bool take = cand && st <= thr_st;
        const unsigned bl = __ballot_sync(FULL, take);
        if (bl) {
          int at = 0;
          if (lane == 0) at = (int)atomicAdd(&s_sc[SC_GATHER], (uint32_t)__popc(bl));
          at = __shfl_sync(FULL, at, 0) + __popc(bl & lt_mask);
          if (take && at < n_le) s_keys[at] = ((uint64_t)(uint32_t)st << 32) | (uint32_t)s;
        }
      }
      __syncthreads();
      rank_keys(s_keys, n_le, m2, s_vict + take_free);
    } else {
      // Gather: warp by warp in slot order, candidates older than the threshold to
      // [0, n_lt), the first need_eq at it to [n_lt, m2). Keys (stamp, slot) are distinct.
      int c_lt = 0, c_eq = 0;
      for (int b = sw0; b < sw1; b += 32) {
        const int s = b + lane;
        const bool cand = s < sw1 && s_tok[s] >= 0 && !(s_sflag[s] & SF_USED);
        const int32_t st = cand ? s_stamp[s] : 0;
        c_lt += __popc(__ballot_sync(FULL, cand && st < thr_st));
        c_eq += __popc(__ballot_sync(FULL, cand && st == thr_st));
      }
      __syncthreads();  // every warp has read phase 5's counts
      if (lane == 0) s_wsum[warp] = (c_lt << 16) | c_eq;
      __syncthreads();
      {
        const int before = __reduce_add_sync(FULL, lane < warp ? s_wsum[lane] : 0);
        int p_lt = before >> 16, p_eq = before & 0xffff;
        for (int b = sw0; b < sw1; b += 32) {
          const int s = b + lane;
          const bool cand = s < sw1 && s_tok[s] >= 0 && !(s_sflag[s] & SF_USED);
          const int32_t st = cand ? s_stamp[s] : 0;
          const bool lt = cand && st < thr_st, eq = cand && st == thr_st;
          const unsigned bl = __ballot_sync(FULL, lt), be = __ballot_sync(FULL, eq);
          const uint64_t key = ((uint64_t)(uint32_t)st << 32) | (uint32_t)s;
          if (lt) s_keys[p_lt + __popc(bl & lt_mask)] = key;
          if (eq) {
            const int q = p_eq + __popc(be & lt_mask);
            if (q < need_eq) s_keys[n_lt + q] = key;
          }
          p_lt += __popc(bl);
          p_eq += __popc(be);
        }
      }
      __syncthreads();
      if (m2 <= T) {
        rank_keys(s_keys, m2, m2, s_vict + take_free);  // a victim's place is its key's rank
      } else {
        int n = 1;
        while (n < m2) n <<= 1;
        for (int i = m2 + tid; i < n; i += T) s_keys[i] = ~0ull;
        __syncthreads();
        bitonic_sort(s_keys, n);
        for (int j = tid; j < m2; j += T) s_vict[take_free + j] = (int32_t)(s_keys[j] & 0xffffffffu);
      }
    }
  }
  __syncthreads();

  // ---- phase 7: miss j takes victim j; the entry's copy CTA gets its device row. The global
  // writes of this phase (residency bits, plan) come after the barrier arrive: a release
  // arrive first waits for the thread's earlier writes to complete, which would hold the
  // copy CTAs back by a global-memory round trip.
  for (int j = tid; j < m; j += T) {
    const int32_t v = s_vict[j];
    const int32_t i = s_miss[j];
    int32_t d = -1, old_tok = -2;  // -2: no slot taken
    if ((uint32_t)v < (uint32_t)H) {
      old_tok = s_tok[v];
      s_tok[v] = s_tk[i];
      s_stamp[v] = clock;
      s_sflag[v] |= SF_DIRTY;
      d = checked_row(s_dbl[v], g.device_rows, flags);
    } else {
      flags |= HS_FLAG_STATE;  // unreachable by construction; never index with it
    }
    s_out[i] = d;
    s_vict[j] = old_tok;  // the evicted token (-1: a free slot), for the bitmap below
    if (C > 0) {  // the copy CTA owning entry i moves this row
      st_remote(smem + cl.res + 4 * (size_t)(i % per), 1 + i / per, d);
      s_pdst[j] = -1;
    } else {
      s_sc[SC_DIRECT] = 1u;
      int32_t hr = -1;
      if (d >= 0) {
        hr = a.host_cache_locs[(size_t)r * g.max_context + s_tk[i]];
        if (hr < 0 || (int64_t)hr >= g.host_rows) {
          hr = -1;
          flags |= HS_FLAG_HOSTROW;  // destination is zero-filled
        }
      }
      s_psrc[j] = hr;
      s_pdst[j] = d;
    }
  }
  if (C > 0) {  // every outcome is in the copy CTAs' shared memory: publish it to each
    __syncthreads();
    if (tid < C) publish_to(pub, tid + 1);
  }
  for (int j = tid; j < m; j += T) {  // this thread's misses of the loop above
    const int32_t t = s_tk[s_miss[j]], old_tok = s_vict[j];
    if (hint_row && old_tok >= -1) {
      if (old_tok >= 0) atomicAnd(&hint_row[old_tok >> 5], ~(1u << (old_tok & 31)));  // evicted
      atomicOr(&hint_row[t >> 5], 1u << (t & 31));
    }
    if (sa.plan_tok) {  // the miss plan the follower layers replay: token and destination row
      sa.plan_tok[(size_t)r * K + j] = t;
      sa.plan_dst[(size_t)r * K + j] = s_out[s_miss[j]];
    }
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
    if (sa.miss_counts) sa.miss_counts[r] = m;
    if (sa.plan_cnt) sa.plan_cnt[r] = m;
  }

  // ---- phase 9: misses no copy CTA took, the leader layers, straight from host memory
  if (s_sc[SC_DIRECT]) copy_rows(g, s_pools, s_psrc, s_pdst, m, a.copy_layers);
  flush_flags(flags, err_word);
}

// kBatch = false: one step (a plain decode step, or the one verify step a.spec_q); true: the
// a.spec_steps verify steps of a speculative batch in order. Two instances, so the one-step
// kernel carries no loop state.
template <bool kBatch>
__global__ void __launch_bounds__(T, 1)
    resolve_kernel(const Geometry g, const Pools* __restrict__ pools, const ResolveArgs a,
                   uint32_t* __restrict__ err_word) {
  // The eager backup touches only the newest token's rows, which this kernel never reads
  // or writes: let it launch now and run beside the resolve (it orders its own exit).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) Pools s_pools;
  __shared__ StepArgs s_step;  // this step's arguments, read where they are used (no registers held)
  __shared__ __align__(8) uint64_t s_pub;  // copy CTAs: the resolve CTA published this step's outcomes
  const int tid = threadIdx.x;
  const int C = g.copy_ctas;
  const uint32_t rank = C > 0 ? cluster_rank() : 0u;
  const int r = blockIdx.x / (C + 1);  // one cluster of C + 1 CTAs per request
  // The pools table comes in asynchronously after the first release-arrive of barrier phase A
  // (which would otherwise wait for it): no CTA waits for it before it needs a pool address
  // (the copy CTAs before their first row load, the resolve CTA at the end of its phase 0).
  static_assert(sizeof(Pools) % 16 == 0, "the pools table moves in 16-byte pieces");
  const auto load_pools = [&] {
    if (tid < (int)(sizeof(Pools) / 16))
      cp_async16(reinterpret_cast<uint4*>(&s_pools) + tid, reinterpret_cast<const uint4*>(pools) + tid);
    cp_async_commit();
  };
  // A speculative batch's verify steps run here in order, one after the other, over the
  // request's shared slot state (each with its own top-k slice, row table, miss counts and
  // plan slice); a plain step is one pass. The two roles loop apart, so each loop keeps only
  // its own role's registers.
  const int steps = kBatch ? a.spec_steps : 1;
  if (rank > 0) {
    for (int q = 0; q < steps; ++q) {
      if (kBatch && q > 0) {
        // step q - 1 is complete in every CTA of the cluster, and its writes (slot state,
        // clock, residency bits, copied rows) are visible, before this CTA clears its tables
        cluster_arrive();
        cluster_wait();
      }
      if (tid == 0) s_step = step_args(a, kBatch ? q : -1);
      // Barrier phase A: every CTA of the cluster runs, and each copy CTA has cleared its
      // outcome table and counters, before the resolve CTA stores into a copy CTA's shared
      // memory. Only that first remote store waits for it (phase 4); the copy CTAs start
      // their own work at once.
      const CopyLayout cl0 = make_copy_layout(g);
      int32_t* res = reinterpret_cast<int32_t*>(smem + cl0.res);
      for (int e = tid; e < copy_slice(g); e += T) res[e] = -1;
      if (tid < 4) reinterpret_cast<uint32_t*>(smem + cl0.cnt)[tid] = 0u;
      if (q == 0 && tid == 0) {  // one phase per step; phase A orders the initialisation before the first arrival
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_pub)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      }
      cluster_arrive();
      if (q == 0) load_pools();
      __syncthreads();  // the CTA's own clears and step arguments before its threads read them
      // Loaded after the release-arrive, which would otherwise wait for it (plain load: may be
      // host memory); its latency overlaps the prediction's loads.
      const int32_t seq_r = a.seq_lens[r];
      copy_cta(g, s_pools, a, s_step, r, (int)rank, seq_r, smem, &s_pub, (uint32_t)q & 1u, err_word);
    }
    return;
  }
  for (int q = 0; q < steps; ++q) {
    if (kBatch && q > 0) {
      // step q - 1 is complete everywhere before step q reads the state (a CTA barrier when the
      // request has no copy CTAs)
      if (C > 0) {
        cluster_arrive();
        cluster_wait();
      } else {
        __syncthreads();
      }
    }
    if (tid == 0) s_step = step_args(a, kBatch ? q : -1);
    __syncthreads();  // the step arguments (and the pools table) before any thread reads them
    if (C > 0) cluster_arrive();  // phase A
    if (q == 0) load_pools();
    const int32_t seq_r = a.seq_lens[r];  // after the release-arrive, as in the copy CTAs
    resolve_cta(g, s_pools, a, s_step, err_word, smem, &s_pub, r, seq_r);
  }
}

}  // namespace

size_t resolve_smem_bytes(const Geometry& g) {
  const size_t a = make_layout(g).total;
  const size_t b = g.copy_ctas > 0 ? make_copy_layout(g).total : 0;
  return a > b ? a : b;
}

// Raise the kernel's dynamic shared-memory limit to the device maximum beside its static
// shared memory (not to this geometry's size: the attribute is per function and device, so
// a smaller value set for one handle would make launches of a larger, earlier handle
// fail), then choose the copy CTAs. Each request gets C = SMs / max_requests - 1 of them
// (at most 3), so a full batch spreads over the GPU, each staging as many misses as its
// shared memory holds; none when rows are not 16-byte copyable or the cluster does not fit.
cudaError_t resolve_prepare(Geometry& g, int32_t max_requests) {
  int dev = 0, optin = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, resolve_kernel<false>);
  if (e != cudaSuccess) return e;
  const int max_dynamic = optin - (int)fa.sharedSizeBytes;
  g.sms = sms;
  g.copy_ctas = 0;
  g.copy_cap = 0;
  g.bits_smem = 0;
  // The largest layout that fits, in this order: the slot -> row table staged, else read from
  // global memory; then, for the largest top_k, the same with the top-k hash half full
  // instead of a quarter (still at least half empty, so every probe loop ends).
  int half_bits = 0;
  while ((1 << half_bits) < g.K) ++half_bits;
  half_bits += 1;  // 2 * sort_cap buckets: room for the keys and plan aliased onto the hash
  bool fits = false;
  for (int pass = 0; pass < 2 && !fits; ++pass) {
    if (pass == 1) {
      if (g.hash_bits <= half_bits) break;
      g.hash_bits = half_bits;
    }
    for (int d = 1; d >= 0 && !fits; --d) {
      g.dbl_smem = d;
      fits = make_layout(g).total <= (size_t)max_dynamic;
    }
  }
  if (!fits) return cudaErrorInvalidValue;
  cudaFuncAttributes fb{};
  e = cudaFuncGetAttributes(&fb, resolve_kernel<true>);
  if (e != cudaSuccess) return e;
  if (fb.sharedSizeBytes > fa.sharedSizeBytes && make_layout(g).total > (size_t)(optin - (int)fb.sharedSizeBytes))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(resolve_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(resolve_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fb.sharedSizeBytes);
  if (e != cudaSuccess) return e;

  int C = max_requests > 0 ? sms / max_requests - 1 : 0;
  C = C < 0 ? 0 : (C > 3 ? 3 : C);
  if (g.vec != 16) C = 0;
  if (C > 0) {
    Geometry t = g;
    t.copy_ctas = C;
    t.copy_cap = 0;
    t.bits_smem = g.bit_words > 0 && 4 * g.bit_words <= kBitsSmemMax ? 1 : 0;
    const size_t fixed = make_copy_layout(t).total + 64;  // + alignment slack
    if (fixed < (size_t)max_dynamic) {
      size_t cap = ((size_t)max_dynamic - fixed) / (2 + (size_t)g.L * (size_t)g.B);
      if (cap > (size_t)copy_slice(t)) cap = (size_t)copy_slice(t);
      t.copy_cap = (int32_t)cap;
      while (t.copy_cap > 0 && resolve_smem_bytes(t) > (size_t)max_dynamic) --t.copy_cap;
    }
    if (t.copy_cap > 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(C + 1));
      cfg.blockDim = dim3(T);
      cfg.dynamicSmemBytes = resolve_smem_bytes(t);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)(C + 1);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, resolve_kernel<false>, &cfg) == cudaSuccess && clusters > 0) {
        g.copy_ctas = C;
        g.copy_cap = t.copy_cap;
        g.bits_smem = t.bits_smem;
      } else {
        cudaGetLastError();
      }
    }
  }
  return cudaSuccess;
}

cudaError_t launch_resolve(const Geometry& g, const Pools* pools, const ResolveArgs& a, int32_t num_requests,
                           uint32_t* err_word, cudaStream_t stream) {
  const unsigned per_request = (unsigned)(g.copy_ctas + 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_requests * per_request);
  cfg.blockDim = dim3(T);
  cfg.dynamicSmemBytes = resolve_smem_bytes(g);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = per_request;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g.copy_ctas > 0 ? 1 : 0;
  if (a.spec_steps > 0) return cudaLaunchKernelEx(&cfg, resolve_kernel<true>, g, pools, a, err_word);
  return cudaLaunchKernelEx(&cfg, resolve_kernel<false>, g, pools, a, err_word);
}

}  // namespace hs
