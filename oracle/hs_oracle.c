/*
 * CPU ORACLE of the HiSparse decode-step resolver / swap-in.  TEST INFRASTRUCTURE ONLY.
 *
 * This is the plain, single-threaded, obviously-correct definition that the CUDA path
 * is checked against. Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark may load it; the library's product path never does. It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Sources (page title, section):
 *   [SGLang-analysis]  "HiSparse: moving the long-context decode capacity bottleneck from
 *                      GPU memory to CPU memory" - "Per decode step workflow" (steps 3 and
 *                      5: swap-in with the short-sequence fast path; eager backup) and
 *                      "Core: swap-in CUDA kernel" (the kernel parameters top_k_tokens,
 *                      seq_lens, host_cache_locs, device_buffer_locs, lru_slots), and
 *                      "How capacity is computed" (buffer padded by one page reserved for
 *                      the new token).
 *   [SGLang-blog]      "HiSparse: Turbocharging Sparse Attention with Hierarchical Memory"
 *                      - "Efficient swap-in kernel" (find top-k misses, pick LRU victims,
 *                      update the table and fetch the missing rows).
 *   [vLLM-arch]        "vLLM HiSparse local KV offload architecture" - "Hot-row lookup and
 *                      LRU" (resident page, then hot row with an LRU refresh, then a
 *                      victim filled from pinned host memory) and "Performance invariants".
 *   [vLLM-impl]        "vLLM Hybrid HiSparse source implementation analysis" - section 7.2
 *                      (phase 1 resident short-circuit; phase 2 hot hits; phase 3 miss plan
 *                      with corruption tripwires downgraded to a re-miss; the gather that
 *                      zeroes a destination whose source row is out of range), 7.3
 *                      (physical row IDs), 7.4 (IndexShare followers reuse the plan).
 *   [Tair-HSA]         "Hierarchical Sparse Attention" (Alibaba Tair KVCache) - 2.4.3 "LRU
 *                      Diff Kernel" (evict only when the buffer is full, coldest first).
 *   [GLM53]            "vLLM GLM 5.3 optimisation: Hybrid HiSparse Offloading" - "Mixed
 *                      Residency" (resident tokens read in place, hot tokens refresh their
 *                      LRU entry, misses copy one row from pinned host memory).
 *
 * Readings where the pages leave a step open (the plainest reading the rest of the pages
 * supports, with the passage it rests on):
 *   - The LRU state is a per-slot stamp plus a per-request clock; a slow-path call
 *     first advances the clock (c = clock + 1) and stamps every slot it touches with c.
 *     [vLLM-impl] 7.1 keeps a per-slot order and rewrites it every call with the hits at
 *     the most-recent end (7.2 phase 4); a stamp of the call's clock orders the slots the
 *     same way and lives in device memory, so no host value enters the step.
 *   - Victims: slots not hit in this call, free slots first by ascending index, then
 *     occupied slots by ascending (stamp, slot). The j-th miss (top-k array order)
 *     takes the j-th victim. [Tair-HSA] 2.4.3: evict only when the buffer is full, the
 *     coldest first; [vLLM-impl] 7.2 phase 3 hands the misses, compacted in order, the
 *     oldest evictable slots in turn. The lowest slot breaks ties.
 *   - The newest token (seq_len - 1), when not resident and not on the fast path,
 *     resolves to the reserved slot H: [SGLang-analysis] "How capacity is computed" pads
 *     each request's buffer with room for the token the step adds.
 *   - A token >= seq_len outputs -1 (ERR_TOKEN); a repeated valid token keeps its first
 *     occurrence and the later ones output -1 (ERR_DUP). [vLLM-impl] 7.1: padding rows
 *     output -1 for attention to mask; one output row per distinct token keeps every
 *     entry's row distinct.
 *   - Corrupt slot state (stamp outside [0, c-1], token outside [-1, seq_len-2]) is
 *     reset to free with stamp 0 (ERR_STATE): [vLLM-impl] 7.2 phase 3, an out-of-range slot
 *     is downgraded to a re-miss instead of being trusted. If several slots hold a
 *     looked-up token, the lowest slot is the hit (ERR_STATE) and the other holders are not
 *     hits: [vLLM-impl] 7.2 phase 2 sorts each slot into exactly two classes by probing the
 *     top-k hash with its key -- a hit that gives the entry its row, or an evictable slot --
 *     and one entry has one row, so one holder serves it and the rest are evictable with
 *     their stamps. A held token nobody looks up is not probed, so its duplicates stay.
 *   - A miss whose host row is outside the host pool gets a zeroed destination
 *     (ERR_HOSTROW, [vLLM-impl] 7.2, the gather kernel); a physical row outside the device
 *     pool outputs -1 and nothing is written (ERR_DEVROW); seq_len outside
 *     [0, max_context] skips the request (ERR_SEQLEN).
 *
 * Parity pins (tests, not this file): brute-force enumeration of victim choices on tiny
 * inputs, reduction to textbook LRU at top_k = 1, the pages' invariants (injective slot
 * map, occupancy <= H, exact row bytes, misses = |top-k \ hot set|), and special cases.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_ERR_TOKEN 1u
#define OR_ERR_DUP 2u
#define OR_ERR_STATE 4u
#define OR_ERR_HOSTROW 8u
#define OR_ERR_DEVROW 16u
#define OR_ERR_SEQLEN 32u

typedef struct {
  int32_t top_k, hot_slots, row_bytes, num_layers, page_size, max_context, max_pages;
  int64_t host_rows, device_rows;
  int64_t host_row_stride; /* bytes from host row h to h + 1 in one layer's pool; 0 = row_bytes */
} oracle_geom;

/* Host row h of layer l. The host pool layouts of "Hierarchical Sparse Attention" (Alibaba
 * Tair KVCache), 2.4.4 "I/O Transfer Kernel": layer first (one pool per layer, rows
 * row_bytes apart) or page first (one row holds every layer's bytes of a token, the pools
 * given as base + l * row_bytes, rows num_layers * row_bytes apart). Either way the row
 * starts host_row_stride * h bytes into the layer's pool. */
static uint8_t* host_row(const oracle_geom* g, uint8_t* const* host_pools, int32_t l, int64_t h) {
  const int64_t stride = g->host_row_stride > 0 ? g->host_row_stride : g->row_bytes;
  return host_pools[l] + (size_t)h * (size_t)stride;
}

enum { E_PAD = 0, E_BAD, E_DUP, E_VALID, E_RES, E_NEWEST, E_DONE, E_MISS };

typedef struct {
  int32_t occupied;
  int32_t stamp;
  int32_t slot;
} victim_key;

static int cmp_key(const void* a, const void* b) {
  const victim_key* x = (const victim_key*)a;
  const victim_key* y = (const victim_key*)b;
  if (x->occupied != y->occupied) return x->occupied < y->occupied ? -1 : 1;
  if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
  if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
  return 0;
}

static int32_t checked_row(int64_t row, int64_t device_rows, uint32_t* err) {
  if (row < 0 || row >= device_rows) {
    *err |= OR_ERR_DEVROW;
    return -1;
  }
  return (int32_t)row;
}

/* Device row of token t from the resident page table, or -1 when its page is host only.
 * [vLLM-arch] "Hot-row lookup and LRU": the resident page is checked first. */
static int64_t resident_row(const oracle_geom* g, const int32_t* resident_pages, int32_t r, int32_t t) {
  if (!resident_pages || g->page_size <= 0) return -1;
  int32_t p = resident_pages[(int64_t)r * g->max_pages + t / g->page_size];
  if (p < 0) return -1;
  return (int64_t)p * g->page_size + t % g->page_size;
}

/*
 * One decode-step resolve for requests [0, num_requests).
 * Arrays are dense row-major: top_k_tokens [R,K], seq_lens [R],
 * host_cache_locs [R,max_context], device_buffer_locs [R,H+1],
 * device_buffer_tokens / lru_slots [R,H], lru_clock [R], resident_pages [R,max_pages]
 * (or NULL), out_rows [R,K], miss_counts [R] (or NULL).
 * host_pools / device_pools: num_layers pointers to [rows, row_bytes] byte pools.
 * Error bits are OR-ed into *err.
 */
/* One resolve call. spec_q < 0: a plain decode step (seq_lens are the lengths, the one new
 * position is the newest token); spec_q >= 0: verify step spec_q of a speculative batch of
 * spec_n queries (seq_lens are the committed lengths S0). device_buffer_locs rows hold
 * H + spec_n entries (H slots, then the reserved rows). */
static void resolve_call(const oracle_geom* g, int32_t num_requests, const int32_t* top_k_tokens,
                         const int32_t* seq_lens, const int32_t* host_cache_locs,
                         const int32_t* device_buffer_locs, int32_t* device_buffer_tokens,
                         int32_t* lru_slots, int32_t* lru_clock, const int32_t* resident_pages,
                         int32_t* out_rows, int32_t* miss_counts, uint8_t* const* host_pools,
                         uint8_t* const* device_pools, uint32_t* err, int32_t copy_layers,
                         int32_t* plan_tokens, int32_t* plan_dst, int32_t* plan_count, int32_t spec_q,
                         int32_t spec_n) {
  const int32_t K = g->top_k, H = g->hot_slots, B = g->row_bytes;
  int32_t* cls = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  int32_t* first_at = (int32_t*)malloc(sizeof(int32_t) * (size_t)(g->max_context + 1));
  int32_t* lowest_slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(g->max_context + 1));
  int32_t* holders = (int32_t*)malloc(sizeof(int32_t) * (size_t)(g->max_context + 1));
  int32_t* used = (int32_t*)malloc(sizeof(int32_t) * (size_t)H);
  int32_t* misses = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  victim_key* cand = (victim_key*)malloc(sizeof(victim_key) * (size_t)H);
  for (int32_t t = 0; t <= g->max_context; ++t) first_at[t] = -1, lowest_slot[t] = -1, holders[t] = 0;

  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t* tk = top_k_tokens + (int64_t)r * K;
    const int32_t* dbl = device_buffer_locs + (int64_t)r * (H + spec_n);
    const int32_t* hcl = host_cache_locs + (int64_t)r * g->max_context;
    int32_t* tokens = device_buffer_tokens + (int64_t)r * H;
    int32_t* stamps = lru_slots + (int64_t)r * H;
    int32_t* out = out_rows + (int64_t)r * K;
    /* Verify step q of a speculative batch attends over S0 + q + 1 tokens. The batch's
     * positions [S0, S0 + Q) -- S0 the token the last round sampled, then the drafts -- are
     * new to the cache and sit in the reserved rows H + (t - S0)
     * ([vLLM-impl] 7.1: the buffer is (n_spec + 2) x top_k rows; 7.4: each verify step gets
     * its own plan and shares the request's hot state). A plain step's one new position is
     * the newest token, seq_len - 1, in row H. */
    const int32_t S = spec_q < 0 ? seq_lens[r] : seq_lens[r] + spec_q + 1;
    const int32_t base = spec_q < 0 ? S - 1 : seq_lens[r];

    for (int32_t i = 0; i < K; ++i) out[i] = -1;
    if (miss_counts) miss_counts[r] = 0;
    if (plan_count) plan_count[r] = 0;
    if (S < 0 || S > g->max_context) {
      *err |= OR_ERR_SEQLEN;
      continue;
    }

    /* Validate: padding (t < 0) outputs -1; t >= seq_len is an error; a repeated valid
     * token keeps its first occurrence. */
    for (int32_t i = 0; i < K; ++i) {
      int32_t t = tk[i];
      if (t < 0) cls[i] = E_PAD;
      else if (t >= S) { cls[i] = E_BAD; *err |= OR_ERR_TOKEN; }
      else if (first_at[t] >= 0) { cls[i] = E_DUP; *err |= OR_ERR_DUP; }
      else { first_at[t] = i; cls[i] = E_VALID; }
    }
    for (int32_t i = 0; i < K; ++i)
      if (cls[i] == E_VALID) first_at[tk[i]] = -1;

    /* Phase 1: resident tokens resolve in place ([vLLM-impl] 7.2 phase 1; [GLM53]). */
    for (int32_t i = 0; i < K; ++i) {
      if (cls[i] != E_VALID) continue;
      int64_t row = resident_row(g, resident_pages, r, tk[i]);
      if (row >= 0) { out[i] = checked_row(row, g->device_rows, err); cls[i] = E_RES; }
    }

    /* Fast path: the whole sequence fits the buffer, slot t holds token t; nothing moves
     * ([SGLang-analysis] "Per decode step workflow", step 3). The newest token's slot is
     * recorded so the map stays complete when the sequence outgrows the buffer. */
    if (S <= H) {
      for (int32_t i = 0; i < K; ++i)
        if (cls[i] == E_VALID) out[i] = checked_row(dbl[tk[i]], g->device_rows, err);
      if (spec_q < 0) {
        if (S >= 1) tokens[S - 1] = S - 1;
      } else {  /* committed positions only: S0 (the token the last round sampled) and the
                 * ones before it the previous batch may have accepted, never the drafts */
        for (int32_t t = base - spec_n > 0 ? base - spec_n : 0; t <= base; ++t) tokens[t] = t;
      }
      continue;
    }

    /* Slow path: advance this request's clock. */
    const int32_t c = lru_clock[r] + 1;
    lru_clock[r] = c;

    /* New positions live in the reserved rows after the H slots ([SGLang-analysis] "How
     * capacity is computed": the buffer carries an extra page for the new token). */
    for (int32_t i = 0; i < K; ++i)
      if (cls[i] == E_VALID && tk[i] >= base) {
        out[i] = checked_row(dbl[H + (tk[i] - base)], g->device_rows, err);
        cls[i] = E_NEWEST;
      }

    /* Tripwires: corrupt slot state becomes a free slot ([vLLM-impl] 7.2 phase 3). */
    for (int32_t s = 0; s < H; ++s) {
      if (stamps[s] < 0 || stamps[s] > c - 1 || tokens[s] < -1 || tokens[s] >= base) {
        tokens[s] = -1;
        stamps[s] = 0;
        *err |= OR_ERR_STATE;
      }
      used[s] = 0;
    }
    for (int32_t s = 0; s < H; ++s) {
      int32_t t = tokens[s];
      if (t < 0) continue;
      if (holders[t] == 0) lowest_slot[t] = s;
      holders[t] += 1;
    }

    /* Hits refresh their stamp; everything else is a miss, kept in top-k order
     * ([vLLM-arch] "Hot-row lookup and LRU"). */
    int32_t m = 0;
    for (int32_t i = 0; i < K; ++i) {
      if (cls[i] != E_VALID) continue;
      int32_t t = tk[i];
      if (holders[t] > 0) {
        int32_t s = lowest_slot[t];
        if (holders[t] > 1) *err |= OR_ERR_STATE;
        stamps[s] = c;
        used[s] = 1;
        out[i] = checked_row(dbl[s], g->device_rows, err);
        cls[i] = E_DONE;
      } else {
        misses[m++] = i;
        cls[i] = E_MISS;
      }
    }
    for (int32_t s = 0; s < H; ++s)
      if (tokens[s] >= 0) holders[tokens[s]] = 0, lowest_slot[tokens[s]] = -1;
    if (miss_counts) miss_counts[r] = m;
    if (plan_count) plan_count[r] = m;

    /* Victims: among slots not hit now, free slots first (lowest index first), then the
     * oldest stamps, ties to the lowest slot ([Tair-HSA] 2.4.3: evict only when the buffer
     * is full, coldest first). */
    int32_t nc = 0;
    for (int32_t s = 0; s < H; ++s) {
      if (used[s]) continue;
      cand[nc].occupied = tokens[s] >= 0 ? 1 : 0;
      cand[nc].stamp = tokens[s] >= 0 ? stamps[s] : 0;
      cand[nc].slot = s;
      ++nc;
    }
    qsort(cand, (size_t)nc, sizeof(victim_key), cmp_key);

    /* The j-th miss takes the j-th victim; its row is copied from pinned host memory for
     * every layer of the group ([SGLang-blog] "Efficient swap-in kernel"; [vLLM-impl] 7.4:
     * layers that share the indexer share the plan and copy their own bytes). */
    for (int32_t j = 0; j < m; ++j) {
      int32_t i = misses[j];
      int32_t t = tk[i];
      int32_t v = cand[j].slot;
      tokens[v] = t;
      stamps[v] = c;
      int32_t d = checked_row(dbl[v], g->device_rows, err);
      out[i] = d;
      if (plan_tokens) {  /* the miss plan, in miss order: token and destination row */
        plan_tokens[(int64_t)r * K + j] = t;
        plan_dst[(int64_t)r * K + j] = d;
      }
      if (d < 0) continue;
      int64_t h = hcl[t];
      int host_ok = h >= 0 && h < g->host_rows;
      if (!host_ok) *err |= OR_ERR_HOSTROW;
      for (int32_t l = 0; l < copy_layers; ++l) {
        uint8_t* dst = device_pools[l] + (size_t)d * (size_t)B;
        if (host_ok) memcpy(dst, host_row(g, host_pools, l, h), (size_t)B);
        else memset(dst, 0, (size_t)B);
      }
    }
  }
  free(cls); free(first_at); free(lowest_slot); free(holders); free(used); free(misses); free(cand);
}

void oracle_resolve_plan(const oracle_geom* g, int32_t num_requests, const int32_t* top_k_tokens,
                         const int32_t* seq_lens, const int32_t* host_cache_locs,
                         const int32_t* device_buffer_locs, int32_t* device_buffer_tokens,
                         int32_t* lru_slots, int32_t* lru_clock, const int32_t* resident_pages,
                         int32_t* out_rows, int32_t* miss_counts, uint8_t* const* host_pools,
                         uint8_t* const* device_pools, uint32_t* err, int32_t copy_layers,
                         int32_t* plan_tokens, int32_t* plan_dst, int32_t* plan_count) {
  resolve_call(g, num_requests, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs, device_buffer_tokens,
               lru_slots, lru_clock, resident_pages, out_rows, miss_counts, host_pools, device_pools, err,
               copy_layers, plan_tokens, plan_dst, plan_count, -1, 1);
}

void oracle_resolve_spec_plan(const oracle_geom* g, int32_t num_requests, int32_t num_queries,
                              const int32_t* top_k_tokens, const int32_t* committed_lens,
                              const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                              int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                              const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                              uint8_t* const* host_pools, uint8_t* const* device_pools, uint32_t* err,
                              int32_t copy_layers, int32_t* plan_tokens, int32_t* plan_dst, int32_t* plan_count);

/*
 * A speculative batch ([vLLM-arch] speculative decoding: each verify step is resolved and
 * consumed in order, with its own replayable plan rows and the request's shared hot state,
 * so a later step cannot reuse a hot row before the earlier step consumed it; [vLLM-impl]
 * 7.4 and 7.1: one resolve per verify step over a slice of the workspace, buffer of
 * (n_spec + 2) x top_k rows). num_queries = n_spec + 1 verify steps run in order: step q
 * resolves top_k_tokens[q] (each [R, K]) for S0 + q + 1 tokens into out_rows[q] and
 * miss_counts[q] (or NULL), every layer copied. committed_lens are the S0.
 */
void oracle_resolve_spec(const oracle_geom* g, int32_t num_requests, int32_t num_queries,
                         const int32_t* top_k_tokens, const int32_t* committed_lens,
                         const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                         int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                         const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                         uint8_t* const* host_pools, uint8_t* const* device_pools, uint32_t* err) {
  oracle_resolve_spec_plan(g, num_requests, num_queries, top_k_tokens, committed_lens, host_cache_locs,
                           device_buffer_locs, device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows,
                           miss_counts, host_pools, device_pools, err, g->num_layers, NULL, NULL, NULL);
}

/*
 * The same batch for a layer group split into leader and followers ([vLLM-impl] 7.4: with
 * IndexShare the follower layers replay the leader's miss plan; under MTP each verify step
 * is its own resolve over its own slice of the workspace, sharing the request's hot state;
 * [vLLM-arch] speculative decoding: every verify step has its own replayable plan rows).
 * Verify step q copies its misses' rows for layers [0, copy_layers) only and records its
 * miss plan in slice q: plan_tokens / plan_dst [Q, R, K], plan_count [Q, R] (all NULL:
 * none kept). oracle_gather on slice q then copies step q's rows for the followers.
 */
void oracle_resolve_spec_plan(const oracle_geom* g, int32_t num_requests, int32_t num_queries,
                              const int32_t* top_k_tokens, const int32_t* committed_lens,
                              const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                              int32_t* device_buffer_tokens, int32_t* lru_slots, int32_t* lru_clock,
                              const int32_t* resident_pages, int32_t* out_rows, int32_t* miss_counts,
                              uint8_t* const* host_pools, uint8_t* const* device_pools, uint32_t* err,
                              int32_t copy_layers, int32_t* plan_tokens, int32_t* plan_dst, int32_t* plan_count) {
  const int64_t RK = (int64_t)num_requests * g->top_k;
  for (int32_t q = 0; q < num_queries; ++q)
    resolve_call(g, num_requests, top_k_tokens + q * RK, committed_lens, host_cache_locs, device_buffer_locs,
                 device_buffer_tokens, lru_slots, lru_clock, resident_pages, out_rows + q * RK,
                 miss_counts ? miss_counts + (int64_t)q * num_requests : NULL, host_pools, device_pools, err,
                 copy_layers, plan_tokens ? plan_tokens + q * RK : NULL, plan_dst ? plan_dst + q * RK : NULL,
                 plan_count ? plan_count + (int64_t)q * num_requests : NULL, q, num_queries);
}

/* The whole step: every layer of the group gets its miss rows; no plan is kept. */
void oracle_resolve(const oracle_geom* g, int32_t num_requests, const int32_t* top_k_tokens,
                    const int32_t* seq_lens, const int32_t* host_cache_locs,
                    const int32_t* device_buffer_locs, int32_t* device_buffer_tokens,
                    int32_t* lru_slots, int32_t* lru_clock, const int32_t* resident_pages,
                    int32_t* out_rows, int32_t* miss_counts, uint8_t* const* host_pools,
                    uint8_t* const* device_pools, uint32_t* err) {
  resolve_call(g, num_requests, top_k_tokens, seq_lens, host_cache_locs, device_buffer_locs, device_buffer_tokens,
               lru_slots, lru_clock, resident_pages, out_rows, miss_counts, host_pools, device_pools, err,
               g->num_layers, NULL, NULL, NULL, -1, 1);
}

/*
 * Follower gather ([vLLM-impl] 7.4: layers that share the indexer see the same indices and
 * get the same slot plan; each follower copies its own bytes following the leader's plan,
 * with no LRU work; [vLLM-arch] "Performance invariants": compatible layers share one miss
 * plan). The plan is what oracle_resolve_plan recorded: per request, plan_count[r] misses,
 * miss j being token plan_tokens[r][j] bound for device row plan_dst[r][j] (-1: none). For
 * each layer in [first_layer, first_layer + num_layers) the token's host row is copied to
 * that device row, or zeros when the host row is outside the pool (ERR_HOSTROW).
 */
void oracle_gather(const oracle_geom* g, int32_t num_requests, const int32_t* plan_count,
                   const int32_t* plan_tokens, const int32_t* plan_dst, const int32_t* host_cache_locs,
                   int32_t first_layer, int32_t num_layers, uint8_t* const* host_pools,
                   uint8_t* const* device_pools, uint32_t* err) {
  const int32_t K = g->top_k, B = g->row_bytes;
  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t* hcl = host_cache_locs + (int64_t)r * g->max_context;
    for (int32_t j = 0; j < plan_count[r]; ++j) {
      const int32_t t = plan_tokens[(int64_t)r * K + j];
      const int32_t d = plan_dst[(int64_t)r * K + j];
      if (d < 0) continue;
      const int64_t src_row = hcl[t];
      const int src_ok = src_row >= 0 && src_row < g->host_rows;
      if (!src_ok) *err |= OR_ERR_HOSTROW;
      for (int32_t l = first_layer; l < first_layer + num_layers; ++l) {
        uint8_t* to = device_pools[l] + (size_t)d * (size_t)B;
        if (!src_ok) {
          memset(to, 0, (size_t)B);
          continue;
        }
        memcpy(to, host_row(g, host_pools, l, src_row), (size_t)B);
      }
    }
  }
}

/*
 * Eager backup: copy the newest token's row (seq_len - 1) from where the step left it
 * to its host row, for every layer ([SGLang-analysis] "Per decode step workflow", step 5).
 * The row is the resident row when its page is resident, slot seq_len-1 on the fast
 * path, else the reserved slot H.
 */
void oracle_backup(const oracle_geom* g, int32_t num_requests, const int32_t* seq_lens,
                   const int32_t* host_cache_locs, const int32_t* device_buffer_locs,
                   const int32_t* resident_pages, uint8_t* const* host_pools,
                   uint8_t* const* device_pools, uint32_t* err) {
  const int32_t H = g->hot_slots, B = g->row_bytes;
  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t S = seq_lens[r];
    if (S < 0 || S > g->max_context) { *err |= OR_ERR_SEQLEN; continue; }
    if (S == 0) continue;
    const int32_t t = S - 1;
    const int32_t* dbl = device_buffer_locs + (int64_t)r * (H + 1);
    int64_t row = resident_row(g, resident_pages, r, t);
    if (row < 0) row = S <= H ? dbl[t] : dbl[H];
    if (row < 0 || row >= g->device_rows) { *err |= OR_ERR_DEVROW; continue; }
    int64_t h = host_cache_locs[(int64_t)r * g->max_context + t];
    if (h < 0 || h >= g->host_rows) { *err |= OR_ERR_HOSTROW; continue; }
    for (int32_t l = 0; l < g->num_layers; ++l)
      memcpy(host_row(g, host_pools, l, h), device_pools[l] + (size_t)row * (size_t)B, (size_t)B);
  }
}

/*
 * Invalidation of hot slots ([vLLM-impl] section 6, invalidation propagation: when a host
 * block is handed to other content, hot entries that point at its old rows must go; rows
 * rewritten by prefill in this step are cleared exactly). A cleared slot is free again
 * (token -1, stamp 0, as a reset slot), so the next lookup of its token misses and copies
 * the current host row. The clock does not move.
 * Readings: slots are keyed by token, so the exact clear names tokens; only tokens in
 * [0, seq_len - 1) are considered (no valid slot holds any other); requests on the fast
 * path (seq_len <= H) are left alone, since their device rows are the tokens' own rows,
 * which the forward pass rewrites in place; seq_len outside [0, max_context] skips the
 * request (ERR_SEQLEN).
 */
static int invalidation_applies(const oracle_geom* g, int32_t S, uint32_t* err) {
  if (S < 0 || S > g->max_context) {
    *err |= OR_ERR_SEQLEN;
    return 0;
  }
  return S > g->hot_slots;
}

static void clear_slot(int32_t* tokens, int32_t* stamps, int32_t s) {
  tokens[s] = -1;
  stamps[s] = 0;
}

/* The tokens clear[offsets[r] .. offsets[r+1]) of request r leave its hot set. */
void oracle_invalidate_tokens(const oracle_geom* g, int32_t num_requests, const int32_t* seq_lens,
                              const int32_t* offsets, const int32_t* clear,
                              int32_t* device_buffer_tokens, int32_t* lru_slots, uint32_t* err) {
  const int32_t H = g->hot_slots;
  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t S = seq_lens[r];
    if (!invalidation_applies(g, S, err)) continue;
    int32_t* tokens = device_buffer_tokens + (int64_t)r * H;
    int32_t* stamps = lru_slots + (int64_t)r * H;
    for (int32_t k = offsets[r]; k < offsets[r + 1]; ++k) {
      const int32_t t = clear[k];
      if (t < 0 || t >= S - 1) continue;
      for (int32_t s = 0; s < H; ++s)
        if (tokens[s] == t) clear_slot(tokens, stamps, s);
    }
  }
}

/* Every slot whose token's host row (host_cache_locs[r][token]) is one of rows[0..n)
 * leaves the hot set, in every request. */
void oracle_invalidate_host_rows(const oracle_geom* g, int32_t num_requests, const int32_t* seq_lens,
                                 const int32_t* host_cache_locs, const int32_t* rows, int32_t n,
                                 int32_t* device_buffer_tokens, int32_t* lru_slots, uint32_t* err) {
  const int32_t H = g->hot_slots;
  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t S = seq_lens[r];
    if (!invalidation_applies(g, S, err)) continue;
    int32_t* tokens = device_buffer_tokens + (int64_t)r * H;
    int32_t* stamps = lru_slots + (int64_t)r * H;
    const int32_t* hcl = host_cache_locs + (int64_t)r * g->max_context;
    for (int32_t s = 0; s < H; ++s) {
      const int32_t t = tokens[s];
      if (t < 0 || t >= S - 1) continue;
      for (int32_t j = 0; j < n; ++j)
        if (rows[j] == hcl[t]) {
          clear_slot(tokens, stamps, s);
          break;
        }
    }
  }
}

/*
 * Backup after a speculative batch: the first accepted[r] of the batch's positions S0 + j
 * (j < num_queries) are now committed; each one's row goes to its host row, every layer.
 * The row is its resident row when its page is resident, slot S0 + j while the sequence
 * then fit the buffer (S0 + j + 1 <= H), else the reserved row H + j. accepted outside
 * [0, num_queries] or a position past max_context skips the request (ERR_SEQLEN).
 */
void oracle_backup_spec(const oracle_geom* g, int32_t num_requests, int32_t num_queries,
                        const int32_t* committed_lens, const int32_t* accepted, const int32_t* host_cache_locs,
                        const int32_t* device_buffer_locs, const int32_t* resident_pages,
                        uint8_t* const* host_pools, uint8_t* const* device_pools, uint32_t* err) {
  const int32_t H = g->hot_slots, B = g->row_bytes;
  for (int32_t r = 0; r < num_requests; ++r) {
    const int32_t S0 = committed_lens[r], n = accepted[r];
    if (S0 < 0 || n < 0 || n > num_queries || (int64_t)S0 + n > g->max_context) {
      *err |= OR_ERR_SEQLEN;
      continue;
    }
    const int32_t* dbl = device_buffer_locs + (int64_t)r * (H + num_queries);
    for (int32_t j = 0; j < n; ++j) {
      const int32_t t = S0 + j;
      int64_t row = resident_row(g, resident_pages, r, t);
      if (row < 0) row = t + 1 <= H ? dbl[t] : dbl[H + j];
      if (row < 0 || row >= g->device_rows) { *err |= OR_ERR_DEVROW; continue; }
      const int64_t h = host_cache_locs[(int64_t)r * g->max_context + t];
      if (h < 0 || h >= g->host_rows) { *err |= OR_ERR_HOSTROW; continue; }
      for (int32_t l = 0; l < g->num_layers; ++l)
        memcpy(host_row(g, host_pools, l, h), device_pools[l] + (size_t)row * (size_t)B, (size_t)B);
    }
  }
}

/* Per-request GPU bytes of the hot buffer: (n_spec + 2) * top_k rows of row_bytes for
 * each layer ([vLLM-impl] 7.1 region_stride = (max_decode_query_len + 1) * top_k with
 * max_decode_query_len = 1 + n_spec; section 9 gives 2 x 2048 x 656 B x 60 ~ 155 MiB). */
int64_t oracle_hot_bytes_per_request(int32_t top_k, int32_t n_spec, int32_t row_bytes, int32_t layers) {
  return (int64_t)(n_spec + 2) * top_k * row_bytes * layers;
}
