/*
 * Seeded synthetic KV-row bytes: input data for the resolver and its checks.
 *
 * This file holds no part of the resolver's method. It only produces the bytes
 * that stand in for one layer's KV row of one token of one request, as a pure
 * function of (seed, layer, request, token), so that both the CUDA path and the
 * CPU oracle see identical host pools, and a test can regenerate the exact bytes
 * a resolved row must hold.
 *
 * Word stream: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), seeded per row by chaining the mixer over
 * seed, layer, request and token. Everything is integer arithmetic or a single
 * correctly rounded IEEE operation, so x86-64 and aarch64 produce the same bytes
 * (the build passes -ffp-contract=off so no multiply-add is fused).
 *
 * Row formats (the row shapes the pages use):
 *   FMT_U8     : B uniform bytes.
 *   FMT_FP8MLA : 656 bytes = 512 fp8-e4m3 codes (NaN codes 0x7F/0xFF excluded)
 *                + 4 fp32 scales in [2^-8, 1) + 64 bf16 values ~N(0,1)
 *                (vLLM hybrid HiSparse analysis, section 9: 512 B NoPE + 16 B
 *                scales + 128 B RoPE).
 *   FMT_BF16   : B/2 bf16 values ~N(0,1) (576 x bf16 = 1152 B for the bf16 MLA row).
 * The N(0,1) values are an Irwin-Hall sum of four 16-bit uniforms, centred and
 * scaled by sqrt(3) to unit variance (bounded at +-2*sqrt(3)); the kernel never
 * reads the bytes as numbers, so only determinism matters.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <pthread.h>

enum { FMT_U8 = 0, FMT_FP8MLA = 1, FMT_BF16 = 2 };

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t row_state(uint64_t seed, int32_t layer, int32_t request, int32_t token) {
  uint64_t h = sm_mix(seed + SM_GAMMA);
  h = sm_mix(h ^ ((uint64_t)(uint32_t)layer + SM_GAMMA));
  h = sm_mix(h ^ ((uint64_t)(uint32_t)request + 2 * SM_GAMMA));
  h = sm_mix(h ^ ((uint64_t)(uint32_t)token + 3 * SM_GAMMA));
  return h;
}

/* k-th word of the row's splitmix64 stream. */
static inline uint64_t row_word(uint64_t st, uint64_t k) { return sm_mix(st + (k + 1) * SM_GAMMA); }

static inline void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static inline void put_u32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

static inline uint16_t normal_bf16(uint64_t w) {
  int32_t s = (int32_t)(w & 0xFFFF) + (int32_t)((w >> 16) & 0xFFFF) +
              (int32_t)((w >> 32) & 0xFFFF) + (int32_t)((w >> 48) & 0xFFFF);
  double x = (double)(s - 131070) * (1.7320508075688772 / 65536.0);
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even */
  return (uint16_t)(u >> 16);
}

static void make_row(uint64_t seed, int fmt, int32_t row_bytes, int32_t layer, int32_t request,
                     int32_t token, uint8_t* out) {
  uint64_t st = row_state(seed, layer, request, token);
  if (fmt == FMT_FP8MLA && row_bytes == 656) {
    uint64_t k = 0;
    for (int j = 0; j < 512; j += 8) {
      uint64_t w = row_word(st, k++);
      for (int b = 0; b < 8; ++b) {
        uint8_t c = (uint8_t)(w >> (8 * b));
        if ((c & 0x7F) == 0x7F) c = (uint8_t)(c - 1); /* 0x7F->0x7E, 0xFF->0xFE */
        out[j + b] = c;
      }
    }
    for (int j = 0; j < 4; ++j) {
      uint64_t w = row_word(st, k++);
      uint32_t u24 = (uint32_t)(w >> 40);
      double x = (double)u24 * ((1.0 - 1.0 / 256.0) / 16777216.0);
      x = x + 1.0 / 256.0;
      float f = (float)x;
      uint32_t u;
      memcpy(&u, &f, 4);
      put_u32(out + 512 + 4 * j, u);
    }
    for (int j = 0; j < 64; ++j) put_u16(out + 528 + 2 * j, normal_bf16(row_word(st, k++)));
    return;
  }
  if (fmt == FMT_BF16) {
    int32_t n = row_bytes / 2;
    for (int32_t j = 0; j < n; ++j) put_u16(out + 2 * j, normal_bf16(row_word(st, (uint64_t)j)));
    if (row_bytes & 1) out[row_bytes - 1] = (uint8_t)row_word(st, (uint64_t)n);
    return;
  }
  /* FMT_U8 (and any other size): uniform bytes */
  for (int32_t j = 0; j < row_bytes; j += 8) {
    uint64_t w = row_word(st, (uint64_t)(j / 8));
    for (int b = 0; b < 8 && j + b < row_bytes; ++b) out[j + b] = (uint8_t)(w >> (8 * b));
  }
}

/* Rows of `n` tokens of one (layer, request), written back to back into out[n * row_bytes]. */
void rowgen_rows(uint64_t seed, int32_t fmt, int32_t row_bytes, int32_t layer, int32_t request,
                 const int32_t* tokens, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i)
    make_row(seed, fmt, row_bytes, layer, request, tokens[i], out + (size_t)i * (size_t)row_bytes);
}

/* Scatter rows for (layer, request r_i, token t_i) to pool rows dst_rows[i]. */
void rowgen_scatter(uint64_t seed, int32_t fmt, int32_t row_bytes, int32_t layer,
                    const int32_t* requests, const int32_t* tokens, const int64_t* dst_rows,
                    int64_t n, uint8_t* pool) {
  for (int64_t i = 0; i < n; ++i)
    make_row(seed, fmt, row_bytes, layer, requests[i], tokens[i],
             pool + (size_t)dst_rows[i] * (size_t)row_bytes);
}

typedef struct {
  uint64_t seed;
  int32_t fmt, row_bytes, layer, num_requests, max_context;
  int64_t row_stride;
  const int32_t* seq_max;
  const int32_t* host_cache_locs;
  uint8_t* pool;
  int32_t r0, r1;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  for (int32_t r = j->r0; r < j->r1; ++r) {
    const int32_t* loc = j->host_cache_locs + (size_t)r * (size_t)j->max_context;
    for (int32_t t = 0; t < j->seq_max[r]; ++t) {
      int32_t h = loc[t];
      if (h < 0) continue;
      make_row(j->seed, j->fmt, j->row_bytes, j->layer, r, t,
               j->pool + (size_t)h * (size_t)j->row_stride);
    }
  }
  return NULL;
}

/* Fill one layer's host pool: row host_cache_locs[r][t] <- row(layer, r, t) for t < seq_max[r],
 * host row h starting h * row_stride bytes into `pool` (row_stride 0: row_bytes).
 * Work is split by request over up to `nthreads` threads. Returns 0 on success. */
int32_t rowgen_fill_pool(uint64_t seed, int32_t fmt, int32_t row_bytes, int32_t layer,
                         int32_t num_requests, const int32_t* seq_max, const int32_t* host_cache_locs,
                         int32_t max_context, uint8_t* pool, int32_t nthreads, int64_t row_stride) {
  if (row_stride <= 0) row_stride = row_bytes;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > num_requests) nthreads = num_requests > 0 ? num_requests : 1;
  pthread_t th[256];
  fill_job jobs[256];
  int started[256];
  int32_t per = (num_requests + nthreads - 1) / nthreads;
  for (int32_t i = 0; i < nthreads; ++i) {
    fill_job* j = &jobs[i];
    j->seed = seed; j->fmt = fmt; j->row_bytes = row_bytes; j->layer = layer;
    j->num_requests = num_requests; j->max_context = max_context; j->seq_max = seq_max;
    j->host_cache_locs = host_cache_locs; j->pool = pool; j->row_stride = row_stride;
    j->r0 = i * per;
    j->r1 = (i + 1) * per < num_requests ? (i + 1) * per : num_requests;
    started[i] = 0;
    if (j->r0 >= j->r1) continue;
    if (pthread_create(&th[i], NULL, fill_worker, j) == 0) started[i] = 1;
    else fill_worker(j); /* no thread available: do this share inline */
  }
  for (int32_t i = 0; i < nthreads; ++i)
    if (started[i]) pthread_join(th[i], NULL);
  return 0;
}
