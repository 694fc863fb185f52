// Synthetic consumer of the resolver's row table: sparse-MLA decode attention on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Sources (page title, section): "vLLM Hybrid HiSparse source implementation analysis", 7.3
// (the sparse attention kernel reads the pool's flat view through the table of physical
// rows) and 9 (an fp8 sparse-MLA row: 512 B of e4m3 latent, 16 B of four fp32 scales, 128 B
// of bf16 RoPE); "HiSparse: Turbocharging Sparse Attention with Hierarchical Memory" (decode
// attention only over the top-k positions, through the sparse MLA backend).
//
// Per request r and query head h over the valid rows j of out_rows[r]:
//   s[h, j] = sm_scale * (q[h, :512] . latent_j + q[h, 512:] . rope_j), latent_j = e4m3 x scale
//   o[h]    = softmax_j(s[h]) . latent,   lse[h] = log sum_j exp s[h, j]
// (MLA decode with the absorbed projection: keys are the 576-dim rows, values their latent.)
//
// Layout of the work: a CTA of 512 threads takes (request r, quarter u of the 512 value dims,
// split p of the rows) and runs a three-role pipeline over blocks of 64 rows:
//   - producers (warps 5-15) gather each block's 656-B records through the row table (staged
//     in shared memory) straight into registers, 32 rows at a time with the next 32 rows'
//     loads in flight, 16-byte loads of 16 latent codes (plus their block's scale) or of 8
//     RoPE dims each; they dequantise the latent to bf16 (e4m3 -> f16 in hardware, times the
//     scale), copy the RoPE part, and fill one of three swizzled K-major tiles (72 KB each);
//   - one issuer warp (warp 4) runs S = Q . K^T for a block as soon as its tile is full and the
//     softmax has read the previous S (36 MMAs of M 128, N 64, K 16, with Q as the A operand in
//     tensor memory), and O += P . V for the previous block once its probabilities are in (four
//     MMAs of N 128, P as the A operand in tensor memory);
//   - the softmax warpgroup (warps 0-3, one head per thread, tensor-memory lane = head) reads
//     S into registers, runs the online softmax and writes P as bf16 pairs into tensor memory.
// Tensor memory (512 columns): Q (128 heads x 576 bf16, 288 columns), S (128 x 64 fp32), P
// (128 x 64 bf16, 32 columns) and O (128 x 128 fp32). Q in tensor memory leaves shared memory
// to the tiles; the cost is that the four quarter-CTAs of a request each compute S. A
// tcgen05.mma costs about the same up to N 64 (issue-bound), so 64-row blocks halve that cost
// per row. O is rescaled only when a head's block maximum passes its reference maximum by
// more than 2^8 (a lazy rescale: P is computed against the reference and stays below 2^8).
// The roles hand blocks over through mbarriers: tile full (producers -> issuer and softmax),
// S full (issuer -> softmax), S read (softmax -> issuer), P full (softmax -> issuer), P . V done
// (issuer -> producers, which may then refill that tile, and softmax, before it rewrites P or
// rescales O). Every wait is bounded. With more than one split a small kernel merges the
// splits by their log-sum-exp.
#include "hs_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace hs {
namespace {

constexpr int T = 512;           // threads: four warpgroups
constexpr int WG = T / 128;      // warpgroups sharing the tensor-memory lanes (by column) at readout
constexpr int MH = 128;          // MMA M: heads (padded with zero rows)
constexpr int BJ = 64;           // rows per block (MMA N of S, K of P . V)
constexpr int HB = 32;           // rows a producer pass fills (a block is two passes)
constexpr int DQK = 576, DL = 512, ROWB = 656;
constexpr int ATOMS = DQK / 64;  // 9 swizzle atoms of 64 bf16 along the 576 dims
constexpr int NQ = 4;            // CTAs per (request, split): each takes a quarter of the value dims
constexpr int HALF = DL / NQ;    // value dims per CTA (128)
constexpr int ISSUER_WARP = 4;   // warp 4 issues the MMAs; warps 0-3 run the softmax
constexpr int PROD0 = 160;       // first producer thread (warps 5-15)
constexpr int NPROD = T - PROD0;
constexpr int ITEMS_ROW = DL / 16 + (DQK - DL) / 8;     // per row: 32 latent items of 16 dims, 8 RoPE of 8
constexpr int CHUNKS = HB * ITEMS_ROW;                 // producer items per pass
constexpr int PER_PROD = (CHUNKS + NPROD - 1) / NPROD;  // items per producer thread
constexpr int NT = 3;            // tiles in flight
constexpr int ROWS_CAP = 2048;   // a split's row-table entries staged in shared memory
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t Q_COL = 0;    // Q, the A operand of S = Q . K^T: 288 columns of bf16 pairs
constexpr uint32_t S_COL = 288;  // S of the current block, 64 columns (one buffer)
constexpr uint32_t P_COL = 352;  // P of the current block (bf16 pairs), 32 columns (one buffer)
constexpr uint32_t O_COL = 384;  // O, 128 x 128 fp32

// shared memory carve-up (offsets from a 1024-B aligned base)
constexpr uint32_t SKV = 0;                              // NT tiles of 9 atoms x 32 rows x 128 B
constexpr uint32_t KV_TILE = ATOMS * BJ * 128;
constexpr uint32_t SVALID = SKV + NT * KV_TILE;          // NT x 32 int (row valid, per tile)
constexpr uint32_t SROWS = SVALID + NT * BJ * 4;         // the split's rows of the row table
constexpr uint32_t SMEM_USED = SROWS + ROWS_CAP * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;        // + alignment slack
constexpr uint64_t kWaitNs = 100000000ull;               // 100 ms bound on an mbarrier wait
constexpr float kRescaleLog2 = 8.f;                      // reference-maximum slack (log2 units)

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of (row, k) in a K-major tile whose rows are 128 B (64 bf16), swizzled in
// 8-row groups of 1024 B: the 16-B chunk index is XOR-ed with row % 8.
__device__ __forceinline__ uint32_t sw128(int row, int k) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k * 2) >> 4) ^ (row & 7)) << 4) + ((k * 2) & 15));
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets, 128-B swizzle.
__device__ __forceinline__ uint64_t mdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K- or
// MN-major, N and M.
__host__ __device__ constexpr uint32_t idesc(int n, int m, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc(BJ, MH, false);   // S = Q . K^T
constexpr uint32_t kIdescO = idesc(HALF, MH, true);  // O += P . V (V read MN-major)

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// OR of a predicate over warpgroup 0's 128 threads (named barrier 1, so warpgroup 1 is not
// held up).
__device__ __forceinline__ int __syncthreads_or_wg0(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r;
}

// AND of a predicate over warpgroup 0's 128 threads (named barrier 1).
__device__ __forceinline__ int __syncthreads_and_wg0(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r;
}

// Two e4m3 codes (low byte first) to two floats, exactly (e4m3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2(uint16_t codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "h"(codes));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// MMA with A in tensor memory (Q of S, P of P . V): lane m = row m, column c = A[m][2c],
// A[m][2c + 1].
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Bounded wait for the completion of use k of a ring of `depth` barriers (barrier k % depth,
// parity of k / depth); false when the bound ran out or another role gave up (abort set).
__device__ __forceinline__ bool pipe_wait(uint64_t* ring, int depth, int k, volatile int* abort) {
  uint64_t* bar = ring + (k % depth);
  const uint32_t parity = (uint32_t)(k / depth) & 1u;
  const uint64_t t0 = gtime();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (*abort || gtime() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
}

// A producer's items of one pass: item c = (thread - PROD0) + i * NPROD covers row
// c / ITEMS_ROW; item it = c % ITEMS_ROW < 32 is latent dims [16 it, 16 it + 16) (16 codes in
// one load, and the scale of their 128-dim block), else RoPE dims [512 + 8 j, +8), j = it - 32.
// rows: this pass's entries of the row table (shared memory); n: how many are real.
__device__ __forceinline__ uint32_t load_raw(const SparseMlaArgs& a, int pt, const int32_t* rows, int n,
                                             uint4 (&raw)[PER_PROD], float (&scl)[PER_PROD]) {
  uint32_t valid = 0;  // bit i: item i's row is a pool row
#pragma unroll
  for (int i = 0; i < PER_PROD; ++i) {
    const int c = pt + i * NPROD;
    const int row = c / ITEMS_ROW, it = c - row * ITEMS_ROW;
    const int32_t pr = c < CHUNKS && row < n ? rows[row] : -1;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    float sc = 0.f;
    if (pr >= 0 && (int64_t)pr < a.pool_rows) {
      valid |= 1u << i;
      const uint8_t* rec = a.kv_pool + (size_t)pr * ROWB;
      if (it < DL / 16) {
        v = __ldg(reinterpret_cast<const uint4*>(rec) + it);
        sc = __ldg(reinterpret_cast<const float*>(rec + DL) + (it >> 3));
      } else {
        v = __ldg(reinterpret_cast<const uint4*>(rec + DL + 16) + (it - DL / 16));
      }
    }
    raw[i] = v;
    scl[i] = sc;
  }
  return valid;
}

__global__ void __launch_bounds__(T, 1) sparse_mla_kernel(const SparseMlaArgs a, float* __restrict__ part_o,
                                                          float* __restrict__ part_lse, uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint32_t s_taddr;
  // barrier rings: tile full and P . V done per tile (b % NT), S full and P full per buffer
  // (b & 1), Q in tensor memory
  __shared__ __align__(8) uint64_t s_tile_full[NT], s_o_done[NT], s_s_full, s_s_free, s_p_full, s_q_full;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = tid >> 7;
  const int head = tid & (MH - 1);  // this thread's tensor-memory lane
  const int r = blockIdx.x, u = blockIdx.y, p = blockIdx.z;
  const int per = (a.top_k + a.splits - 1) / a.splits;
  const int j_begin = p * per, j_end = min(a.top_k, j_begin + per);
  const int nblk = j_end > j_begin ? (j_end - j_begin + BJ - 1) / BJ : 0;

  if (tid == 0) {
    for (int k = 0; k < NT; ++k) {
      bar_init(&s_tile_full[k], NPROD);
      bar_init(&s_o_done[k], 1);
    }
    bar_init(&s_s_full, 1);
    bar_init(&s_s_free, MH);
    bar_init(&s_p_full, MH);
    bar_init(&s_q_full, MH);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_taddr)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tbase = s_taddr;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's tensor-memory lanes
  float m_run = -INFINITY, l_run = 0.f;
  if (wg == 0) {
    // Q of request r into tensor memory, one head per lane (zero past the last head): the A
    // operand of S = Q . K^T, column c holding dims 2c and 2c + 1
    const int h = tid;
    const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)r * a.num_heads + h) * DQK);
    for (int c0 = 0; c0 < DQK / 2; c0 += 16) {
      float v[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 w = h < a.num_heads ? __ldg(src + (c0 * 2) / 8 + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = __uint_as_float(w.x);
        v[4 * k + 1] = __uint_as_float(w.y);
        v[4 * k + 2] = __uint_as_float(w.z);
        v[4 * k + 3] = __uint_as_float(w.w);
      }
      tmem_st16(tbase + lane_off + Q_COL + c0, v);
    }
    tc_before();
    bar_arrive(&s_q_full);
  }

  if (tid >= PROD0) {
    // ---- producers: gather and dequantise block b into tile b % NT once P . V of block b - NT
    // has read it, 32 rows per pass; the next pass's records load while this one is stored
    const int pt = tid - PROD0;
    // the split's part of the row table, once, so each block's record loads wait on nothing else
    // (a split of more than ROWS_CAP rows reads them from the row table in global memory)
    const int32_t* g_rows = a.out_rows + (size_t)r * a.top_k + j_begin;
    int32_t* s_rows = reinterpret_cast<int32_t*>(base + SROWS);
    const bool staged = j_end - j_begin <= ROWS_CAP;
    if (staged)
      for (int i = pt; i < j_end - j_begin; i += NPROD) s_rows[i] = __ldg(g_rows + i);
    asm volatile("bar.sync 2, %0;" ::"n"(NPROD) : "memory");  // producers only
    const int32_t* rows_src = staged ? s_rows : g_rows;
    // pass k fills rows [32 (k & 1), 32 (k & 1) + 32) of block k / 2
    const auto pass_rows = [&](int k) { return rows_src + k * HB; };
    const auto pass_n = [&](int k) { return min(HB, j_end - j_begin - k * HB); };
    uint4 raw[PER_PROD];
    float scl[PER_PROD];
    uint32_t vmask = 0;
    if (nblk > 0) vmask = load_raw(a, pt, pass_rows(0), pass_n(0), raw, scl);
    const auto to_bf16 = [](uint32_t codes2x2, float sc) {  // four codes to two bf16 pairs
      const float2 v0 = e4m3x2((uint16_t)(codes2x2 & 0xFFFFu)), v1 = e4m3x2((uint16_t)(codes2x2 >> 16));
      __nv_bfloat162 b0 = __floats2bfloat162_rn(v0.x * sc, v0.y * sc), b1 = __floats2bfloat162_rn(v1.x * sc, v1.y * sc);
      return make_uint2(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1));
    };
    // dequantise this thread's items of rows [32 half, 32 half + 32) of a block into its tile
    const auto fill = [&](uint8_t* tile, int half) {
#pragma unroll
      for (int i = 0; i < PER_PROD; ++i) {
        const int c = pt + i * NPROD;
        if (c >= CHUNKS) continue;
        const int hrow = c / ITEMS_ROW, it = c - hrow * ITEMS_ROW;
        const int row = half * HB + hrow;
        const uint4 v = raw[i];
        if (it < DL / 16) {
          const int d = 16 * it;
          const uint2 p0 = to_bf16(v.x, scl[i]), p1 = to_bf16(v.y, scl[i]);
          const uint2 p2 = to_bf16(v.z, scl[i]), p3 = to_bf16(v.w, scl[i]);
          *reinterpret_cast<uint4*>(tile + (d >> 6) * (BJ * 128) + sw128(row, d & 63)) = make_uint4(p0.x, p0.y, p1.x, p1.y);
          *reinterpret_cast<uint4*>(tile + ((d + 8) >> 6) * (BJ * 128) + sw128(row, (d + 8) & 63)) =
              make_uint4(p2.x, p2.y, p3.x, p3.y);
        } else {
          const int d = DL + 8 * (it - DL / 16);
          *reinterpret_cast<uint4*>(tile + (d >> 6) * (BJ * 128) + sw128(row, d & 63)) = v;
        }
      }
    };
    const int npass = (j_end - j_begin + HB - 1) / HB;
    for (int b = 0; b < nblk; ++b) {
      if (b >= NT && !pipe_wait(s_o_done, NT, b - NT, abort)) break;
      uint8_t* tile = base + SKV + (b % NT) * KV_TILE;
      int32_t* valid = reinterpret_cast<int32_t*>(base + SVALID) + (b % NT) * BJ;
      for (int half = 0; half < 2; ++half) {
        const int k = 2 * b + half;
        fill(tile, half);
        // a row's validity, from the thread that holds its first item
#pragma unroll
        for (int i = 0; i < PER_PROD; ++i) {
          const int c = pt + i * NPROD;
          if (c < CHUNKS && c % ITEMS_ROW == 0) valid[half * HB + c / ITEMS_ROW] = (int32_t)((vmask >> i) & 1u);
        }
        if (k + 1 < npass) vmask = load_raw(a, pt, pass_rows(k + 1), pass_n(k + 1), raw, scl);
        else vmask = load_raw(a, pt, pass_rows(k + 1), 0, raw, scl);  // past the end: zero rows
      }
      fence_async_smem();
      bar_arrive(&s_tile_full[b % NT]);
    }
  } else if (warp == ISSUER_WARP) {
    // ---- issuer: S of block b as soon as its tile is full (Q from tensor memory), then
    // P . V of block b - 1
    const bool q_in = __all_sync(0xffffffffu, nblk == 0 || pipe_wait(&s_q_full, 1, 0, abort));
    for (int b = 0; q_in && b <= nblk; ++b) {
      if (b < nblk) {
        bool go = pipe_wait(s_tile_full, NT, b, abort);
        go = go && (b == 0 || pipe_wait(&s_s_free, 1, b - 1, abort));  // the softmax holds S of b - 1
        if (!__all_sync(0xffffffffu, go)) break;  // the warp leaves together
        tc_after();
        if (lane == 0) {
          const uint64_t dkv0 = mdesc(smem_u32(base + SKV + (b % NT) * KV_TILE), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < ATOMS * 4; ++kk) {
            const int at = kk >> 2, w = kk & 3;
            mma_ta(tbase + S_COL, tbase + Q_COL + 8 * kk, dkv0 + (uint64_t)((at * (BJ * 128) + w * 32) >> 4), kIdescS,
                   kk > 0);
          }
          commit(&s_s_full);
        }
        __syncwarp();
      }
      if (b >= 1) {
        const int pb = b - 1;
        if (!__all_sync(0xffffffffu, pipe_wait(&s_p_full, 1, pb, abort))) break;
        tc_after();
        if (lane == 0) {
          const uint64_t dv0 =
              mdesc(smem_u32(base + SKV + (pb % NT) * KV_TILE + (u * (HALF / 64)) * (BJ * 128)), BJ * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < BJ / 16; ++kk)
            mma_ta(tbase + O_COL, tbase + P_COL + 8 * kk, dv0 + (uint64_t)((kk * 2048) >> 4), kIdescO,
                   (pb > 0 || kk > 0) ? 1u : 0u);
          commit(&s_o_done[pb % NT]);
        }
        __syncwarp();
      }
    }
  } else if (wg == 0) {
    // ---- softmax: warpgroup 0, one head per thread
    const float sl2 = a.sm_scale * 1.4426950408889634f;  // scores in log2 units
    for (int b = 0; b < nblk; ++b) {
      // every exit is taken by the whole warpgroup (it meets at named barrier 1 below)
      bool got = pipe_wait(s_tile_full, NT, b, abort);
      got = got && pipe_wait(&s_s_full, 1, b, abort);
      if (!__syncthreads_and_wg0(got)) break;
      tc_after();
      float s[BJ];
      {
        const int32_t* valid = reinterpret_cast<const int32_t*>(base + SVALID) + (b % NT) * BJ;
#pragma unroll
        for (int q = 0; q < BJ / 16; ++q) {
          float t[16];
          tmem_ld16(tbase + lane_off + S_COL + 16 * q, t);
#pragma unroll
          for (int j = 0; j < 16; ++j) s[16 * q + j] = valid[16 * q + j] ? t[j] * sl2 : -INFINITY;
        }
      }
      tc_before();
      bar_arrive(&s_s_free);  // S is in registers: the next block's S may overwrite it
      float bm = -INFINITY;
#pragma unroll
      for (int j = 0; j < BJ; ++j) bm = fmaxf(bm, s[j]);
      // Lazy rescale: a head keeps its reference maximum until the block's maximum exceeds it
      // by more than kRescaleLog2, so P stays below 2^kRescaleLog2 (exact in bf16 and fp32) and
      // O in tensor memory is rescaled only on those rare jumps.
      const float m_new = bm > m_run + kRescaleLog2 || m_run == -INFINITY ? fmaxf(m_run, bm) : m_run;
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);  // m_run = -inf: O is still 0
      // P . V of block b - 1 must be done before P is rewritten (one buffer) and before O is
      // scaled
      if (!__syncthreads_and_wg0(b == 0 || pipe_wait(s_o_done, NT, b - 1, abort))) break;
      tc_after();
      if (__syncthreads_or_wg0(b > 0 && alpha != 1.f)) {
        for (int c = 0; c < HALF; c += 16) {
          float v[16];
          tmem_ld16(tbase + lane_off + O_COL + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= alpha;
          tmem_st16(tbase + lane_off + O_COL + c, v);
        }
      }
      float psum = 0.f;
#pragma unroll
      for (int q = 0; q < BJ / 32; ++q) {
        float pk[16];  // bf16 pairs, bit-cast, for 16 tensor-memory columns of P
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = m_new == -INFINITY ? 0.f : exp2f(s[32 * q + j] - m_new);
          const float p1 = m_new == -INFINITY ? 0.f : exp2f(s[32 * q + j + 1] - m_new);
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          psum += __low2float(pb) + __high2float(pb);  // the normaliser sums what P . V uses
          pk[j >> 1] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&pb));
        }
        tmem_st16(tbase + lane_off + P_COL + 16 * q, pk);
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      tc_before();
      bar_arrive(&s_p_full);
    }
  }
  // every role is done issuing; wait for the last P . V, then read O out
  bool ok = !*abort;
  if (ok && nblk > 0 && !pipe_wait(s_o_done, NT, nblk - 1, abort)) ok = false;
  ok = __syncthreads_and(ok && !*abort);
  tc_after();
  if (!ok) {  // outputs are not valid: flag it and leave them alone
    if (tid == 0) atomicOr(err, HS_FLAG_TIMEOUT);
    // give any MMA still in flight one more bound before the tensor memory is released
    s_abort = 0;
    if (nblk > 0) pipe_wait(s_o_done, NT, nblk - 1, abort);
    tc_before();
    __syncthreads();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS) : "memory");
    return;
  }
  // write this split's normalised output and log-sum-exp: warpgroup 0 holds each head's l and
  // m (handed over through the first tile, unused now); every warpgroup reads a quarter of the
  // columns of its lanes
  float* s_l = reinterpret_cast<float*>(base + SKV);
  float* s_m = s_l + MH;
  if (wg == 0) {
    s_l[tid] = l_run;
    s_m[tid] = m_run;
  }
  __syncthreads();
  l_run = s_l[head];
  m_run = s_m[head];
  const bool live = head < a.num_heads;
  const size_t row_out = (((size_t)p * gridDim.x + r) * a.num_heads + head);  // [split][r][h]
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  for (int c = wg * (HALF / WG); c < (wg + 1) * (HALF / WG); c += 16) {
    float v[16];
    if (nblk > 0) {
      tmem_ld16(tbase + lane_off + O_COL + c, v);
    } else {
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    if (live) {
      float* dst = part_o + row_out * DL + u * HALF + c;
#pragma unroll
      for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
    }
  }
  if (live && u == 0 && wg == 0)
    part_lse[row_out] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
  tc_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS) : "memory");
}

// Merge the splits of each (request, head): weights exp(lse_p - lse), lse = log sum exp lse_p.
__global__ void __launch_bounds__(T) combine_kernel(const SparseMlaArgs a, const float* __restrict__ part_o,
                                                    const float* __restrict__ part_lse) {
  const int rh = blockIdx.x;  // r * num_heads + h
  const int R = gridDim.x / a.num_heads;
  const size_t stride = (size_t)R * a.num_heads;
  float mx = -INFINITY;
  for (int p = 0; p < a.splits; ++p) mx = fmaxf(mx, part_lse[p * stride + rh]);
  float z = 0.f;
  for (int p = 0; p < a.splits; ++p) z += mx == -INFINITY ? 0.f : expf(part_lse[p * stride + rh] - mx);
  for (int d = threadIdx.x; d < DL; d += T) {
    float acc = 0.f;
    for (int p = 0; p < a.splits; ++p) {
      const float w = mx == -INFINITY ? 0.f : expf(part_lse[p * stride + rh] - mx) / z;
      acc += w * part_o[(p * stride + rh) * DL + d];
    }
    a.o[(size_t)rh * DL + d] = acc;
  }
  if (threadIdx.x == 0) a.lse[rh] = mx == -INFINITY ? -INFINITY : mx + logf(z);
}

}  // namespace

static_assert(SMEM_BYTES <= 227 * 1024, "the consumer's shared memory exceeds a CTA's limit");

size_t sparse_mla_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_sparse_mla(const SparseMlaArgs& a, int32_t num_requests, float* part_o, float* part_lse,
                              uint32_t* err, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const bool direct = a.splits == 1;
  sparse_mla_kernel<<<dim3(num_requests, NQ, a.splits), T, SMEM_BYTES, stream>>>(
      a, direct ? a.o : part_o, direct ? a.lse : part_lse, err);
  e = cudaGetLastError();
  if (e != cudaSuccess || direct) return e;
  combine_kernel<<<num_requests * a.num_heads, T, 0, stream>>>(a, part_o, part_lse);
  return cudaGetLastError();
}

}  // namespace hs
