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
// Layout of the work. A pair of CTAs in one thread-block cluster takes (request r, split p of
// the rows) and walks the split in blocks of 64 rows:
//   - the S-CTA (even cluster rank) holds Q (128 heads x 576, in f16) in tensor memory and computes
//     S = Q . K^T of each block (36 MMAs of M 128, N 64, K 16) into one of two S buffers; its
//     two softmax warpgroups (each 32 of the block's rows, one head per thread) run the
//     online softmax and write P as f16 straight into the O-CTA's shared memory (distributed
//     shared memory, asynchronous stores that complete on the O-CTA's mbarrier), with each
//     head's rescale factor;
//   - the O-CTA (the odd rank after it) holds O (128 heads x 512 fp32, all of its tensor memory) and adds
//     P . V of each block (8 MMAs of N 256, P read from shared memory); its corrector
//     warpgroup rescales O in the rare blocks that raise a head's reference maximum, and at the
//     end every warp reads O out, normalised by the S-CTA's row sums.
// So S is computed once per row and O once per value dim: no CTA repeats another's product.
// In each CTA a loader warp brings the half-blocks of 32 records into a ring of shared-memory
// buffers (eight four-row tensor gathers per half-block, mbarrier completion; the S-CTA whole
// 656-B records, the O-CTA their 528 B of latent codes and scales) through the split's row
// table staged in shared memory once, and dequantisation warps turn them into the CTA's own f16
// tile (the S-CTA all 576 dims as K, the O-CTA the 512 latent dims as V: e4m3 -> f16 in
// hardware, times the row's scale in f16; bf16 RoPE rounded to f16), swizzled K-major, two
// tiles in flight. The pair exchanges only P: shared memory between two CTAs moves ~41 GB/s
// per direction, well below what each SM reads from L2. Q comes into shared memory as nine
// swizzled 2-D tensor boxes, requested at kernel start (over the K tiles, before the first
// block), and moves into tensor memory from there. The roles hand blocks over through mbarriers
// (the two CTAs' through mbarriers in the partner's shared memory); every wait is bounded and
// an abort flag makes the other roles stop. O is rescaled only when a head's block maximum
// passes its reference maximum by more than 2^8 (a lazy rescale: P stays below 2^8). Splits
// merge by their log-sum-exp: two splits inside the kernel, the two pairs of a request sharing
// a four-CTA cluster whose O-CTAs each merge half of the value dims (when every request's
// cluster fits the device at once); otherwise, and for other split counts, in a small second
// kernel. Clusters of two CTAs serve one split and the fallback.
#include "hs_internal.h"

#include <cuda.h>  // CUtensorMap and its encoder's types (the encoder is fetched through the runtime)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

namespace hs {
namespace {

constexpr int T = 512;           // threads per CTA
constexpr int MH = 128;          // MMA M: heads (padded with zero rows)
constexpr int BJ = 64;           // rows per block (MMA N of S, K of P . V)
constexpr int HB = 32;           // rows per half-block (one loader step, one ring buffer)
constexpr int DQK = 576, DL = 512, ROWB = 656;
constexpr int KATOMS = DQK / 64;  // swizzle atoms of 64 f16 in a K tile (9) and a V tile (8)
constexpr int VATOMS = DL / 64;
constexpr int NT = 2;            // K / V tiles in flight
constexpr int NR = 3;            // raw half-block buffers in flight
constexpr uint32_t TMEM_COLS = 512;
// S-CTA tensor memory: Q (the A operand of S, f16 pairs) and two S buffers
constexpr uint32_t Q_COL = 0, S_COL = 288;
// Each CTA loads and dequantises what its own operand needs: the S-CTA whole records (656 B,
// K = all 576 dims), the O-CTA their latent codes and scales (528 B, V = the 512 latent dims).
// Shared memory between the CTAs moves only ~41 GB/s per direction, far below what the two
// SMs read from L2, so the pair exchanges P and nothing else.
constexpr int S_REC = ROWB, O_REC = DL + 16;          // bytes of a record in the raw buffers
// The loader gathers four records per tensor copy (rows of the pool seen as a 2-D tensor of
// 8-byte elements, one row per record); each group of four lands 128-byte aligned.
constexpr int S_GRP = (4 * S_REC + 127) / 128 * 128, O_GRP = (4 * O_REC + 127) / 128 * 128;
constexpr int S_SLOT = HB / 4 * S_GRP, O_SLOT = HB / 4 * O_GRP;  // a ring buffer: one half-block
constexpr int S_ITEMS = DL / 16 + (DQK - DL) / 8;     // dequantisation items per row: 16 codes or 8 RoPE dims
constexpr int O_ITEMS = DL / 16;
// S-CTA warps: 0-7 softmax (two warpgroups), 8 issuer, 9 loader, 10-15 dequantisation
constexpr int S_ISSUER = 8, S_LOADER = 9, S_DEQW0 = 10, S_NDEQW = T / 32 - S_DEQW0;
// O-CTA warps: 0-3 corrector, 4 issuer, 5 loader, 6-15 dequantisation
constexpr int O_ISSUER = 4, O_LOADER = 5, O_DEQW0 = 6, O_NDEQW = T / 32 - O_DEQW0;

// shared memory carve-up (offsets from a 1024-B aligned base); the two roles use different parts
constexpr uint32_t KV_ATOM = BJ * 128;                 // one swizzle atom of a tile: 64 rows x 128 B
constexpr uint32_t K_TILE = KATOMS * KV_ATOM, V_TILE = VATOMS * KV_ATOM;
constexpr uint32_t QBOX = MH * 128;                     // a staged Q box: 128 heads x 64 dims (128 B), swizzled
constexpr int QPITCH = DQK * 2 + 16;                   // the staging area's extent per head
constexpr uint32_t S_TILES = 0;                         // S-CTA: NT K tiles
constexpr uint32_t S_QSTAGE = 0;                        //        Q staged over them before the first block
constexpr uint32_t S_RAW = MH * QPITCH;                 //        NR raw buffers
constexpr uint32_t S_MX = S_RAW + NR * S_SLOT;         //        block maxima of the two warpgroups
constexpr uint32_t S_L1 = S_MX + 2 * MH * 4;            //        warpgroup 1's row sums at the end
constexpr uint32_t S_END = S_L1 + MH * 4;
constexpr uint32_t O_TILES = 0;                         // O-CTA: NT V tiles
constexpr uint32_t O_RAW = O_TILES + NT * V_TILE;       //        NR raw buffers
constexpr uint32_t O_P = (O_RAW + NR * O_SLOT + 1023u) & ~1023u;  // two P buffers, 128 x 64 f16
constexpr uint32_t P_BUF = MH * BJ * 2;
constexpr uint32_t O_ALPHA = O_P + 2 * P_BUF;           //        two blocks' rescale factors
constexpr uint32_t P_BYTES = P_BUF + MH * 4;            // what the S-CTA sends per block
constexpr uint32_t O_FIN = O_ALPHA + 2 * MH * 4;        //        the S-CTA's final l and m per head
constexpr uint32_t O_XLSE = O_FIN + 2 * MH * 4;         //        fused merge: the other split's lse per head
constexpr uint32_t O_END = O_XLSE + MH * 4;
constexpr int ROWS_CAP = 2048;                          // a split's row-table entries staged in shared memory
constexpr uint32_t SROWS = (S_END > O_END ? S_END : O_END);  // both: the split's rows of the row table
constexpr uint32_t SMEM_USED = SROWS + ROWS_CAP * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;       // + alignment slack
constexpr uint64_t kWaitNs = 100000000ull;              // 100 ms bound on an mbarrier wait
constexpr uint32_t kSuspendNs = 20000;                  // a waiting thread sleeps up to this long per try
                                                        // (it wakes when the phase completes), so waiting
                                                        // warps leave the issue slots to the working ones
constexpr float kRescaleLog2 = 8.f;                     // reference-maximum slack (log2 units)
constexpr int EPI_PITCH = 36;                           // floats per staged row of the read-out (16-B aligned,
                                                        // and 8 lanes' 16-B stores hit distinct banks)
static_assert(16 * 32 * EPI_PITCH * 4 <= NT * V_TILE, "the read-out staging fits the V tiles' space");
static_assert(S_RAW >= NT * K_TILE, "the staged Q covers the K tiles only");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of (row, k) in a K-major tile whose rows are 128 B (64 f16), swizzled in
// 8-row groups of 1024 B: the 16-B chunk index is XOR-ed with row % 8.
__device__ __forceinline__ uint32_t sw128(int row, int k) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k * 2) >> 4) ^ (row & 7)) << 4) + ((k * 2) & 15));
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets, 128-B swizzle.
__device__ __forceinline__ uint64_t mdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, f16 A and B, A K-major, B K- or
// MN-major, N and M.
__host__ __device__ constexpr uint32_t idesc(int n, int m, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc(BJ, MH, false);  // S = Q . K^T
constexpr uint32_t kIdescO = idesc(256, MH, true);  // O[:, n0:n0+256] += P . V (V read MN-major)

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

// OR / AND of a predicate over the first n threads of the CTA (named barrier 1; n a multiple of 32).
// Named barrier 1 serves the softmax / corrector warpgroups, 2 the dequantisation warps.
template <int id = 1>
__device__ __forceinline__ int sync_or(bool pred, int n) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %3, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(n), "n"(id)
      : "memory");
  return r;
}
template <int id = 1>
__device__ __forceinline__ int sync_and(bool pred, int n) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %3, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(n), "n"(id)
      : "memory");
  return r;
}
template <int id = 1>
__device__ __forceinline__ void sync_n(int n) {
  asm volatile("bar.sync %1, %0;" ::"r"(n), "n"(id) : "memory");
}

// Two e4m3 codes (low byte first) to an f16 pair, exactly (e4m3 is a subset of f16), times the
// row's scale in f16.
__device__ __forceinline__ uint32_t to_f16x2(uint16_t codes, __half2 sc) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "h"(codes));
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), sc);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// A bf16 pair (low half first) to an f16 pair, rounded to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// MMA with A in tensor memory (Q of S): lane m = row m, column c = A[m][2c], A[m][2c + 1].
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
// MMA with A and B in shared memory (P of P . V, and V).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// The partner CTA's copy of a shared-memory address (distributed shared memory).
__device__ __forceinline__ uint32_t remote(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void bar_arrive_remote(uint32_t raddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}
__device__ __forceinline__ void st_remote_f32(uint32_t raddr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}
// Asynchronous stores into the partner CTA's shared memory that complete their bytes on the
// partner's mbarrier (no fence or arrival of the storing thread needed).
__device__ __forceinline__ void st_async16(uint32_t raddr, uint4 v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   raddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t raddr, float v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
               "r"(__float_as_uint(v)), "r"(rbar)
               : "memory");
}
// Arrive on the mbarrier at this shared-memory offset in the cluster CTAs of `mask` once the
// MMAs issued so far are done.
__device__ __forceinline__ void commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                   "r"(smem_u32(bar)),
               "h"(mask)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Bounded wait for the completion of use k of a ring of `depth` barriers (barrier k % depth,
// parity of k / depth); false when the bound ran out or another role gave up (abort set).
// cluster: the barrier is arrived on from the partner CTA (acquire at cluster scope).
template <bool cluster = false>
__device__ __forceinline__ bool pipe_wait(uint64_t* ring, int depth, int k, volatile int* abort) {
  uint64_t* bar = ring + (k % depth);
  const uint32_t parity = (uint32_t)(k / depth) & 1u;
  const uint64_t t0 = gtime();
  for (;;) {
    uint32_t done;
    if (cluster)
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(done)
          : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(done)
          : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
          : "memory");
    if (done) return true;
    if (*abort || gtime() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
}

struct Barriers {
  uint64_t raw_full[NR];                // loader -> dequantisation: a ring buffer's records have landed
  uint64_t raw_free[NR];                // every dequantisation warp is done with a ring buffer
  uint64_t tile_full[NT];               // dequantisation -> issuer: the tile is written
  uint64_t tile_free[NT];               // the MMAs that read the tile are done
  uint64_t q_raw;                       // S-CTA: Q's boxes have landed in the staging area
  uint64_t q_full;                      // S-CTA: Q in tensor memory (its staging area is free)
  uint64_t s_full[2], s_free[2];        // S-CTA: S written by the MMAs; read by the softmax
  uint64_t p_free[2];                   // S-CTA, arrived by the O-CTA: P buffer free again
  uint64_t p_full[2];                   // O-CTA, arrived by the S-CTA: P and the factors written
  uint64_t pv_go[2];                    // O-CTA: O rescaled (if needed); P . V may go
  uint64_t mma_done;                    // O-CTA: the MMAs it issued so far are done
  uint64_t fin;                         // O-CTA, arrived by the S-CTA: final l and m written
  uint64_t xch;                         // fused merge, O-CTA: the other split's O-CTA wrote its half for this one
};

// The loader warp: half-block k's 32 records into ring buffer k % NR once every dequantisation
// warp is done with half-block k - NR, as eight four-row tensor gathers (lane g < 8: records
// 4g .. 4g + 3) that complete on raw_full; the S-CTA's tensor map spans whole records, the
// O-CTA's their first DL + 16 bytes (latent codes, scales). Rows outside the pool (and the
// rows past the split's end) are gathered as pool row 0 -- the dequantisation writes zeros for
// them -- so every gather moves the same bytes; an empty pool gathers nothing.
template <bool kS>
__device__ __forceinline__ void run_loader(const SparseMlaArgs& a, const CUtensorMap* tmap, const int32_t* rows,
                                           int n_rows, int nblk, uint8_t* raw, Barriers& bs, int lane,
                                           volatile int* abort) {
  constexpr int REC = kS ? S_REC : O_REC, GRP = kS ? S_GRP : O_GRP, SLOT = kS ? S_SLOT : O_SLOT;
  const bool any = a.pool_rows > 0;
  const int halves = 2 * nblk;
  for (int k = 0; k < halves; ++k) {
    if (k >= NR && !__all_sync(0xffffffffu, pipe_wait(bs.raw_free, NR, k - NR, abort))) break;
    const int j = HB * k + lane;
    const int32_t pr = j < n_rows ? rows[j] : -1;
    const int32_t y = pr >= 0 && (int64_t)pr < a.pool_rows ? pr : 0;  // lane l: record l's pool row
    int32_t y4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y4[i] = __shfl_sync(0xffffffffu, y, (4 * lane + i) & 31);
    if (lane == 0) bar_arrive_tx(&bs.raw_full[k % NR], any ? HB * REC : 0);
    if (any && lane < HB / 4)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
          "%4, %5, %6}], [%7];" ::"r"(smem_u32(raw + (k % NR) * SLOT + lane * GRP)),
          "l"(tmap), "r"(0), "r"(y4[0]), "r"(y4[1]), "r"(y4[2]), "r"(y4[3]), "r"(smem_u32(&bs.raw_full[k % NR]))
          : "memory");
  }
}

// One dequantisation warp's part of a half-block: items it = wq, wq + NW, ... of each of the
// 32 rows (lane = row of the half), so its 16-B reads of the raw records (272 or 400 B apart)
// and its tile stores (8 rows spread over a 128-B line by the swizzle) hit distinct banks.
// Latent items (16 codes): e4m3 -> f16 times the row's scale; RoPE items (S only, 8 dims):
// bf16 -> f16. Rows outside the pool are written as zeros.
template <bool kS>
__device__ __forceinline__ void dequant_half(const uint8_t* __restrict__ rec, uint8_t* __restrict__ tile, int row,
                                             bool valid, int wq) {
  constexpr int ITEMS = kS ? S_ITEMS : O_ITEMS;
  constexpr int NW = kS ? S_NDEQW : O_NDEQW;
  // Gather groups are 128-B aligned, so records 4 apart sit at the same bank offset: rows with
  // bit 2 set take their items in an order rotated by four, which moves their reads to the
  // other half of the banks (their tile stores stay spread by the swizzle).
  const int rot = (row & 4) ? 4 : 0;
  const uint32_t rb = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
  const int x = row & 7;
  const auto at = [&](int d) {  // byte offset of (row, dim d) in the tile
    return (uint32_t)((d >> 6) * KV_ATOM) + rb + ((uint32_t)(((d & 63) >> 3) ^ x) << 4);
  };
#pragma unroll
  for (int it0 = 0; it0 < ITEMS; it0 += NW) {
    if (it0 + wq < ITEMS) {
      const int it = it0 + wq + rot < ITEMS ? it0 + wq + rot : it0 + wq + rot - ITEMS;
      if (it < DL / 16) {
        const int d = 16 * it;
        uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
        if (valid) {
          const uint4 v = *reinterpret_cast<const uint4*>(rec + d);
          const __half2 sc = __float2half2_rn(*reinterpret_cast<const float*>(rec + DL + 4 * (d >> 7)));
          o0 = make_uint4(to_f16x2((uint16_t)(v.x & 0xFFFFu), sc), to_f16x2((uint16_t)(v.x >> 16), sc),
                          to_f16x2((uint16_t)(v.y & 0xFFFFu), sc), to_f16x2((uint16_t)(v.y >> 16), sc));
          o1 = make_uint4(to_f16x2((uint16_t)(v.z & 0xFFFFu), sc), to_f16x2((uint16_t)(v.z >> 16), sc),
                          to_f16x2((uint16_t)(v.w & 0xFFFFu), sc), to_f16x2((uint16_t)(v.w >> 16), sc));
        }
        *reinterpret_cast<uint4*>(tile + at(d)) = o0;
        *reinterpret_cast<uint4*>(tile + at(d + 8)) = o1;
      } else {
        const int e = it - DL / 16;  // RoPE dims DL + 8e .. (S only)
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          const uint4 w = *reinterpret_cast<const uint4*>(rec + DL + 16 + 16 * e);
          v = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
        }
        *reinterpret_cast<uint4*>(tile + at(DL + 8 * e)) = v;
      }
    }
  }
}

// A dequantisation warp's loop over half-blocks. In the S-CTA it waits, before its first tile
// store, until Q has left the staging area (which the K tiles overlay). Each warp goes at its
// own pace: it frees the ring buffer when done with it, and its lane 0 arrives on tile_full
// after the block's second half.
template <bool kS>
__device__ __forceinline__ void run_dequant(const SparseMlaArgs& a, const int32_t* rows, int n_rows, int nblk,
                                            const uint8_t* raw, uint8_t* tiles, Barriers& bs, int wq, int lane,
                                            volatile int* abort) {
  constexpr int REC = kS ? S_REC : O_REC, GRP = kS ? S_GRP : O_GRP, SLOT = kS ? S_SLOT : O_SLOT;
  constexpr uint32_t TB = kS ? K_TILE : V_TILE;
  const int halves = 2 * nblk;
  for (int k = 0; k < halves; ++k) {
    const int b = k >> 1;
    bool ok = true;
    if (kS && k == 0) ok = pipe_wait(&bs.q_full, 1, 0, abort);
    if ((k & 1) == 0 && b >= NT) ok = ok && pipe_wait(bs.tile_free, NT, b - NT, abort);
    ok = ok && pipe_wait(bs.raw_full, NR, k, abort);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int j = HB * k + lane;
    const int32_t pr = j < n_rows ? rows[j] : -1;
    dequant_half<kS>(raw + (k % NR) * SLOT + (lane >> 2) * GRP + (lane & 3) * REC, tiles + (b % NT) * TB,
                     (k & 1) * HB + lane, pr >= 0 && (int64_t)pr < a.pool_rows, wq);
    fence_async_smem();  // the tile's generic writes before the tensor core reads it
    __syncwarp();
    if (lane == 0) {
      bar_arrive(&bs.raw_free[k % NR]);
      if (k & 1) bar_arrive(&bs.tile_full[b % NT]);
    }
  }
}

// kCluster 2: one CTA pair per (request, split); 4: the two splits of a request as two pairs of
// one cluster, whose O-CTAs merge the splits at the end (no merge kernel).
template <int kCluster>
__global__ void __launch_bounds__(T, 1) sparse_mla_kernel(const SparseMlaArgs a, const __grid_constant__ CUtensorMap tm_s,
                                                          const __grid_constant__ CUtensorMap tm_o,
                                                          const __grid_constant__ CUtensorMap tm_q,
                                                          float* __restrict__ part_o, float* __restrict__ part_lse,
                                                          uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) Barriers bs;
  __shared__ int s_abort;
  __shared__ int s_issued;  // blocks whose MMAs the issuer started (the last commit to wait for)
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t crank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  const uint32_t rank = crank & 1u;     // 0: S-CTA, 1: O-CTA
  const uint32_t partner = crank ^ 1u;  // the other CTA of this pair
  const int r = blockIdx.x / kCluster;
  const int p = kCluster == 4 ? (int)(crank >> 1) : (int)blockIdx.y;
  const int per = (a.top_k + a.splits - 1) / a.splits;
  const int j_begin = p * per, j_end = min(a.top_k, j_begin + per);
  const int nblk = j_end > j_begin ? (j_end - j_begin + BJ - 1) / BJ : 0;

  if (tid == 0) {
    const int ndeqw = rank == 0 ? S_NDEQW : O_NDEQW;
    for (int k = 0; k < NR; ++k) {
      bar_init(&bs.raw_full[k], 1);  // the loader's arrival with the gathers' bytes
      bar_init(&bs.raw_free[k], ndeqw);
    }
    for (int k = 0; k < NT; ++k) {
      bar_init(&bs.tile_full[k], ndeqw);
      bar_init(&bs.tile_free[k], 1);
    }
    bar_init(&bs.q_raw, 1);   // the issuing thread's arrival with the boxes' bytes
    bar_init(&bs.q_full, 8);  // one arrival per warp of the two softmax warpgroups
    bar_init(&bs.mma_done, 1);
    for (int k = 0; k < 2; ++k) {
      bar_init(&bs.s_full[k], 1);
      bar_init(&bs.s_free[k], 8);
      bar_init(&bs.p_free[k], 1);
      bar_init(&bs.p_full[k], 1);  // the O-CTA's expect_tx; the S-CTA's st.async bytes complete it
      bar_init(&bs.pv_go[k], 4);  // one per corrector warp
    }
    bar_init(&bs.fin, 4);
    bar_init(&bs.xch, 1);  // fused merge: one release by the other split's O-CTA
    s_abort = 0;
    s_issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (rank == 0 && nblk > 0) {
      // S-CTA: Q of request r into the staging area (over the K tiles) as nine tensor boxes of
      // 128 heads x 64 dims, 128 B per head with its 16-B chunks swizzled by head % 8; issued
      // first, so that they land while the row table is staged. Heads past num_heads read as
      // zeros.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // q_raw's init, seen by the copies
      bar_arrive_tx(&bs.q_raw, (DQK / 64) * QBOX);
      for (int bx = 0; bx < DQK / 64; ++bx)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
            "[%4];" ::"r"(smem_u32(base + S_QSTAGE + bx * QBOX)),
            "l"(&tm_q), "r"(64 * bx), "r"(r * a.num_heads), "r"(smem_u32(&bs.q_raw))
            : "memory");
    }
    // O-CTA: the bytes blocks 0 and 1 will bring (P and the rescale factors)
    if (rank == 1)
      for (int k = 0; k < 2 && k < nblk; ++k) bar_arrive_tx(&bs.p_full[k], P_BYTES);
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
  // The split's part of the row table, once, into shared memory (a split longer than ROWS_CAP
  // rows is read from the row table in global memory).
  const int n_rows = j_end - j_begin;
  const int32_t* g_rows = a.out_rows + (size_t)r * a.top_k + j_begin;
  int32_t* s_rows = reinterpret_cast<int32_t*>(base + SROWS);
  const bool staged = n_rows <= ROWS_CAP;
  if (staged)
    for (int i = tid; i < n_rows; i += T) s_rows[i] = __ldg(g_rows + i);
  const int32_t* rows = staged ? s_rows : g_rows;
  // Both CTAs' barriers are initialised (and the rows staged) before either arrives on the other's.
  __syncthreads();
  cluster_sync_all();
  const uint32_t tbase = s_taddr;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's tensor-memory lanes
  const int head = (warp & 3) * 32 + lane;                        // = its tensor-memory lane

  if (rank == 0) {
    // ================================ S-CTA ================================
    uint8_t* tiles = base + S_TILES;
    uint8_t* raw = base + S_RAW;
    if (warp < 8) {
      // ---- softmax: warpgroup wg takes rows [32 wg, 32 wg + 32) of each block, one head per
      // thread; first, Q of request r into tensor memory (warpgroup wg the columns
      // [144 wg, 144 wg + 144)), the A operand of S = Q . K^T, column c holding dims 2c, 2c + 1
      const int wg = warp >> 2;
      if (nblk > 0) {
        // Q's staged boxes (requested at kernel start; the swizzle makes the per-head reads
        // below hit distinct banks): each thread converts its head's half of the row
        // (warpgroup wg the columns [144 wg, 144 wg + 144)) to f16 pairs in tensor memory, the
        // A operand of S = Q . K^T, column c holding dims 2c, 2c + 1.
        const uint8_t* qs = base + S_QSTAGE;
        const bool landed = sync_and(pipe_wait(&bs.q_raw, 1, 0, abort), 2 * MH);  // every softmax thread takes part
        const bool live = landed && head < a.num_heads;
        const uint8_t* src = qs + head * 128;
#pragma unroll 6
        for (int c = 36 * wg; c < 36 * wg + 36; c += 2) {  // two 16-B chunks: 16 dims, 8 columns
          uint4 x = make_uint4(0u, 0u, 0u, 0u), y = x;
          if (live) {
            x = *reinterpret_cast<const uint4*>(src + (c >> 3) * QBOX + ((((c & 7)) ^ (head & 7)) << 4));
            y = *reinterpret_cast<const uint4*>(src + ((c + 1) >> 3) * QBOX + ((((c + 1) & 7) ^ (head & 7)) << 4));
          }
          x = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
          y = make_uint4(bf16x2_to_f16x2(y.x), bf16x2_to_f16x2(y.y), bf16x2_to_f16x2(y.z), bf16x2_to_f16x2(y.w));
          asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                           tbase + lane_off + Q_COL + 4 * c),
                       "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w)
                       : "memory");
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bs.q_full);
      }
      float* s_mx = reinterpret_cast<float*>(base + S_MX);
      const uint32_t r_pbuf = remote(base + O_P, partner), r_alpha = remote(base + O_ALPHA, partner);
      const float sl2 = a.sm_scale * 1.4426950408889634f;  // scores in log2 units
      float m_run = -INFINITY, l_run = 0.f;
      for (int b = 0; b < nblk; ++b) {
        // this warpgroup's rows' validity from the row table (lane i: row 32 wg + i), loaded
        // before the wait so its latency hides behind it
        const int j = BJ * b + HB * wg + lane;
        const int32_t pr = j < n_rows ? rows[j] : -1;
        const uint32_t vm = __ballot_sync(0xffffffffu, pr >= 0 && (int64_t)pr < a.pool_rows);
        // every exit is taken by both warpgroups together (they meet at named barrier 1)
        if (!sync_and(pipe_wait(bs.s_full, 2, b, abort), 2 * MH)) break;
        tc_after();
        float s[HB];
#pragma unroll
        for (int q = 0; q < HB / 16; ++q) {
          float t[16];
          tmem_ld16(tbase + lane_off + S_COL + BJ * (b & 1) + HB * wg + 16 * q, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[16 * q + i] = ((vm >> (16 * q + i)) & 1u) ? t[i] * sl2 : -INFINITY;
        }
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bs.s_free[b & 1]);  // S is in registers: the MMAs of block b + 2 may overwrite it
        float bm = -INFINITY;
#pragma unroll
        for (int i = 0; i < HB; ++i) bm = fmaxf(bm, s[i]);
        s_mx[wg * MH + head] = bm;
        sync_n(2 * MH);
        bm = fmaxf(s_mx[head], s_mx[MH + head]);
        // Lazy rescale: a head keeps its reference maximum until the block's maximum exceeds it
        // by more than kRescaleLog2, so P stays below 2^kRescaleLog2 (well inside f16's range)
        // and O is rescaled only on those rare jumps.
        const float m_new = bm > m_run + kRescaleLog2 || m_run == -INFINITY ? fmaxf(m_run, bm) : m_run;
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);  // m_run = -inf: O is still 0
        // the O-CTA's P buffer b & 1 is free once its P . V of block b - 2 is done
        if (!sync_and(b < 2 || pipe_wait<true>(bs.p_free, 2, b - 2, abort), 2 * MH)) break;
        float psum = 0.f;
        const uint32_t pbuf = r_pbuf + (b & 1) * P_BUF;
        const uint32_t rbar = remote(&bs.p_full[b & 1], partner);
#pragma unroll
        for (int c = 0; c < HB / 8; ++c) {  // four 16-B chunks of 8 f16: rows 32 wg + 8c ..
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = m_new == -INFINITY ? 0.f : exp2f(s[8 * c + 2 * i] - m_new);
            const float p1 = m_new == -INFINITY ? 0.f : exp2f(s[8 * c + 2 * i + 1] - m_new);
            const __half2 pb = __floats2half2_rn(p0, p1);
            psum += __low2float(pb) + __high2float(pb);  // the normaliser sums what P . V uses
            w[i] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          st_async16(pbuf + sw128(head, HB * wg + 8 * c), make_uint4(w[0], w[1], w[2], w[3]), rbar);
        }
        if (wg == 0) st_async_f32(r_alpha + 4 * ((b & 1) * MH + head), alpha, rbar);
        l_run = l_run * alpha + psum;
        m_run = m_new;
      }
      // the row sums of both warpgroups, and the reference maxima, to the O-CTA
      float* s_l1 = reinterpret_cast<float*>(base + S_L1);
      if (wg == 1) s_l1[head] = l_run;
      sync_n(2 * MH);
      if (wg == 0) {
        const uint32_t fin = remote(base + O_FIN, partner);
        st_remote_f32(fin + 4 * head, l_run + s_l1[head]);
        st_remote_f32(fin + 4 * (MH + head), m_run);
        __syncwarp();
        if (lane == 0) bar_arrive_remote(remote(&bs.fin, partner));
      }
    } else if (warp == S_ISSUER) {
      // ---- issuer: S of block b once its tile is full and the softmax has read S of b - 2
      bool go = __all_sync(0xffffffffu, nblk == 0 || pipe_wait(&bs.q_full, 1, 0, abort));
      for (int b = 0; go && b < nblk; ++b) {
        bool ok = pipe_wait(bs.tile_full, NT, b, abort);
        ok = ok && (b < 2 || pipe_wait(bs.s_free, 2, b - 2, abort));
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_after();
        if (lane == 0) {
          const uint64_t dk0 = mdesc(smem_u32(tiles + (b % NT) * K_TILE), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < KATOMS * 4; ++kk) {
            const int at = kk >> 2, w = kk & 3;
            mma_ta(tbase + S_COL + BJ * (b & 1), tbase + Q_COL + 8 * kk,
                   dk0 + (uint64_t)((at * KV_ATOM + w * 32) >> 4), kIdescS, kk > 0);
          }
          commit(&bs.s_full[b & 1]);
          commit(&bs.tile_free[b % NT]);
          s_issued = b + 1;
        }
        __syncwarp();
      }
    } else if (warp == S_LOADER) {
      run_loader<true>(a, &tm_s, rows, n_rows, nblk, raw, bs, lane, abort);
    } else {
      run_dequant<true>(a, rows, n_rows, nblk, raw, tiles, bs, warp - S_DEQW0, lane, abort);
    }
  } else {
    // ================================ O-CTA ================================
    uint8_t* tiles = base + O_TILES;
    uint8_t* raw = base + O_RAW;
    const float* alpha_buf = reinterpret_cast<const float*>(base + O_ALPHA);
    if (warp < 4) {
      // ---- corrector: block b's P and factors are in; if a head's reference maximum rose,
      // rescale O once P . V of block b - 1 is done; then P . V of block b may go
      for (int b = 0; b < nblk; ++b) {
        if (!sync_and(pipe_wait<true>(bs.p_full, 2, b, abort), MH)) break;
        const float f = alpha_buf[(b & 1) * MH + head];
        // this buffer's next phase is block b + 2: its bytes come only after P . V of block b
        if (tid == 0 && b + 2 < nblk) bar_arrive_tx(&bs.p_full[b & 1], P_BYTES);
        if (sync_or(b > 0 && f != 1.f, MH)) {
          if (!sync_and(pipe_wait(bs.tile_free, NT, b - 1, abort), MH)) break;
          tc_after();
          for (int c = 0; c < DL; c += 16) {
            float v[16];
            tmem_ld16(tbase + lane_off + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= f;
            tmem_st16(tbase + lane_off + c, v);
          }
          tc_before();
        }
        __syncwarp();
        if (lane == 0) bar_arrive(&bs.pv_go[b & 1]);
      }
    } else if (warp == O_ISSUER) {
      // ---- issuer: O += P . V of block b once its tile is full and O is ready for it; then
      // the P buffer of block b - 1 goes back to the S-CTA when its MMAs are done
      for (int b = 0; b < nblk; ++b) {
        bool ok = pipe_wait(bs.tile_full, NT, b, abort);
        ok = ok && pipe_wait(bs.pv_go, 2, b, abort);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_after();
        fence_async_smem();
        if (lane == 0) {
          const uint64_t dp0 = mdesc(smem_u32(base + O_P + (b & 1) * P_BUF), 16, 1024);
          const uint64_t dv0 = mdesc(smem_u32(tiles + (b % NT) * V_TILE), KV_ATOM, 1024);
#pragma unroll
          for (int kk = 0; kk < BJ / 16; ++kk)
#pragma unroll
            for (int nh = 0; nh < 2; ++nh)
              mma_ss(tbase + 256 * nh, dp0 + (uint64_t)((kk * 32) >> 4),
                     dv0 + (uint64_t)((nh * 4 * KV_ATOM + kk * 2048) >> 4), kIdescO, (b > 0 || kk > 0) ? 1u : 0u);
          commit(&bs.tile_free[b % NT]);
          commit_multicast(&bs.p_free[b & 1], (uint16_t)(1u << partner));  // the S-CTA's P buffer is free once these are done
          commit(&bs.mma_done);
          s_issued = b + 1;
        }
        __syncwarp();
      }
    } else if (warp == O_LOADER) {
      run_loader<false>(a, &tm_o, rows, n_rows, nblk, raw, bs, lane, abort);
    } else {
      run_dequant<false>(a, rows, n_rows, nblk, raw, tiles, bs, warp - O_DEQW0, lane, abort);
    }
  }

  __syncthreads();
  // this CTA's MMAs of every block are done; the O-CTA also has the S-CTA's totals, the S-CTA
  // the O-CTA's last P-buffer releases (its last arrivals here)
  bool ok = !*abort && (nblk == 0 || pipe_wait(bs.tile_free, NT, nblk - 1, abort));
  if (rank == 1) {
    ok = ok && pipe_wait<true>(&bs.fin, 1, 0, abort);
  } else {
    for (int b = nblk >= 2 ? nblk - 2 : 0; b < nblk; ++b) ok = ok && pipe_wait<true>(bs.p_free, 2, b, abort);
  }
  ok = __syncthreads_and(ok && !*abort);
  tc_after();
  if (rank == 1 && ok) {
    // O out, normalised: warp w holds heads 32 (w & 3) .. + 31 (its tensor-memory lanes) and
    // reads its columns 32 at a time; each 32 x 32 piece goes through the warp's own staging
    // rows in shared memory (the V tiles' space, free now) so that every global store writes
    // whole 128-byte lines: 8 lanes per row, 4 rows per instruction.
    const float* fin = reinterpret_cast<const float*>(base + O_FIN);
    const float l = fin[head], m = fin[MH + head];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    const int nreq = (int)(gridDim.x / kCluster);
    const int head0 = (warp & 3) * 32;
    float* stg = reinterpret_cast<float*>(base + O_TILES) + warp * (32 * EPI_PITCH);
    // columns c .. c + 31 of the warp's heads, normalised, into its staging rows
    auto stage = [&](int c) {
      float v[32];
      if (nblk > 0) {
        tmem_ld16(tbase + lane_off + c, *reinterpret_cast<float(*)[16]>(v));
        tmem_ld16(tbase + lane_off + c + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(stg + lane * EPI_PITCH + i) =
            make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
      __syncwarp();
    };
    // the staged piece at column c, as is, to rows [h][DL] from `rows`
    auto put = [&](float* rows, int c) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3), q4 = lane & 7;  // row of the piece, four-float column
        if (head0 + rr < a.num_heads)
          *reinterpret_cast<float4*>(rows + (size_t)(head0 + rr) * DL + c + 4 * q4) =
              *reinterpret_cast<const float4*>(stg + rr * EPI_PITCH + 4 * q4);
      }
      __syncwarp();
    };
    float* own_rows = part_o + (((size_t)p * nreq + r) * a.num_heads) * DL;  // [split][r][h][DL]
    if (kCluster == 2) {
      const int c0 = (warp >> 2) * (DL / 4);  // a quarter of the columns per warp
      for (int c = c0; c < c0 + DL / 4; c += 32) {
        stage(c);
        put(own_rows, c);
      }
      if (head < a.num_heads && warp < 4) part_lse[((size_t)p * nreq + r) * a.num_heads + head] = lse;
    } else {
      // Both splits of request r in this cluster: the O-CTA of split p merges columns
      // [256 p, 256 p + 256) of both and hands the other 256 columns of its own output, and its
      // lse, to the other split's O-CTA. Warp w takes 64 columns of each half (w >> 2 picks them).
      const int q = 1 - p;
      const uint32_t xo = crank ^ 2u;  // the other split's O-CTA
      const int cj = (warp >> 2) * (DL / 8);
      for (int c = DL / 2 * q + cj; c < DL / 2 * q + cj + DL / 8; c += 32) {
        stage(c);
        put(own_rows, c);
      }
      if (warp < 4) st_remote_f32(remote(base + O_XLSE, xo) + 4 * head, lse);
      // every thread's hand-off stores before one release at cluster scope
      __syncthreads();
      if (tid == 0) {
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        bar_arrive_remote(remote(&bs.xch, xo));
      }
      const bool go = __all_sync(0xffffffffu, pipe_wait<true>(&bs.xch, 1, 0, abort));
      if (!go && lane == 0) atomicOr(err, HS_FLAG_TIMEOUT);
      // the two splits' weights for this lane's head and the merged lse (the merge kernel's
      // arithmetic, in split order)
      const float other = reinterpret_cast<const float*>(base + O_XLSE)[head];
      const float l0 = p == 0 ? lse : other, l1 = p == 0 ? other : lse;
      const float mx = fmaxf(fmaxf(-INFINITY, l0), l1);
      float w0 = 0.f, w1 = 0.f, lse_all = -INFINITY;
      if (mx != -INFINITY) {
        const float z = expf(l0 - mx) + expf(l1 - mx);
        const float iz = 1.f / z;
        w0 = expf(l0 - mx) * iz;
        w1 = expf(l1 - mx) * iz;
        lse_all = mx + logf(z);
      }
      const float* other_rows = part_o + (((size_t)q * nreq + r) * a.num_heads) * DL;
      float* out_rows = a.o + ((size_t)r * a.num_heads) * DL;
      for (int c = DL / 2 * p + cj; go && c < DL / 2 * p + cj + DL / 8; c += 32) {
        // the other split's piece first (from L2), so its latency overlaps the staging
        float4 ys[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + (lane >> 3), q4 = lane & 7;
          ys[i] = head0 + rr < a.num_heads
                      ? __ldcg(reinterpret_cast<const float4*>(other_rows + (size_t)(head0 + rr) * DL + c + 4 * q4))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        stage(c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + (lane >> 3), q4 = lane & 7;
          const size_t at = (size_t)(head0 + rr) * DL + c + 4 * q4;
          const float wa = __shfl_sync(0xffffffffu, w0, rr), wb = __shfl_sync(0xffffffffu, w1, rr);
          if (head0 + rr < a.num_heads) {
            const float4 x = *reinterpret_cast<const float4*>(stg + rr * EPI_PITCH + 4 * q4);
            const float4 y = ys[i];
            const float4 v0 = p == 0 ? x : y, v1 = p == 0 ? y : x;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            acc.x += wa * v0.x;
            acc.y += wa * v0.y;
            acc.z += wa * v0.z;
            acc.w += wa * v0.w;
            acc.x += wb * v1.x;
            acc.y += wb * v1.y;
            acc.z += wb * v1.z;
            acc.w += wb * v1.w;
            *reinterpret_cast<float4*>(out_rows + at) = acc;
          }
        }
        __syncwarp();
      }
      if (go && p == 0 && warp < 4 && head < a.num_heads) a.lse[(size_t)r * a.num_heads + head] = lse_all;
    }
  }
  if (!ok) {
    // outputs are not valid: flag it, and give any MMA still in flight one more bound before
    // the tensor memory is released
    if (tid == 0) atomicOr(err, HS_FLAG_TIMEOUT);
    __syncthreads();
    if (tid == 0) s_abort = 0;
    __syncthreads();
    const int n = s_issued;
    if (n > 0) {
      if (rank == 0)
        pipe_wait(bs.s_full, 2, n - 1, abort);
      else
        pipe_wait(&bs.mma_done, 1, n - 1, abort);
    }
  }
  tc_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS) : "memory");
  // the merge kernel (if any) may launch; it waits for this grid's completion before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the partner no longer reads or arrives on this CTA's shared memory
  cluster_sync_all();
}

// Merge the splits of each (request, head): weights exp(lse_p - lse), lse = log sum exp lse_p.
// One thread per four consecutive output dims, so every thread issues its splits' loads
// together (the merge is a pass over the splits' partial outputs, bound by memory latency and
// bandwidth, not arithmetic).
constexpr int COMBINE_T = 256;
__global__ void __launch_bounds__(COMBINE_T) combine_kernel(const SparseMlaArgs a, int rh_total,
                                                            const float* __restrict__ part_o,
                                                            const float* __restrict__ part_lse) {
  // launched as a programmatic dependent of the attention kernel: wait until that grid has
  // finished and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int g = blockIdx.x * COMBINE_T + threadIdx.x;  // (r * num_heads + h) * 128 + quarter-dim index
  const int rh = g >> 7, c4 = g & 127;
  if (rh >= rh_total) return;
  const size_t stride = (size_t)rh_total;
  float mx = -INFINITY;
  for (int p = 0; p < a.splits; ++p) mx = fmaxf(mx, __ldg(part_lse + p * stride + rh));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (mx != -INFINITY) {
    for (int p = 0; p < a.splits; ++p) z += expf(__ldg(part_lse + p * stride + rh) - mx);
    const float inv = 1.f / z;
    for (int p = 0; p < a.splits; ++p) {
      const float w = expf(__ldg(part_lse + p * stride + rh) - mx) * inv;
      const float4 v = __ldg(reinterpret_cast<const float4*>(part_o + (p * stride + rh) * DL) + c4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
  reinterpret_cast<float4*>(a.o + (size_t)rh * DL)[c4] = acc;
  if (c4 == 0) a.lse[rh] = mx == -INFINITY ? -INFINITY : mx + logf(z);
}

}  // namespace

static_assert(SMEM_BYTES <= 227 * 1024, "the consumer's shared memory exceeds a CTA's limit");

size_t sparse_mla_smem_bytes() { return SMEM_BYTES; }

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched once through the runtime (no link against the
// driver library).
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// The pool as a 2-D tensor of 8-byte elements, one row per record (656 B = 82 elements), read
// `box_bytes` at a time from the start of a row (one row per box: the gathers pick the rows).
cudaError_t pool_map(CUtensorMap* m, const uint8_t* pool, int64_t rows, int box_bytes) {
  EncodeTiled fn = encoder();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)(ROWB / 8), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ROWB};
  const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 8), 1u};
  const cuuint32_t elem[2] = {1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(pool), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Q ([rows = requests x heads][576] bf16) as a 2-D tensor read in boxes of 128 rows x 64 dims
// (128 B), swizzled in 128-byte rows (the 16-B chunk index XOR-ed with the row % 8); rows past
// the end read as zeros.
cudaError_t q_map(CUtensorMap* m, const uint16_t* q, int64_t rows) {
  EncodeTiled fn = encoder();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)DQK, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)DQK * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)MH};
  const cuuint32_t elem[2] = {1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(q), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

namespace {

// The kernel's launch: a cluster of kCluster CTAs per request and split group, with the dynamic
// shared memory it needs.
template <int kCluster>
cudaLaunchConfig_t mla_config(int32_t num_requests, int splits, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = kCluster == 4 ? dim3(4u * (unsigned)num_requests, 1u)  // both splits' pairs of a request
                              : dim3(2u * (unsigned)num_requests, (unsigned)splits);  // a pair per (request, split)
  cfg.blockDim = dim3(T);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Four-CTA clusters of this kernel that the device holds at once (queried once per device).
int fused_clusters_resident() {
  static std::mutex mu;
  static int cached[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = mla_config<4>(1, 2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_kernel<4>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cached[dev] = n;
    known[dev] = true;
  }
  return cached[dev];
}

// Two splits merge inside the kernel when every request's four-CTA cluster fits at once.
bool merge_in_kernel(int32_t num_requests, int splits) {
  return splits == 2 && fused_clusters_resident() >= num_requests;
}

}  // namespace

int sparse_mla_launches(int32_t num_requests, int splits) {
  if (cudaFuncSetAttribute(sparse_mla_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return splits == 1 ? 1 : 2;
  }
  return splits == 1 || merge_in_kernel(num_requests, splits) ? 1 : 2;
}

cudaError_t launch_sparse_mla(const SparseMlaArgs& a, int32_t num_requests, float* part_o, float* part_lse,
                              uint32_t* err, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(sparse_mla_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  CUtensorMap tm_s, tm_o, tm_q;  // an empty pool is never gathered from
  memset(&tm_s, 0, sizeof(tm_s));
  memset(&tm_o, 0, sizeof(tm_o));
  if ((e = q_map(&tm_q, a.q, (int64_t)num_requests * a.num_heads)) != cudaSuccess) return e;
  if (a.pool_rows > 0) {
    if ((e = pool_map(&tm_s, a.kv_pool, a.pool_rows, S_REC)) != cudaSuccess) return e;
    if ((e = pool_map(&tm_o, a.kv_pool, a.pool_rows, O_REC)) != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  // two splits whose four-CTA clusters all fit at once: merged inside the kernel
  if (merge_in_kernel(num_requests, a.splits)) {
    const cudaLaunchConfig_t cfg = mla_config<4>(num_requests, 2, stream, attr);
    return cudaLaunchKernelEx(&cfg, sparse_mla_kernel<4>, a, tm_s, tm_o, tm_q, part_o, part_lse, err);
  }
  const bool direct = a.splits == 1;
  const cudaLaunchConfig_t cfg = mla_config<2>(num_requests, a.splits, stream, attr);
  e = cudaLaunchKernelEx(&cfg, sparse_mla_kernel<2>, a, tm_s, tm_o, tm_q, direct ? a.o : part_o,
                         direct ? a.lse : part_lse, err);
  if (e != cudaSuccess || direct) return e;
  const int rh_total = num_requests * a.num_heads;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3((unsigned)((rh_total * (DL / 4) + COMBINE_T - 1) / COMBINE_T));
  mc.blockDim = dim3(COMBINE_T);
  mc.stream = stream;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  mc.attrs = pdl;
  mc.numAttrs = 1;
  return cudaLaunchKernelEx(&mc, combine_kernel, a, rh_total, (const float*)part_o, (const float*)part_lse);
}

}  // namespace hs
