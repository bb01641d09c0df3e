// Paged prefill attention for sm_103a: causal multi-query attention of each sequence's
// newest tokens over its paged context, on the 5th-generation tensor cores (tcgen05).
//
// Sequence s owns query rows query_start[s] .. query_start[s+1]-1, its newest q_len tokens
// at positions p = ctx - q_len .. ctx - 1 (their K/V rows are already in the cache); the
// token at position p attends to positions 0 .. p, K/V found block by block through the
// table (daiw.org "Paged Attention", section 回顾与衔接: a FlashAttention-style kernel
// has to read the block table; chenyuan1125 "vllm-pagedattention", section 它和
// FlashAttention…: prefill works on large blocks of queries).
//
// Design: one CTA per (pair of 128-row query tiles, sequence, kv head), 384 threads in
// three roles that run concurrently and hand work over through mbarriers:
// * A query tile's rows are (token, query head of the kv head) pairs, 128 / G tokens x G
//   heads, so every K/V tile is read once for all heads of the group (GQA), and both
//   query tiles of the CTA share the K/V tiles.
// * Two loader warps: Q of both tiles once, then 64-key K tiles (one warp) and V tiles
//   (the other) into a four-stage ring, in the 128-byte swizzled layout the tcgen05
//   descriptors read.  A query tile that lies wholly inside its sequence comes by TMA (a
//   3-D tensor map over q: d, head, token; a token's G heads are adjacent rows of the
//   tile), one copy per 64-column half; a tile that runs past its sequence comes by
//   16-byte cp.async, zero-filled past the last token.  (Loading every Q row that way,
//   with an integer division by G per 16-byte copy, held each CTA for about 19000 cycles
//   before its first K tile.)  Whole K/V blocks come by TMA (a 4-D tensor map over the
//   cache: d, row, kv head, block; one copy per block and 64-column half); the ragged last
//   block and the blocks past the context by cp.async with zero fill, so no row past the
//   context is ever read (its V row must be zero: P is 0 there, and 0 x NaN is NaN).
//   Block-table entries are looked up four tiles ahead.  One thread issuing TMA copies
//   moves only about 26 GB/s per SM, so K and V each get their own issuer.  A stage of
//   the ring is free again once P V of both query tiles has read it (the same barrier
//   tells the softmax that P V is done).
// * Two MMA warps, one issuing thread per query tile: S = Q K^T into tensor memory (two
//   buffers per tile, alternate key tiles), and O += P V with P read from tensor memory
//   (the A operand, packed two values a column over the first half of its own S buffer)
//   and O kept there across the whole key range.  S of a tile's next keys is issued before
//   the current P V, so the tensor cores compute it while that tile's softmax runs, and the
//   two tiles interleave on the tensor cores.  The S MMA that refills a buffer comes after
//   the P V that read its P, and the tensor pipe runs one thread's MMAs in order: neither
//   the MMA thread nor the softmax waits for the other over a buffer, which took two
//   barrier waits off each step of the MMA thread's critical path.
// * Two softmax warpgroups, one per query tile, one thread per row (= tensor-memory
//   lane): read the row of S, mask causally, keep the running maximum m and sum l in
//   exp2 units, write the row of P (input type) over the row of S just read.
//   O is rescaled only when a row's maximum grows by more than 8 (in log2 units), so
//   P <= 2^8 and the rescale (a read-modify-write of the row in tensor memory) is rare
//   after the first tiles; the final O / l uses the same m, so the result is exact
//   softmax.  The rows of out leave through shared memory (the idle K/V ring) so that
//   every store instruction of a warp writes whole rows; storing them one row per thread,
//   as the tensor-memory lanes hold them, cost about 8 % of the from-scratch time.
// Every mbarrier wait is bounded (about 1 s) and checks a shared abort flag, so a stuck
// role ends the CTA with PA_DEVERR_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace prefill {

constexpr int kTiles = 2;       // query tiles per CTA (softmax warpgroups)
constexpr int kRows = 128;      // rows of a query tile (MMA M, tensor-memory lanes)
constexpr int kKeys = 64;       // keys of a K/V tile (MMA N of S, K of P V)
constexpr int kStages = 4;      // K/V ring
constexpr int kTableAhead = 4;  // tiles the loader looks block-table entries up ahead
constexpr int kLoadWarp = 8;    // loads Q and the K tiles
constexpr int kLoadWarpV = 11;  // loads the V tiles
constexpr int kMmaWarp = 9;     // MMA issue for tile 0; tile 1 has the next warp
constexpr int kThreads = 384;   // 2 x 128 softmax threads, two loader warps, two MMA warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;  // log2 growth of a row's maximum that forces a rescale of O

struct Params {
  CUtensorMap kmap;  // the caches as [num_blocks][Hkv][B][d] 16-bit, box (64, B, 1, 1)
  CUtensorMap vmap;
  CUtensorMap qmap;  // q as [tokens][Hq][d], box (64, G, 128 / G): one query tile's half
  int q_tma;         // qmap is valid (G divides 128, q 16-byte aligned)
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;  // [n + 1]
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, tpt;  // tpt = tokens per query tile = 128 / G
  int max_blocks_per_seq, block_size, num_blocks;
  int ncb;  // query blocks (of kTiles x tpt tokens) of the longest sequence
  float scale_log2;
  unsigned* err;
};

template <int D>
struct Smem {
  uint8_t q[kTiles][kRows * D * 2];            // K-major, 128-byte swizzle; 1024-byte aligned
  uint8_t k[kStages][kKeys * D * 2];           // [64-column half][64 keys][128 B]
  uint8_t v[kStages][kKeys * D * 2];
  unsigned long long q_full;
  unsigned long long kv_full[kStages];
  unsigned long long s_full[kTiles][2];
  unsigned long long p_full[kTiles][2];
  unsigned long long o_done[kTiles][kStages];  // P V of tile kt done (frees stage kt % kStages)
  unsigned long long fin;  // the MMA thread's last commit
  uint32_t tmem;
  int bad;    // a block id of this CTA's keys is out of range
  int abort;  // a wait gave up: every role stops
};

// Byte offset of (row, 16-byte chunk) in a [rows][D] 16-bit tile stored K-major with the
// 128-byte swizzle: chunk c lives in the 64-element column block c / 8 (blocks rows * 128
// bytes apart), row r at r * 128 inside it, the chunk index XORed with r % 8.  TMA with
// the 128-byte swizzle writes the same pattern into a 1024-byte aligned box.
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  return static_cast<uint32_t>((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// tcgen05 shared-memory matrix descriptor with the 128-byte swizzle (version 1 = sm_100
// family): lbo / sbo in bytes.  K-major operands: sbo = 1024 (8-row groups), lbo unused.
// MN-major operands: lbo = distance between 64-element MN blocks, sbo = 1024.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFF) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// tcgen05 instruction descriptor, kind::f16: fp32 accumulate, A and B of the same 16-bit
// type (bf16 or fp16), A K-major, B K-major or MN-major, M, N.
template <typename T>
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 7) |
         ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns (32 packed 16-bit values) written to this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// tcgen05.mma with A from tensor memory (lane = row, column c = elements 2c and 2c + 1).
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t db,
                                           uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(db), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
      : "memory");
}

// The same 32 columns written back.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// One arrival on `bar` once every cp.async this thread has issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2^x by the special-function unit (approximate, subnormal results flushed to zero; the
// arguments here are <= 8 and results below 2^-126 only lose weights that small).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 3-D tiled TMA load through the tensor map at `map` (a kernel parameter); completion
// counted in bytes on `bar`.  x * the element size is a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ Params p) {
  constexpr int CH = D / 8;                  // 16-byte chunks of a 16-bit row
  constexpr int KS1 = D / 16;                // MMA k-steps of S = Q K^T
  constexpr int KS2 = kKeys / 16;            // MMA k-steps of P V
  constexpr uint32_t kTileCols = 256;        // TMEM columns per query tile:
  constexpr uint32_t kColS = kKeys;          //   S of keys kt in [64 (kt % 2), + 64), its P over
                                             //   the first 32 of those columns,
  constexpr uint32_t kColO = 2 * kKeys;      //   O [128, 128 + D)
  constexpr uint32_t kTmemCols = kTiles * kTileCols;
  constexpr uint32_t kHalf = kKeys * 128;    // bytes of a 64-column half of a K/V tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw + (((raw_addr + 1023) & ~1023u) - raw_addr));

  pdl_wait_primary();
  pdl_launch_dependents();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launch order: the later half of every sequence's query blocks (the most keys) first,
  // then the earlier half, latest block first within each; the blocks of one (sequence,
  // kv head) stay together within a half, so they share their K/V in L2.  The long CTAs no
  // longer come last: 986 -> 1001 TFLOP/s on 2048-token prompts from scratch.
  const int s = blockIdx.y, g = blockIdx.z % p.num_kv_heads, half = blockIdx.z / p.num_kv_heads;
  const int nearly = p.ncb - static_cast<int>(gridDim.x);  // blocks in the earlier half
  if (half == 1 && static_cast<int>(blockIdx.x) >= nearly) return;  // (uniform over the CTA)
  const int cb = (half == 0 ? p.ncb : nearly) - 1 - static_cast<int>(blockIdx.x);
  const int qs = __ldg(p.query_start + s), qlen = __ldg(p.query_start + s + 1) - qs;
  const int tpt = p.tpt, G = p.group;
  const int tok0 = cb * kTiles * tpt;
  if (tok0 >= qlen) return;  // (uniform over the CTA)
  const int ctx = __ldg(p.context_lens + s);
  T* outp = reinterpret_cast<T*>(p.out);
  if (ctx < 1 || ctx > p.max_blocks_per_seq * p.block_size || qlen > ctx) {
    const int ntok = min(kTiles * tpt, qlen - tok0);
    for (int i = tid; i < ntok * G * CH; i += kThreads) {
      const int r = i / CH, c = i % CH;
      reinterpret_cast<uint4*>(outp + ((static_cast<size_t>(qs + tok0 + r / G) * p.num_q_heads +
                                        g * G + r % G) * D))[c] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) atomicOr(p.err, kErrBadContext);
    return;
  }
  // keys each query tile needs: 0 .. the position of its last token
  int nt[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int ntok = min(tpt, qlen - (tok0 + t * tpt));
    nt[t] = ntok > 0 ? (ctx - qlen + tok0 + t * tpt + ntok - 1) / kKeys + 1 : 0;
  }
  const int n = max(nt[0], nt[1]);

  // ---- set-up: barriers, tensor memory ----
  if (tid == 0) {
    mbar_init(smem_addr(&sm.q_full), 33);  // TMA expect-tx + 32 copy lanes
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_addr(&sm.kv_full[i]), 66);  // per loader: TMA expect-tx + 32 copy lanes
    }
    for (int t = 0; t < kTiles; ++t)
      for (int b = 0; b < 2; ++b) {
        mbar_init(smem_addr(&sm.s_full[t][b]), 1);
        mbar_init(smem_addr(&sm.p_full[t][b]), kRows);
      }
    for (int t = 0; t < kTiles; ++t)
      for (int i = 0; i < kStages; ++i) mbar_init(smem_addr(&sm.o_done[t][i]), 1);
    mbar_init(smem_addr(&sm.fin), kTiles);
    fence_mbar_init();
    sm.bad = 0;
    sm.abort = 0;
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&sm.tmem)), "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  // a bounded wait; on failure every role stops (the flag is checked inside the waits)
  auto wait = [&](unsigned long long& bar, int parity) -> bool {
    if (mbar_wait_bounded(smem_addr(&bar), static_cast<uint32_t>(parity), &sm.abort)) return true;
    if (atomicExch(&sm.abort, 1) == 0) atomicOr(p.err, kErrTimeout);
    return false;
  };

  if (warp == kLoadWarp || warp == kLoadWarpV) {
    // ===== loaders: Q once (the K loader), then the K (or V) tiles of the ring =====
    // Two warps, because one thread issuing TMA copies moves only about 26 GB/s per SM:
    // with one loader a 64-key step of both query tiles (32 KB of K and V) took about 2200
    // cycles to issue, against about 1300 cycles of tensor work.
    const bool is_v = warp == kLoadWarpV;
    if (!is_v) {
      // Q of both tiles: a whole tile (tpt tokens x G heads = 128 rows, each token's G rows
      // contiguous in q) by TMA, one copy per 64-column half; a tile that runs past the
      // sequence by 16-byte copies, zero-filled past its last token (token-major, no
      // divisions: for one token the G x D values are contiguous)
      uint32_t tma_bytes = 0;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const int first = tok0 + t * tpt;
        if (first >= qlen) continue;
        if (p.q_tma && first + tpt <= qlen) {
          tma_bytes += kRows * D * 2;
          continue;
        }
        for (int tl = 0; tl < tpt; ++tl) {
          const int tok = first + tl;
          const bool live = tok < qlen;
          const uint8_t* src =
              p.q + (static_cast<size_t>(qs + (live ? tok : 0)) * p.num_q_heads + g * G) * D * 2;
          for (int u = lane; u < G * CH; u += 32) {
            const int r = tl * G + u / CH, c = u % CH;
            cp_async16(smem_addr(sm.q[t]) + swz(kRows, r, c), src + u * 16, live ? 16u : 0u);
          }
        }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_addr(&sm.q_full), tma_bytes);
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          const int first = tok0 + t * tpt;
          if (!(p.q_tma && first < qlen && first + tpt <= qlen)) continue;
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(smem_addr(sm.q[t]) + h * kRows * 128, &p.qmap, h * 64, g * G, qs + first,
                        smem_addr(&sm.q_full));
        }
      }
      cp_async_arrive(smem_addr(&sm.q_full));
    }
    const uint8_t* cache = is_v ? p.v_cache : p.k_cache;
    const CUtensorMap* tmap = is_v ? &p.vmap : &p.kmap;
    const int B = p.block_size, nbk = kKeys / B;
    const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
    // Block-table entries, lane j holding block j of a tile, looked up kTableAhead tiles
    // before the tile is issued: a lookup is a dependent load from global memory, and
    // waiting for it at each tile made the loader the slowest role (about 2500 cycles a
    // tile, against about 1300 of tensor work for both query tiles).
    auto lookup = [&](int kt) -> int {
      const int lb = kt * nbk + lane;
      return (lane < nbk && kt < n && lb * B < ctx) ? __ldg(trow + lb) : -1;
    };
    int ahead[kTableAhead];
#pragma unroll
    for (int i = 0; i < kTableAhead; ++i) ahead[i] = lookup(i);
    for (int kt = 0; kt < n; ++kt) {
      const int st = kt % kStages;
      // this tile's blocks (lane j: block j), and the lookup kTableAhead tiles on
      const int my_e = ahead[0];
#pragma unroll
      for (int i = 0; i + 1 < kTableAhead; ++i) ahead[i] = ahead[i + 1];
      ahead[kTableAhead - 1] = lookup(kt + kTableAhead);
      if (kt >= kStages && !(wait(sm.o_done[0][st], ((kt - kStages) / kStages) & 1) &&
                             wait(sm.o_done[1][st], ((kt - kStages) / kStages) & 1)))
        break;
      const uint32_t kb = smem_addr(is_v ? sm.v[st] : sm.k[st]);
      uint32_t full_mask = 0;  // blocks that come whole by TMA
      for (int j = 0; j < nbk; ++j) {
        const int e = __shfl_sync(0xffffffffu, my_e, j);
        const int rows = min(B, max(0, ctx - (kt * nbk + j) * B));
        if (rows == B && e >= 0 && e < p.num_blocks) full_mask |= 1u << j;
      }
      if (lane == 0) {  // whole blocks by TMA
        mbar_arrive_expect_tx(smem_addr(&sm.kv_full[st]),
                              static_cast<uint32_t>(__popc(full_mask)) * B * D * 2);
      }
      {
        // lane (j, h) copies block j's 64-column half h (the copies of a tile issue side by
        // side)
        constexpr int NH = D / 64;
        const int j = lane / NH, h = lane % NH;
        const int e = __shfl_sync(0xffffffffu, my_e, j < nbk ? j : 0);
        if (j < nbk && (full_mask >> j & 1))
          tma_load_4d(kb + h * kHalf + j * B * 128, tmap, h * 64, 0, g, e, smem_addr(&sm.kv_full[st]));
      }
      // the ragged block and blocks past the context: rows by cp.async, zero-filled
      for (int j = 0; j < nbk; ++j) {
        if (full_mask >> j & 1) continue;
        const int lb = kt * nbk + j, rows = min(B, max(0, ctx - lb * B));
        const int e = __shfl_sync(0xffffffffu, my_e, j);
        const bool ok = e >= 0 && e < p.num_blocks;
        if (rows > 0 && !ok && lane == 0) sm.bad = 1;
        for (int i = lane; i < B * CH; i += 32) {
          const int r = i / CH, c = i % CH;
          const bool live = ok && r < rows;
          const size_t src =
              (((static_cast<size_t>(live ? e : 0) * p.num_kv_heads + g) * B + (live ? r : 0)) * D + c * 8) * 2;
          cp_async16(kb + swz(kKeys, j * B + r, c), cache + src, live ? 16u : 0u);
        }
      }
      cp_async_arrive(smem_addr(&sm.kv_full[st]));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ============ MMA issue: one thread per query tile (issue cost is per thread) ============
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16<T>(kRows, kKeys, false);
      constexpr uint32_t id_o = idesc_f16<T>(kRows, D, true);
      // Descriptors built once: the start address is the low field (address / 16, 14
      // bits; shared addresses here stay below 256 KB), so a byte offset o inside a tile is
      // a plain add of o / 16 -- the issue loop is then a few adds per MMA.
      constexpr uint32_t kStageBytes = kKeys * D * 2;
      const uint64_t dq0 = desc_sw128(smem_addr(sm.q[0]), 16, 1024);
      const uint64_t dq1 = desc_sw128(smem_addr(sm.q[1]), 16, 1024);
      const uint64_t dk0 = desc_sw128(smem_addr(sm.k[0]), 16, 1024);
      const uint64_t dv0 = desc_sw128(smem_addr(sm.v[0]), kKeys * 128, 1024);
      auto issue_s = [&](int t, int kt) -> bool {
        const int b = kt & 1;
        // S buffer b last held S and P of the keys two tiles back, whose P V this thread
        // issued before this S: the tensor pipe runs them in order
        const uint32_t d = tmem + t * kTileCols + b * kColS;
        const uint64_t qd = t == 0 ? dq0 : dq1;
        const uint64_t kd = dk0 + (((kt % kStages) * kStageBytes) >> 4);
        mma_f16(d, qd, kd, id_s, false);
#pragma unroll
        for (int ks = 1; ks < KS1; ++ks) {
          // k-step ks: 16 columns = 32 bytes within 64-column block ks / 4
          mma_f16(d, qd + (((ks >> 2) * kRows * 128 + (ks & 3) * 32) >> 4),
                  kd + (((ks >> 2) * kKeys * 128 + (ks & 3) * 32) >> 4), id_s, true);
        }
        mma_commit(smem_addr(&sm.s_full[t][b]));
        return true;
      };
      auto issue_pv = [&](int t, int kt) -> bool {
        const int b = kt & 1;
        if (!wait(sm.p_full[t][b], (kt >> 1) & 1)) return false;
        tc_fence_after();
        const uint64_t vd = dv0 + (((kt % kStages) * kStageBytes) >> 4);
        const uint32_t o = tmem + t * kTileCols + kColO;
        const uint32_t pa = tmem + t * kTileCols + b * kColS;
        mma_f16_ts(o, pa, vd, id_o, kt > 0);
#pragma unroll
        for (int ks = 1; ks < KS2; ++ks)  // P from tensor memory: 16 keys = 8 columns
          mma_f16_ts(o, pa + ks * 8, vd + ((ks * 16 * 128) >> 4), id_o, true);
        return true;
      };
      auto kv_ready = [&](int kt) -> bool {
        if (!wait(sm.kv_full[kt % kStages], (kt / kStages) & 1)) return false;
        fence_async_smem();  // rows the loader's lanes copied (generic proxy) -> tensor cores
        return true;
      };
      // S of the next keys goes in before P V of the current ones, so the tensor cores
      // compute it while this tile's softmax runs.  A thread whose tile needs no more keys
      // still releases each stage, after it has landed (one commit per stage and use).
      const int t = warp - kMmaWarp;
      bool ok = wait(sm.q_full, 0);
      if (ok) fence_async_smem();
      ok = ok && kv_ready(0);
      ok = ok && (nt[t] == 0 || issue_s(t, 0));
      for (int kt = 0; ok && kt < n; ++kt) {
        if (kt + 1 < n) {
          ok = kv_ready(kt + 1);
          ok = ok && (kt + 1 >= nt[t] || issue_s(t, kt + 1));
        }
        ok = ok && (kt >= nt[t] || issue_pv(t, kt));
        if (ok) mma_commit(smem_addr(&sm.o_done[t][kt % kStages]));
      }
      mma_commit(smem_addr(&sm.fin));  // every MMA this thread issued
      wait(sm.fin, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax: warpgroup t, one thread per row =================
    const int t = warp >> 2, r = tid & (kRows - 1);
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + t * kTileCols;
    const int tok = tok0 + t * tpt + r / G;
    const bool row_ok = r / G < tpt && tok < qlen;
    const int pos = row_ok ? ctx - qlen + tok : -1;
    const int pos_lo = ctx - qlen + tok0 + t * tpt;  // the tile's first position
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    auto wwait = [&](unsigned long long& bar, int parity) -> bool {  // warp-uniform result
      return __all_sync(0xffffffffu, wait(bar, parity)) != 0;
    };
    for (int kt = 0; kt < nt[t]; ++kt) {
      const int b = kt & 1;
      if (!(ok = wwait(sm.s_full[t][b], (kt >> 1) & 1))) break;
      tc_fence_after();
      float sv[kKeys];
      {
        float tmp[32];
        tmem_ld32(tl + b * kColS, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = tmp[i];
        tmem_ld32(tl + b * kColS + 32, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[32 + i] = tmp[i];
      }
      // causal mask on the raw scores (key kt*64 + i > pos), then the maximum over eight
      // independent partial chains; scores stay unscaled (the scale is positive, so the
      // maximum commutes with it) and P = 2^(s * scale - m) is one FFMA per element
      if (kt * kKeys + kKeys - 1 > pos_lo) {
        const int lim = pos - kt * kKeys;
#pragma unroll
        for (int i = 0; i < kKeys; ++i)
          if (i > lim) sv[i] = -INFINITY;
      }
      float pm[4];  // four chains of three-input maxima
#pragma unroll
      for (int j = 0; j < 4; ++j) pm[j] = fmaxf(sv[2 * j], sv[2 * j + 1]);
#pragma unroll
      for (int i = 8; i < kKeys; i += 8)
#pragma unroll
        for (int j = 0; j < 4; ++j) pm[j] = fmax3(pm[j], sv[i + 2 * j], sv[i + 2 * j + 1]);
      const float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
      const float m_new = fmaxf(m_used, mx * p.scale_log2);
      const bool need = kt > 0 && m_new > m_used + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        // rescale O (rows whose maximum grew too far) once P V of tile kt - 1 is done
        if (!(ok = wwait(sm.o_done[t][(kt - 1) % kStages], ((kt - 1) / kStages) & 1))) break;
        tc_fence_after();
        const float alpha = need ? ex2(m_used - m_new) : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(tl + kColO + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tl + kColO + c0, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        if (need) {
          l_run *= alpha;
          m_used = m_new;
        }
      }
      if (kt == 0) m_used = m_new;
      // P = 2^(s * scale - m) (0 for a row with nothing unmasked yet), rounded, packed two
      // per column over the S columns just read (P V reads it there); the row sum over
      // eight partial chains
      // (a row with nothing unmasked yet has every score at -inf, so any finite offset
      // gives it P = 0; packed FP32 pairs halve the FMA and add counts)
      // P goes over this thread's own row of S, already in registers (the P V that last
      // read this buffer ran before the S MMA that filled it)
      const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(neg_m, neg_m);
      float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = __ffma2_rn(make_float2(sv[32 * h + i], sv[32 * h + i + 1]), sc2, nm2);
          const float2 e = make_float2(ex2(x.x), ex2(x.y));
          ps[(i >> 1) & 3] = __fadd2_rn(ps[(i >> 1) & 3], e);
          pk[i >> 1] = pack2<T>(e.x, e.y);
        }
        tmem_st16(tl + b * kColS + 16 * h, pk);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      const float2 s01 = __fadd2_rn(ps[0], ps[1]), s23 = __fadd2_rn(ps[2], ps[3]);
      const float2 sall = __fadd2_rn(s01, s23);
      l_run += sall.x + sall.y;
      tc_fence_before();  // the P stores before the MMA thread reads them
      mbar_arrive(smem_addr(&sm.p_full[t][b]));
    }
    if (ok && nt[t] > 0) {
      const int last = nt[t] - 1;
      ok = wwait(sm.o_done[t][last % kStages], (last / kStages) & 1);
    }
    // ---- out = O / l, after every role is done (the loader's bad-block flag is final) ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool good = ok && sm.abort == 0 && sm.bad == 0;
    const float inv = 1.f / l_run;
    // The rows go out through shared memory (the K/V ring, idle now that every P V is
    // done), so that each store instruction of a warp writes whole rows: a warp's 32 rows
    // are 32 / G tokens x G heads (or 32 heads of one token) and rows of adjacent heads are
    // adjacent in out.  Row r's 16-byte chunk c sits at chunk c ^ (r % 16) of its 2 D-byte
    // staging row, so that neither the writes nor the reads collide in a bank much.
    const uint32_t stage = smem_addr(sm.k[0]) + static_cast<uint32_t>(warp) * 32 * D * 2;
    const int rw = r & 31;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float o[32];
      if (nt[t] > 0 && sm.abort == 0) tmem_ld32(tl + kColO + c0, o);  // (warp-uniform)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (good && nt[t] > 0) {
          w.x = pack2<T>(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
          w.y = pack2<T>(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
          w.z = pack2<T>(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
          w.w = pack2<T>(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
        }
        const int ch = c0 / 8 + c;  // 16-byte chunk of the row
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         stage + rw * D * 2 + ((ch ^ (rw & (CH - 1))) << 4)),
                     "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                     : "memory");
      }
    }
    __syncwarp();
    // piece i of the warp: row i / CH, chunk i % CH
#pragma unroll 4
    for (int i = lane; i < 32 * CH; i += 32) {
      const int rr = i / CH, ch = i % CH;
      const int rrow = (r - rw) + rr;  // the row in the tile
      const int tk = tok0 + t * tpt + rrow / G;
      if (rrow / G < tpt && tk < qlen) {
        uint4 w;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(stage + rr * D * 2 + ((ch ^ (rr & (CH - 1))) << 4)));
        reinterpret_cast<uint4*>(outp + (static_cast<size_t>(qs + tk) * p.num_q_heads + g * G + rrow % G) * D)[ch] = w;
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && sm.bad) atomicOr(p.err, kErrBadBlock);
    return;
  }
  // loader and MMA warps: the two CTA-wide barriers of the softmax epilogue
  tc_fence_before();
  __syncthreads();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int D, typename T>
int launch(const Params& prm, int max_query_len, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<D>) + 1024;
  auto* kern = prefill_kernel<D, T>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return -3;
  cudaLaunchConfig_t cfg = {};
  const int per_cta = kTiles * prm.tpt;
  const int ncb = (max_query_len + per_cta - 1) / per_cta;
  Params q = prm;
  q.ncb = ncb;
  // x: a block within its half (the later half has ceil(ncb / 2)), y: sequence,
  // z: half x kv head
  cfg.gridDim = dim3((ncb + 1) / 2, prm.num_seqs, 2 * prm.num_kv_heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, q) != cudaSuccess) return -3;
  return 0;
}

}  // namespace prefill

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the driver
// library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool kv_cache_map(CUtensorMap* map, const void* base, int elem_bytes, int num_blocks, int hkv,
                  int bs, int d) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn || (elem_bytes != 1 && elem_bytes != 2)) return false;
  const cuuint64_t eb = static_cast<cuuint64_t>(elem_bytes);
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(bs),
                              static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * eb,
                                 static_cast<cuuint64_t>(bs) * d * eb,
                                 static_cast<cuuint64_t>(hkv) * bs * d * eb};
  const int row_bytes = d * elem_bytes;
  const cuuint32_t box_x = static_cast<cuuint32_t>((row_bytes < 128 ? row_bytes : 128) / elem_bytes);
  const cuuint32_t box[4] = {box_x, static_cast<cuuint32_t>(bs), 1u, 1u};
  const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
            4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q as [tokens][Hq][d] 16-bit with a box of one query tile's 64-column half: (64, G,
// 128 / G).  `tokens` bounds the rows a launch may read (num_seqs x max_query_len); only
// tiles that lie wholly inside their sequence are read through it.
static bool q_map(CUtensorMap* map, const void* q, int hq, int d, int g, long long tokens) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn || prefill::kRows % g != 0 || tokens < 1) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hq) * d * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(prefill::kRows / g)};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int prefill_launch(const PrefillArgs& a, cudaStream_t stream) {
  prefill::Params p;
  if (!kv_cache_map(&p.kmap, a.k_cache, 2, a.num_blocks, a.num_kv_heads, a.block_size,
                    a.head_dim) ||
      !kv_cache_map(&p.vmap, a.v_cache, 2, a.num_blocks, a.num_kv_heads, a.block_size,
                    a.head_dim))
    return -3;
  p.q = static_cast<const uint8_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.query_start = a.query_start;
  p.out = static_cast<uint8_t*>(a.out);
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.tpt = prefill::kRows / p.group;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * prefill::kLog2e;
  p.q_tma = q_map(&p.qmap, a.q, a.num_q_heads, a.head_dim, p.group,
                  static_cast<long long>(a.num_seqs) * a.max_query_len)
                ? 1 : 0;
  p.err = a.err;
  if (a.head_dim == 128)
    return a.bf16 ? prefill::launch<128, __nv_bfloat16>(p, a.max_query_len, stream)
                  : prefill::launch<128, __half>(p, a.max_query_len, stream);
  if (a.head_dim == 64)
    return a.bf16 ? prefill::launch<64, __nv_bfloat16>(p, a.max_query_len, stream)
                  : prefill::launch<64, __half>(p, a.max_query_len, stream);
  return -1;
}

}  // namespace pa
