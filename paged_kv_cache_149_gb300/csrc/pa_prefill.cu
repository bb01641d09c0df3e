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
// Design (one CTA per (query block, sequence, kv head); 4 warps, one thread per query row):
// * The CTA's 128 query rows are (token, query head of the kv head) pairs: 128 / G tokens x
//   G heads, so every K/V tile is read once for all G heads of a kv head (GQA).  Q sits in
//   shared memory, K-major with the 128-byte swizzle (the layout tcgen05 descriptors read).
// * Key tiles of 64 tokens are gathered through the table by 16-byte cp.async into a
//   double-buffered ring, in the same swizzled layout: K is the K-major B operand of
//   S = Q K^T, V (keys x d, d contiguous) the MN-major B operand of P V.  Rows past the
//   context are zero-filled, never read.
// * Per tile: one thread issues S = Q K^T (tcgen05.mma kind::f16, M 128, N 64, fp32 in
//   tensor memory) and commits it to an mbarrier; every thread reads its own row of S with
//   tcgen05.ld (row = TMEM lane: no shuffles), applies the causal mask and the online
//   softmax in exp2, and writes its row of P (rounded to the input type) into the K
//   buffer just consumed; then one thread issues P V (M 128, N d) into a second TMEM
//   region, and every thread folds its row of P V into its fp32 O held in registers.
// * Every mbarrier wait is bounded (about 1 s, PA_DEVERR_TIMEOUT); tiles entirely in the
//   future of every row of the CTA are never loaded.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace prefill {

constexpr int kThreads = 128;  // one per query row
constexpr int kRows = 128;     // query rows of a CTA (MMA M)
constexpr int kKeys = 64;      // keys of a tile (MMA N of S, K of P V)
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;  // [n + 1]
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, tq;  // tq = tokens per CTA = 128 / G
  int max_blocks_per_seq, block_size, log2_block, num_blocks;
  float scale_log2;
  unsigned* err;
};

// P of a tile ([128 rows][64 keys], 16 KB) takes the place of the tile's K when K is at
// least as large (d >= 128), else a buffer of its own.
template <int D>
constexpr bool kAliasP = kKeys * D >= kRows * kKeys;

template <int D>
struct Smem {
  uint8_t q[kRows * D * 2];            // K-major, 128-byte swizzle; 1024-byte aligned
  uint8_t kv[2][2][kKeys * D * 2];     // [buffer][K, V]
  uint8_t p[kAliasP<D> ? 1024 : kRows * kKeys * 2];
  unsigned long long bar_s, bar_o;     // S and P V done (one phase per tile)
  uint32_t tmem;                       // tensor-memory base address
  int bad;                             // a block id of this CTA's tiles is out of range
};

// Byte offset of (row, 16-byte chunk) in a [rows][D] 16-bit tile stored K-major with the
// 128-byte swizzle: chunk c lives in the 64-element column block c / 8 (blocks rows * 128
// bytes apart), row r at r * 128 inside it, the chunk index XORed with r % 8.
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  return static_cast<uint32_t>((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// tcgen05 shared-memory matrix descriptor with the 128-byte swizzle (version 1 = sm_100
// family): lbo / sbo in bytes.  K-major operands: sbo = 1024 (8-row groups), lbo unused.
// MN-major operands: lbo = distance between 64-element MN blocks, sbo = 1024 (8-row K
// groups).
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Wait for the phase of `bar` with parity `par`, bounded by kWaitLimitNs.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t par) {
  if (mbar_try_wait(bar, par)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, par)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const __grid_constant__ Params p) {
  constexpr int CH = D / 8;            // 16-byte chunks per row
  constexpr int KS1 = D / 16;          // MMA k-steps of S = Q K^T
  constexpr int KS2 = kKeys / 16;      // MMA k-steps of P V
  constexpr uint32_t kColS = 0;        // TMEM columns: S [0, 64), P V [64, 64 + D)
  constexpr uint32_t kColO = kKeys;
  constexpr uint32_t kTmemCols = kKeys + D <= 128 ? 128 : 256;  // power of two >= 64 + D
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw + (((raw_addr + 1023) & ~1023u) - raw_addr));

  pdl_wait_primary();
  pdl_launch_dependents();

  const int tid = threadIdx.x, warp = tid >> 5;
  const int s = blockIdx.y, g = blockIdx.z;
  const int tb = gridDim.x - 1 - blockIdx.x;  // later token blocks (more keys) first
  const int qs = __ldg(p.query_start + s), qlen = __ldg(p.query_start + s + 1) - qs;
  const int tok0 = tb * p.tq;
  if (tok0 >= qlen) return;  // (uniform over the CTA)
  const int ctx = __ldg(p.context_lens + s);
  const int ntok = min(p.tq, qlen - tok0);
  const int G = p.group;
  T* outp = reinterpret_cast<T*>(p.out);
  if (ctx < 1 || ctx > p.max_blocks_per_seq * p.block_size || qlen > ctx) {
    for (int i = tid; i < ntok * G * CH; i += kThreads) {
      const int r = i / CH, c = i % CH;
      reinterpret_cast<uint4*>(outp + ((static_cast<size_t>(qs + tok0 + r / G) * p.num_q_heads +
                                        g * G + r % G) * D))[c] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) atomicOr(p.err, kErrBadContext);
    return;
  }

  // ---- this thread's row: (token tid / G, head tid % G) ----
  const bool row_ok = tid < ntok * G;
  const int pos = row_ok ? ctx - qlen + tok0 + tid / G : -1;
  const long long row_off =
      row_ok ? (static_cast<long long>(qs + tok0 + tid / G) * p.num_q_heads + g * G + tid % G) * D
             : -1;
  const int pos_lo = ctx - qlen + tok0, pos_hi = ctx - qlen + tok0 + ntok - 1;
  const int ntiles = pos_hi / kKeys + 1;

  // ---- set-up: barriers, tensor memory, Q into shared memory ----
  if (tid == 0) {
    mbar_init(smem_addr(&sm.bar_s), 1);
    mbar_init(smem_addr(&sm.bar_o), 1);
    fence_mbar_init();
    sm.bad = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&sm.tmem)), "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (row_ok ? row_off : 0) * 2);
#pragma unroll 4
    for (int c = 0; c < CH; ++c) {
      const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sm.q + swz(kRows, tid, c)) = v;
    }
  }

  const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
  auto issue_tile = [&](int kt, int b) {
    const uint32_t kbase = smem_addr(sm.kv[b][0]);
    const uint32_t vbase = smem_addr(sm.kv[b][1]);
    for (int e = tid; e < kKeys * CH; e += kThreads) {
      const int row = e / CH, c = e % CH;
      const int t = kt * kKeys + row;
      const bool live = t < ctx;
      int blk = 0;
      if (live) {
        blk = __ldg(trow + (t >> p.log2_block));
        if (blk < 0 || blk >= p.num_blocks) {
          sm.bad = 1;
          blk = 0;
        }
      }
      const size_t src = ((static_cast<size_t>(blk) * p.num_kv_heads + g) * p.block_size +
                          (live ? (t & (p.block_size - 1)) : 0)) * D + c * 8;
      const uint32_t so = swz(kKeys, row, c);
      cp_async16(kbase + so, p.k_cache + src * 2, live ? 16u : 0u);
      cp_async16(vbase + so, p.v_cache + src * 2, live ? 16u : 0u);
    }
    cp_async_commit();
  };
  __syncthreads();  // (sm.bad cleared before any copy sets it)
  issue_tile(0, 0);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = sm.tmem;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;  // this warp's TMEM lanes

  float o[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  constexpr uint32_t id_s = idesc_f16<T>(kRows, kKeys, false);
  constexpr uint32_t id_o = idesc_f16<T>(kRows, D, true);

  for (int kt = 0; kt < ntiles && ok; ++kt) {
    const int b = kt & 1;
    if (kt + 1 < ntiles) {
      issue_tile(kt + 1, b ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    // the tile's copies (generic proxy) before the tensor cores read it (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t qa = smem_addr(sm.q), kb = smem_addr(sm.kv[b][0]), vb = smem_addr(sm.kv[b][1]);

    // ---- S = Q K^T ----
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < KS1; ++ks) {
        const uint32_t koff = (ks & 3) * 32;  // 16 columns = 32 bytes within a 64-column block
        mma_f16(tmem + kColS,
                desc_sw128(qa + (ks >> 2) * kRows * 128 + koff, 16, 1024),
                desc_sw128(kb + (ks >> 2) * kKeys * 128 + koff, 16, 1024), id_s, ks > 0);
      }
      mma_commit(smem_addr(&sm.bar_s));
    }
    ok = wait_bounded(smem_addr(&sm.bar_s), kt & 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }

    // ---- this row of S: mask, online softmax, P into the K buffer ----
    float sv[kKeys];
    {
      float tmp[32];
      tmem_ld32(tmem + lane_base + kColS, tmp);
#pragma unroll
      for (int i = 0; i < 32; ++i) sv[i] = tmp[i];
      tmem_ld32(tmem + lane_base + kColS + 32, tmp);
#pragma unroll
      for (int i = 0; i < 32; ++i) sv[32 + i] = tmp[i];
    }
    const bool needs_mask = kt * kKeys + kKeys - 1 > pos_lo;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kKeys; ++i) {
      float v = sv[i] * p.scale_log2;
      if (needs_mask && kt * kKeys + i > pos) v = -INFINITY;
      sv[i] = v;
      mx = fmaxf(mx, v);
    }
    const float m_new = fmaxf(m_run, mx);
    // (a row whose keys are all masked so far keeps m = -inf; its weights stay 0)
    const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
    m_run = m_new;
    float rs = 0.f;
    uint8_t* prow = kAliasP<D> ? sm.kv[b][0] : sm.p;  // P [128][64], K-major: one column block
#pragma unroll
    for (int c = 0; c < kKeys / 8; ++c) {
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[j] = m_new == -INFINITY ? 0.f : exp2f(sv[8 * c + j] - m_new);
        rs += e[j];
      }
      uint4 w;
      w.x = pack2<T>(e[0], e[1]);
      w.y = pack2<T>(e[2], e[3]);
      w.z = pack2<T>(e[4], e[5]);
      w.w = pack2<T>(e[6], e[7]);
      *reinterpret_cast<uint4*>(prow + swz(kRows, tid, c)) = w;
    }
    l_run = l_run * alpha + rs;
    if (alpha != 1.f) {
#pragma unroll
      for (int i = 0; i < D; ++i) o[i] *= alpha;
    }
    // P (generic writes) before the tensor cores read it; every S read is done
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // ---- P V into its own TMEM columns, then O += P V ----
    if (tid == 0) {
      const uint32_t pa = smem_addr(kAliasP<D> ? sm.kv[b][0] : sm.p);
#pragma unroll
      for (int ks = 0; ks < KS2; ++ks)
        mma_f16(tmem + kColO, desc_sw128(pa + ks * 32, 16, 1024),
                desc_sw128(vb + ks * 16 * 128, kKeys * 128, 1024), id_o, ks > 0);
      mma_commit(smem_addr(&sm.bar_o));
    }
    ok = wait_bounded(smem_addr(&sm.bar_o), kt & 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float tmp[32];
      tmem_ld32(tmem + lane_base + kColO + c0, tmp);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[c0 + i] += tmp[i];
    }
    // every P V read and every thread's use of buffer b is done before it is refilled
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }
  if (!ok) {  // a wait gave up: flag it; let the copies land before leaving
    cp_async_wait<0>();
    if (tid == 0) atomicOr(p.err, kErrTimeout);
  }

  // ---- out = O / l ----
  const bool bad = sm.bad != 0 || !ok;
  if (row_ok) {
    uint4* dst = reinterpret_cast<uint4*>(outp + row_off);
    const float inv = 1.f / l_run;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (!bad) {
        w.x = pack2<T>(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
        w.y = pack2<T>(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
        w.z = pack2<T>(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
        w.w = pack2<T>(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
      }
      dst[c] = w;
    }
  }
  if (sm.bad && tid == 0) atomicOr(p.err, kErrBadBlock);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

template <int D, typename T>
int launch(const Params& prm, int max_query_len, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<D>) + 1024;
  auto* kern = prefill_kernel<D, T>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return -3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_query_len + prm.tq - 1) / prm.tq, prm.num_seqs, prm.num_kv_heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return -3;
  return 0;
}

}  // namespace prefill

int prefill_launch(const PrefillArgs& a, cudaStream_t stream) {
  prefill::Params p;
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
  p.tq = prefill::kRows / p.group;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.log2_block = a.block_size == 8 ? 3 : (a.block_size == 16 ? 4 : 5);
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * prefill::kLog2e;
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
