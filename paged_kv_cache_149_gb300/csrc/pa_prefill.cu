// Paged prefill attention for sm_103a: causal multi-query attention of each sequence's
// newest tokens over its paged context.
//
// Sequence s owns query rows query_start[s] .. query_start[s+1]-1, its newest q_len tokens
// at positions p = ctx - q_len .. ctx - 1 (their K/V rows are already in the cache); the
// token at position p attends to positions 0 .. p, K/V found block by block through the
// table (daiw.org "Paged Attention", section 回顾与衔接: a FlashAttention-style kernel
// has to read the block table; chenyuan1125 "vllm-pagedattention", section 它和
// FlashAttention…: prefill works on large blocks of queries).
//
// Design (one CTA per (query block, sequence, kv head); 4 warps):
// * The CTA's 64 query rows are (token, query head of the kv head) pairs: TQ = 64 / G
//   tokens x G heads, so every K/V tile is read once for all G heads of a kv head (GQA).
//   Each warp owns 16 rows; its Q rows stay in registers as MMA A fragments.
// * Key tiles of 64 tokens (four 16-row groups, each one block row range found through the
//   table) are copied by all 128 threads with 16-byte cp.async into a double-buffered,
//   swizzled shared-memory ring (rows past the context are zero-filled, never read).
// * Per tile, warp-level tensor-core MMAs (m16n8k16, fp32 accumulate): S = Q K^T, online
//   softmax per row in exp2 (the causal mask only on tiles that reach past a row's
//   position), P rounded to the input type straight from the S accumulators into A
//   fragments, O += P V with V through ldmatrix.trans.  Tiles entirely in the future of
//   every row of the CTA are never loaded.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace prefill {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 64;   // query rows of a CTA
constexpr int kKeys = 64;   // keys of a tile
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;  // [n + 1]
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, tq;  // tq = tokens per CTA = 64 / G
  int max_blocks_per_seq, block_size, log2_block, num_blocks;
  float scale_log2;
  unsigned* err;
};

template <int D>
struct Smem {
  uint8_t kv[2][2][kKeys * D * 2];  // [buffer][K, V][tile], 1024-byte aligned
  int bad;                          // a block id of this CTA's tiles is out of range
};

// Byte offset of (row, 16-byte chunk) in a [kKeys][D] tile: chunk c of a row lives in
// column half c / 8 (128 bytes of each row per half), and the 128-byte swizzle permutes the
// chunks of a row so that ldmatrix reads are conflict-free.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kKeys * 128) + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const __grid_constant__ Params p) {
  constexpr int KS = D / 16;      // k-steps of Q K^T
  constexpr int NK = kKeys / 8;   // n-tiles of S (8 keys each)
  constexpr int ND = D / 8;       // n-tiles of O (8 d each)
  constexpr int CH = D / 8;       // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw + (((raw_addr + 1023) & ~1023u) - raw_addr));

  pdl_wait_primary();
  pdl_launch_dependents();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.y, g = blockIdx.z;
  const int tb = gridDim.x - 1 - blockIdx.x;  // later token blocks (more keys) first
  const int qs = __ldg(p.query_start + s), qlen = __ldg(p.query_start + s + 1) - qs;
  const int tok0 = tb * p.tq;
  if (tok0 >= qlen) return;  // (uniform over the CTA)
  const int ctx = __ldg(p.context_lens + s);
  const int ntok = min(p.tq, qlen - tok0);  // tokens of this CTA
  const int G = p.group;
  T* outp = reinterpret_cast<T*>(p.out);
  const bool bad_ctx = ctx < 1 || ctx > p.max_blocks_per_seq * p.block_size || qlen > ctx;
  if (bad_ctx) {  // zeros for this CTA's rows, and a flag
    for (int i = tid; i < ntok * G * D / 8; i += kThreads) {
      const int r = i / (D / 8), c = i % (D / 8);
      const int t = r / G, hh = r % G;
      reinterpret_cast<uint4*>(outp + ((static_cast<size_t>(qs + tok0 + t) * p.num_q_heads +
                                        g * G + hh) * D))[c] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) atomicOr(p.err, kErrBadContext);
    return;
  }
  if (tid == 0) sm.bad = 0;
  __syncthreads();  // (before any copy can set it)

  // ---- this warp's 16 rows: r = 16*warp + {r0, r0+8}; row = (token r / G, head r % G) ----
  const int r0 = lane >> 2, qc = 2 * (lane & 3);
  const int rows_used = ntok * G;
  int pos[2];             // position of each of this lane's two rows (-1: an unused row)
  long long qrow_off[2];  // element offset of the row's q / out vector (-1: unused)
  for (int i = 0; i < 2; ++i) {
    const int r = 16 * warp + r0 + 8 * i;
    if (r < rows_used) {
      const int t = r / G, hh = r % G;
      pos[i] = ctx - qlen + tok0 + t;
      qrow_off[i] = (static_cast<long long>(qs + tok0 + t) * p.num_q_heads + g * G + hh) * D;
    } else {
      pos[i] = -1;
      qrow_off[i] = -1;
    }
  }
  // Q as A fragments: a0 (row r0, k 2lq..), a1 (row r0+8), a2 (row r0, k +8), a3 (row r0+8)
  uint32_t qa[KS][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int col = 16 * ks + qc;
      qa[ks][0] = qrow_off[0] >= 0 ? __ldg(q32 + (qrow_off[0] + col) / 2) : 0u;
      qa[ks][1] = qrow_off[1] >= 0 ? __ldg(q32 + (qrow_off[1] + col) / 2) : 0u;
      qa[ks][2] = qrow_off[0] >= 0 ? __ldg(q32 + (qrow_off[0] + col + 8) / 2) : 0u;
      qa[ks][3] = qrow_off[1] >= 0 ? __ldg(q32 + (qrow_off[1] + col + 8) / 2) : 0u;
    }
  }

  // key tiles this CTA needs: 0 .. (highest position of its rows) / 64
  const int pos_hi = ctx - qlen + tok0 + ntok - 1;
  const int pos_lo = ctx - qlen + tok0;
  const int ntiles = pos_hi / kKeys + 1;

  // ---- copy of key tile kt into buffer b (all threads) ----
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
      const uint32_t so = swz(row, c);
      const bool ok = live && blk >= 0;
      cp_async16(kbase + so, p.k_cache + src * 2, ok ? 16u : 0u);
      cp_async16(vbase + so, p.v_cache + src * 2, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  const int lrow = lane & 7, lmat = lane >> 3;

  issue_tile(0, 0);
  for (int kt = 0; kt < ntiles; ++kt) {
    const int b = kt & 1;
    if (kt + 1 < ntiles) {
      issue_tile(kt + 1, b ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile kt has landed for every thread
    const uint32_t kb = smem_addr(sm.kv[b][0]);
    const uint32_t vb = smem_addr(sm.kv[b][1]);

    // ---- S = Q K^T: 16 rows x 64 keys ----
    float sc[NK][4];
#pragma unroll
    for (int nk = 0; nk < NK; ++nk) sc[nk][0] = sc[nk][1] = sc[nk][2] = sc[nk][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < NK / 2; ++np) {
        // B fragments of two n-tiles (keys 16np..16np+15), k = d chunks 2ks, 2ks+1
        uint32_t bf[4];
        ldsm_x4(kb + swz(16 * np + lrow + ((lmat >> 1) << 3), 2 * ks + (lmat & 1)), bf);
        mma16816<T>(sc[2 * np], qa[ks], bf[0], bf[1]);
        mma16816<T>(sc[2 * np + 1], qa[ks], bf[2], bf[3]);
      }
    }
    // ---- causal mask, online softmax (rows r0: c0,c1; r0+8: c2,c3) ----
    const bool needs_mask = kt * kKeys + kKeys - 1 > pos_lo;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nk = 0; nk < NK; ++nk) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        const int key = kt * kKeys + 8 * nk + qc + (e & 1);
        float v = sc[nk][e] * p.scale_log2;
        if (needs_mask && key > pos[i]) v = -INFINITY;
        sc[nk][e] = v;
        mx[i] = fmaxf(mx[i], v);
      }
    }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float m_new = fmaxf(m_run[i], mx[i]);
      // (a row with every key masked so far keeps m = -inf; its weights stay 0)
      alpha[i] = m_new == -INFINITY ? 1.f : exp2f(m_run[i] - m_new);
      m_run[i] = m_new;
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pa[NK / 2][4];  // P as A fragments: k-step kk covers keys 16kk..16kk+15
#pragma unroll
    for (int nk = 0; nk < NK; ++nk) {
      float pr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        pr[e] = m_run[i] == -INFINITY ? 0.f : exp2f(sc[nk][e] - m_run[i]);
        rs[i] += pr[e];
      }
      // C layout of n-tile nk (keys 8nk + qc, +1) is A layout of k-step nk/2, half nk%2
      pa[nk >> 1][(nk & 1) * 2 + 0] = pack2<T>(pr[0], pr[1]);  // row r0
      pa[nk >> 1][(nk & 1) * 2 + 1] = pack2<T>(pr[2], pr[3]);  // row r0 + 8
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
      l_run[i] = l_run[i] * alpha[i] + rs[i];
    }
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      o[nd][0] *= alpha[0];
      o[nd][1] *= alpha[0];
      o[nd][2] *= alpha[1];
      o[nd][3] *= alpha[1];
    }
    // ---- O += P V: k = 64 keys (4 k-steps), n = d ----
#pragma unroll
    for (int kk = 0; kk < NK / 2; ++kk) {
      // the A fragment registers a0..a3 are (r0, k lo), (r0+8, k lo), (r0, k hi), (r0+8, k hi)
      const uint32_t a[4] = {pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]};
#pragma unroll
      for (int np = 0; np < ND / 2; ++np) {
        // B fragments of two n-tiles (d 16np..16np+15), k = keys 16kk..16kk+15, V^T
        uint32_t bf[4];
        ldsm_x4_t(vb + swz(16 * kk + lrow + ((lmat & 1) << 3), 2 * np + (lmat >> 1)), bf);
        mma16816<T>(o[2 * np], a, bf[0], bf[1]);
        mma16816<T>(o[2 * np + 1], a, bf[2], bf[3]);
      }
    }
    __syncthreads();  // every warp is done with buffer b before it is refilled
  }

  // ---- out = O / l ----
  const bool bad = sm.bad != 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (qrow_off[i] < 0) continue;
    const float inv = 1.f / l_run[i];
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      // (a bad block's rows were read from block 0, whatever it holds: zeros, not 0 * O)
      const uint32_t v = bad ? 0u : pack2<T>(o[nd][2 * i] * inv, o[nd][2 * i + 1] * inv);
      *reinterpret_cast<uint32_t*>(outp + qrow_off[i] + 8 * nd + qc) = v;
    }
  }
  if (bad && tid == 0) atomicOr(p.err, kErrBadBlock);
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
