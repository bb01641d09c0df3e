// Paged decode attention for sm_103a.
//
// Per sequence s and query head h (kv head g = h / G):
//   z_t = scale * <q[s,h], K_s[t,g]>,  out[s,h] = sum_t softmax(z)_t V_s[t,g],  t < ctx_s
// with K_s[t] = k_cache[block_tables[s][t / B], g, t % B, :] (daiw.org "Paged Attention",
// sections 直觉 and 定义; chenyuan1125 "vllm-pagedattention", section 页表真正解开的…: the
// kernel finds each K/V block through the table and does score, softmax and weighted sum
// block by block).
//
// Design (GB300: 152 SMs, HBM-bound at <= 1 FLOP/byte per query head):
// * Work unit = a 16-token "stage" (K and V rows) of one (sequence, kv head, head chunk)
//   pair, plus a fixed charge per pair.  The batch's units are cut into gridDim.x equal
//   contiguous shares, one per persistent CTA (one CTA per SM), so SMs finish together.  A pair cut between CTAs is merged with a log-sum-exp reduction by the CTA holding
//   its first piece, once the later pieces (written first thing by the next CTAs) are
//   published (split-KV: the rescaling identity of online softmax that chenyuan1125,
//   section 它和 FlashAttention…, names as FlashAttention's technique).  The launch is
//   cooperative, so all CTAs are resident; a CTA only waits for higher-numbered CTAs.  Cut points depend on
//   logical positions and context lengths only, so permuting physical blocks (and the
//   table with them) gives bit-identical output.
// * One producer warp: lane i owns stage i of a batch of up to 8 stages, waits for its
//   ring slot (stage kk belongs to consumer warp kk % 8, which owns a private set of
//   slots and takes them in order), and issues TMA tensor copies (cp.async.bulk.tensor, 128-byte swizzle) of
//   the stage's K and V rows; the next batch's block-table entries load meanwhile.  A
//   2-slot side ring carries each pair's q rows (1-D bulk copy).
// * Eight consumer warps take stages round-robin.  Warp-level tensor-core MMAs
//   (m16n8k16, fp32 accumulate) with the pair's query heads as the N = 8 (or 16) columns:
//   S^T = K Q^T (rows = the stage's 16 tokens), then O^T += V^T P^T (rows = d) with
//   P = 2^(S - m) rounded to the input type and moved into B-fragment layout by an
//   in-register transpose (movmatrix).  Each warp keeps its own running max/sum (online
//   softmax); the eight warps merge at the end of each segment.  Swizzled smem makes
//   every ldmatrix conflict-free.
// * Every mbarrier wait is bounded (about 1 s) and sets PA_DEVERR_TIMEOUT on expiry;
//   exits after a failed wait are decided collectively so no warp is left at a barrier.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <random>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace decode {

constexpr int kStageTok = 16;
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kBatch = 8;                        // stages the producer issues together
constexpr int kMaxHeads = 16;                    // query heads per work pair (MMA rows)
constexpr int kBarConsumers = 1;                 // named barrier id for the consumers
constexpr float kLog2e = 1.4426950408889634f;
// A pair costs its stages plus this many stage-equivalents of fixed work (q load, the
// eight-warp merge and the output write at its end).  Charging it when cutting the batch
// into per-SM shares keeps SMs whose shares hold many short pairs from finishing last.
constexpr int kSegCost = 5;

template <int D>
struct Geo {
  static constexpr int kHalves = D / 64;                    // 128-byte column halves of a row
  static constexpr int kBoxBytes = kStageTok * 128;         // 16 rows of one half
  static constexpr int kKBytes = kHalves * kBoxBytes;       // K rows of a stage
  static constexpr int kStageBytes = 2 * kKBytes;           // K then V
  // Ring slots per consumer warp; each warp owns its slots, so every slot has a single
  // consumer that takes its rounds in order and mbarrier parity waits are exact.
  static constexpr int kSlotsPerWarp = (192 * 1024) / (kStageBytes * 8);
  static constexpr int kStages = kSlotsPerWarp * 8;
  static constexpr int kKSteps = D / 16;                    // MMA k-steps of Q K^T
  static constexpr int kNTiles = D / 8;                     // MMA n-tiles of P V
};

struct Params {
  const uint8_t* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, heads_per_pair, head_chunks;
  int max_blocks_per_seq, block_size, log2_block, num_blocks, max_ctx;
  int seg_cost;  // work units charged per pair on top of its stages (see Walk)
  float scale_log2;
  unsigned long long* flags;  // [grid]: epoch once the CTA's leading piece is written
  unsigned long long epoch;   // unique per call
  float* part_acc;  // [grid][2][kMaxHeads][D]
  float* part_ml;   // [grid][2][kMaxHeads][2]  (m, l); l < 0 marks a piece with a bad block
  unsigned* err;
};

__device__ __forceinline__ int pair_stages(int ctx, int max_ctx) {
  return (ctx >= 1 && ctx <= max_ctx) ? (ctx + kStageTok - 1) / kStageTok : 1;
}

// Deterministic walk over this CTA's share [w, w1) of the batch's work units.  Pair p of
// sequence s weighs ns(s) + seg_cost units: seg_cost leading units of fixed work, then one
// unit per 16-token stage.  Sequence s holds pairs_per_seq such pairs.
struct Walk {
  const int32_t* ctx_lens;
  int pairs_per_seq, max_ctx, seg_cost;
  int s;
  long long pre;  // first unit of sequence s
  long long w, w0, w1;
  bool first_done;  // a segment of this share has been returned already
};

struct Seg {
  int s, pair, ctx, ns;
  int j0, j1;          // stage range within the pair
  int ta, tb;          // token range [ta, tb)
  bool bad_ctx;        // context length outside [1, max_ctx]
  bool whole;          // the pair is not cut
  bool cta_first;      // first segment of this CTA's share
  long long pair_end;  // one past the pair's last unit
};

__device__ __forceinline__ bool next_seg(Walk& wk, Seg& sg) {
  while (wk.w < wk.w1) {
    const int ctx = __ldg(wk.ctx_lens + wk.s);
    const int ns = pair_stages(ctx, wk.max_ctx);
    const long long pw = ns + wk.seg_cost;
    const long long units = static_cast<long long>(wk.pairs_per_seq) * pw;
    if (wk.w >= wk.pre + units) {
      wk.pre += units;
      ++wk.s;
      continue;
    }
    const long long local = wk.w - wk.pre;
    const int pair = static_cast<int>(local / pw);
    const long long pstart = wk.pre + pair * pw;
    const long long end_w = min(wk.w1, pstart + pw);
    const int j0 = static_cast<int>(max(0ll, local - pair * pw - wk.seg_cost));
    const int j1 = static_cast<int>(max(0ll, end_w - pstart - wk.seg_cost));
    wk.w = end_w;
    if (j1 <= j0) continue;  // this share holds only the pair's fixed-cost units
    sg.s = wk.s;
    sg.ctx = ctx;
    sg.ns = ns;
    sg.pair = pair;
    sg.j0 = j0;
    sg.j1 = j1;
    sg.bad_ctx = !(ctx >= 1 && ctx <= wk.max_ctx);
    sg.ta = j0 * kStageTok;
    sg.tb = sg.bad_ctx ? sg.ta : min(j1 * kStageTok, ctx);
    sg.whole = (j0 == 0 && j1 == ns);
    sg.cta_first = !wk.first_done;
    wk.first_done = true;
    sg.pair_end = pstart + pw;
    return true;
  }
  return false;
}

// Owner CTA of unit x when W units are cut into G shares, the first W % G one larger.
__device__ __forceinline__ int owner_of(long long x, long long W, int G) {
  const long long q = W / G, r = W % G;
  if (x < r * (q + 1)) return static_cast<int>(x / (q + 1));
  return static_cast<int>(r + (x - r * (q + 1)) / q);
}

struct PairHeads {
  int kvh, h0, nh;
};

__device__ __forceinline__ PairHeads pair_heads(const Params& p, int pair) {
  PairHeads ph;
  ph.kvh = pair / p.head_chunks;
  const int hc = pair - ph.kvh * p.head_chunks;
  ph.h0 = ph.kvh * p.group + hc * p.heads_per_pair;
  ph.nh = min(p.heads_per_pair, p.group - hc * p.heads_per_pair);
  return ph;
}

// Batches (<= kBatch stages) of the segments of this CTA's share, skipping pairs with an
// invalid context length (those carry no pipeline traffic).
struct Batch {
  int s, kvh, h0, nh, ca, cb;
  bool seg_start;
};

struct BatchIt {
  Walk wk;
  Seg sg;
  int cpos;
  bool have_seg;
};

__device__ __forceinline__ bool next_batch(BatchIt& it, Batch& b, const Params& p) {
  for (;;) {
    if (it.have_seg && it.cpos < it.sg.tb) {
      const PairHeads ph = pair_heads(p, it.sg.pair);
      b.s = it.sg.s;
      b.kvh = ph.kvh;
      b.h0 = ph.h0;
      b.nh = ph.nh;
      b.ca = it.cpos;
      b.cb = min(it.cpos + kBatch * kStageTok, it.sg.tb);
      b.seg_start = (it.cpos == it.sg.ta);
      it.cpos = b.cb;
      return true;
    }
    if (!next_seg(it.wk, it.sg)) return false;
    it.have_seg = !it.sg.bad_ctx;
    it.cpos = it.sg.ta;
  }
}

// Block-table entries of stage `lane` of batch `b`: x = the block holding the stage's
// first token, y = the next block when the stage spans two blocks (block_size 8).
__device__ __forceinline__ int2 stage_entries(const Batch& b, int lane, const Params& p) {
  int2 e = make_int2(0, 0);
  const int nst = (b.cb - b.ca + kStageTok - 1) / kStageTok;
  if (lane < nst) {
    const int t0 = b.ca + lane * kStageTok;
    const int nt = min(kStageTok, b.cb - t0);
    const int32_t* trow = p.block_tables + static_cast<size_t>(b.s) * p.max_blocks_per_seq;
    const int j0 = t0 >> p.log2_block;
    e.x = __ldg(trow + j0);
    if ((t0 & (p.block_size - 1)) + nt > p.block_size) e.y = __ldg(trow + j0 + 1);
  }
  return e;
}

// 2-D TMA tile load (box of the tensor map at column x, row y) into swizzled smem.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
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

// Transpose of an 8x8 matrix of 16-bit values held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D += A * B, m16n8k16, fp32 accumulate.
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

// Byte offset of (row, 16-byte chunk) in a stage's K or V rows: chunk c of the row lives
// in column half c / 8, and the 128-byte swizzle permutes chunks within each row.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kStageTok * 128) + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void st_release_gpu(unsigned long long* addr, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* addr) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(addr) : "memory");
  return v;
}

// Spin (bounded by kWaitLimitNs) until *flag holds this call's epoch.
__device__ __forceinline__ bool wait_flag_bounded(const unsigned long long* flag,
                                                  unsigned long long epoch) {
  if (ld_acquire_gpu(flag) == epoch) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) == epoch) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Merge the pieces of a cut pair held by CTAs c..c_last (c's piece in slot `first_slot`,
// the others in slot 0): M = max m_i, L = sum l_i 2^(m_i - M), out = sum acc_i 2^(m_i - M) / L,
// pieces taken in CTA order (deterministic).  Zeros when a piece saw a bad block or a
// wait for a piece gave up.
template <int D, typename T>
__device__ void merge_pieces(const Params& p, int c, int first_slot, int c_last, int nh, bool failed,
                             T* out_rows, int tid, int nthreads) {
  for (int i = tid; i < nh * D; i += nthreads) {
    const int h = i / D;
    const int d = i - h * D;
    float M = -INFINITY;
    bool bad = failed;
    for (int cc = c; cc <= c_last; ++cc) {
      const size_t base = static_cast<size_t>(cc) * 2 + (cc == c ? first_slot : 0);
      const float* ml = p.part_ml + (base * kMaxHeads + h) * 2;
      M = fmaxf(M, __ldcg(ml));
      bad |= __ldcg(ml + 1) < 0.f;
    }
    float L = 0.f, o = 0.f;
    for (int cc = c; cc <= c_last; ++cc) {
      const size_t base = static_cast<size_t>(cc) * 2 + (cc == c ? first_slot : 0);
      const float* ml = p.part_ml + (base * kMaxHeads + h) * 2;
      const float w = exp2f(__ldcg(ml) - M);
      L += __ldcg(ml + 1) * w;
      o += __ldcg(p.part_acc + (base * kMaxHeads + h) * D + d) * w;
    }
    out_rows[h * D + d] = from_float<T>(bad ? 0.f : o / L);
  }
}

template <int D>
struct Smem {
  uint8_t ring[Geo<D>::kStages][Geo<D>::kStageBytes];  // 1024-byte aligned
  uint8_t qbuf[2][kMaxHeads * D * 2];
  float xo[kConsumerWarps][4][D];  // per-warp O rows, 4 heads per exchange round
  float xm[kConsumerWarps][kMaxHeads], xl[kConsumerWarps][kMaxHeads];
  long long scan[kThreads / 32];
  long long start_pre;
  int start_s;
  int slot_bad[Geo<D>::kStages];
  int abort_flag;
  unsigned long long full[Geo<D>::kStages], empty[Geo<D>::kStages];
  unsigned long long qfull[2], qempty[2];
};

template <int D, int NTH, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
  using G_ = Geo<D>;
  constexpr int S = G_::kStages;
  constexpr int R = G_::kSlotsPerWarp;
  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle pattern repeats every 1024 bytes: align the ring to it
  const uint32_t raw_addr = smem_addr(smem_raw);
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw + (((raw_addr + 1023) & ~1023u) - raw_addr));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int pairs_per_seq = p.num_kv_heads * p.head_chunks;

  // ---- setup: total units W, this CTA's share, and the sequence where it starts ----
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(&sm.full[i]), 1);
      mbar_init(smem_addr(&sm.empty[i]), 1);  // the consuming warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&sm.qfull[i]), 1);
      mbar_init(smem_addr(&sm.qempty[i]), kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  const int per = (p.num_seqs + kThreads - 1) / kThreads;
  const int sa = min(p.num_seqs, tid * per), sb = min(p.num_seqs, sa + per);
  long long mine = 0;
  for (int s = sa; s < sb; ++s)
    mine += static_cast<long long>(pairs_per_seq) *
            (pair_stages(__ldg(p.context_lens + s), p.max_ctx) + p.seg_cost);
  long long incl = mine;  // inclusive scan of `mine` over the block
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  long long before = 0, W = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) before += sm.scan[w];
    W += sm.scan[w];
  }
  const long long excl = before + incl - mine;
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const long long qd = W / G, rm = W % G;
  const long long w0 = c * qd + min(static_cast<long long>(c), rm);
  const long long w1 = w0 + qd + (c < rm ? 1 : 0);
  if (w0 < w1 && excl <= w0 && w0 < excl + mine) {
    long long pre = excl;
    int s = sa;
    for (;; ++s) {
      const long long u = static_cast<long long>(pairs_per_seq) *
                          (pair_stages(__ldg(p.context_lens + s), p.max_ctx) + p.seg_cost);
      if (w0 < pre + u) break;
      pre += u;
    }
    sm.start_s = s;
    sm.start_pre = pre;
  }
  __syncthreads();

  Walk walk;
  walk.ctx_lens = p.context_lens;
  walk.pairs_per_seq = pairs_per_seq;
  walk.max_ctx = p.max_ctx;
  walk.seg_cost = p.seg_cost;
  walk.first_done = false;
  walk.s = (w0 < w1) ? sm.start_s : 0;
  walk.pre = (w0 < w1) ? sm.start_pre : 0;
  walk.w = w0;
  walk.w0 = w0;
  walk.w1 = w1;
  const volatile int* abort_flag = &sm.abort_flag;

  if (warp == kConsumerWarps) {
    // =============================== producer warp ===============================
    BatchIt it;
    it.wk = walk;
    it.cpos = 0;
    it.have_seg = false;
    Batch cur, nxt;
    bool has_cur = next_batch(it, cur, p);
    int2 e_cur = has_cur ? stage_entries(cur, lane, p) : make_int2(0, 0);
    const int box_rows = min(p.block_size, kStageTok);
    const uint32_t box_bytes = box_rows * 128;
    uint32_t k = 0, qi = 0;
    bool ok = true, issued = false;
    while (ok && has_cur) {
      issued = false;
      const bool has_nxt = next_batch(it, nxt, p);
      const int2 e_nxt = has_nxt ? stage_entries(nxt, lane, p) : make_int2(0, 0);
      if (cur.seg_start) {  // the pair's q rows, contiguous in q
        if (lane == 0) {
          const uint32_t qs = qi & 1;
          ok = mbar_wait_bounded(smem_addr(&sm.qempty[qs]), ((qi >> 1) & 1) ^ 1, abort_flag);
          if (ok) {
            const uint32_t bytes = cur.nh * D * 2;
            mbar_arrive_expect_tx(smem_addr(&sm.qfull[qs]), bytes);
            bulk_g2s(smem_addr(sm.qbuf[qs]),
                     p.q + (static_cast<size_t>(cur.s) * p.num_q_heads + cur.h0) * D * 2, bytes,
                     smem_addr(&sm.qfull[qs]));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++qi;
        if (!ok) break;
      }
      const int nst = (cur.cb - cur.ca + kStageTok - 1) / kStageTok;
      if (lane < nst) {
        const int t0 = cur.ca + lane * kStageTok;
        const int nt = min(kStageTok, cur.cb - t0);
        const int row0 = t0 & (p.block_size - 1);
        const bool two = row0 + nt > p.block_size;  // block_size 8: a second block
        const bool bad = e_cur.x < 0 || e_cur.x >= p.num_blocks ||
                         (two && (e_cur.y < 0 || e_cur.y >= p.num_blocks));
        const uint32_t kk = k + lane;
        const uint32_t u = kk / kConsumerWarps;  // round-robin: warp kk % 8, its u-th stage
        const uint32_t slot = (kk % kConsumerWarps) * R + u % R;
        ok = mbar_wait_bounded(smem_addr(&sm.empty[slot]), ((u / R) & 1) ^ 1, abort_flag);
        if (ok) {
          const uint32_t fbar = smem_addr(&sm.full[slot]);
          if (bad) {
            sm.slot_bad[slot] = 1;
            mbar_arrive(fbar);
          } else {
            sm.slot_bad[slot] = 0;
            const int nboxes = two ? 2 : 1;
            mbar_arrive_expect_tx(fbar, 2 * G_::kHalves * nboxes * box_bytes);
            const uint32_t base = smem_addr(sm.ring[slot]);
            const int y0 = (e_cur.x * p.num_kv_heads + cur.kvh) * p.block_size + row0;
            const int y1 = (e_cur.y * p.num_kv_heads + cur.kvh) * p.block_size;
#pragma unroll
            for (int hf = 0; hf < G_::kHalves; ++hf) {
              const uint32_t kd = base + hf * G_::kBoxBytes;
              const uint32_t vd = kd + G_::kKBytes;
              tma_load_2d(kd, &tmap_k, hf * 64, y0, fbar);
              tma_load_2d(vd, &tmap_v, hf * 64, y0, fbar);
              if (two) {
                tma_load_2d(kd + box_bytes, &tmap_k, hf * 64, y1, fbar);
                tma_load_2d(vd + box_bytes, &tmap_v, hf * 64, y1, fbar);
              }
            }
          }
          issued = true;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      k += nst;
      cur = nxt;
      e_cur = e_nxt;
      has_cur = has_nxt;
    }
    if (!ok) {
      // A wait gave up: stop everyone, then let the copies already issued land (the last
      // S stages before this batch, plus this batch's stages whose lanes issued them).
      int zero = 0;
      const volatile int* never = &zero;
      if (lane == 0) {
        sm.abort_flag = 1;
        atomicOr(p.err, kErrTimeout);
      }
      auto slot_of = [&](uint32_t kk) { return (kk % kConsumerWarps) * R + (kk / kConsumerWarps) % R; };
      auto parity_of = [&](uint32_t kk) { return ((kk / kConsumerWarps) / R) & 1; };
      if (issued) mbar_wait_bounded(smem_addr(&sm.full[slot_of(k + lane)]), parity_of(k + lane), never);
      if (lane == 0) {
        const uint32_t first = k > static_cast<uint32_t>(S) ? k - S : 0;
        for (uint32_t kk = first; kk < k; ++kk)
          mbar_wait_bounded(smem_addr(&sm.full[slot_of(kk)]), parity_of(kk), never);
        for (uint32_t qq = qi > 2 ? qi - 2 : 0; qq < qi; ++qq)
          mbar_wait_bounded(smem_addr(&sm.qfull[qq & 1]), (qq >> 1) & 1, never);
      }
    }
    return;
  }

  // ================================ consumer warps ================================
  // Control flow of the eight consumer warps stays identical: every exit taken after a
  // failed wait is decided collectively at a named barrier (bar.red.or).
  constexpr int KS = G_::kKSteps;
  constexpr int MT = D / 16;  // m-tiles of O^T (16 rows of d each)
  const int cw = warp;
  const int r0 = lane >> 2;        // MMA row of this lane (query head r0, and r0 + 8)
  const int qc = 2 * (lane & 3);   // MMA column pair of this lane
  const int lrow = lane & 7;       // ldmatrix: row within an 8x8 matrix
  const int lmat = lane >> 3;      // ldmatrix: which of the four matrices

  uint32_t k = 0, qi = 0;
  bool ok = true;
  Seg sg;
  while (next_seg(walk, sg)) {
    const PairHeads ph = pair_heads(p, sg.pair);
    T* out_rows =
        reinterpret_cast<T*>(p.out) + (static_cast<size_t>(sg.s) * p.num_q_heads + ph.h0) * D;
    if (sg.bad_ctx) {  // no pipeline traffic for this pair: zeros and a flag
      for (int i = tid; i < ph.nh * D / 8; i += kConsumerThreads)
        reinterpret_cast<uint4*>(out_rows)[i] = make_uint4(0, 0, 0, 0);
      if (tid == 0) atomicOr(p.err, kErrBadContext);
      continue;
    }

    // ---- Q^T of the pair as MMA B fragments: column n = head 8*nt + (lane >> 2) ----
    // (heads >= nh are zero)
    uint32_t qb[KS][NTH][2];
    {
      const uint32_t qs = qi & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(smem_addr(&sm.qfull[qs]),
                                                            (qi >> 1) & 1, abort_flag));
      const uint8_t* qbuf = sm.qbuf[qs];
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt) {
        const int h = nt * 8 + r0;
        const bool hv = ok && h < ph.nh;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int col = 16 * ks + qc;
          qb[ks][nt][0] = hv ? *reinterpret_cast<const uint32_t*>(qbuf + (h * D + col) * 2) : 0u;
          qb[ks][nt][1] = hv ? *reinterpret_cast<const uint32_t*>(qbuf + (h * D + col + 8) * 2) : 0u;
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(smem_addr(&sm.qempty[qs]));
      if (!ok) sm.abort_flag = 1;
      ++qi;
    }
    // This lane's softmax columns: heads hc0 = 8*nt + qc and hc0 + 1 of every n-tile.
    float m_run[NTH][2], l_run[NTH][2];
    float o[MT][NTH][4];  // O^T: rows d = 16*mt + r0 (+8), columns = heads
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }
    bool seg_bad = false;

    const int nstage = (sg.tb - sg.ta + kStageTok - 1) / kStageTok;
    // this warp's stages: global index k + i with (k + i) % 8 == cw
    for (int i = (cw - static_cast<int>(k % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
         ok && i < nstage; i += kConsumerWarps) {
      const uint32_t u = (k + i) / kConsumerWarps;  // this warp's u-th stage
      const uint32_t slot = cw * R + u % R;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(smem_addr(&sm.full[slot]), (u / R) & 1, abort_flag));
      if (!ok) break;
      const int nt_tok = min(kStageTok, sg.tb - (sg.ta + i * kStageTok));
      bool zeroed = false;
      if (sm.slot_bad[slot]) {
        seg_bad = true;
      } else {
        const uint32_t kb = smem_addr(sm.ring[slot]);
        const uint32_t vb = kb + G_::kKBytes;
        // ---- S^T = K Q^T: rows = the stage's 16 tokens, columns = heads ----
        float sacc[NTH][4], sodd[NTH][4];
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) sacc[nt][j] = sodd[nt][j] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a[4];  // rows tok 0-7 / 8-15, d chunks 2ks / 2ks+1
          ldsm_x4(kb + swz(lrow + ((lmat & 1) << 3), 2 * ks + (lmat >> 1)), a);
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt) {
            if (ks & 1)
              mma16816<T>(sodd[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
            else
              mma16816<T>(sacc[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
          }
        }
        // ---- online softmax per head (column) over the 16 tokens (rows) ----
        // c0,c1: token r0, heads qc, qc+1; c2,c3: token r0 + 8, same heads
        const bool v_lo = r0 < nt_tok, v_hi = r0 + 8 < nt_tok;
        uint32_t pb[NTH][2];
        float alpha[NTH][2];
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          float x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float v = (sacc[nt][j] + sodd[nt][j]) * p.scale_log2;
            x[j] = (j < 2 ? v_lo : v_hi) ? v : -INFINITY;
          }
          float pr[4];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float mx = fmaxf(x[c], x[c + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[nt][c], mx);
            alpha[nt][c] = exp2f(m_run[nt][c] - m_new);  // 0 on the first stage
            pr[c] = exp2f(x[c] - m_new);
            pr[c + 2] = exp2f(x[c + 2] - m_new);
            float sum = pr[c] + pr[c + 2];
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l_run[nt][c] = l_run[nt][c] * alpha[nt][c] + sum;
            m_run[nt][c] = m_new;
          }
          // P^T as B fragments: transpose the (token x head) 8x8 blocks in registers
          pb[nt][0] = movmatrix_t(pack2<T>(pr[0], pr[1]));  // tokens 0-7
          pb[nt][1] = movmatrix_t(pack2<T>(pr[2], pr[3]));  // tokens 8-15
        }
        bool all_one = true;
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) all_one = all_one && alpha[nt][0] == 1.f && alpha[nt][1] == 1.f;
        if (!__all_sync(0xffffffffu, all_one)) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
              o[mt][nt][0] *= alpha[nt][0];
              o[mt][nt][1] *= alpha[nt][1];
              o[mt][nt][2] *= alpha[nt][0];
              o[mt][nt][3] *= alpha[nt][1];
            }
        }
        // ---- rows past the context may hold anything (even NaN): zero them in V ----
        if (nt_tok < kStageTok) {
          const int per_half = (kStageTok - nt_tok) * 8;  // 16-byte chunks per column half
          for (int e = lane; e < per_half * G_::kHalves; e += 32) {
            const int hf = e / per_half;
            const int rem = e - hf * per_half;
            const uint32_t addr = vb + hf * G_::kBoxBytes + (nt_tok + rem / 8) * 128 + (rem % 8) * 16;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
          }
          zeroed = true;
          __syncwarp();
        }
        // ---- O^T += V^T P^T: rows = d (16 per m-tile), k = tokens, columns = heads ----
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a[4];  // V^T: d chunks 2mt / 2mt+1, tokens 0-7 / 8-15
          ldsm_x4_t(vb + swz(lrow + ((lmat >> 1) << 3), 2 * mt + (lmat & 1)), a);
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt) mma16816<T>(o[mt][nt], a, pb[nt][0], pb[nt][1]);
        }
      }
      // generic-proxy stores (the zeroed rows) must be ordered before the next TMA write
      if (zeroed) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
    }
    k += nstage;
    if (!ok) sm.abort_flag = 1;

    // ---------------- segment end: merge the 8 warps, write out ----------------
    if (bar_red_or(kBarConsumers, kConsumerThreads, !ok)) {
      ok = false;
      break;
    }
    if (r0 == 0) {  // lanes 0..3 hold the running max/sum of heads 8*nt + qc, + 1
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          sm.xm[cw][nt * 8 + qc + c] = m_run[nt][c];
          sm.xl[cw][nt * 8 + qc + c] = l_run[nt][c];
        }
    }
    const int slot_out = sg.cta_first ? 0 : 1;
    float* pacc = p.part_acc + (static_cast<size_t>(blockIdx.x) * 2 + slot_out) * kMaxHeads * D;
    float* pml = p.part_ml + (static_cast<size_t>(blockIdx.x) * 2 + slot_out) * kMaxHeads * 2;
    bool any_bad = false;
    // Exchange O four heads at a time: round r covers heads 4r..4r+3.
    const int rounds = (ph.nh + 3) / 4;
    for (int round = 0; round < rounds; ++round) {
      if (round > 0) named_bar_sync(kBarConsumers, kConsumerThreads);  // previous reads done
      const int rbase = round * 4;
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int h = nt * 8 + qc + c;
          if (h >= rbase && h < rbase + 4) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              sm.xo[cw][h - rbase][16 * mt + r0] = o[mt][nt][c];
              sm.xo[cw][h - rbase][16 * mt + r0 + 8] = o[mt][nt][c + 2];
            }
          }
        }
      }
      any_bad = bar_red_or(kBarConsumers, kConsumerThreads, seg_bad);
      const int rows = min(4, ph.nh - rbase);
      for (int idx = tid; idx < rows * (D / 4); idx += kConsumerThreads) {
        const int hr = idx / (D / 4);
        const int h = rbase + hr;
        const int d4 = (idx - hr * (D / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.xm[w][h]);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float wt = exp2f(sm.xm[w][h] - M);  // 0 for warps without stages here
          L += sm.xl[w][h] * wt;
          const float4 x4 = *reinterpret_cast<const float4*>(&sm.xo[w][hr][d4]);
          acc.x += x4.x * wt;
          acc.y += x4.y * wt;
          acc.z += x4.z * wt;
          acc.w += x4.w * wt;
        }
        if (sg.whole) {
          uint2 packed = make_uint2(0u, 0u);  // zeros for a pair with a bad block
          if (!any_bad) {
            const float inv = 1.f / L;
            packed.x = pack2<T>(acc.x * inv, acc.y * inv);
            packed.y = pack2<T>(acc.z * inv, acc.w * inv);
          }
          *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
        } else {
          *reinterpret_cast<float4*>(pacc + h * D + d4) = acc;
          if (d4 == 0) {
            pml[h * 2 + 0] = M;
            pml[h * 2 + 1] = any_bad ? -1.f : L;
          }
        }
      }
    }
    if (!sg.whole) {
      __threadfence();  // this thread's partial writes, before the piece is published or merged
      named_bar_sync(kBarConsumers, kConsumerThreads);
      if (sg.j0 > 0) {
        // A later piece of a cut pair (this share's first segment): publish it.
        if (tid == 0) st_release_gpu(p.flags + blockIdx.x, p.epoch);
      } else {
        // The first piece (this share's last segment): wait for the later pieces, which
        // the next CTAs wrote at the start of their shares, then merge in CTA order.
        const int c_last = owner_of(sg.pair_end - 1, W, G);
        bool waited_ok = true;
        if (tid == 0) {
          for (int cc = blockIdx.x + 1; cc <= c_last && waited_ok; ++cc)
            waited_ok = wait_flag_bounded(p.flags + cc, p.epoch);
          if (!waited_ok) atomicOr(p.err, kErrTimeout);
        }
        const bool failed = bar_red_or(kBarConsumers, kConsumerThreads, !waited_ok);
        merge_pieces<D, T>(p, blockIdx.x, slot_out, c_last, ph.nh, failed, out_rows, tid,
                           kConsumerThreads);
      }
    }
    if (tid == 0 && any_bad) atomicOr(p.err, kErrBadBlock);
  }
  if (!ok && tid == 0) atomicOr(p.err, kErrTimeout);
}

// Tensor map over one cache viewed as rows of D elements: [num_blocks * Hkv * B, D],
// boxes of 64 columns x min(B, 16) rows, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, bool bf16, int head_dim, long long rows,
                    int box_rows) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int NTH, typename T>
int launch(const Params& prm, const CUtensorMap& mk, const CUtensorMap& mv, int grid,
           cudaStream_t stream) {
  const size_t smem = sizeof(Smem<D>) + 1024;  // + alignment slack for the ring
  auto* kern = decode_kernel<D, NTH, T>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return -3;
  // Cooperative launch: every CTA is resident at once, so a CTA may wait (bounded) for the
  // pieces that higher-numbered CTAs write at the start of their shares.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm, mk, mv) != cudaSuccess) return -3;
  return 0;
}

}  // namespace decode

int decode_heads_per_pair(int num_q_heads, int num_kv_heads) {
  const int g = num_q_heads / num_kv_heads;
  return g < decode::kMaxHeads ? g : decode::kMaxHeads;
}

size_t decode_workspace_bytes(int grid, int /*heads_per_pair*/, int head_dim) {
  const size_t flags = static_cast<size_t>(grid) * sizeof(unsigned long long);
  const size_t acc = static_cast<size_t>(grid) * 2 * decode::kMaxHeads * head_dim * sizeof(float);
  const size_t ml = static_cast<size_t>(grid) * 2 * decode::kMaxHeads * 2 * sizeof(float);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return up(flags) + up(acc) + up(ml);
}

// Epochs tag the pieces of one call: a flag in the (caller-owned, never cleared) workspace
// counts only when it holds the current call's epoch.  64-bit values, random high half.
static unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{
      (static_cast<unsigned long long>(std::random_device{}()) << 32) ^
      static_cast<unsigned long long>(
          std::chrono::steady_clock::now().time_since_epoch().count())};
  return counter.fetch_add(1, std::memory_order_relaxed) + 1;
}

int decode_launch(const DecodeArgs& a, int grid, cudaStream_t stream) {
  decode::Params p;
  p.q = static_cast<const uint8_t*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<uint8_t*>(a.out);
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.heads_per_pair = decode_heads_per_pair(a.num_q_heads, a.num_kv_heads);
  p.head_chunks = (p.group + p.heads_per_pair - 1) / p.heads_per_pair;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.log2_block = a.block_size == 8 ? 3 : (a.block_size == 16 ? 4 : 5);
  p.num_blocks = a.num_blocks;
  p.max_ctx = a.max_blocks_per_seq * a.block_size;
  p.seg_cost = decode::kSegCost;
  p.scale_log2 = a.scale * decode::kLog2e;
  p.err = a.err;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.flags = reinterpret_cast<unsigned long long*>(ws);
  ws += up(static_cast<size_t>(grid) * sizeof(unsigned long long));
  p.epoch = next_epoch();
  p.part_acc = reinterpret_cast<float*>(ws);
  ws += up(static_cast<size_t>(grid) * 2 * decode::kMaxHeads * a.head_dim * sizeof(float));
  p.part_ml = reinterpret_cast<float*>(ws);

  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * a.block_size;
  const int box_rows = a.block_size < decode::kStageTok ? a.block_size : decode::kStageTok;
  CUtensorMap mk, mv;
  if (!decode::make_cache_map(&mk, a.k_cache, a.bf16, a.head_dim, rows, box_rows) ||
      !decode::make_cache_map(&mv, a.v_cache, a.bf16, a.head_dim, rows, box_rows))
    return -3;
  // heads of a pair are MMA columns: one n-tile of 8, or two for up to 16
#define PA_DECODE_CASE(DD, NN)                                                        \
  if (a.head_dim == DD && (p.heads_per_pair > 8) == (NN == 2))                        \
    return a.bf16 ? decode::launch<DD, NN, __nv_bfloat16>(p, mk, mv, grid, stream)    \
                  : decode::launch<DD, NN, __half>(p, mk, mv, grid, stream);
  PA_DECODE_CASE(128, 1)
  PA_DECODE_CASE(128, 2)
  PA_DECODE_CASE(64, 1)
  PA_DECODE_CASE(64, 2)
#undef PA_DECODE_CASE
  return -1;
}

}  // namespace pa
