// Paged decode attention for sm_103a.
//
// Per sequence s and query head h (kv head g = h / G):
//   z_t = scale * <q[s,h], K_s[t,g]>,  out[s,h] = sum_t softmax(z)_t V_s[t,g],  t < ctx_s
// with K_s[t] = k_cache[block_tables[s][t / B], g, t % B, :] (daiw.org "Paged Attention",
// sections 直觉 and 定义; chenyuan1125 "vllm-pagedattention", section 页表真正解开的…: the
// kernel finds each K/V block through the table and does score, softmax and weighted sum
// block by block).
//
// Design (GB300 has 152 SMs; decode is HBM-bound at <= 1 FLOP/byte per head group):
// * Work unit = a 16-token "stage" of one (sequence, kv head[, head chunk]) pair.  The
//   units of the whole batch are cut into gridDim.x equal contiguous shares, one per
//   persistent CTA (one CTA per SM), so every SM streams the same number of bytes and
//   there is no tail of idle SMs.  A pair cut between CTAs is merged afterwards by a
//   log-sum-exp reduction (split-KV; the rescaling identity of online softmax that
//   chenyuan1125, section 它和 FlashAttention…, names as FlashAttention's technique).
//   Cut points depend on logical positions and context lengths only, so permuting
//   physical blocks gives bit-identical output.
// * Warp specialisation: one producer warp walks the CTA's share and issues 1-D
//   cp.async.bulk copies of each stage's K rows, then V rows, into a ring of smem slots
//   guarded by mbarriers (full: transaction bytes; empty: consumer arrivals).  Only the
//   valid rows of a tail block are copied.  One q copy per pair goes through a 2-slot
//   side ring.
// * Eight consumer warps, in two groups taking alternate stages.  K stage: 8 lanes per
//   token, each lane holds 16 (or 8) q values per head in fp32 (pre-scaled by
//   scale*log2 e), packed fp32x2 FMAs, 3 xor-shuffles per head.  Scores of a chunk of
//   up to 256 tokens go to smem; one warp per head turns them into exp2 weights with a
//   running max/sum (online softmax across chunks).  V stage: each lane owns D/32
//   output columns for every head; accumulators are rescaled once per chunk.
// * Every mbarrier wait is bounded (about 1 s) and sets PA_DEVERR_TIMEOUT on expiry.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace decode {

constexpr int kStageTok = 16;
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kChunk = 256;                      // tokens per softmax chunk
constexpr int kMaxHeads = 8;                     // query heads per work pair
constexpr int kBarConsumers = 1;                 // named barrier id for the consumers
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Geo {
  static constexpr int kStageBytes = kStageTok * D * 2;  // one stage of K (or V) rows
  static constexpr int kStages = (128 * 1024) / kStageBytes;
  static constexpr int kNch = D / 64;  // 16-byte chunks per lane in a K row (8 lanes/token)
  static constexpr int kVe = D / 32;   // output columns per lane in the V stage
};

struct SplitRec {
  int seq;         // -1: this CTA starts no split pair
  int pair;        // kv head * head_chunks + head chunk
  int c_last;      // last CTA holding a piece of the pair
  int first_slot;  // partial slot of the starting CTA's piece
};

struct Params {
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, heads_per_pair, head_chunks;
  int max_blocks_per_seq, block_size, num_blocks, max_ctx;
  float scale_log2;
  SplitRec* recs;
  float* part_acc;  // [grid][2][GP][D]
  float* part_ml;   // [grid][2][GP][2]  (m, l); l < 0 marks a piece with a bad block
  unsigned* err;
};

__device__ __forceinline__ int pair_stages(int ctx, int max_ctx) {
  return (ctx >= 1 && ctx <= max_ctx) ? (ctx + kStageTok - 1) / kStageTok : 1;
}

// Deterministic walk over this CTA's share [w, w1) of the batch's stage units.
// Units of sequence s: pairs_per_seq * ns(s); pair p owns units [p*ns, (p+1)*ns).
struct Walk {
  const int32_t* ctx_lens;
  int pairs_per_seq, max_ctx;
  int s;
  long long pre;  // first unit of sequence s
  long long w, w0, w1;
};

struct Seg {
  int s, pair, ctx, ns;
  int j0, j1;      // stage range within the pair
  int ta, tb;      // token range [ta, tb)
  bool bad_ctx;    // context length outside [1, max_ctx]
  bool whole;      // the pair is not cut
  bool cta_first;  // first segment of this CTA's share
  long long pair_end;  // one past the pair's last unit
};

__device__ __forceinline__ bool next_seg(Walk& wk, Seg& sg) {
  while (wk.w < wk.w1) {
    const int ctx = __ldg(wk.ctx_lens + wk.s);
    const int ns = pair_stages(ctx, wk.max_ctx);
    const long long units = static_cast<long long>(wk.pairs_per_seq) * ns;
    if (wk.w >= wk.pre + units) {
      wk.pre += units;
      ++wk.s;
      continue;
    }
    const long long local = wk.w - wk.pre;
    sg.s = wk.s;
    sg.ctx = ctx;
    sg.ns = ns;
    sg.pair = static_cast<int>(local / ns);
    sg.j0 = static_cast<int>(local % ns);
    const long long left = wk.w1 - wk.w;
    sg.j1 = static_cast<int>(left < ns - sg.j0 ? sg.j0 + left : ns);
    sg.bad_ctx = !(ctx >= 1 && ctx <= wk.max_ctx);
    sg.ta = sg.j0 * kStageTok;
    sg.tb = sg.bad_ctx ? sg.ta : min(sg.j1 * kStageTok, ctx);
    sg.whole = (sg.j0 == 0 && sg.j1 == ns);
    sg.cta_first = (wk.w == wk.w0);
    sg.pair_end = wk.pre + static_cast<long long>(sg.pair + 1) * ns;
    wk.w += sg.j1 - sg.j0;
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

template <int D, int GP>
struct Smem {
  uint8_t ring[Geo<D>::kStages][Geo<D>::kStageBytes];
  uint8_t qbuf[2][kMaxHeads * D * 2];
  float logits[2][kChunk][GP];
  float xacc[kConsumerWarps][GP][D];
  float m_run[GP], l_run[GP], alpha[GP];
  long long scan[kThreads / 32];
  long long start_pre;
  int start_s;
  int slot_bad[Geo<D>::kStages];
  int abort_flag;
  unsigned long long full[Geo<D>::kStages], empty[Geo<D>::kStages];
  unsigned long long qfull[2], qempty[2];
};

template <int D, int GP, typename T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const Params p) {
  using G_ = Geo<D>;
  constexpr int S = G_::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<D, GP>& sm = *reinterpret_cast<Smem<D, GP>*>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int pairs_per_seq = p.num_kv_heads * p.head_chunks;

  // Let the merge kernel launch early; it waits for this grid before reading anything.
  pdl_launch_dependents();

  // ---- setup: total units W, this CTA's share, and the sequence where it starts ----
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(&sm.full[i]), 1);
      mbar_init(smem_addr(&sm.empty[i]), 4);  // the owning group's four warps
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
    mine += static_cast<long long>(pairs_per_seq) * pair_stages(__ldg(p.context_lens + s), p.max_ctx);
  // inclusive scan of `mine` over the block: shuffles within warps, then warp totals
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long v = __shfl_up_sync(0xffffffffu, incl, o);
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
      const long long u =
          static_cast<long long>(pairs_per_seq) * pair_stages(__ldg(p.context_lens + s), p.max_ctx);
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
  walk.s = (w0 < w1) ? sm.start_s : 0;
  walk.pre = (w0 < w1) ? sm.start_pre : 0;
  walk.w = w0;
  walk.w0 = w0;
  walk.w1 = w1;

  const volatile int* abort_flag = &sm.abort_flag;
  const size_t kv_head_stride = static_cast<size_t>(p.block_size) * D * 2;  // bytes

  if (warp == kConsumerWarps) {
    // =============================== producer warp ===============================
    uint32_t k = 0, qi = 0;
    bool ok = true;
    Seg sg;
    while (ok && next_seg(walk, sg)) {
      if (sg.bad_ctx) continue;
      const int kvh = sg.pair / p.head_chunks;
      const int hc = sg.pair % p.head_chunks;
      const int h0 = kvh * p.group + hc * p.heads_per_pair;
      const int nh = min(p.heads_per_pair, p.group - hc * p.heads_per_pair);
      // q rows of the pair's heads (contiguous in q)
      if (lane == 0) {
        const uint32_t qs = qi & 1;
        ok = mbar_wait_bounded(smem_addr(&sm.qempty[qs]), ((qi >> 1) & 1) ^ 1, abort_flag);
        if (ok) {
          const uint32_t bytes = nh * D * 2;
          mbar_arrive_expect_tx(smem_addr(&sm.qfull[qs]), bytes);
          bulk_g2s(smem_addr(sm.qbuf[qs]),
                   p.q + (static_cast<size_t>(sg.s) * p.num_q_heads + h0) * D * 2, bytes,
                   smem_addr(&sm.qfull[qs]));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++qi;
      const int32_t* trow = p.block_tables + static_cast<size_t>(sg.s) * p.max_blocks_per_seq;
      for (int ca = sg.ta; ok && ca < sg.tb; ca += kChunk) {
        const int cb = min(ca + kChunk, sg.tb);
        const int fb = ca / p.block_size;
        const int nblk = (cb - 1) / p.block_size - fb + 1;  // <= 32 for B >= 8
        int ent = (lane < nblk) ? __ldg(trow + fb + lane) : 0;
        const bool ent_ok = (ent >= 0 && ent < p.num_blocks);
        if (!ent_ok) ent = 0;
        const unsigned bad_mask = __ballot_sync(0xffffffffu, !ent_ok && lane < nblk);
        const int nst = (cb - ca + kStageTok - 1) / kStageTok;
        for (int pass = 0; ok && pass < 2; ++pass) {
          const uint8_t* cache = pass == 0 ? p.k_cache : p.v_cache;
          for (int st = 0; st < nst; ++st, ++k) {
            const int t0 = ca + st * kStageTok;
            const int nt = min(kStageTok, cb - t0);
            const int i0 = t0 / p.block_size - fb;
            const int row0 = t0 % p.block_size;
            const int rows0 = min(nt, p.block_size - row0);
            const int blk0 = __shfl_sync(0xffffffffu, ent, i0);
            const int blk1 = __shfl_sync(0xffffffffu, ent, min(i0 + 1, 31));
            const bool bad = ((bad_mask >> i0) & 1u) || (rows0 < nt && ((bad_mask >> (i0 + 1)) & 1u));
            if (lane == 0) {
              const uint32_t slot = k % S;
              ok = mbar_wait_bounded(smem_addr(&sm.empty[slot]), ((k / S) & 1) ^ 1, abort_flag);
              if (ok) {
                const uint32_t fbar = smem_addr(&sm.full[slot]);
                if (bad) {
                  sm.slot_bad[slot] = 1;
                  mbar_arrive(fbar);
                } else {
                  sm.slot_bad[slot] = 0;
                  mbar_arrive_expect_tx(fbar, nt * D * 2);
                  const uint8_t* src0 = cache +
                      (static_cast<size_t>(blk0) * p.num_kv_heads + kvh) * kv_head_stride +
                      static_cast<size_t>(row0) * D * 2;
                  bulk_g2s(smem_addr(sm.ring[slot]), src0, rows0 * D * 2, fbar);
                  if (rows0 < nt) {  // block_size 8: the stage spans two blocks
                    const uint8_t* src1 =
                        cache + (static_cast<size_t>(blk1) * p.num_kv_heads + kvh) * kv_head_stride;
                    bulk_g2s(smem_addr(sm.ring[slot]) + rows0 * D * 2, src1, (nt - rows0) * D * 2,
                             fbar);
                  }
                }
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // A wait gave up: stop everyone, then let copies already in flight land.
      sm.abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
      int zero = 0;
      const volatile int* never = &zero;
      const uint32_t first = k > static_cast<uint32_t>(S) ? k - S : 0;
      for (uint32_t kk = first; kk < k; ++kk)
        mbar_wait_bounded(smem_addr(&sm.full[kk % S]), (kk / S) & 1, never);
      for (uint32_t qq = qi > 2 ? qi - 2 : 0; qq < qi; ++qq)
        mbar_wait_bounded(smem_addr(&sm.qfull[qq & 1]), (qq >> 1) & 1, never);
    }
    return;
  }

  // ================================ consumer warps ================================
  // Control flow of the eight consumer warps must stay identical: every exit taken
  // after a failed wait is decided collectively at a named barrier (bar.red.or).
  const int cw = warp;        // 0..7
  const int grp = cw >> 2;    // stage-parity group
  const int wi = cw & 3;      // warp within group
  const int ktok = wi * 4 + (lane >> 3);  // K stage: token of this lane
  const int sub = lane & 7;               // K stage: lane within the token's 8
  constexpr int NCH = G_::kNch;
  constexpr int VE = G_::kVe;

  float qf[GP][NCH][8];
  float acc[GP][VE];
  uint32_t k = 0, qi = 0, chunk_no = 0;
  bool ok = true;
  Seg sg;
  int rec_seq = -1, rec_pair = 0, rec_last = 0, rec_slot = 0;

  while (next_seg(walk, sg)) {
    const int kvh = sg.pair / p.head_chunks;
    const int hc = sg.pair % p.head_chunks;
    const int h0 = kvh * p.group + hc * p.heads_per_pair;
    const int nh = min(p.heads_per_pair, p.group - hc * p.heads_per_pair);
    T* out_rows = reinterpret_cast<T*>(p.out) + (static_cast<size_t>(sg.s) * p.num_q_heads + h0) * D;

    if (sg.bad_ctx) {  // no pipeline traffic for this pair: zeros and a flag
      for (int i = tid; i < nh * D / 8; i += kConsumerThreads)
        reinterpret_cast<uint4*>(out_rows)[i] = make_uint4(0, 0, 0, 0);
      if (tid == 0) atomicOr(p.err, kErrBadContext);
      continue;
    }

    // ---- q of this pair: smem slot -> fp32 registers, pre-scaled by scale*log2(e) ----
    {
      const uint32_t qs = qi & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(smem_addr(&sm.qfull[qs]), (qi >> 1) & 1, abort_flag));
      if (ok) {
        const uint8_t* qb = sm.qbuf[qs];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
#pragma unroll
          for (int cch = 0; cch < NCH; ++cch) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (h < nh) raw = *reinterpret_cast<const uint4*>(qb + (h * D + (sub + 8 * cch) * 8) * 2);
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack2<T>(wv[e]);
              qf[h][cch][2 * e] = f.x * p.scale_log2;
              qf[h][cch][2 * e + 1] = f.y * p.scale_log2;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.qempty[qs]));
      } else {
        sm.abort_flag = 1;
      }
      ++qi;
    }
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[h][e] = 0.f;
    bool seg_bad = false;

    for (int ca = sg.ta; ca < sg.tb; ca += kChunk) {
      const int cb = min(ca + kChunk, sg.tb);
      const int nst = (cb - ca + kStageTok - 1) / kStageTok;
      const int buf = chunk_no & 1;
      ++chunk_no;

      // ---------------------------- K stages: scores ----------------------------
      for (int st = 0; ok && st < nst; ++st) {
        const uint32_t kk = k + st;
        if (static_cast<int>(kk & 1) != grp) continue;
        const uint32_t slot = kk % S;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&sm.full[slot]), (kk / S) & 1, abort_flag));
        if (!ok) break;
        const int nt = min(kStageTok, cb - (ca + st * kStageTok));
        if (sm.slot_bad[slot]) {
          seg_bad = true;
        } else {
          const uint8_t* row = sm.ring[slot] + ktok * D * 2;
          float2 dot[GP];
#pragma unroll
          for (int h = 0; h < GP; ++h) dot[h] = make_float2(0.f, 0.f);
#pragma unroll
          for (int cch = 0; cch < NCH; ++cch) {
            const uint4 raw = *reinterpret_cast<const uint4*>(row + (sub + 8 * cch) * 16);
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kv = unpack2<T>(wv[e]);
#pragma unroll
              for (int h = 0; h < GP; ++h)
                dot[h] = ffma2(make_float2(qf[h][cch][2 * e], qf[h][cch][2 * e + 1]), kv, dot[h]);
            }
          }
          float sc[GP];
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            float v = dot[h].x + dot[h].y;
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            sc[h] = v;
          }
          if (ktok < nt) {
            float mine_sc = sc[0];
#pragma unroll
            for (int h = 1; h < GP; ++h)
              if (sub == h) mine_sc = sc[h];
            if (sub < GP) sm.logits[buf][st * kStageTok + ktok][sub] = mine_sc;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
      }
      if (!ok) sm.abort_flag = 1;
      if (bar_red_or(kBarConsumers, kConsumerThreads, !ok)) {
        ok = false;
        break;
      }
      k += nst;

      // ------------------- online softmax over the chunk, per head -------------------
      if (cw < nh) {
        const int h = cw;
        const int ntok = cb - ca;
        float mx = -INFINITY;
        for (int i = lane; i < ntok; i += 32) mx = fmaxf(mx, sm.logits[buf][i][h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const bool first = (ca == sg.ta);
        const float m_old = first ? -INFINITY : sm.m_run[h];
        const float m_new = fmaxf(m_old, mx);
        const float alpha = first ? 0.f : exp2f(m_old - m_new);
        float sum = 0.f;
        for (int i = lane; i < ntok; i += 32) {
          const float e = exp2f(sm.logits[buf][i][h] - m_new);
          sm.logits[buf][i][h] = e;
          sum += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
          sm.l_run[h] = first ? sum : sm.l_run[h] * alpha + sum;
          sm.m_run[h] = m_new;
          sm.alpha[h] = alpha;
        }
      }
      named_bar_sync(kBarConsumers, kConsumerThreads);

      // ------------------------- V stages: weighted sum -------------------------
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float a = sm.alpha[h];
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[h][e] *= a;
      }
      for (int st = 0; ok && st < nst; ++st) {
        const uint32_t kk = k + st;
        if (static_cast<int>(kk & 1) != grp) continue;
        const uint32_t slot = kk % S;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&sm.full[slot]), (kk / S) & 1, abort_flag));
        if (!ok) break;
        const int nt = min(kStageTok, cb - (ca + st * kStageTok));
        if (!sm.slot_bad[slot]) {
          for (int t = wi; t < nt; t += 4) {
            const uint8_t* vrow = sm.ring[slot] + t * D * 2 + lane * VE * 2;
            float pw[GP];
            const float* prow = sm.logits[buf][st * kStageTok + t];
            if constexpr (GP >= 4) {
#pragma unroll
              for (int h = 0; h < GP; h += 4) {
                const float4 p4 = *reinterpret_cast<const float4*>(prow + h);
                pw[h] = p4.x; pw[h + 1] = p4.y; pw[h + 2] = p4.z; pw[h + 3] = p4.w;
              }
            } else if constexpr (GP == 2) {
              const float2 p2 = *reinterpret_cast<const float2*>(prow);
              pw[0] = p2.x; pw[1] = p2.y;
            } else {
              pw[0] = prow[0];
            }
            if constexpr (VE == 4) {
              const uint2 raw = *reinterpret_cast<const uint2*>(vrow);
              const float2 v01 = unpack2<T>(raw.x), v23 = unpack2<T>(raw.y);
#pragma unroll
              for (int h = 0; h < GP; ++h) {
                const float2 ph = make_float2(pw[h], pw[h]);
                const float2 a01 = ffma2(ph, v01, make_float2(acc[h][0], acc[h][1]));
                const float2 a23 = ffma2(ph, v23, make_float2(acc[h][2], acc[h][3]));
                acc[h][0] = a01.x; acc[h][1] = a01.y; acc[h][2] = a23.x; acc[h][3] = a23.y;
              }
            } else {
              const uint32_t raw = *reinterpret_cast<const uint32_t*>(vrow);
              const float2 v01 = unpack2<T>(raw);
#pragma unroll
              for (int h = 0; h < GP; ++h) {
                const float2 a01 =
                    ffma2(make_float2(pw[h], pw[h]), v01, make_float2(acc[h][0], acc[h][1]));
                acc[h][0] = a01.x; acc[h][1] = a01.y;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
      }
      if (!ok) sm.abort_flag = 1;
      k += nst;
    }

    // ---------------- segment end: combine the 8 warps, write out ----------------
    if (bar_red_or(kBarConsumers, kConsumerThreads, !ok)) {
      ok = false;
      break;
    }
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
      for (int e = 0; e < VE; ++e) sm.xacc[cw][h][lane * VE + e] = acc[h][e];
    const bool any_bad = bar_red_or(kBarConsumers, kConsumerThreads, seg_bad);
    const int slot_out = sg.cta_first ? 0 : 1;
    float* pacc = p.part_acc + (static_cast<size_t>(blockIdx.x) * 2 + slot_out) * GP * D;
    float* pml = p.part_ml + (static_cast<size_t>(blockIdx.x) * 2 + slot_out) * GP * 2;
    for (int i = tid; i < nh * (D / 4); i += kConsumerThreads) {
      const int h = i / (D / 4);
      const int d4 = (i % (D / 4)) * 4;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float4 x = *reinterpret_cast<const float4*>(&sm.xacc[w][h][d4]);
        o.x += x.x; o.y += x.y; o.z += x.z; o.w += x.w;
      }
      if (sg.whole) {
        const float inv = any_bad ? 0.f : 1.f / sm.l_run[h];
        uint2 packed;
        packed.x = pack2<T>(o.x * inv, o.y * inv);
        packed.y = pack2<T>(o.z * inv, o.w * inv);
        *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
      } else {
        *reinterpret_cast<float4*>(pacc + h * D + d4) = o;
        if (d4 == 0) {
          pml[h * 2 + 0] = sm.m_run[h];
          pml[h * 2 + 1] = any_bad ? -1.f : sm.l_run[h];
        }
      }
    }
    if (tid == 0 && any_bad) atomicOr(p.err, kErrBadBlock);
    if (!sg.whole && sg.j0 == 0) {  // this CTA holds the first piece of a cut pair
      rec_seq = sg.s;
      rec_pair = sg.pair;
      rec_last = owner_of(sg.pair_end - 1, W, G);
      rec_slot = slot_out;
    }
  }
  if (!ok && tid == 0) atomicOr(p.err, kErrTimeout);
  if (tid == 0) {
    SplitRec r;
    r.seq = ok ? rec_seq : -1;
    r.pair = rec_pair;
    r.c_last = rec_last;
    r.first_slot = rec_slot;
    p.recs[blockIdx.x] = r;
  }
}

// Merge the pieces of every cut pair: M = max m_i, L = sum l_i 2^(m_i - M),
// out = sum acc_i 2^(m_i - M) / L, pieces taken in CTA order (deterministic).
template <int D, int GP, typename T>
__global__ void __launch_bounds__(128) merge_kernel(const Params p) {
  pdl_wait_primary();
  const SplitRec r = p.recs[blockIdx.x];
  if (r.seq < 0) return;
  const int kvh = r.pair / p.head_chunks;
  const int hc = r.pair % p.head_chunks;
  const int h0 = kvh * p.group + hc * p.heads_per_pair;
  const int nh = min(p.heads_per_pair, p.group - hc * p.heads_per_pair);
  T* out_rows = reinterpret_cast<T*>(p.out) + (static_cast<size_t>(r.seq) * p.num_q_heads + h0) * D;
  for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
    const int h = i / D;
    const int d = i % D;
    float M = -INFINITY;
    bool bad = false;
    for (int cc = blockIdx.x; cc <= r.c_last; ++cc) {
      const int slot = (cc == static_cast<int>(blockIdx.x)) ? r.first_slot : 0;
      const float* ml = p.part_ml + ((static_cast<size_t>(cc) * 2 + slot) * GP + h) * 2;
      M = fmaxf(M, ml[0]);
      bad |= ml[1] < 0.f;
    }
    float L = 0.f, o = 0.f;
    for (int cc = blockIdx.x; cc <= r.c_last; ++cc) {
      const int slot = (cc == static_cast<int>(blockIdx.x)) ? r.first_slot : 0;
      const size_t base = static_cast<size_t>(cc) * 2 + slot;
      const float* ml = p.part_ml + (base * GP + h) * 2;
      const float w = exp2f(ml[0] - M);
      L += ml[1] * w;
      o += p.part_acc[base * GP * D + h * D + d] * w;
    }
    const float v = bad ? 0.f : o / L;
    out_rows[h * D + d] = from_float<T>(v);
  }
}

template <int D, int GP>
constexpr size_t smem_bytes() {
  return sizeof(Smem<D, GP>);
}

template <int D, int GP, typename T>
int launch(const Params& prm, int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes<D, GP>();
  auto* kern = decode_kernel<D, GP, T>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return -3;
  kern<<<grid, kThreads, smem, stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return -3;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, merge_kernel<D, GP, T>, prm) != cudaSuccess) return -3;
  return 0;
}

}  // namespace decode

size_t decode_workspace_bytes(int grid, int heads_per_pair, int head_dim) {
  int gp = 1;
  while (gp < heads_per_pair) gp <<= 1;
  const size_t recs = static_cast<size_t>(grid) * sizeof(decode::SplitRec);
  const size_t acc = static_cast<size_t>(grid) * 2 * gp * head_dim * sizeof(float);
  const size_t ml = static_cast<size_t>(grid) * 2 * gp * 2 * sizeof(float);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return up(recs) + up(acc) + up(ml);
}

int decode_launch(const DecodeArgs& a, int grid, cudaStream_t stream) {
  decode::Params p;
  p.q = static_cast<const uint8_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<uint8_t*>(a.out);
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.heads_per_pair = p.group < decode::kMaxHeads ? p.group : decode::kMaxHeads;
  p.head_chunks = (p.group + p.heads_per_pair - 1) / p.heads_per_pair;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.max_ctx = a.max_blocks_per_seq * a.block_size;
  p.scale_log2 = a.scale * decode::kLog2e;
  p.err = a.err;
  int gp = 1;
  while (gp < p.heads_per_pair) gp <<= 1;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.recs = reinterpret_cast<decode::SplitRec*>(ws);
  ws += up(static_cast<size_t>(grid) * sizeof(decode::SplitRec));
  p.part_acc = reinterpret_cast<float*>(ws);
  ws += up(static_cast<size_t>(grid) * 2 * gp * a.head_dim * sizeof(float));
  p.part_ml = reinterpret_cast<float*>(ws);

#define PA_DECODE_CASE(DD, GG)                                                   \
  if (a.head_dim == DD && gp == GG) {                                            \
    return a.bf16 ? decode::launch<DD, GG, __nv_bfloat16>(p, grid, stream)       \
                  : decode::launch<DD, GG, __half>(p, grid, stream);             \
  }
  PA_DECODE_CASE(128, 1)
  PA_DECODE_CASE(128, 2)
  PA_DECODE_CASE(128, 4)
  PA_DECODE_CASE(128, 8)
  PA_DECODE_CASE(64, 1)
  PA_DECODE_CASE(64, 2)
  PA_DECODE_CASE(64, 4)
  PA_DECODE_CASE(64, 8)
#undef PA_DECODE_CASE
  return -1;
}

}  // namespace pa
