#ifndef PA_DECODE_KERNEL_CUH_
#define PA_DECODE_KERNEL_CUH_
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
// * A "pair" is one kv head (or a chunk of up to 16 of its query heads) of one sequence.
//   The pairs of a sequence are taken in groups of gs (the largest power of two <= 8 that
//   divides the pair count); a "family" is one sequence's group.  A family's work is
//   ns(s) units of 16 tokens (32 over FP8 / INT4 blocks) x gs pairs (a "stage" is one
//   unit of one pair: its K rows and V rows), plus a fixed charge.  The batch's stages, in
//   (family, unit, pair) order, are cut into gridDim.x equal contiguous shares, one per
//   persistent CTA (one per SM).
// * Warp w of a CTA works on pair w / P of every family (P = 8 / gs warps per pair, each
//   taking every P-th unit).  With 8 or more kv heads (gs = 8) a warp owns one kv head
//   outright: it streams its pair's stages straight across family boundaries and never
//   waits for another warp.  With fewer, the P warps of a pair merge their partial
//   softmax states through shared memory under a named barrier of their own.
// * Loads: each warp copies its own stages, kAhead ahead of the one it computes, with
//   16-byte cp.async copies (every lane copies a slice of the stage's K and V rows) into a
//   private ring of swizzled shared-memory slots, and waits with cp.async.wait_group.
//   Spreading the copies over all eight warps keeps enough bytes in flight per SM to reach
//   the HBM limit; a single issuing warp, with TMA or with cp.async, streams about 26 GB/s
//   per SM on GB300.  Rows past the context are zero-filled by the copy itself (source
//   size 0) and never read.
// * Math per stage on warp-level tensor cores (m16n8k16, fp32 accumulate) with the pair's
//   query heads as the N = 8 (or 16) columns: S^T = K Q^T (rows = the stage's tokens, 16
//   per m-tile), then O^T += V^T P^T (rows = d) with P = 2^(S - m) rounded to the MMA type
//   and moved into B-fragment layout by an in-register transpose (movmatrix); online
//   softmax with a running max and sum per head.  The swizzles make every fragment load
//   conflict-free.  FP8 and INT4 codes are widened to f16 exactly in registers.
// * Whole stages (every row inside the context, no pass split between blocks) copy from
//   one base address per block with constant offsets; others take a per-row path.
// * A pair cut between CTAs (split-KV) leaves one partial softmax state (O, m, l) per
//   piece in the workspace.  A CTA counts its pieces in on per-pair counters: a piece
//   whose family is not the share's last right after it is stored (one warp per pair),
//   the share's last one when the whole share is streamed (no copies left in flight, so
//   a fence is cheap).  The CTA that brings a pair's count to its number of pieces
//   merges them in CTA order with a log-sum-exp reduction (the rescaling identity of
//   online softmax that chenyuan1125, section 它和 FlashAttention…, names as
//   FlashAttention's technique), after its share.  No CTA ever waits for another.  Cut points depend on logical positions and context lengths only, and
//   the merge order is fixed, so permuting physical blocks gives bit-identical output.
// * Launched as a programmatic dependent of the kernel before it in the stream: while
//   that kernel drains, the grid plans its shares from the context lengths and block
//   tables and warms L2 with each warp's first blocks; q, the caches and the workspace
//   are touched only after griddepcontrol.wait.
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <random>
#include <type_traits>

#include "pa_arrive.h"
#include "pa_common.cuh"
#include "pa_internal.h"

// Diagnostics (pa_decode_timeline).  pa_decode_timed.cu defines PA_DECODE_TIMELINE before
// including this file, which compiles the 16-bit kernel once more under another name, with
// a `timeline` argument -- null, or [grid][kWarps][3] globaltimer readings (ns) -- into
// which lane 0 of each warp writes when the programmatic wait released (0), when its
// streaming is done (1) and at its end (2).  Everywhere else the stamps are empty
// statements, so the kernels that serve calls are compiled without them: an extra argument
// or Params field, or a stamp in the stage loop, measurably slowed the FP8 and 16-bit
// kernels.
#ifdef PA_DECODE_TIMELINE
#define PA_DECODE_KERNEL decode_kernel_timed
#define PA_DECODE_LAUNCH launch_timed
#define PA_DECODE_TIMELINE_ARG , unsigned long long* timeline
#define PA_DECODE_TIMELINE_PASS , timeline
#define PA_DECODE_STAMP(k)                                                                     \
  do {                                                                                        \
    if (timeline != nullptr && lane == 0)                                                     \
      timeline[(static_cast<size_t>(blockIdx.x) * kWarps + warp) * 3 + (k)] = global_timer_ns(); \
  } while (0)
#else
#define PA_DECODE_KERNEL decode_kernel
#define PA_DECODE_LAUNCH launch
#define PA_DECODE_TIMELINE_ARG
#define PA_DECODE_TIMELINE_PASS
#define PA_DECODE_STAMP(k)
#endif

namespace pa {
namespace decode {

constexpr int kStageTok = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxHeads = 16;  // query heads per pair (MMA columns)
constexpr float kLog2e = 1.4426950408889634f;
// Stage-equivalents (16-token stages) charged per family on top of its stages when
// cutting the batch into per-SM shares: a family switch (a new table row, the pair-end
// writes) costs time, and when families are larger than shares a family start in a share
// also means one more cut piece to count in and merge at the share's end.  So the charge
// is kSegCostFew stages when the batch has no more families than shares, falling towards
// kSegCostMany as families outnumber shares (seg_cost_for).  On GB300 (one box, 16-bit
// blocks, charge 16 / 32 / 48 / 64): 64 sequences of 128..2048 tokens (64 families)
// 53.4 / 52.8 / 51.8 / 51.4 us; 256 MHA sequences (1024 families) 385.9 / 387.7 / 391.5 /
// 395.7 us; 8 sequences of 8-32 K tokens flat within 1 us.
constexpr int kSegCostFew = 64;
constexpr int kSegCostMany = 16;

// The charge for `families` families cut into `shares` shares, in 16-token stages.
inline int seg_cost_for(long long families, int shares) {
  const long long f = families > shares ? families : shares;
  return kSegCostMany + static_cast<int>((kSegCostFew - kSegCostMany) * static_cast<long long>(shares) / f);
}

// Cached K/V formats: 16-bit values, FP8 (E4M3) codes with one scale per cache, INT4
// codes (two per byte) with one float32 scale per row.
constexpr int kKv16 = 0;
constexpr int kKvFp8 = 1;
constexpr int kKvInt4 = 2;

// A stage of quantised blocks holds 32 tokens, so the per-stage work that does not scale
// with bytes (softmax reductions, bookkeeping) is paid once per 32 tokens.  INT4 stages
// carry the rows' scales after the codes (K scales, then V scales).
template <int D, int KV = kKv16>
struct Geo {
  static constexpr int kTok = KV == kKv16 ? kStageTok : 2 * kStageTok;  // tokens per stage
  static constexpr int kRowBytes = KV == kKv16 ? 2 * D : (KV == kKvFp8 ? D : D / 2);
  static constexpr int kRowChunks = kRowBytes / 16;         // 16-byte chunks per row
  static constexpr int kKBytes = kTok * kRowBytes;          // K rows of a stage
  static constexpr int kScaleBytes = KV == kKvInt4 ? 4 * kTok : 0;  // K (or V) row scales
  static constexpr int kStageBytes = 2 * kKBytes + 2 * kScaleBytes;  // K, V, K scales, V scales
  // Ring slots per warp (192 KB in all, at most 32) and how many stages ahead a warp loads.
  static constexpr int kSlots0 = (192 * 1024) / (kStageBytes * kWarps);
  static constexpr int kSlots = kSlots0 > 32 ? 32 : kSlots0;
  static constexpr int kAhead = kSlots - 1;
  static constexpr int kRowsPerPass = 32 / kRowChunks;      // rows one warp-wide copy covers
  static constexpr int kPasses = kTok / kRowsPerPass;       // copies per lane per K (or V)
  static constexpr int kMaxSpan = kTok / 8;                 // blocks a stage can span (B >= 8)
  static constexpr int kKSteps = D / 16;                    // MMA k-steps of K Q^T
};

struct Params {
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  // Fused cache write (pa_decode_append*), else null: the newest token of each sequence,
  // [n][Hkv][D] 16-bit.  Its row is attended from here (quantised first for FP8 / INT4
  // blocks) and stored at position ctx - 1.
  const uint8_t* key_new;
  const uint8_t* value_new;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint8_t* out;
  int num_seqs, num_q_heads, num_kv_heads, group, heads_per_pair, head_chunks;
  int gs, log2_gs, ngroups, phases;  // pairs per family, families per sequence, warps per pair
  int max_blocks_per_seq, block_size, log2_block, num_blocks, max_ctx;
  int log2_stage;  // tokens per stage: 16 (16-bit blocks) or 32 (FP8 blocks)
  int seg_cost;    // stage units charged per family on top of its stages
  float scale_log2;
  float out_scale;  // FP8 blocks: v_scale, applied to every output row (else 1)
  float k_quant, v_quant;  // FP8 blocks: k_scale, v_scale for the fused step's newest rows
  // INT4 blocks: float32 scale of each cached row, [num_blocks][Hkv][B] (else null)
  const float* k_scales;
  const float* v_scales;
  // [grid][gs]: arrivals at cut pair (first CTA, pi): epoch tag << 24 | pieces counted in
  unsigned long long* counters;
  unsigned long long epoch;  // 40-bit tag, different from the previous call's
  float* part_acc;  // [grid][2][gs][heads_per_pair][D]
  float* part_ml;   // [grid][2][gs][heads_per_pair][2]  (m, l); l < 0: the piece saw a bad block
  unsigned* err;
};

// Units (stages per pair) of a sequence; an invalid context length counts one.
__device__ __forceinline__ int pair_stages(int ctx, const Params& p) {
  return (ctx >= 1 && ctx <= p.max_ctx) ? ((ctx - 1) >> p.log2_stage) + 1 : 1;
}

// Family (sequence s, pair group g) and its place in the batch's stage order.
struct Fam {
  int s, g, ctx, ns;
  bool ok;        // 1 <= ctx <= max_ctx
  long long pre;  // first stage unit of the family
  long long fw;   // its weight: ns * gs + seg_cost
};

__device__ __forceinline__ void fam_load(Fam& f, const Params& p) {
  f.ctx = __ldg(p.context_lens + f.s);
  f.ok = f.ctx >= 1 && f.ctx <= p.max_ctx;
  f.ns = pair_stages(f.ctx, p);
  f.fw = static_cast<long long>(f.ns) * p.gs + p.seg_cost;
}

__device__ __forceinline__ void fam_next(Fam& f, const Params& p) {
  f.pre += f.fw;
  if (++f.g == p.ngroups) {
    f.g = 0;
    if (++f.s < p.num_seqs) fam_load(f, p);
  }
}

__device__ __forceinline__ bool fam_valid(const Fam& f) { return f.ok; }

// ceil(x / 2^k) for any sign of x.
__device__ __forceinline__ long long ceil_shift(long long x, int k) {
  return x > 0 ? (x + (1ll << k) - 1) >> k : -((-x) >> k);
}

// Units [x, y) of pair pi of family f whose stages lie in the share [w0, w1).
__device__ __forceinline__ int2 unit_range(const Fam& f, int pi, long long w0, long long w1,
                                           const Params& p) {
  const long long base = f.pre + p.seg_cost + pi;
  const long long a = ceil_shift(w0 - base, p.log2_gs), b = ceil_shift(w1 - base, p.log2_gs);
  return make_int2(static_cast<int>(max(0ll, min(static_cast<long long>(f.ns), a))),
                   static_cast<int>(max(0ll, min(static_cast<long long>(f.ns), b))));
}

// Does this share hold a piece of the pair: some of its units, or none while the pair runs
// on both sides of the share (an empty middle piece, published so the merge can count on it)?
__device__ __forceinline__ bool has_piece(int2 r, int ns) {
  return r.x < r.y || (r.x > 0 && r.x < ns);
}

// Share [w0, w1) of CTA c when W units are cut into G shares, the first W % G one larger.
__device__ __forceinline__ void share_of(int c, long long W, int G, long long& w0, long long& w1) {
  const long long q = W / G, r = W % G;
  w0 = c * q + min(static_cast<long long>(c), r);
  w1 = w0 + q + (c < r ? 1 : 0);
}

// Owner CTA of stage unit x.
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

// This warp's stages in order: for every family of the share, the units of its pair with
// unit index = its phase (mod P).  Families with an invalid context carry no stages.
struct Stage {
  int s, kvh, t0, nt;  // sequence, kv head, first token, valid tokens (1..tokens per stage)
  bool last;           // holds the context's last token
};

struct StageIt {
  Fam f;
  int kvh, j, jb;
};

__device__ __forceinline__ void stage_it_enter(StageIt& it, int pi, int phase, long long w0,
                                               long long w1, const Params& p) {
  const int2 r = unit_range(it.f, pi, w0, w1, p);
  if (!fam_valid(it.f) || r.x >= r.y) {
    it.j = it.jb = 0;
    return;
  }
  it.kvh = pair_heads(p, it.f.g * p.gs + pi).kvh;
  it.j = r.x + (phase - r.x % p.phases + p.phases) % p.phases;
  it.jb = r.y;
}

__device__ __forceinline__ bool next_stage(StageIt& it, int pi, int phase, long long w0, long long w1,
                                           Stage& st, const Params& p) {
  for (;;) {
    if (it.j < it.jb) {
      st.s = it.f.s;
      st.kvh = it.kvh;
      st.t0 = it.j << p.log2_stage;
      st.nt = min(1 << p.log2_stage, it.f.ctx - st.t0);
      st.last = st.t0 + st.nt == it.f.ctx;
      it.j += p.phases;
      return true;
    }
    fam_next(it.f, p);
    if (it.f.s >= p.num_seqs || it.f.pre >= w1) return false;
    stage_it_enter(it, pi, phase, w0, w1, p);
  }
}

// Block-table entries of a stage: e[k] = the k-th block holding its tokens (the entry of
// block t0 / B + k); entries past the stage's last token repeat e[0] and are not read.
template <int NE>
__device__ __forceinline__ void stage_entries(const Stage& st, const Params& p, int (&e)[NE]) {
  const int32_t* trow = p.block_tables + static_cast<size_t>(st.s) * p.max_blocks_per_seq;
  const int j0 = st.t0 >> p.log2_block;
  const int jl = (st.t0 + st.nt - 1) >> p.log2_block;
  e[0] = __ldg(trow + j0);
#pragma unroll
  for (int k = 1; k < NE; ++k) e[k] = j0 + k <= jl ? __ldg(trow + j0 + k) : e[0];
}

// 16-byte global -> shared copy through L2 only; the bytes past src_bytes (0 or 16) are
// zero-filled, and src_bytes = 0 reads nothing.
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

// FP8 stages: a row is D bytes.  At D = 128 the 16-byte chunk c of row r sits at c ^ (r % 8)
// so that the fragment loads below (eight lanes: four chunks of two rows, or one chunk of
// eight rows) hit distinct banks; at D = 64 rows are packed as they come.
template <int D>
__device__ __forceinline__ uint32_t swz8(int row, int chunk) {
  return D == 128 ? static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4))
                  : static_cast<uint32_t>(row * D + (chunk << 4));
}

// Row of O^T held in MMA accumulator row r (0..15) of m-tile mt.  16-bit blocks: d = 16 mt
// + r.  Quantised blocks (QK) permute d so that every lane builds its V fragments from
// contiguous bytes: rows r and r + 8 are the adjacent d = (D/8)(r % 8) + 2 mt and that + 1.
template <int D, bool QK>
__device__ __forceinline__ int drow(int mt, int r) {
  return QK ? (r & 7) * (D / 8) + 2 * mt + (r >> 3) : 16 * mt + r;
}

// Two E4M3 values (low byte first) -> f16x2, exact (every E4M3 value is an f16 normal):
// from the low or the high half of a 32-bit word.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(r)
      : "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2_hi(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}"
      : "=r"(r)
      : "r"(w));
  return r;
}

// INT4 stages: a row is D / 2 bytes.  The V fragment loads read, per half-warp, the same
// bytes of rows c, c + 2, c + 4, c + 6; the K fragment loads and the copies read or write
// whole consecutive rows.  At D = 128 (64-byte rows) row r sits in row slot
// r ^ ((r >> 1) & 1) with its 16-byte chunks XORed by 2 ((r >> 2) & 1); at D = 64
// (32-byte rows) row r sits in slot r ^ ((r >> 2) & 1).  Either way those four rows fall
// on distinct banks and consecutive rows stay whole and contiguous.
template <int D>
__device__ __forceinline__ uint32_t swz4(int row, int chunk) {
  return D == 128
             ? static_cast<uint32_t>(64 * (row ^ ((row >> 1) & 1)) + 16 * (chunk ^ (2 * ((row >> 2) & 1))))
             : static_cast<uint32_t>(32 * (row ^ ((row >> 2) & 1)) + 16 * chunk);
}

// Shared-memory offset, within a stage's K (or V) rows, of the 16-byte chunk `ch` that a
// lane copies in pass j (its row rsub + j * rows-per-pass), in closed form: the XOR
// patterns of swz / swz8 / swz4 reduce to a lane-dependent base and a per-pass constant.
template <int D, int KV, int ROWB>
__device__ __forceinline__ uint32_t copy_dst(int rsub, int ch, int j) {
  if constexpr (ROWB == 256) {  // 16-bit rows of 128 values, two rows a pass
    return static_cast<uint32_t>((ch >> 3) * 2048 + rsub * 128 + 256 * j +
                                 ((16 * ((ch & 7) ^ rsub)) ^ (32 * (j & 3))));
  } else if constexpr (ROWB == 128) {  // 128-byte rows (16-bit d = 64, FP8 d = 128), four a pass
    return static_cast<uint32_t>(128 * rsub + 512 * j + ((16 * (ch ^ rsub)) ^ (64 * (j & 1))));
  } else if constexpr (KV == 2) {  // INT4 rows: a pass spans 512 bytes of whole rows
    return swz4<D>(rsub, ch) + 512u * j;
  } else {  // FP8 rows of 64 bytes, packed
    return static_cast<uint32_t>(64 * rsub + 16 * ch + 512 * j);
  }
}

// INT4 nibbles -> f16x2 with one logic operation, exact: the nibble u (= code + 8) at
// bits 0-3 and 16-19 of w (i4x2_lo) or at bits 4-7 and 20-23 (i4x2_hi) is placed in the
// mantissa of 1024.0 (0x6400), which reads 1024 + u, or 1024 + 16 u.  The offsets never
// pass through these registers: the products are exact in the fp32 accumulators, and the
// kernel removes them there.  For K the high nibbles meet q / 16, so a score gains
// 1032 Q_lo + 72 Q_hi (Q_lo, Q_hi: the sums of q over the low- and high-nibble d), which
// the score accumulators start from minus.  For V a low-nibble output row holds
// O + 1032 W and a high-nibble row 16 (O + 72 W), W = the sum of the weights that entered
// P V, taken out at the pair end.
__device__ __forceinline__ uint32_t i4x2_lo(uint32_t w) { return (w & 0x000F000Fu) | 0x64006400u; }
__device__ __forceinline__ uint32_t i4x2_hi(uint32_t w) { return (w & 0x00F000F0u) | 0x64006400u; }

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// 2^x on the SFU (ex2.approx, subnormal results flushed to zero; 2^-inf = 0).  The
// softmax only takes it of x <= 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A piece of a cut pair as every holder of a piece sees it: the CTAs holding its first and
// last pieces, where the first CTA stored its piece (slot 0 when the pair's family is that
// CTA's first family), and the pair's sequence and heads.
struct CutPiece {
  int c_first, c_last, first_slot, s, h0, nh;
};

__device__ __forceinline__ CutPiece cut_piece(const Fam& f, int pi, const PairHeads& ph,
                                              long long W, int G, const Params& p) {
  CutPiece cp;
  const long long first_unit = f.pre + p.seg_cost + pi;
  const long long last_unit = first_unit + static_cast<long long>(f.ns - 1) * p.gs;
  cp.c_first = owner_of(first_unit, W, G);
  cp.c_last = owner_of(last_unit, W, G);
  long long w0f, w1f;
  share_of(cp.c_first, W, G, w0f, w1f);
  cp.first_slot = w0f >= f.pre ? 0 : 1;
  cp.s = f.s;
  cp.h0 = ph.h0;
  cp.nh = ph.nh;
  return cp;
}

// Count one piece in at a pair's counter (pa_arrive.h): the count this arrival makes
// (n: it completed the pair, and the counter is back at zero), or -1 if it gave up.  The
// loop retries only when another arrival changed the counter in between, so it ends after
// at most one try per piece.
struct DeviceCas {
  __device__ unsigned long long operator()(unsigned long long* a, unsigned long long e,
                                           unsigned long long d) const {
    return atomicCAS(a, e, d);
  }
};
struct DeviceLoad {
  __device__ unsigned long long operator()(unsigned long long* a) const {
    return *reinterpret_cast<volatile unsigned long long*>(a);
  }
};

__device__ __forceinline__ int arrive(unsigned long long* ctr, unsigned long long epoch, int n) {
  return arrive_count(ctr, epoch, n, DeviceCas(), DeviceLoad());
}

// Merge the pieces of a cut pair held by CTAs c..c_last (c's piece in slot `first_slot`,
// the others in slot 0), pieces taken in CTA order so the result is deterministic:
//   M = max m_i,  w_i = 2^(m_i - M) (0 for an empty piece),  L = sum l_i w_i,
//   out = sum w_i acc_i / L
// (the log-sum-exp rescaling of online softmax); zeros when a piece saw a bad block.
// merge_staged computes the same sums in the same order with the same fused multiply-adds,
// so a pair's output does not depend on which of the two merges it.
template <int D, typename T, bool QK>
__device__ void merge_pieces(const Params& p, int pi, int c, int first_slot, int c_last, int nh,
                             T* out_rows, int gt, int gthreads) {
  constexpr int C4 = D / 4;  // 4-float chunks per head row
  const int hpp = p.heads_per_pair;
  const int hstep = gthreads / C4;  // heads the group covers side by side
  const int d4 = (gt % C4) * 4;
  auto piece_of = [&](int cc) {
    return (static_cast<size_t>(cc) * 2 + (cc == c ? first_slot : 0)) * p.gs + pi;
  };
  for (int h = gt / C4; h < nh; h += hstep) {
    float M = -INFINITY;
    bool bad = false;
    for (int cc = c; cc <= c_last; ++cc) {
      const float* ml = p.part_ml + (piece_of(cc) * hpp + h) * 2;
      M = fmaxf(M, __ldcg(ml));
      bad |= __ldcg(ml + 1) < 0.f;
    }
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = c; cc <= c_last; ++cc) {
      const size_t pc = piece_of(cc);
      const float* ml = p.part_ml + (pc * hpp + h) * 2;
      const float m = __ldcg(ml), l = __ldcg(ml + 1);
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      L = fmaf(l, w, L);
      const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_acc + (pc * hpp + h) * D + d4));
      O.x = fmaf(a.x, w, O.x);
      O.y = fmaf(a.y, w, O.y);
      O.z = fmaf(a.z, w, O.z);
      O.w = fmaf(a.w, w, O.w);
    }
    uint2 packed = make_uint2(0u, 0u);
    if (!bad) {
      const float inv = QK ? p.out_scale / L : 1.f / L;
      packed.x = pack2<T>(O.x * inv, O.y * inv);
      packed.y = pack2<T>(O.z * inv, O.w * inv);
    }
    *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
  }
}

// Wait for the phase of `bar` with parity `parity`, bounded by kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}


// merge_staged when every piece of both pairs fits in the ring at once: every piece's O
// by one bulk copy, the (m, l) by plain loads behind them, a single round trip.
template <int D, typename T, bool QK>
__device__ bool merge_staged_once(const Params& p, int pi, const CutPiece& job0,
                                  const CutPiece& job1, int njobs, uint32_t ring,
                                  uint8_t* ring_ptr, uint32_t bar, uint32_t& bar_phase, int lane) {
  const int hpp = p.heads_per_pair;
  const int np0 = job0.c_last - job0.c_first + 1;
  const int np1 = njobs > 1 ? job1.c_last - job1.c_first + 1 : 0;
  const uint32_t rb0 = job0.nh * D * 4, rb1 = job1.nh * D * 4;
  const uint32_t acc_bytes = np0 * rb0 + np1 * rb1;
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(bar, acc_bytes);
  __syncwarp();
  // the ring was last read through the generic proxy; the bulk copies write it through
  // the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  for (int i = lane; i < np0 + np1; i += 32) {
    const bool first = i < np0;
    const CutPiece& cp = first ? job0 : job1;
    const int cc = cp.c_first + (first ? i : i - np0);
    const size_t piece = (static_cast<size_t>(cc) * 2 + (cc == cp.c_first ? cp.first_slot : 0)) * p.gs + pi;
    const uint32_t off = first ? i * rb0 : np0 * rb0 + (i - np0) * rb1;
    bulk_g2s(ring + off, p.part_acc + piece * hpp * D, first ? rb0 : rb1, bar);
  }
  float2* ml = reinterpret_cast<float2*>(ring_ptr + acc_bytes);
  {
    int k = 0;
    for (int j = 0; j < njobs; ++j) {
      const CutPiece& cp = j == 0 ? job0 : job1;
      const int np = cp.c_last - cp.c_first + 1;
      for (int i = lane; i < np * cp.nh; i += 32) {
        const int cc = cp.c_first + i / cp.nh, h = i % cp.nh;
        const size_t piece = (static_cast<size_t>(cc) * 2 + (cc == cp.c_first ? cp.first_slot : 0)) * p.gs + pi;
        const float* src = p.part_ml + (piece * hpp + h) * 2;
        ml[k + i] = make_float2(__ldcg(src), __ldcg(src + 1));
      }
      k += np * cp.nh;
    }
  }
  __syncwarp();  // (the (m, l) stores, before lanes read other lanes' entries)
  // Pass 1, one lane per (job, head): M, the weights in place of the m_i, and L in place
  // of the first piece's l (negative for a bad piece: zeros out).
  {
    int moff = 0;
    for (int j = 0; j < njobs; ++j) {
      const CutPiece& cp = j == 0 ? job0 : job1;
      const int np = cp.c_last - cp.c_first + 1;
      for (int h = lane; h < cp.nh; h += 32) {
        float M = -INFINITY;
        bool bad = false;
        for (int i = 0; i < np; ++i) {
          const float2 v = ml[moff + i * cp.nh + h];
          M = fmaxf(M, v.x);
          bad |= v.y < 0.f;
        }
        float L = 0.f;
        for (int i = 0; i < np; ++i) {
          float2 v = ml[moff + i * cp.nh + h];
          const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M);
          L = fmaf(v.y, w, L);
          v.x = w;
          ml[moff + i * cp.nh + h] = v;
        }
        ml[moff + h].y = bad ? -1.f : L;
      }
      moff += np * cp.nh;
    }
  }
  const bool landed = mbar_wait_limit(bar, bar_phase);  // (bounded; never expected to expire)
  bar_phase ^= 1u;
  if (!landed) {
    if (lane == 0) atomicOr(p.err, kErrTimeout);
    return true;
  }
  __syncwarp();
  // Pass 2: out = sum_i w_i acc_i / L, pieces in CTA order.
  constexpr int C4 = D / 4;
  int aoff = 0, moff = 0;
  for (int j = 0; j < njobs; ++j) {
    const CutPiece& cp = j == 0 ? job0 : job1;
    const int np = cp.c_last - cp.c_first + 1;
    T* out_rows = reinterpret_cast<T*>(p.out) + (static_cast<size_t>(cp.s) * p.num_q_heads + cp.h0) * D;
    const float* acc = reinterpret_cast<const float*>(ring_ptr + aoff);
    for (int idx = lane; idx < cp.nh * C4; idx += 32) {
      const int h = idx / C4, d4 = (idx % C4) * 4;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int i = 0; i < np; ++i) {
        const float w = ml[moff + i * cp.nh + h].x;
        const float4 a = *reinterpret_cast<const float4*>(acc + (i * cp.nh + h) * D + d4);
        O.x = fmaf(a.x, w, O.x);
        O.y = fmaf(a.y, w, O.y);
        O.z = fmaf(a.z, w, O.z);
        O.w = fmaf(a.w, w, O.w);
      }
      const float L = ml[moff + h].y;
      uint2 packed = make_uint2(0u, 0u);
      if (L >= 0.f) {
        const float inv = QK ? p.out_scale / L : 1.f / L;
        packed.x = pack2<T>(O.x * inv, O.y * inv);
        packed.y = pack2<T>(O.z * inv, O.w * inv);
      }
      *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
    }
    aoff += np * cp.nh * D * 4;
    moff += np * cp.nh;
  }
  return true;
}

// One warp merges the cut pairs it completed (up to two) through its own ring, which is
// idle once the share is streamed.  When everything fits, merge_staged_once stages it in
// one round trip.  Otherwise every piece's (m, l) comes in by plain loads (one round trip
// for all pieces of both pairs), then every piece's O by one bulk copy per piece, as many
// pieces at a time as the ring holds, so a pair cut into any number of pieces is merged in
// ring-sized chunks.  The pieces are folded in CTA order:
//   M = max m_i,  w_i = 2^(m_i - M),  L = sum l_i w_i,  out = sum w_i acc_i / L,
// with the same fused multiply-adds as merge_pieces, so a pair's output does not depend on
// which CTA merges it.  Returns false, having done nothing, when the (m, l) of the pieces
// do not fit in half the ring (a pair cut into thousands of pieces): merge_pieces then.
template <int D, typename T, bool QK>
__device__ bool merge_staged_chunked(const Params& p, int pi, const CutPiece& job0,
                                     const CutPiece& job1, int njobs, uint32_t ring,
                                     uint8_t* ring_ptr, int ring_bytes, uint32_t bar,
                                     uint32_t& bar_phase, int lane);

template <int D, typename T, bool QK>
__device__ __forceinline__ bool merge_staged(const Params& p, int pi, const CutPiece& job0,
                                             const CutPiece& job1, int njobs, uint32_t ring,
                                             uint8_t* ring_ptr, int ring_bytes, uint32_t bar,
                                             uint32_t& bar_phase, int lane) {
  int mlen = 0;  // (m, l) entries of every piece of every job
  for (int j = 0; j < njobs; ++j) {
    const CutPiece& cp = j == 0 ? job0 : job1;
    mlen += (cp.c_last - cp.c_first + 1) * cp.nh;
  }
  const uint32_t ml_bytes = (static_cast<uint32_t>(mlen) * 8u + 127u) & ~127u;
  const int np0 = job0.c_last - job0.c_first + 1;
  const int np1 = njobs > 1 ? job1.c_last - job1.c_first + 1 : 0;
  const uint32_t acc_bytes = np0 * job0.nh * D * 4 + np1 * job1.nh * D * 4;
  if (acc_bytes + ml_bytes <= static_cast<uint32_t>(ring_bytes))
    return merge_staged_once<D, T, QK>(p, pi, job0, job1, njobs, ring, ring_ptr, bar, bar_phase,
                                       lane);
  return merge_staged_chunked<D, T, QK>(p, pi, job0, job1, njobs, ring, ring_ptr, ring_bytes, bar,
                                        bar_phase, lane);
}

template <int D, typename T, bool QK>
__device__ bool merge_staged_chunked(const Params& p, int pi, const CutPiece& job0,
                                     const CutPiece& job1, int njobs, uint32_t ring,
                                     uint8_t* ring_ptr, int ring_bytes, uint32_t bar,
                                     uint32_t& bar_phase, int lane) {
  constexpr int C4 = D / 4;  // 4-float chunks of a head row
  constexpr int NI = 4;      // a lane's chunks of a pair's rows per round (128 a warp)
  const int hpp = p.heads_per_pair;
  auto piece_of = [&](const CutPiece& cp, int cc) {
    return (static_cast<size_t>(cc) * 2 + (cc == cp.c_first ? cp.first_slot : 0)) * p.gs + pi;
  };
  int mlen = 0;  // (m, l) entries of every piece of every job
  for (int j = 0; j < njobs; ++j) {
    const CutPiece& cp = j == 0 ? job0 : job1;
    mlen += (cp.c_last - cp.c_first + 1) * cp.nh;
  }
  const uint32_t ml_bytes = (static_cast<uint32_t>(mlen) * 8u + 127u) & ~127u;
  if (2 * static_cast<int>(ml_bytes) > ring_bytes) return false;
  // (m, l) of every piece at the start of the ring; the O chunks after them.
  float2* ml = reinterpret_cast<float2*>(ring_ptr);
  const uint32_t acc0 = ml_bytes;
  const int acc_room = ring_bytes - static_cast<int>(ml_bytes);
  __syncwarp();  // (every lane is done with the ring's last stage)
  {
    int k = 0;
    for (int j = 0; j < njobs; ++j) {
      const CutPiece& cp = j == 0 ? job0 : job1;
      const int np = cp.c_last - cp.c_first + 1;
      for (int i = lane; i < np * cp.nh; i += 32) {
        const int cc = cp.c_first + i / cp.nh, h = i % cp.nh;
        const float* src = p.part_ml + (piece_of(cp, cc) * hpp + h) * 2;
        ml[k + i] = make_float2(__ldcg(src), __ldcg(src + 1));
      }
      k += np * cp.nh;
    }
  }
  __syncwarp();  // (the (m, l) stores, before lanes read other lanes' entries)
  // Pass 1, one lane per (job, head): M = max m_i, then each piece's weight 2^(m_i - M)
  // (0 for an empty piece) in place of m_i, and L = sum l_i 2^(m_i - M) in place of the
  // first piece's l (bad pieces, l < 0, make L negative: the head's output is zeros).
  {
    int moff = 0;
    for (int j = 0; j < njobs; ++j) {
      const CutPiece& cp = j == 0 ? job0 : job1;
      const int np = cp.c_last - cp.c_first + 1;
      for (int h = lane; h < cp.nh; h += 32) {
        float M = -INFINITY;
        bool bad = false;
        for (int i = 0; i < np; ++i) {
          const float2 v = ml[moff + i * cp.nh + h];
          M = fmaxf(M, v.x);
          bad |= v.y < 0.f;
        }
        float L = 0.f;
        for (int i = 0; i < np; ++i) {
          float2 v = ml[moff + i * cp.nh + h];
          const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M);
          L = fmaf(v.y, w, L);
          v.x = w;
          ml[moff + i * cp.nh + h] = v;
        }
        ml[moff + h].y = bad ? -1.f : L;  // (read back below only through this slot)
      }
      moff += np * cp.nh;
    }
  }
  // Pass 2, per job and round of 128 output chunks: out = sum_i w_i acc_i / L, pieces in
  // CTA order, staged in chunks.
  int moff = 0;
  for (int j = 0; j < njobs; ++j) {
    const CutPiece& cp = j == 0 ? job0 : job1;
    const int np = cp.c_last - cp.c_first + 1;
    const uint32_t rb = static_cast<uint32_t>(cp.nh) * D * 4;  // O bytes of one piece
    const int cap = acc_room / static_cast<int>(rb);          // pieces a chunk holds
    for (int base = 0; base < cp.nh * C4; base += 32 * NI) {
    float4 O[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) O[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < np; c0 += cap) {
      const int nc = min(cap, np - c0);
      __syncwarp();  // (every lane is done reading the previous chunk)
      // the ring was last read through the generic proxy; the bulk copies write it
      // through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nc) * rb);
      __syncwarp();
      for (int i = lane; i < nc; i += 32)
        bulk_g2s(ring + acc0 + i * rb, p.part_acc + piece_of(cp, cp.c_first + c0 + i) * hpp * D,
                 rb, bar);
      const bool landed = mbar_wait_limit(bar, bar_phase);  // (bounded; never expected to expire)
      bar_phase ^= 1u;
      if (!landed) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        // the copies may still land: leave the ring (and the rest of the merge) alone
        return true;
      }
      const float* acc = reinterpret_cast<const float*>(ring_ptr + acc0);
#pragma unroll
      for (int it = 0; it < NI; ++it) {
        const int idx = base + lane + 32 * it;
        if (idx >= cp.nh * C4) continue;
        const int h = idx / C4, d4 = (idx % C4) * 4;
#pragma unroll 4
        for (int i = 0; i < nc; ++i) {
          const float w = ml[moff + (c0 + i) * cp.nh + h].x;
          const float4 a = *reinterpret_cast<const float4*>(acc + (i * cp.nh + h) * D + d4);
          O[it].x = fmaf(a.x, w, O[it].x);
          O[it].y = fmaf(a.y, w, O[it].y);
          O[it].z = fmaf(a.z, w, O[it].z);
          O[it].w = fmaf(a.w, w, O[it].w);
        }
      }
    }
    T* out_rows = reinterpret_cast<T*>(p.out) + (static_cast<size_t>(cp.s) * p.num_q_heads + cp.h0) * D;
#pragma unroll
    for (int it = 0; it < NI; ++it) {
      const int idx = base + lane + 32 * it;
      if (idx >= cp.nh * C4) continue;
      const int h = idx / C4, d4 = (idx % C4) * 4;
      const float L = ml[moff + h].y;
      uint2 packed = make_uint2(0u, 0u);
      if (L >= 0.f) {
        const float inv = QK ? p.out_scale / L : 1.f / L;
        packed.x = pack2<T>(O[it].x * inv, O[it].y * inv);
        packed.y = pack2<T>(O[it].z * inv, O[it].w * inv);
      }
      *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
    }
    }
    moff += np * cp.nh;
  }
  return true;
}

// A pair whose arrival gave up (no merge will come): zeros for its output rows.
template <int D, typename T>
__device__ void zero_pair(const Params& p, const CutPiece& cp, int gt, int gthreads) {
  T* out_rows = reinterpret_cast<T*>(p.out) + (static_cast<size_t>(cp.s) * p.num_q_heads + cp.h0) * D;
  for (int i = gt; i < cp.nh * D / 8; i += gthreads)
    reinterpret_cast<uint4*>(out_rows)[i] = make_uint4(0u, 0u, 0u, 0u);
}

template <int D, int KV>
struct Smem {
  uint8_t ring[kWarps][Geo<D, KV>::kSlots][Geo<D, KV>::kStageBytes];  // 1024-byte aligned
  // quantised blocks, fused step: the newest token's 16-bit K and V rows, per ring slot
  uint8_t newrow[kWarps][Geo<D, KV>::kSlots][KV == kKv16 ? 16 : 4 * D];
  float xo[kWarps][4][D];  // per-warp O rows, 4 heads per exchange round
  float xm[kWarps][kMaxHeads], xl[kWarps][kMaxHeads];
  long long scan[kWarps];
  long long start_pre;
  int start_s;
  int last[kWarps];  // per pair group: this CTA's arrival completed the pair
  unsigned long long merge_bar[kWarps];  // per warp: the staged merge's copies, one phase a chunk
};

// Q^T of a pair as MMA B fragments (column n = head 8*nt + lane / 4; heads >= nh are zero).
template <int D, int NTH>
__device__ __forceinline__ void load_q(const Params& p, int s, int h0, int nh, int lane,
                                       uint32_t (&qb)[D / 16][NTH][2]) {
  const int r0 = lane >> 2, qc = 2 * (lane & 3);
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
      p.q + (static_cast<size_t>(s) * p.num_q_heads + h0) * D * 2);
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt) {
    const int h = nt * 8 + r0;
    const bool hv = h < nh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int col = 16 * ks + qc;
      qb[ks][nt][0] = hv ? __ldg(qrow + (h * D + col) / 2) : 0u;
      qb[ks][nt][1] = hv ? __ldg(qrow + (h * D + col + 8) / 2) : 0u;
    }
  }
}

// The same for FP8 blocks, as f16 (the type the E4M3 values are widened to), with d in the
// order the K fragments use: k-step ks takes d = (D/4) t + 4 ks + {0, 1} into b0 and
// + {2, 3} into b1, t = lane % 4.  bf16 queries are rounded to f16 (exact within the f16
// normal range).
template <int D, int NTH, typename T>
__device__ __forceinline__ void load_q8(const Params& p, int s, int h0, int nh, int lane,
                                        uint32_t (&qb)[D / 16][NTH][2]) {
  const int r0 = lane >> 2, t = lane & 3;
  const uint2* qrow = reinterpret_cast<const uint2*>(
      p.q + (static_cast<size_t>(s) * p.num_q_heads + h0) * D * 2);
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt) {
    const int h = nt * 8 + r0;
    const bool hv = h < nh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint2 w = hv ? __ldg(qrow + (h * D + (D / 4) * t + 4 * ks) / 4) : make_uint2(0u, 0u);
      if (std::is_same<T, __half>::value) {
        qb[ks][nt][0] = w.x;
        qb[ks][nt][1] = w.y;
      } else {
        const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y);
        qb[ks][nt][0] = pack2<__half>(a.x, a.y);
        qb[ks][nt][1] = pack2<__half>(b.x, b.y);
      }
    }
  }
}

// Q^T for INT4 blocks, as f16, in the d order the K fragments use: k-steps 2j and 2j + 1
// take the eight d = (D/4) t + 8 j + {0..7} of word j of a K row, k-step 2j + e getting
// d + 2e and d + 2e + 4 in b0 and d + 2e + 1 and d + 2e + 5 in b1 (t = lane % 4).  b1
// meets the high nibbles (1024 + 16 u), so it holds q / 16 (exact unless q / 16 is an f16
// subnormal, |q| < 2^-10).
template <int D, int NTH, typename T>
__device__ __forceinline__ void load_q4(const Params& p, int s, int h0, int nh, int lane,
                                        uint32_t (&qb)[D / 16][NTH][2]) {
  const int r0 = lane >> 2, t = lane & 3;
  const uint4* qrow = reinterpret_cast<const uint4*>(
      p.q + (static_cast<size_t>(s) * p.num_q_heads + h0) * D * 2);
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt) {
    const int h = nt * 8 + r0;
    const bool hv = h < nh;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const uint4 w = hv ? __ldg(qrow + (h * D + (D / 4) * t + 8 * j) / 8) : make_uint4(0u, 0u, 0u, 0u);
      const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y), c = unpack2<T>(w.z),
                   d = unpack2<T>(w.w);  // d + 0,1 / 2,3 / 4,5 / 6,7
      qb[2 * j][nt][0] = pack2<__half>(a.x, c.x);
      qb[2 * j][nt][1] = pack2<__half>(a.y * 0.0625f, c.y * 0.0625f);
      qb[2 * j + 1][nt][0] = pack2<__half>(b.x, d.x);
      qb[2 * j + 1][nt][1] = pack2<__half>(b.y * 0.0625f, d.y * 0.0625f);
    }
  }
}

// The next family (after f) where pair pi has units to compute; false at the share's end.
__device__ __forceinline__ bool next_busy_fam(Fam f, int pi, long long w0, long long w1,
                                              const Params& p, Fam& out) {
  for (;;) {
    fam_next(f, p);
    if (f.s >= p.num_seqs || f.pre >= w1) return false;
    const int2 r = unit_range(f, pi, w0, w1, p);
    if (fam_valid(f) && r.x < r.y) {
      out = f;
      return true;
    }
  }
}

// KV = kKvFp8: K/V blocks hold E4M3 codes (scales folded into scale_log2 and out_scale).
// KV = kKvInt4: K/V blocks hold INT4 codes with a float32 scale per row: a token's K scale
// multiplies its scores, its V scale its weights in P V.  Both quantised formats run the
// MMAs in f16 on values widened exactly, with 32-token stages and the permuted d order of
// O (drow).  The fused step (key_new) quantises the newest rows in the kernel.
// NEW: compiled for the fused step (key_new set); a plain decode runs a copy compiled
// without that code, which uses fewer instructions and registers in the stage loop.
template <int D, int NTH, typename T, int KV, bool NEW>
__global__ void __launch_bounds__(kThreads, 1) PA_DECODE_KERNEL(const __grid_constant__ Params p
                                                                  PA_DECODE_TIMELINE_ARG) {
  constexpr bool F8 = KV == kKvFp8;
  constexpr bool I4 = KV == kKvInt4;
  constexpr bool QK = KV != kKv16;  // quantised blocks
  using G_ = Geo<D, KV>;
  using TM = typename std::conditional<QK, __half, T>::type;  // MMA operand type
  constexpr int R = G_::kSlots;
  constexpr int KS = G_::kKSteps;
  constexpr int ST = G_::kTok;  // tokens per stage
  constexpr int U = ST / 16;    // 16-token m-tiles per stage
  constexpr int MT = D / 16;  // m-tiles of O^T (16 rows of d each)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  Smem<D, KV>& sm = *reinterpret_cast<Smem<D, KV>*>(smem_raw + (((raw_addr + 1023) & ~1023u) - raw_addr));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int P = p.phases;
  const int pi = warp / P;     // this warp's pair within each family
  const int phase = warp % P;  // and its units: unit index = phase (mod P)
  const int gt = phase * 32 + lane;  // thread index within the pair's P warps
  const int gthreads = P * 32;
  // the pair's P warps: their own named barrier (ids 1..8), or just the warp when P = 1
  auto gsync = [&]() {
    if (P == 1) __syncwarp();
    else named_bar_sync(1 + pi, gthreads);
  };
  auto gor = [&](bool v) -> bool {
    return P == 1 ? (__any_sync(0xffffffffu, v) != 0) : bar_red_or(1 + pi, gthreads, v);
  };

  // The next kernel in the stream may start launching.  Everything up to the first copy
  // reads only context_lens and block_tables (the share, the first family, the first
  // stages' table entries), which no kernel of this library writes; it runs while the
  // kernel before this one drains.  The wait comes before anything touches q, the caches
  // or the workspace.
  pdl_launch_dependents();

  if (lane == 0) {
    mbar_init(smem_addr(&sm.merge_bar[warp]), 1);
    fence_mbar_init();
  }

  // ---- setup: total units W, this CTA's share [w0, w1), and its first family ----
  const int per = (p.num_seqs + kThreads - 1) / kThreads;
  const int sa = min(p.num_seqs, tid * per), sb = min(p.num_seqs, sa + per);
  long long mine = 0;
  for (int s = sa; s < sb; ++s)
    mine += static_cast<long long>(p.ngroups) *
            (static_cast<long long>(pair_stages(__ldg(p.context_lens + s), p)) * p.gs +
             p.seg_cost);
  long long incl = mine;  // inclusive scan of `mine` over the block
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  long long before = 0, W = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += sm.scan[w];
    W += sm.scan[w];
  }
  const long long excl = before + incl - mine;
  const int G = gridDim.x;
  const int c = blockIdx.x;
  long long w0, w1;
  share_of(c, W, G, w0, w1);
  if (w0 < w1 && excl <= w0 && w0 < excl + mine) {
    long long pre = excl;
    int s = sa;
    for (;; ++s) {
      const long long u = static_cast<long long>(p.ngroups) *
                          (static_cast<long long>(pair_stages(__ldg(p.context_lens + s), p)) *
                               p.gs + p.seg_cost);
      if (w0 < pre + u) break;
      pre += u;
    }
    sm.start_s = s;
    sm.start_pre = pre;
  }
  __syncthreads();
  if (w0 >= w1) return;  // more CTAs than units: nothing here (uniform over the CTA)

  Fam first;
  first.s = sm.start_s;
  first.g = 0;
  first.pre = sm.start_pre;
  fam_load(first, p);
  while (w0 >= first.pre + first.fw) {  // the family holding unit w0
    first.pre += first.fw;
    ++first.g;
  }

  // ---- this warp's copy stream: kAhead stages in flight ahead of the one computed ----
  const uint32_t ring = smem_addr(sm.ring[warp][0]);
  const int ch = lane % G_::kRowChunks;    // this lane's 16-byte column chunk of a row
  const int rsub = lane / G_::kRowChunks;  // and its first row
  StageIt sit;
  sit.f = first;
  stage_it_enter(sit, pi, phase, w0, w1, p);
  constexpr int NE = G_::kMaxSpan;
  Stage nxt;
  bool nxt_ok = next_stage(sit, pi, phase, w0, w1, nxt, p);
  int nxt_e[NE];
#pragma unroll
  for (int k = 0; k < NE; ++k) nxt_e[k] = 0;
  if (nxt_ok) stage_entries<NE>(nxt, p, nxt_e);
  uint32_t issued = 0;   // stages this warp has issued (slot = count % R)
  uint32_t badbits = 0;  // slots whose stage has an out-of-range block id

  auto issue_one = [&]() {
    if (nxt_ok) {
      const uint32_t slot = issued % R;
      bool bad = false;
#pragma unroll
      for (int k = 0; k < NE; ++k) bad = bad || nxt_e[k] < 0 || nxt_e[k] >= p.num_blocks;
      badbits = bad ? (badbits | (1u << slot)) : (badbits & ~(1u << slot));
      if (!bad) {
        const uint32_t dst = ring + slot * G_::kStageBytes;
        const int row0 = nxt.t0 & (p.block_size - 1);
        size_t rbase[NE];  // first cache row of (block e[k], kv head)
#pragma unroll
        for (int k = 0; k < NE; ++k)
          rbase[k] = static_cast<size_t>((nxt_e[k] * p.num_kv_heads + nxt.kvh) * p.block_size);
        // A whole stage whose rows a pass never splits between blocks (rows per pass <= B):
        // each pass's block and row offset are constants for the block size, so the copies
        // need one base address per block.
        auto copy_whole = [&](auto lbc) {
          constexpr int LB = decltype(lbc)::value;
          constexpr int B = 1 << LB;
          constexpr int RPP = G_::kRowsPerPass;
          constexpr int NEU = ST / B > 1 ? ST / B : 1;
          const uint8_t* gk[NEU];
          const uint8_t* gv[NEU];
#pragma unroll
          for (int k = 0; k < NEU; ++k) {
            const size_t off = (rbase[k] + row0 + rsub) * G_::kRowBytes + ch * 16;
            gk[k] = p.k_cache + off;
            gv[k] = p.v_cache + off;
          }
#pragma unroll
          for (int j = 0; j < G_::kPasses; ++j) {
            const int kk = min(NEU - 1, (RPP * j) >> LB);
            const ptrdiff_t goff = static_cast<ptrdiff_t>(RPP * j - kk * B) * G_::kRowBytes;
            const uint32_t so = dst + copy_dst<D, KV, G_::kRowBytes>(rsub, ch, j);
            cp_async16(so, gk[kk] + goff, 16u);
            cp_async16(so + G_::kKBytes, gv[kk] + goff, 16u);
          }
        };
        const bool whole_stage = nxt.nt == ST && G_::kRowsPerPass <= p.block_size &&
                                 !(!QK && NEW && nxt.last);
        if (whole_stage) {
          if (p.log2_block == 3) copy_whole(std::integral_constant<int, 3>());
          else if (p.log2_block == 4) copy_whole(std::integral_constant<int, 4>());
          else copy_whole(std::integral_constant<int, 5>());
        } else {
#pragma unroll
        for (int j = 0; j < G_::kPasses; ++j) {
          const int row = rsub + j * G_::kRowsPerPass;
          const int r = row0 + row;
          const bool live = row < nxt.nt;
          const int kk = r >> p.log2_block;  // which of the stage's blocks
          size_t rb = rbase[0];
#pragma unroll
          for (int k = 1; k < NE; ++k) rb = kk == k ? rbase[k] : rb;
          // rows past the context: zero-filled, nothing read (the source stays in block e[0])
          const size_t grow = !live ? rbase[0] : rb + (r & (p.block_size - 1));
          const size_t src = grow * G_::kRowBytes + ch * 16;
          const uint32_t so = I4 ? swz4<D>(row, ch) : (F8 ? swz8<D>(row, ch) : swz(row, ch));
          if (!QK && NEW && nxt.last && row == nxt.nt - 1) {
            // the newest token: from the step's input (the cache row is written later)
            const size_t nsrc = ((static_cast<size_t>(nxt.s) * p.num_kv_heads + nxt.kvh) * D + ch * 8) * 2;
            cp_async16(dst + so, p.key_new + nsrc, 16u);
            cp_async16(dst + G_::kKBytes + so, p.value_new + nsrc, 16u);
          } else {
            cp_async16(dst + so, p.k_cache + src, live ? 16u : 0u);
            cp_async16(dst + G_::kKBytes + so, p.v_cache + src, live ? 16u : 0u);
          }
        }
        }
        if constexpr (QK) {
          // fused step: the newest token's 16-bit K and V rows into this slot's scratch
          // (quantised when the stage is computed)
          constexpr int CR = D / 8;  // 16-byte chunks of a 16-bit row
          if (NEW && nxt.last && lane < 2 * CR) {
            const int isv = lane >= CR ? 1 : 0, c = lane % CR;
            const size_t nsrc = ((static_cast<size_t>(nxt.s) * p.num_kv_heads + nxt.kvh) * D + c * 8) * 2;
            cp_async16(smem_addr(sm.newrow[warp][slot]) + isv * 2 * D + 16 * c,
                       (isv ? p.value_new : p.key_new) + nsrc, 16u);
          }
        }
        if constexpr (I4) {
          // the rows' scales: lanes 0-7 copy K's, 8-15 V's, four tokens (16 bytes) each; a
          // token past the context gets scale 0 (its codes are zero-filled too)
          constexpr int SC = G_::kTok / 4;  // 16-byte chunks of one stage's K scales
          if (lane < 2 * SC) {
            const int cc = lane % SC;
            const int r = row0 + 4 * cc;
            const int kk = r >> p.log2_block;
            size_t rb = rbase[0];
#pragma unroll
            for (int k = 1; k < NE; ++k) rb = kk == k ? rbase[k] : rb;
            const int live = max(0, min(4, nxt.nt - 4 * cc));
            const size_t srow = live ? rb + (r & (p.block_size - 1)) : rbase[0];
            const float* sbase = lane < SC ? p.k_scales : p.v_scales;
            cp_async16(dst + 2 * G_::kKBytes + (lane < SC ? 0 : G_::kScaleBytes) + 16 * cc,
                       sbase + srow, 4u * live);
          }
        }
      }
      ++issued;
      nxt_ok = next_stage(sit, pi, phase, w0, w1, nxt, p);
      if (nxt_ok) stage_entries<NE>(nxt, p, nxt_e);
    }
    cp_async_commit();  // one group per call, empty or not
  };
  // Warm L2 with the blocks of this warp's first 4 * kAhead stages (INT4: kAhead stages,
  // whose blocks already come as many small prefetches) of its first pair, while the
  // kernel before this one drains: one lane per block, one bulk prefetch per block's K
  // rows and V rows (and INT4 scales) of the pair's kv head.  On GB300 the 16-bit decode
  // of 64 sequences of 128..2048 tokens took 53.3 / 52.6 / 51.4 / 56.1 us with 1 / 2 / 4
  // / 8 times kAhead stages (8: the prefetches start to evict each other from L2); INT4
  // took 36.8 us with 1 and 37.9 us with 4.
  if (nxt_ok) {
    const int j0 = nxt.t0 >> p.log2_block;
    constexpr int kPre = (I4 ? 1 : 4) * G_::kAhead * ST;  // tokens to warm
    const int tl = min(p.max_ctx, min(__ldg(p.context_lens + nxt.s), nxt.t0 + kPre)) - 1;
    const int nbk = (tl >> p.log2_block) - j0 + 1;
    if (lane < nbk) {
      const int e = __ldg(p.block_tables + static_cast<size_t>(nxt.s) * p.max_blocks_per_seq + j0 + lane);
      if (e >= 0 && e < p.num_blocks) {
        const size_t row = (static_cast<size_t>(e) * p.num_kv_heads + nxt.kvh) * p.block_size;
        const uint32_t bytes = static_cast<uint32_t>(p.block_size) * G_::kRowBytes;
        prefetch_l2(p.k_cache + row * G_::kRowBytes, bytes);
        prefetch_l2(p.v_cache + row * G_::kRowBytes, bytes);
        if constexpr (I4) {
          prefetch_l2(p.k_scales + row, 4u * p.block_size);
          prefetch_l2(p.v_scales + row, 4u * p.block_size);
        }
      }
    }
  }
  // the kernel before this one (say the cache write) has finished and its writes are
  // visible past this point
  pdl_wait_primary();
  PA_DECODE_STAMP(0);
#pragma unroll
  for (int a = 0; a < G_::kAhead; ++a) issue_one();

  const int r0 = lane >> 2;        // MMA row of this lane
  const int qc = 2 * (lane & 3);   // MMA column pair of this lane
  const int lrow = lane & 7;       // ldmatrix: row within an 8x8 matrix
  const int lmat = lane >> 3;      // ldmatrix: which of the four matrices

  // q of the first family where this pair computes; later ones are loaded a family ahead
  uint32_t qn[KS][NTH][2];
  {
    const int2 r = unit_range(first, pi, w0, w1, p);
    Fam qf;
    bool have = fam_valid(first) && r.x < r.y;
    if (have) qf = first;
    else have = next_busy_fam(first, pi, w0, w1, p, qf);
    if (have) {
      const PairHeads ph = pair_heads(p, qf.g * p.gs + pi);
      if (I4) load_q4<D, NTH, T>(p, qf.s, ph.h0, ph.nh, lane, qn);
      else if (F8) load_q8<D, NTH, T>(p, qf.s, ph.h0, ph.nh, lane, qn);
      else load_q<D, NTH>(p, qf.s, ph.h0, ph.nh, lane, qn);
    }
  }

  uint32_t used = 0;  // stages this warp has computed
  bool cta_first = true;
  // This warp's pieces of cut pairs (at most two: in the share's first and last families),
  // counted in after the share is streamed.
  CutPiece cut_a, cut_b;
  int ncut = 0;
  int early = 0, early_last = 0, early_lost = 0;  // pieces counted in before the share's end
  for (Fam f = first; f.s < p.num_seqs && f.pre < w1; fam_next(f, p), cta_first = false) {
    const int2 r = unit_range(f, pi, w0, w1, p);
    if (!has_piece(r, f.ns)) continue;
    const PairHeads ph = pair_heads(p, f.g * p.gs + pi);
    T* out_rows =
        reinterpret_cast<T*>(p.out) + (static_cast<size_t>(f.s) * p.num_q_heads + ph.h0) * D;
    if (!fam_valid(f)) {  // invalid context length: the unit-0 holder writes zeros
      if (r.x == 0 && r.x < r.y) {
        for (int i = gt; i < ph.nh * D / 8; i += gthreads)
          reinterpret_cast<uint4*>(out_rows)[i] = make_uint4(0, 0, 0, 0);
        if (gt == 0) atomicOr(p.err, kErrBadContext);
      }
      continue;
    }
    const bool computes = r.x < r.y;  // (an empty middle piece computes nothing)
    uint32_t qb[KS][NTH][2];
    if (computes) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          qb[ks][nt][0] = qn[ks][nt][0];
          qb[ks][nt][1] = qn[ks][nt][1];
        }
      Fam qf;
      if (next_busy_fam(f, pi, w0, w1, p, qf)) {
        const PairHeads lh = pair_heads(p, qf.g * p.gs + pi);
        if (I4) load_q4<D, NTH, T>(p, qf.s, lh.h0, lh.nh, lane, qn);
        else if (F8) load_q8<D, NTH, T>(p, qf.s, lh.h0, lh.nh, lane, qn);
        else load_q<D, NTH>(p, qf.s, lh.h0, lh.nh, lane, qn);
      }
    }

    // INT4: each score starts from -(1032 Q_lo + 72 Q_hi) of its head, from the f16 q
    // values the MMAs use (lane (r0, t) holds column r0's b fragments for its t; sums over
    // t, then each lane takes its columns qc, qc + 1).  W: this lane's share of the
    // weights that entered P V (see i4x2_lo).
    float kofs[NTH][2], wsum[NTH][2];
    if constexpr (I4) {
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt) {
        wsum[nt][0] = wsum[nt][1] = 0.f;
        kofs[nt][0] = kofs[nt][1] = 0.f;
        if (!computes) continue;
        float ql = 0.f, qh = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const float2 a = unpack2<__half>(qb[ks][nt][0]), b = unpack2<__half>(qb[ks][nt][1]);
          ql += a.x + a.y;
          qh += b.x + b.y;  // (q / 16)
        }
        float c = 1032.f * ql + 1152.f * qh;  // 72 * 16 = 1152
        c += __shfl_xor_sync(0xffffffffu, c, 1);
        c += __shfl_xor_sync(0xffffffffu, c, 2);
        kofs[nt][0] = -__shfl_sync(0xffffffffu, c, 4 * qc);
        kofs[nt][1] = -__shfl_sync(0xffffffffu, c, 4 * (qc + 1));
      }
    }

    // This lane's softmax columns: heads 8*nt + qc and + 1 of every n-tile.
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

    const int j_first = r.x + (phase - r.x % P + P) % P;
    for (int j = j_first; j < r.y; j += P) {
      issue_one();                   // stage used + kAhead goes in flight
      const uint32_t slot = used % R;
      ++used;
      cp_async_wait<G_::kAhead>();   // this lane's copies of stage `used` have landed
      __syncwarp();                  // ... and every other lane's
      const int nt_tok = min(ST, f.ctx - j * ST);
      if (badbits & (1u << slot)) {
        seg_bad = true;
      } else {
        const uint32_t kb = ring + slot * G_::kStageBytes;
        const uint32_t vb = kb + G_::kKBytes;
        if constexpr (QK) {
          if (NEW && j == f.ns - 1) {
            // Fused step: the newest token (stage row nt_tok - 1) is quantised from the
            // step's input with the cache-write arithmetic; the codes (and INT4 scales)
            // replace the stage row and go to the cache slot at position ctx - 1.  No other
            // reader of that slot exists in the call.
            const int t = f.ctx - 1, nr = nt_tok - 1;
            const int blk = __ldg(p.block_tables + static_cast<size_t>(f.s) * p.max_blocks_per_seq +
                                  (t >> p.log2_block));
            const size_t grow = (static_cast<size_t>(blk) * p.num_kv_heads + ph.kvh) * p.block_size +
                                (t & (p.block_size - 1));
            const uint8_t* nrow = sm.newrow[warp][slot];
            uint8_t* stage = sm.ring[warp][slot];
            if constexpr (F8) {
              constexpr int CK = D / 16;  // 16-code chunks of a row
              if (lane < 2 * CK) {
                const int isv = lane >= CK ? 1 : 0, c = lane % CK;
                const uint4* src = reinterpret_cast<const uint4*>(nrow + isv * 2 * D + 32 * c);
                const uint4 codes = quantize16_e4m3<T>(src[0], src[1], isv ? p.v_quant : p.k_quant);
                *reinterpret_cast<uint4*>(stage + isv * G_::kKBytes + swz8<D>(nr, c)) = codes;
                reinterpret_cast<uint4*>(const_cast<uint8_t*>(isv ? p.v_cache : p.k_cache))[grow * CK + c] = codes;
              }
            } else {
#pragma unroll
              for (int isv = 0; isv < 2; ++isv) {
                float x[D / 32];
                int4_row_values<T, D>(reinterpret_cast<const T*>(nrow + isv * 2 * D), lane, x);
                float sc;
                const uint32_t packed = int4_quantize_lane<D>(x, sc);
                uint8_t* gcodes = const_cast<uint8_t*>(isv ? p.v_cache : p.k_cache) + grow * (D / 2);
                if constexpr (D == 128) {
                  *reinterpret_cast<uint16_t*>(stage + isv * G_::kKBytes + swz4<D>(nr, lane >> 3) +
                                               2 * (lane & 7)) = static_cast<uint16_t>(packed);
                  reinterpret_cast<uint16_t*>(gcodes)[lane] = static_cast<uint16_t>(packed);
                } else {
                  stage[isv * G_::kKBytes + swz4<D>(nr, lane >> 4) + (lane & 15)] = static_cast<uint8_t>(packed);
                  gcodes[lane] = static_cast<uint8_t>(packed);
                }
                if (lane == 0) {
                  *reinterpret_cast<float*>(stage + 2 * G_::kKBytes + isv * G_::kScaleBytes + 4 * nr) = sc;
                  const_cast<float*>(isv ? p.v_scales : p.k_scales)[grow] = sc;
                }
              }
            }
            __syncwarp();  // the stage row is rewritten before any lane reads it
          }
        }
        // ---- S^T = K Q^T: rows = the stage's tokens (U m-tiles of 16), columns = heads ----
        float sacc[U][NTH][4], sodd[U][NTH][4];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              sacc[u][nt][e] = I4 ? kofs[nt][e & 1] : 0.f;
              sodd[u][nt][e] = 0.f;
            }
        // INT4: the K and V scales of this lane's rows 16u + r0 and 16u + r0 + 8
        float ksc[U][2], vsc[U][2];
        if constexpr (I4) {
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const uint32_t sa = kb + 2 * G_::kKBytes + 4 * (16 * u + r0 + 8 * hr);
              ksc[u][hr] = lds_f32(sa);
              vsc[u][hr] = lds_f32(sa + G_::kScaleBytes);
            }
        }
        if constexpr (I4) {
          // K rows 16u + r0 and + 8, bytes [(D/8) t, (D/8)(t+1)): word j holds the eight d
          // of k-steps 2j and 2j + 1 (the order load_q4 gives q)
          constexpr int KW = D / 32;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            uint32_t kw[2][KW];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int row = 16 * u + r0 + 8 * hr;
              if constexpr (KW == 4) {
                const uint32_t addr = kb + swz4<D>(row, lane & 3);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(kw[hr][0]), "=r"(kw[hr][1]), "=r"(kw[hr][2]), "=r"(kw[hr][3])
                             : "r"(addr));
              } else {
                const uint32_t addr = kb + swz4<D>(row, (lane & 3) >> 1) + 8 * (lane & 1);
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                             : "=r"(kw[hr][0]), "=r"(kw[hr][1])
                             : "r"(addr));
              }
            }
#pragma unroll
            for (int jw = 0; jw < KW; ++jw)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const uint32_t w0 = e ? kw[0][jw] >> 8 : kw[0][jw];
                const uint32_t w1 = e ? kw[1][jw] >> 8 : kw[1][jw];
                uint32_t a[4];
                a[0] = i4x2_lo(w0);
                a[1] = i4x2_lo(w1);
                a[2] = i4x2_hi(w0);
                a[3] = i4x2_hi(w1);
                const int ks = 2 * jw + e;
#pragma unroll
                for (int nt = 0; nt < NTH; ++nt) {
                  if (ks & 1)
                    mma16816<TM>(sodd[u][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
                  else
                    mma16816<TM>(sacc[u][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
                }
              }
          }
        } else if constexpr (F8) {
          // K rows 16u + r0 and + 8, bytes [(D/4) t, (D/4)(t+1)): word ks of a row holds the
          // four d of k-step ks (the order load_q8 gives q)
#pragma unroll
          for (int u = 0; u < U; ++u) {
            uint32_t kw[2][KS];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
              for (int i = 0; i < KS / 4; ++i) {
                const uint32_t addr = kb + swz8<D>(16 * u + r0 + 8 * hr, (KS / 4) * (lane & 3) + i);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(kw[hr][4 * i]), "=r"(kw[hr][4 * i + 1]), "=r"(kw[hr][4 * i + 2]),
                               "=r"(kw[hr][4 * i + 3])
                             : "r"(addr));
              }
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              uint32_t a[4];
              a[0] = e4m3x2_f16x2(kw[0][ks]);
              a[1] = e4m3x2_f16x2(kw[1][ks]);
              a[2] = e4m3x2_f16x2_hi(kw[0][ks]);
              a[3] = e4m3x2_f16x2_hi(kw[1][ks]);
#pragma unroll
              for (int nt = 0; nt < NTH; ++nt) {
                if (ks & 1)
                  mma16816<TM>(sodd[u][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
                else
                  mma16816<TM>(sacc[u][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
              }
            }
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];  // rows tok 0-7 / 8-15, d chunks 2ks / 2ks+1
            ldsm_x4(kb + swz(lrow + ((lmat & 1) << 3), 2 * ks + (lmat >> 1)), a);
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
              if (ks & 1)
                mma16816<TM>(sodd[0][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
              else
                mma16816<TM>(sacc[0][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
            }
          }
        }
        // ---- online softmax per head (column) over the stage's tokens (rows) ----
        // m-tile u: c0,c1 = token 16u + r0, heads qc, qc+1; c2,c3 = token 16u + r0 + 8
        uint32_t pb[U][NTH][2];
        float alpha[NTH][2];
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          float x[U][4];
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float v = (sacc[u][nt][e] + sodd[u][nt][e]) *
                              (I4 ? ksc[u][e >> 1] * p.scale_log2 : p.scale_log2);
              x[u][e] = 16 * u + r0 + (e < 2 ? 0 : 8) < nt_tok ? v : -INFINITY;
            }
          float pr[U][4];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float mx = fmaxf(x[0][cc], x[0][cc + 2]);
#pragma unroll
            for (int u = 1; u < U; ++u) mx = fmaxf(mx, fmaxf(x[u][cc], x[u][cc + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[nt][cc], mx);
            alpha[nt][cc] = fast_exp2(m_run[nt][cc] - m_new);  // 0 on the first stage
            float sum = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              pr[u][cc] = fast_exp2(x[u][cc] - m_new);
              pr[u][cc + 2] = fast_exp2(x[u][cc + 2] - m_new);
              sum = u == 0 ? pr[u][cc] + pr[u][cc + 2] : sum + (pr[u][cc] + pr[u][cc + 2]);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l_run[nt][cc] = l_run[nt][cc] * alpha[nt][cc] + sum;
            m_run[nt][cc] = m_new;
          }
          // P^T as B fragments: transpose the (token x head) 8x8 blocks in registers
          float wst0 = 0.f, wst1 = 0.f;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            // (INT4: each token's weight times its V scale; the sums l keep the weights,
            // W the rounded products that enter P V)
            const float v0 = I4 ? vsc[u][0] : 1.f, v1 = I4 ? vsc[u][1] : 1.f;
            const uint32_t w01 = pack2<TM>(pr[u][0] * v0, pr[u][1] * v0);  // tokens 16u + 0-7
            const uint32_t w23 = pack2<TM>(pr[u][2] * v1, pr[u][3] * v1);  // tokens 16u + 8-15
            if constexpr (I4) {
              const float2 f01 = unpack2<__half>(w01), f23 = unpack2<__half>(w23);
              wst0 += f01.x + f23.x;
              wst1 += f01.y + f23.y;
            }
            pb[u][nt][0] = movmatrix_t(w01);
            pb[u][nt][1] = movmatrix_t(w23);
          }
          if constexpr (I4) {
            wsum[nt][0] = fmaf(wsum[nt][0], alpha[nt][0], wst0);
            wsum[nt][1] = fmaf(wsum[nt][1], alpha[nt][1], wst1);
          }
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
        // ---- O^T += V^T P^T: rows = d (16 per m-tile), k = tokens, columns = heads ----
        // (V rows past the context were zero-filled by the copy, so 0 * garbage cannot occur)
        if constexpr (I4) {
          // k-step u: V rows (tokens) 16u + {2t, 2t+1, 2t+8, 2t+9}, bytes [(D/16) r0,
          // (D/16)(r0+1)) = d [(D/8) r0, (D/8)(r0+1)).  Byte permutes interleave the rows of
          // tokens 2t and 2t + 1 (and 2t + 8, 2t + 9) so that each nibble pair of an A
          // register is one d of the two tokens; word i's d 8i + 2m and 8i + 2m + 1 are
          // m-tile 4i + m's rows r0 and r0 + 8 (see drow).
          constexpr int VW = D / 64;  // 32-bit words of this lane's bytes of one V row
          const int tq = lane & 3;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            uint32_t vw[4][VW];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int row = 16 * u + 2 * tq + (k & 1) + 8 * (k >> 1);
              if constexpr (VW == 2) {
                const uint32_t addr = vb + swz4<D>(row, r0 >> 1) + 8 * (r0 & 1);
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                             : "=r"(vw[k][0]), "=r"(vw[k][1])
                             : "r"(addr));
              } else {
                const uint32_t addr = vb + swz4<D>(row, r0 >> 2) + 4 * (r0 & 3);
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(vw[k][0]) : "r"(addr));
              }
            }
#pragma unroll
            for (int i = 0; i < VW; ++i) {
              const uint32_t z[4] = {__byte_perm(vw[0][i], vw[1][i], 0x5410u),    // tokens 2t, 2t+1
                                     __byte_perm(vw[0][i], vw[1][i], 0x7632u),
                                     __byte_perm(vw[2][i], vw[3][i], 0x5410u),    // 2t+8, 2t+9
                                     __byte_perm(vw[2][i], vw[3][i], 0x7632u)};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint32_t x = (m & 1) ? z[m >> 1] >> 8 : z[m >> 1];
                const uint32_t y = (m & 1) ? z[2 + (m >> 1)] >> 8 : z[2 + (m >> 1)];
                uint32_t a[4];
                a[0] = i4x2_lo(x);
                a[1] = i4x2_hi(x);
                a[2] = i4x2_lo(y);
                a[3] = i4x2_hi(y);
#pragma unroll
                for (int nt = 0; nt < NTH; ++nt)
                  mma16816<TM>(o[4 * i + m][nt], a, pb[u][nt][0], pb[u][nt][1]);
              }
            }
          }
        } else if constexpr (F8) {
          // k-step u: V rows (tokens) 16u + {2t, 2t+1, 2t+8, 2t+9}, bytes [(D/8) r0,
          // (D/8)(r0+1)): m-tile mt takes bytes 2 mt and 2 mt + 1 (its rows r0 and r0 + 8,
          // see drow); a byte permute pairs the two tokens of each A register before widening
          constexpr int VW = D / 32;  // 32-bit words of this lane's bytes of one V row
          const int tq = lane & 3;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            uint32_t vw[4][VW];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int row = 16 * u + 2 * tq + (k & 1) + 8 * (k >> 1);
              if constexpr (VW == 4) {
                const uint32_t addr = vb + swz8<D>(row, r0);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(vw[k][0]), "=r"(vw[k][1]), "=r"(vw[k][2]), "=r"(vw[k][3])
                             : "r"(addr));
              } else {
                const uint32_t addr = vb + swz8<D>(row, r0 >> 1) + 8 * (r0 & 1);
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                             : "=r"(vw[k][0]), "=r"(vw[k][1])
                             : "r"(addr));
              }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
              const uint32_t lo = __byte_perm(vw[0][mt >> 1], vw[1][mt >> 1], sel);  // 2t, 2t+1
              const uint32_t hi = __byte_perm(vw[2][mt >> 1], vw[3][mt >> 1], sel);  // 2t+8, 2t+9
              uint32_t a[4];
              a[0] = e4m3x2_f16x2(lo);
              a[1] = e4m3x2_f16x2_hi(lo);
              a[2] = e4m3x2_f16x2(hi);
              a[3] = e4m3x2_f16x2_hi(hi);
#pragma unroll
              for (int nt = 0; nt < NTH; ++nt) mma16816<TM>(o[mt][nt], a, pb[u][nt][0], pb[u][nt][1]);
            }
          }
        } else {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t a[4];  // V^T: d chunks 2mt / 2mt+1, tokens 0-7 / 8-15
            ldsm_x4_t(vb + swz(lrow + ((lmat >> 1) << 3), 2 * mt + (lmat & 1)), a);
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) mma16816<TM>(o[mt][nt], a, pb[0][nt][0], pb[0][nt][1]);
          }
        }
        if (!QK && NEW && j == f.ns - 1) {
          // fused cache write: the newest token's K and V rows, from the slot, to position
          // ctx - 1 of the sequence (lanes take the 16-byte chunks of K, then of V)
          constexpr int CH = G_::kRowChunks;
          const int t = f.ctx - 1;
          const int blk = __ldg(p.block_tables + static_cast<size_t>(f.s) * p.max_blocks_per_seq +
                                (t >> p.log2_block));
          if (lane < 2 * CH && blk >= 0 && blk < p.num_blocks) {
            const int c16 = lane % CH;
            const uint32_t from = (lane < CH ? kb : vb) + swz(nt_tok - 1, c16);
            const size_t to_bytes = ((static_cast<size_t>(blk) * p.num_kv_heads + ph.kvh) * p.block_size +
                                     (t & (p.block_size - 1))) * G_::kRowBytes + c16 * 16;
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(from));
            reinterpret_cast<uint4*>(const_cast<uint8_t*>(lane < CH ? p.k_cache : p.v_cache))[to_bytes / 16] = v;
          }
        }
      }
      __syncwarp();  // every lane is done with the slot before a later stage refills it
    }

    if constexpr (I4) {
      // take the V offsets out of O (see i4x2_lo), W summed over the lanes of a column
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float w = wsum[nt][cc];
          w += __shfl_xor_sync(0xffffffffu, w, 4);
          w += __shfl_xor_sync(0xffffffffu, w, 8);
          w += __shfl_xor_sync(0xffffffffu, w, 16);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            o[mt][nt][cc] = fmaf(-1032.f, w, o[mt][nt][cc]);                 // low-nibble d
            o[mt][nt][cc + 2] = fmaf(o[mt][nt][cc + 2], 0.0625f, -72.f * w);  // high-nibble d
          }
        }
    }
    const bool whole = r.x == 0 && r.y == f.ns;
    const int slot_out = cta_first ? 0 : 1;
    const size_t piece = (static_cast<size_t>(c) * 2 + slot_out) * p.gs + pi;
    float* pacc = p.part_acc + piece * p.heads_per_pair * D;
    float* pml = p.part_ml + piece * p.heads_per_pair * 2;

    if (P == 1) {
      // ---------- pair end, one warp per pair: everything stays in registers ----------
      // Lane (r0, qc) holds O^T rows d = 16*mt + r0 (+8) for heads h = 8*nt + qc (+1), and
      // the running max/sum of those heads.
      const bool any_bad = __any_sync(0xffffffffu, seg_bad);
      if (!whole) {
        // A piece of a cut pair: store (O, m, l) in [head][d] order; it is counted in
        // below or after the share is streamed, and merged after the share.
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int h = nt * 8 + qc + cc;
            if (h < ph.nh) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                pacc[h * D + drow<D, QK>(mt, r0)] = o[mt][nt][cc];
                pacc[h * D + drow<D, QK>(mt, r0 + 8)] = o[mt][nt][cc + 2];
              }
              if (r0 == 0) {  // an empty piece (m = -inf) gets l = 0: weight 0 in the merge
                pml[h * 2 + 0] = m_run[nt][cc];
                pml[h * 2 + 1] = any_bad ? -1.f : (m_run[nt][cc] == -INFINITY ? 0.f : l_run[nt][cc]);
              }
            }
          }
        CutPiece& cpr = ncut == 0 ? cut_a : cut_b;
        cpr = cut_piece(f, pi, ph, W, G, p);
        if (f.pre + f.fw < w1) {
          // More of the share follows (this is its first family, or a middle one): count
          // the piece in now, so that the share's end has one arrival and merge fewer.
          // The pair's other pieces lie in earlier shares, so this arrival rarely
          // completes it; if it does, the merge waits for the share's end.
          __syncwarp();
          const int n = cpr.c_last - cpr.c_first + 1;
          int got = 0;
          if (lane == 0) {
            __threadfence();
            got = arrive(p.counters + static_cast<size_t>(cpr.c_first) * p.gs + pi, p.epoch, n);
            if (got == n) __threadfence();
          }
          got = __shfl_sync(0xffffffffu, got, 0);
          early |= 1 << ncut;
          if (got == n) early_last |= 1 << ncut;
          else if (got < 0) early_lost |= 1 << ncut;
        }
        ++ncut;
        if (lane == 0 && any_bad) atomicOr(p.err, kErrBadBlock);
        continue;
      }
      const bool bad = any_bad;
      // out = O / l, rounded; transposed in registers (movmatrix) so that each lane stores
      // two adjacent d of one head: lane (r0, qc) writes out[h = 8*nt + r0][16*mt + qc (+8)].
      if (QK) {
        // rows r0 and r0 + 8 of an m-tile are the adjacent d = drow(mt, r0), + 1: each lane
        // stores its two heads' pairs directly
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const float inv = bad ? 0.f : p.out_scale / l_run[nt][cc];
            const int h = nt * 8 + qc + cc;
            if (h < ph.nh) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                *reinterpret_cast<uint32_t*>(out_rows + h * D + drow<D, QK>(mt, r0)) =
                    pack2<T>(o[mt][nt][cc] * inv, o[mt][nt][cc + 2] * inv);
            }
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
          const float i0 = bad ? 0.f : 1.f / l_run[nt][0];
          const float i1 = bad ? 0.f : 1.f / l_run[nt][1];
          const int h = nt * 8 + r0;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t lo = movmatrix_t(pack2<T>(o[mt][nt][0] * i0, o[mt][nt][1] * i1));
            const uint32_t hi = movmatrix_t(pack2<T>(o[mt][nt][2] * i0, o[mt][nt][3] * i1));
            if (h < ph.nh) {
              *reinterpret_cast<uint32_t*>(out_rows + h * D + 16 * mt + qc) = lo;
              *reinterpret_cast<uint32_t*>(out_rows + h * D + 16 * mt + 8 + qc) = hi;
            }
          }
        }
      }
      if (lane == 0 && any_bad) atomicOr(p.err, kErrBadBlock);
      continue;
    }

    // ---------------- pair end, P warps per pair: merge them, write out ----------------
    gsync();  // the previous pair end's reads of xo/xm/xl are done
    if (r0 == 0) {  // lanes 0..3 hold the running max/sum of heads 8*nt + qc, + 1
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          sm.xm[warp][nt * 8 + qc + cc] = m_run[nt][cc];
          sm.xl[warp][nt * 8 + qc + cc] = l_run[nt][cc];
        }
    }
    const bool any_bad = gor(seg_bad);  // (also orders the xm/xl writes before the reads)
    const int wbase = pi * P;  // first warp of the pair
    // Exchange O four heads at a time: round r covers heads 4r..4r+3.
    const int rounds = (ph.nh + 3) / 4;
    for (int round = 0; round < rounds; ++round) {
      if (round > 0) gsync();  // previous round's reads done
      const int rbase = round * 4;
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int h = nt * 8 + qc + cc;
          if (h >= rbase && h < rbase + 4) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              sm.xo[warp][h - rbase][drow<D, QK>(mt, r0)] = o[mt][nt][cc];
              sm.xo[warp][h - rbase][drow<D, QK>(mt, r0 + 8)] = o[mt][nt][cc + 2];
            }
          }
        }
      }
      gsync();
      const int rows = min(4, ph.nh - rbase);
      for (int idx = gt; idx < rows * (D / 4); idx += gthreads) {
        const int hr = idx / (D / 4);
        const int h = rbase + hr;
        const int d4 = (idx - hr * (D / 4)) * 4;
        float M = -INFINITY;
        for (int w = wbase; w < wbase + P; ++w) M = fmaxf(M, sm.xm[w][h]);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = wbase; w < wbase + P; ++w) {
          const float wt = exp2f(sm.xm[w][h] - M);  // 0 for a warp without units here
          L += sm.xl[w][h] * wt;
          const float4 x4 = *reinterpret_cast<const float4*>(&sm.xo[w][hr][d4]);
          acc.x += x4.x * wt;
          acc.y += x4.y * wt;
          acc.z += x4.z * wt;
          acc.w += x4.w * wt;
        }
        if (whole) {
          uint2 packed = make_uint2(0u, 0u);  // zeros for a pair with a bad block
          if (!any_bad) {
            const float inv = QK ? p.out_scale / L : 1.f / L;
            packed.x = pack2<T>(acc.x * inv, acc.y * inv);
            packed.y = pack2<T>(acc.z * inv, acc.w * inv);
          }
          *reinterpret_cast<uint2*>(out_rows + h * D + d4) = packed;
        } else {
          // An empty piece (no units here) has M = -inf, and the weights above are NaN:
          // store acc = 0, l = 0 so that its weight in the merge, 2^(-inf - M'), is 0.
          const bool empty = M == -INFINITY;
          *reinterpret_cast<float4*>(pacc + h * D + d4) = empty ? make_float4(0.f, 0.f, 0.f, 0.f) : acc;
          if (d4 == 0) {
            pml[h * 2 + 0] = M;
            pml[h * 2 + 1] = any_bad ? -1.f : (empty ? 0.f : L);
          }
        }
      }
    }
    if (!whole) {
      (ncut == 0 ? cut_a : cut_b) = cut_piece(f, pi, ph, W, G, p);
      ++ncut;
    }
    if (gt == 0 && any_bad) atomicOr(p.err, kErrBadBlock);
  }
  cp_async_wait<0>();  // (only empty groups can be left; leave none behind)
  PA_DECODE_STAMP(1);

  // ---- count this share's pieces in; the last arrival at a pair merges its pieces ----
  // (ncut is the same in every warp of a pair.)  Lanes 0 and 1 of the pair's first warp
  // count in its two pieces side by side, each after a fence ordering the piece's stores
  // before its arrival; an arrival that completes a pair fences again before the merge's
  // loads.  An arrival that gives up (pa_arrive.h) flags the call and zeros the pair.
  if (ncut > 0) {
    gsync();  // every thread of the pair has stored its parts of the pieces
    int bits = 0, lost = 0;
    if (gt < ncut && !(early & (1 << gt))) {
      const CutPiece& cp = gt == 0 ? cut_a : cut_b;
      __threadfence();
      const int n = cp.c_last - cp.c_first + 1;
      const int got = arrive(p.counters + static_cast<size_t>(cp.c_first) * p.gs + pi, p.epoch, n);
      if (got == n) {
        __threadfence();
        bits = 1 << gt;
      } else if (got < 0) {
        atomicOr(p.err, kErrTimeout);
        lost = 1 << gt;
      }
    }
    __syncwarp();
    bits = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(bits)));
    lost = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(lost)));
    bits |= early_last;
    lost |= early_lost;
    if (early_lost && gt == 0) atomicOr(p.err, kErrTimeout);
    if (P > 1) {
      if (gt == 0) sm.last[pi] = bits | (lost << 2);
      gsync();
      bits = sm.last[pi] & 3;
      lost = sm.last[pi] >> 2;
    }
    for (int k = 0; k < ncut; ++k)
      if (lost & (1 << k)) zero_pair<D, T>(p, k == 0 ? cut_a : cut_b, gt, gthreads);
    if (P == 1 && bits) {
      const int nj = (bits & 1) + ((bits >> 1) & 1);
      const CutPiece& j0 = (bits & 1) ? cut_a : cut_b;
      uint32_t phase = 0;
      if (merge_staged<D, T, QK>(p, pi, j0, cut_b, nj, ring, sm.ring[warp][0], R * G_::kStageBytes,
                                 smem_addr(&sm.merge_bar[warp]), phase, lane))
        bits = 0;
    }
    for (int k = 0; k < ncut; ++k) {
      if (!(bits & (1 << k))) continue;
      const CutPiece& cp = k == 0 ? cut_a : cut_b;
      T* out_rows =
          reinterpret_cast<T*>(p.out) + (static_cast<size_t>(cp.s) * p.num_q_heads + cp.h0) * D;
      merge_pieces<D, T, QK>(p, pi, cp.c_first, cp.first_slot, cp.c_last, cp.nh, out_rows, gt,
                         gthreads);
    }
  }
  PA_DECODE_STAMP(2);
}

template <int D, int NTH, typename T, int KV, bool NEW>
int PA_DECODE_LAUNCH(const Params& prm, int grid, cudaStream_t stream PA_DECODE_TIMELINE_ARG) {
  const size_t smem = sizeof(Smem<D, KV>) + 1024;  // + alignment slack for the ring
  auto* kern = PA_DECODE_KERNEL<D, NTH, T, KV, NEW>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), smem)) return -3;
  // a programmatic dependent of the previous kernel in the stream (see pdl_wait_primary)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm PA_DECODE_TIMELINE_PASS) != cudaSuccess) return -3;
  return 0;
}

#ifndef PA_DECODE_TIMELINE
// Every kernel of one K/V format, for the plain decode (NEW false) or the fused step (NEW
// true): head_dim 128 or 64, one n-tile of heads or two, bf16 or fp16.  Each (format, NEW)
// is instantiated in a translation unit of its own, so that the six compile in parallel:
// pa_decode.cu, pa_decode_fp8.cu, pa_decode_int4.cu (plain decode) and pa_decode_append.cu,
// pa_decode_append_fp8.cu, pa_decode_append_int4.cu (fused step).
template <int KV, bool NEW>
int launch_format(const Params& p, int grid, int head_dim, bool bf16, cudaStream_t stream) {
#define PA_DECODE_CASE(DD, NN)                                                   \
  if (head_dim == DD && (p.heads_per_pair > 8) == (NN == 2))                     \
    return bf16 ? launch<DD, NN, __nv_bfloat16, KV, NEW>(p, grid, stream)        \
                : launch<DD, NN, __half, KV, NEW>(p, grid, stream);
  PA_DECODE_CASE(128, 1)
  PA_DECODE_CASE(128, 2)
  PA_DECODE_CASE(64, 1)
  PA_DECODE_CASE(64, 2)
#undef PA_DECODE_CASE
  return -1;
}
extern template int launch_format<kKv16, false>(const Params&, int, int, bool, cudaStream_t);
extern template int launch_format<kKv16, true>(const Params&, int, int, bool, cudaStream_t);
extern template int launch_format<kKvFp8, false>(const Params&, int, int, bool, cudaStream_t);
extern template int launch_format<kKvFp8, true>(const Params&, int, int, bool, cudaStream_t);
extern template int launch_format<kKvInt4, false>(const Params&, int, int, bool, cudaStream_t);
extern template int launch_format<kKvInt4, true>(const Params&, int, int, bool, cudaStream_t);
#endif

}  // namespace decode

// The stamped 16-bit kernel (pa_decode_timed.cu): head_dim 128, up to 8 heads a pair.
int decode_launch_timed(const decode::Params& p, int grid, bool bf16, cudaStream_t stream,
                        unsigned long long* timeline);

}  // namespace pa

#endif  // PA_DECODE_KERNEL_CUH_
