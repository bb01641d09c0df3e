// Paged decode attention for sm_103a: host side and the 16-bit plain-decode instantiations
// of the kernel in pa_decode_kernel.cuh (whose header comment describes the design).
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <random>

#include "pa_decode_kernel.cuh"

namespace pa {
int decode_heads_per_pair(int num_q_heads, int num_kv_heads) {
  const int g = num_q_heads / num_kv_heads;
  return g < decode::kMaxHeads ? g : decode::kMaxHeads;
}

// Pairs per family: the largest power of two <= 8 dividing the pair count of a sequence.
static int pair_group_size(int num_q_heads, int num_kv_heads) {
  const int hpp = decode_heads_per_pair(num_q_heads, num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  const int pairs = num_kv_heads * ((group + hpp - 1) / hpp);
  int gs = 8;
  while (pairs % gs) gs >>= 1;
  return gs;
}

size_t decode_workspace_bytes(int grid, int num_q_heads, int num_kv_heads, int head_dim) {
  const size_t gs = pair_group_size(num_q_heads, num_kv_heads);
  const size_t hpp = decode_heads_per_pair(num_q_heads, num_kv_heads);
  const size_t ctrs = static_cast<size_t>(grid) * gs * sizeof(unsigned long long);
  const size_t acc = static_cast<size_t>(grid) * 2 * gs * hpp * head_dim * sizeof(float);
  const size_t ml = static_cast<size_t>(grid) * 2 * gs * hpp * 2 * sizeof(float);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return up(ctrs) + up(acc) + up(ml);
}

// Epoch tags of the pair counters: 40 bits, a different value on every call (random start).
static unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{
      (static_cast<unsigned long long>(std::random_device{}()) << 8) ^
      static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count())};
  return (counter.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 40) - 1);
}

// The diagnostic timeline buffer of this host thread (pa_decode_timeline), or null.
static thread_local unsigned long long* t_timeline = nullptr;
static thread_local size_t t_timeline_bytes = 0;

void decode_set_timeline(void* buffer, size_t bytes) {
  t_timeline = static_cast<unsigned long long*>(buffer);
  t_timeline_bytes = buffer ? bytes : 0;
}

int decode_launch(const DecodeArgs& a, int grid, cudaStream_t stream) {
  // a timeline buffer set: the stamped copy of the 16-bit kernel (pa_decode_timed.cu), for
  // head_dim 128 and up to 8 query heads a pair only
  if (t_timeline &&
      (a.kv_fp8 || a.kv_int4 || a.head_dim != 128 ||
       decode_heads_per_pair(a.num_q_heads, a.num_kv_heads) > 8 ||
       t_timeline_bytes < static_cast<size_t>(grid) * decode::kWarps * 3 * sizeof(unsigned long long)))
    return -1;
  decode::Params p;
  p.q = static_cast<const uint8_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.key_new = static_cast<const uint8_t*>(a.key_new);
  p.value_new = static_cast<const uint8_t*>(a.value_new);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<uint8_t*>(a.out);
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.heads_per_pair = decode_heads_per_pair(a.num_q_heads, a.num_kv_heads);
  p.head_chunks = (p.group + p.heads_per_pair - 1) / p.heads_per_pair;
  p.gs = pair_group_size(a.num_q_heads, a.num_kv_heads);
  p.log2_gs = p.gs == 8 ? 3 : (p.gs == 4 ? 2 : (p.gs == 2 ? 1 : 0));
  p.ngroups = a.num_kv_heads * p.head_chunks / p.gs;
  p.phases = decode::kWarps / p.gs;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.log2_block = a.block_size == 8 ? 3 : (a.block_size == 16 ? 4 : 5);
  p.num_blocks = a.num_blocks;
  p.max_ctx = a.max_blocks_per_seq * a.block_size;
  const bool quantised = a.kv_fp8 || a.kv_int4;
  p.log2_stage = quantised ? 5 : 4;  // 32-token stages over quantised blocks, 16 over 16-bit ones
  // per-family charge (the same charge in tokens for 32-token stages)
  p.seg_cost = decode::seg_cost_for(static_cast<long long>(a.num_seqs) * p.ngroups, grid) >>
               (p.log2_stage - 4);
  // FP8 blocks: scores are k_scale * <q, codes>, outputs v_scale * (weighted codes)
  p.scale_log2 = a.scale * (a.kv_fp8 ? a.k_scale : 1.f) * decode::kLog2e;
  p.out_scale = a.kv_fp8 ? a.v_scale : 1.f;
  p.k_quant = a.k_scale;
  p.v_quant = a.v_scale;
  // INT4 blocks: a scale per row, applied in the kernel
  p.k_scales = static_cast<const float*>(a.k_scales);
  p.v_scales = static_cast<const float*>(a.v_scales);
  p.err = a.err;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.counters = reinterpret_cast<unsigned long long*>(ws);
  ws += up(static_cast<size_t>(grid) * p.gs * sizeof(unsigned long long));
  p.epoch = next_epoch();
  p.part_acc = reinterpret_cast<float*>(ws);
  ws += up(static_cast<size_t>(grid) * 2 * p.gs * p.heads_per_pair * a.head_dim * sizeof(float));
  p.part_ml = reinterpret_cast<float*>(ws);

  // The fused step runs kernels compiled with the newest rows' write; a plain decode runs
  // copies compiled without it.  On GB300 (decode alone, one box) that took the INT4 decode
  // of 64 sequences from 37.3 to 36.1 us and of 256 MHA sequences from 229.3 to 218.0 us,
  // FP8 from 35.2 to 34.2 us (64 sequences; 199.8 against 200.9 us on 256), 16-bit blocks
  // from 51.4 to 51.2 and 381.2 to 378.5 us.
  const bool fused = a.key_new != nullptr;
  if (a.kv_fp8)
    return fused ? decode::launch_format<decode::kKvFp8, true>(p, grid, a.head_dim, a.bf16, stream)
                 : decode::launch_format<decode::kKvFp8, false>(p, grid, a.head_dim, a.bf16, stream);
  if (a.kv_int4)
    return fused ? decode::launch_format<decode::kKvInt4, true>(p, grid, a.head_dim, a.bf16, stream)
                 : decode::launch_format<decode::kKvInt4, false>(p, grid, a.head_dim, a.bf16, stream);
  if (t_timeline) return decode_launch_timed(p, grid, a.bf16, stream, t_timeline);
  return fused ? decode::launch_format<decode::kKv16, true>(p, grid, a.head_dim, a.bf16, stream)
               : decode::launch_format<decode::kKv16, false>(p, grid, a.head_dim, a.bf16, stream);
}

namespace decode {
template int launch_format<kKv16, false>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode

}  // namespace pa
