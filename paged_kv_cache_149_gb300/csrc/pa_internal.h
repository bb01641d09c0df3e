// Internal interface between the C ABI layer (pa_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace pa {

struct DecodeArgs {
  const void* q;
  const void* k_cache;  // written only by the fused cache write (key_new != null)
  const void* v_cache;
  const void* key_new;  // pa_decode_append: newest token per sequence [n][Hkv][d], else null
  const void* value_new;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  void* workspace;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, num_blocks;
  float scale;
  bool bf16;       // q / out type (and the cache type unless kv_fp8)
  bool kv_fp8;     // caches hold FP8 E4M3 codes with scales k_scale, v_scale
  float k_scale = 1.f, v_scale = 1.f;
  bool kv_int4 = false;  // caches hold INT4 codes [NB][Hkv][B][d/2] with a scale per row
  const void* k_scales = nullptr;  // INT4: float32 [NB][Hkv][B]
  const void* v_scales = nullptr;
  unsigned* err;  // device address of the per-device error word
};

// Workspace bytes for `grid` persistent CTAs and this head layout.
size_t decode_workspace_bytes(int grid, int num_q_heads, int num_kv_heads, int head_dim);
// Heads a decode work pair covers (query heads per kv head, at most 16).
int decode_heads_per_pair(int num_q_heads, int num_kv_heads);
// Launch the decode kernel; 0 or a negative PA_ERR_* code.
int decode_launch(const DecodeArgs& a, int grid, cudaStream_t stream);
// Diagnostics: every 16-bit decode launch of this host thread stamps its warps' phases
// into `buffer` (device, [grid][8][3] unsigned long long) until called with NULL.
void decode_set_timeline(void* buffer, size_t bytes);

struct PrefillArgs {
  const void* q;  // [num_q_rows, Hq, d]
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;  // [num_seqs + 1]
  void* out;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
      num_blocks, max_query_len;
  float scale;
  bool bf16;
  unsigned* err;
};

// Launch the paged prefill kernel; 0 or a negative PA_ERR_* code.
int prefill_launch(const PrefillArgs& a, cudaStream_t stream);

int reshape_and_cache_launch(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, unsigned* err,
                             cudaStream_t stream);

// row_bytes: bytes of one cached row (head_dim x element size)
int copy_blocks_launch(void* k_cache, void* v_cache, const int32_t* block_mapping, int num_pairs,
                       int num_blocks, int num_kv_heads, int row_bytes, int block_size,
                       unsigned* err, cudaStream_t stream);
int reshape_and_cache_fp8_launch(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_blocks, int num_kv_heads, int head_dim, int block_size,
                                 float k_scale, float v_scale, bool bf16, unsigned* err,
                                 cudaStream_t stream);
// INT4 cache write of num_tokens rows' tokens through slot_mapping.
int cache_int4_launch(const void* key, const void* value, void* k_codes, void* v_codes,
                      float* k_scales, float* v_scales, const int64_t* slot_mapping,
                      int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                      int block_size, bool bf16, unsigned* err, cudaStream_t stream);
int swap_blocks_launch(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                       const int32_t* block_mapping, int num_pairs, int src_num_blocks,
                       int dst_num_blocks, int num_kv_heads, int row_bytes, int block_size,
                       unsigned* err, cudaStream_t stream);

// A cache [num_blocks][Hkv][B][d] of elem_bytes-byte values (2: fp16/bf16, 1: FP8 codes)
// as a 4-D tensor (d, row, kv head, block) read in boxes of (128 bytes of d, B, 1, 1): the
// 128-byte swizzle when a row is 128 bytes or more, none for 64-byte rows.  False when the
// driver's encoder is missing or rejects the tensor.
bool kv_cache_map(CUtensorMap* map, const void* base, int elem_bytes, int num_blocks, int hkv,
                  int bs, int d);

// Raise a kernel's dynamic shared-memory limit once per device; false on failure.
bool ensure_smem_attr(const void* func, size_t bytes);

}  // namespace pa
