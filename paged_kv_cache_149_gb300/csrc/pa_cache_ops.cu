// Cache writes and block copies: exact 16-byte moves of 16-bit K/V rows.
//
// reshape_and_cache: a new token's K/V row goes into its slot of the sequence's last
// block (chenyuan1125 "vllm-pagedattention", section 页表真正解开的…; horeb.top, section
// 分配策略): k_cache[slot / B, h, slot % B, :] = key[i, h, :].
// copy_blocks: the copy behind copy-on-write of a still-shared last block (chenyuan1125,
// section 一块内存，如何安全地属于多条序列; horeb.top, section 内存共享：写时复制).
// swap_blocks: a preempted request's blocks move whole to CPU memory and back (aiqz.cc
// "vLLM PagedAttention engine", section 连续批处理：随到随走的新秩序).  The same block
// copy serves both: copy_blocks within one pool, swap_blocks between a device pool and a
// page-locked host pool that the GPU reads and writes directly over NVLink-C2C.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// One CTA per token: the token's Hkv rows of K and of V, 16 bytes per thread step.
__global__ void __launch_bounds__(128) reshape_and_cache_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, long long num_slots,
    int num_kv_heads, int vec_per_row, int block_size, unsigned* err) {
  // a programmatic dependent of the previous kernel (say the last decode step, which may
  // still read the cache): wait for it before touching anything, then let the next start
  pdl_wait_primary();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const long long slot = slot_mapping[i];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const long long blk = slot / block_size;
  const int row = static_cast<int>(slot % block_size);
  const int n = num_kv_heads * vec_per_row;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int h = j / vec_per_row;
    const int c = j - h * vec_per_row;
    const size_t src = (static_cast<size_t>(i) * num_kv_heads + h) * vec_per_row + c;
    const size_t dst =
        ((static_cast<size_t>(blk) * num_kv_heads + h) * block_size + row) * vec_per_row + c;
    k_cache[dst] = key[src];
    v_cache[dst] = value[src];
  }
}

// FP8 cache write: each 16-bit input x becomes the E4M3 code of x / scale, the division in
// IEEE float32 and the rounding to nearest-even with magnitudes above 448 clamped (the
// hardware's satfinite conversion).  A thread makes one 16-byte chunk of codes (16
// values, 32 input bytes).  One CTA per token, as above.
template <typename T>
__global__ void __launch_bounds__(128) reshape_and_cache_fp8_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, long long num_slots,
    int num_kv_heads, int chunks_per_row, int block_size, float k_scale, float v_scale,
    unsigned* err) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const long long slot = slot_mapping[i];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const long long blk = slot / block_size;
  const int row = static_cast<int>(slot % block_size);
  const int n = num_kv_heads * chunks_per_row;
  for (int j = threadIdx.x; j < 2 * n; j += blockDim.x) {
    const bool is_v = j >= n;
    const int jj = is_v ? j - n : j;
    const int h = jj / chunks_per_row;
    const int c = jj - h * chunks_per_row;
    const float scale = is_v ? v_scale : k_scale;
    // 16 inputs = two 16-byte vectors of the 16-bit row
    const uint4* src = (is_v ? value : key) +
                       ((static_cast<size_t>(i) * num_kv_heads + h) * chunks_per_row + c) * 2;
    const size_t dst =
        ((static_cast<size_t>(blk) * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
    (is_v ? v_cache : k_cache)[dst] = quantize16_e4m3<T>(src[0], src[1], scale);
  }
}

// INT4 rows: one warp quantises one d-value row (a token's K or V for one kv head) with
// int4_quantize_lane; the codes go to the row's D / 2 bytes (element 2i in the low nibble
// of byte i) and the scale beside the block's codes.
template <typename T, int D>
__device__ __forceinline__ void quantize_row_int4(const T* __restrict__ src, uint8_t* __restrict__ codes,
                                                  float* __restrict__ scale, int lane) {
  float x[D / 32];
  int4_row_values<T, D>(src, lane, x);
  float s;
  const uint32_t packed = int4_quantize_lane<D>(x, s);
  if constexpr (D / 32 == 4) reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
  else codes[lane] = static_cast<uint8_t>(packed);
  if (lane == 0) *scale = s;
}

// grid = the rows' tokens; warps take the 2 * Hkv rows (K then V) of their token.
template <typename T, int D>
__global__ void __launch_bounds__(256) cache_int4_kernel(
    const T* __restrict__ key, const T* __restrict__ value, uint8_t* __restrict__ k_codes,
    uint8_t* __restrict__ v_codes, float* __restrict__ k_scales, float* __restrict__ v_scales,
    const int64_t* __restrict__ slot_mapping, int num_blocks, int num_kv_heads, int block_size,
    unsigned* err) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const long long slot = slot_mapping[i];
  if (slot < 0) return;
  if (slot >= static_cast<long long>(num_blocks) * block_size) {
    if (threadIdx.x == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const long long blk = slot / block_size;
  const int row = static_cast<int>(slot % block_size);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < 2 * num_kv_heads; j += blockDim.x >> 5) {
    const bool is_v = j >= num_kv_heads;
    const int h = is_v ? j - num_kv_heads : j;
    const T* src = (is_v ? value : key) + (static_cast<size_t>(i) * num_kv_heads + h) * D;
    const size_t r = (static_cast<size_t>(blk) * num_kv_heads + h) * block_size + row;
    quantize_row_int4<T, D>(src, (is_v ? v_codes : k_codes) + r * (D / 2),
                            (is_v ? v_scales : k_scales) + r, lane);
  }
}

}  // namespace

int cache_int4_launch(const void* key, const void* value, void* k_codes, void* v_codes,
                      float* k_scales, float* v_scales, const int64_t* slot_mapping,
                      int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                      int block_size, bool bf16, unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_tokens);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto* kc = static_cast<uint8_t*>(k_codes);
  auto* vc = static_cast<uint8_t*>(v_codes);
  cudaError_t e = cudaErrorInvalidValue;
#define PA_INT4_CASE(TT, DD)                                                                      \
  e = cudaLaunchKernelEx(&cfg, cache_int4_kernel<TT, DD>, static_cast<const TT*>(key),            \
                         static_cast<const TT*>(value), kc, vc, k_scales, v_scales, slot_mapping, \
                         num_blocks, num_kv_heads, block_size, err)
  if (head_dim == 128) {
    if (bf16) PA_INT4_CASE(__nv_bfloat16, 128); else PA_INT4_CASE(__half, 128);
  } else if (head_dim == 64) {
    if (bf16) PA_INT4_CASE(__nv_bfloat16, 64); else PA_INT4_CASE(__half, 64);
  }
#undef PA_INT4_CASE
  return e == cudaSuccess ? 0 : -3;
}

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per thread before its stores

// grid = (pairs, chunks of a block, 2 caches): block mapping[p][1] of the destination
// pool := block mapping[p][0] of the source pool.  Each thread has kCopyUnroll loads in
// flight (host memory across the chip-to-chip link answers slower than HBM).  The source
// and destination blocks of a pair never overlap (distinct pools, or, within one pool, a
// checked pair list).  A pair with an id outside its pool is skipped and flagged.
__global__ void __launch_bounds__(kCopyThreads) block_copy_kernel(
    const uint4* __restrict__ src_k, const uint4* __restrict__ src_v, uint4* __restrict__ dst_k,
    uint4* __restrict__ dst_v, const int32_t* __restrict__ mapping, int src_blocks,
    int dst_blocks, size_t block_vecs, unsigned* err) {
  const int pair = blockIdx.x;
  const int src = mapping[2 * pair];
  const int dst = mapping[2 * pair + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(err, kErrBadPair);
    return;
  }
  const uint4* s = (blockIdx.z == 0 ? src_k : src_v) + static_cast<size_t>(src) * block_vecs;
  uint4* d = (blockIdx.z == 0 ? dst_k : dst_v) + static_cast<size_t>(dst) * block_vecs;
  const size_t step = static_cast<size_t>(gridDim.y) * kCopyThreads;
  for (size_t j0 = static_cast<size_t>(blockIdx.y) * kCopyThreads + threadIdx.x; j0 < block_vecs;
       j0 += step * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (j0 + u * step < block_vecs) v[u] = s[j0 + u * step];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (j0 + u * step < block_vecs) d[j0 + u * step] = v[u];
  }
}

int block_copy_launch(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                      const int32_t* mapping, int num_pairs, int src_blocks, int dst_blocks,
                      int num_kv_heads, int row_bytes, int block_size, unsigned* err,
                      cudaStream_t stream) {
  if (num_pairs == 0) return 0;
  const size_t block_vecs = static_cast<size_t>(num_kv_heads) * block_size * row_bytes / 16;
  const size_t per_cta = static_cast<size_t>(kCopyThreads) * kCopyUnroll;
  int chunks = static_cast<int>((block_vecs + per_cta - 1) / per_cta);
  if (chunks > 64) chunks = 64;
  block_copy_kernel<<<dim3(num_pairs, chunks, 2), kCopyThreads, 0, stream>>>(
      static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v), static_cast<uint4*>(dst_k),
      static_cast<uint4*>(dst_v), mapping, src_blocks, dst_blocks, block_vecs, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

int reshape_and_cache_launch(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, unsigned* err,
                             cudaStream_t stream) {
  if (num_tokens == 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_tokens);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, reshape_and_cache_kernel, static_cast<const uint4*>(key),
      static_cast<const uint4*>(value), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      slot_mapping, static_cast<long long>(num_blocks) * block_size, num_kv_heads, head_dim / 8,
      block_size, err);
  return e == cudaSuccess ? 0 : -3;
}

int reshape_and_cache_fp8_launch(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_blocks, int num_kv_heads, int head_dim, int block_size,
                                 float k_scale, float v_scale, bool bf16, unsigned* err,
                                 cudaStream_t stream) {
  if (num_tokens == 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_tokens);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long slots = static_cast<long long>(num_blocks) * block_size;
  const cudaError_t e =
      bf16 ? cudaLaunchKernelEx(&cfg, reshape_and_cache_fp8_kernel<__nv_bfloat16>,
                                static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                                static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                slot_mapping, slots, num_kv_heads, head_dim / 16, block_size,
                                k_scale, v_scale, err)
           : cudaLaunchKernelEx(&cfg, reshape_and_cache_fp8_kernel<__half>,
                                static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                                static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                slot_mapping, slots, num_kv_heads, head_dim / 16, block_size,
                                k_scale, v_scale, err);
  return e == cudaSuccess ? 0 : -3;
}

int copy_blocks_launch(void* k_cache, void* v_cache, const int32_t* block_mapping, int num_pairs,
                       int num_blocks, int num_kv_heads, int row_bytes, int block_size,
                       unsigned* err, cudaStream_t stream) {
  return block_copy_launch(k_cache, v_cache, k_cache, v_cache, block_mapping, num_pairs,
                           num_blocks, num_blocks, num_kv_heads, row_bytes, block_size, err, stream);
}

int swap_blocks_launch(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                       const int32_t* block_mapping, int num_pairs, int src_num_blocks,
                       int dst_num_blocks, int num_kv_heads, int row_bytes, int block_size,
                       unsigned* err, cudaStream_t stream) {
  return block_copy_launch(src_k, src_v, dst_k, dst_v, block_mapping, num_pairs, src_num_blocks,
                           dst_num_blocks, num_kv_heads, row_bytes, block_size, err, stream);
}

}  // namespace pa
