// C ABI of libpa.so: argument validation, per-device state (SM count, error word) and
// dispatch to the kernels.  Every check that can be made on the host is made here,
// before anything is launched; the kernels only guard against values that live in
// device memory (block ids, context lengths, slots).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// One error word per device; kernels OR PA_DEVERR_* bits into it.
__device__ unsigned int g_device_error;

struct DeviceInfo {
  int sm_count = 0;
  int max_smem_optin = 0;
  unsigned* err = nullptr;  // device address of g_device_error on this device
};

std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_devices;
std::set<std::pair<int, const void*>> g_smem_done;

// Per-device facts, gathered once per device with that device current.
bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo di;
    void* p = nullptr;
    if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess)
      return false;
    di.err = static_cast<unsigned*>(p);
    it = g_devices.emplace(dev, di).first;
  }
  *out = it->second;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok(int num_kv_heads, int head_dim, int block_size) {
  return num_kv_heads >= 1 && (head_dim == 64 || head_dim == 128) &&
         (block_size == 8 || block_size == 16 || block_size == 32);
}

// The address a kernel uses for p: p itself for device or managed memory, the mapped
// device address for page-locked host memory registered with CUDA, NULL otherwise.
void* device_view(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged)
    return const_cast<void*>(p);
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

}  // namespace

namespace pa {

bool ensure_smem_attr(const void* func, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_smem_done.count({dev, func})) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return false;
  g_smem_done.insert({dev, func});
  return true;
}

}  // namespace pa

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_ARG: return "invalid argument";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_POOL_EXHAUSTED: return "block pool exhausted";
    case PA_ERR_UNKNOWN_SEQ: return "unknown (or already live) sequence id";
    case PA_ERR_WRONG_TIER: return "sequence is in the other pool (swapped out / resident)";
    default: return status > 0 ? "ok (positive result)" : "unknown status";
  }
}

int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                         cudaStream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || !shape_ok(num_kv_heads, head_dim, block_size) ||
      (dtype != PA_FP16 && dtype != PA_BF16))
    return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  return pa::reshape_and_cache_launch(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                      num_blocks, num_kv_heads, head_dim, block_size, di.err,
                                      stream);
}

size_t pa_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim) {
  if (num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0 ||
      (head_dim != 64 && head_dim != 128))
    return 0;
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  return pa::decode_workspace_bytes(di.sm_count, num_q_heads, num_kv_heads, head_dim);
}

namespace {

// pa_decode and pa_decode_append: argument checks, then one launch.
int decode_call(const void* q, const void* key_new, const void* value_new, const void* k_cache,
                const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                int head_dim, int block_size, int num_blocks, float scale, void* out,
                void* workspace, size_t workspace_bytes, pa_dtype dtype, cudaStream_t stream,
                bool kv_fp8 = false, float k_scale = 1.f, float v_scale = 1.f,
                const float* k_scales = nullptr, const float* v_scales = nullptr) {
  const bool kv_int4 = k_scales != nullptr || v_scales != nullptr;
  if (kv_int4 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
    return PA_ERR_ARG;
  if (kv_fp8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) ||
                 !(v_scale > 0.f)))
    return PA_ERR_ARG;
  if (num_seqs < 0 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      !shape_ok(num_kv_heads, head_dim, block_size) || num_q_heads < num_kv_heads ||
      num_q_heads % num_kv_heads != 0 || !std::isfinite(scale) ||
      (dtype != PA_FP16 && dtype != PA_BF16) ||
      static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL ||
      static_cast<long long>(num_blocks) * num_kv_heads * block_size > 0x7fffffffLL)
    return PA_ERR_ARG;  // (the last bound keeps cache row indices within 32 bits)
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ARG;
  if ((key_new != nullptr) != (value_new != nullptr)) return PA_ERR_ARG;
  if (key_new && (!aligned16(key_new) || !aligned16(value_new))) return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  const size_t need =
      pa::decode_workspace_bytes(di.sm_count, num_q_heads, num_kv_heads, head_dim);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  pa::DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.key_new = key_new;
  a.value_new = value_new;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.workspace = workspace;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.bf16 = dtype == PA_BF16;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.kv_int4 = kv_int4;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.err = di.err;
  return pa::decode_launch(a, di.sm_count, stream);
}

}  // namespace

int pa_decode_timeline(void* buffer, size_t bytes) {
  if (buffer && (reinterpret_cast<uintptr_t>(buffer) & 7u)) return PA_ERR_ARG;
  pa::decode_set_timeline(buffer, bytes);
  return PA_OK;
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
              int head_dim, int block_size, int num_blocks, float scale, void* out,
              void* workspace, size_t workspace_bytes, pa_dtype dtype, cudaStream_t stream) {
  return decode_call(q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream);
}

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                  int head_dim, int block_size, int num_blocks, float scale, float k_scale,
                  float v_scale, void* out, void* workspace, size_t workspace_bytes,
                  pa_dtype dtype, cudaStream_t stream) {
  return decode_call(q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream, true,
                     k_scale, v_scale);
}

int pa_decode_append_fp8(const void* q, const void* key_new, const void* value_new,
                         void* k_cache, void* v_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float scale, float k_scale, float v_scale, void* out,
                         void* workspace, size_t workspace_bytes, pa_dtype dtype,
                         cudaStream_t stream) {
  if (num_seqs > 0 && (!key_new || !value_new)) return PA_ERR_ARG;
  // one launch: the warp that computes a sequence's last stage quantises its newest rows
  return decode_call(q, key_new, value_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream, true,
                     k_scale, v_scale);
}

int pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, float k_scale,
                             float v_scale, pa_dtype dtype, cudaStream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || !shape_ok(num_kv_heads, head_dim, block_size) ||
      (dtype != PA_FP16 && dtype != PA_BF16) || !std::isfinite(k_scale) ||
      !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
    return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  return pa::reshape_and_cache_fp8_launch(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                          num_blocks, num_kv_heads, head_dim, block_size, k_scale,
                                          v_scale, dtype == PA_BF16, di.err, stream);
}

// ---- INT4 K/V blocks: codes [NB][Hkv][B][d/2] (two per byte) + float32 scales [NB][Hkv][B] ----

namespace {
bool int4_arrays_ok(const void* kc, const void* vc, const void* ks, const void* vs) {
  return kc && vc && ks && vs && aligned16(kc) && aligned16(vc) && aligned16(ks) && aligned16(vs);
}
}  // namespace

int pa_reshape_and_cache_int4(const void* key, const void* value, void* k_codes, void* v_codes,
                              float* k_scales, float* v_scales, const int64_t* slot_mapping,
                              int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                              int block_size, pa_dtype dtype, cudaStream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || !shape_ok(num_kv_heads, head_dim, block_size) ||
      (dtype != PA_FP16 && dtype != PA_BF16))
    return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value) ||
      !int4_arrays_ok(k_codes, v_codes, k_scales, v_scales))
    return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  return pa::cache_int4_launch(key, value, k_codes, v_codes, k_scales, v_scales, slot_mapping,
                               num_tokens, num_blocks, num_kv_heads, head_dim, block_size,
                               dtype == PA_BF16, di.err, stream);
}

int pa_decode_int4(const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                   const float* v_scales, const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int num_blocks, float scale, void* out,
                   void* workspace, size_t workspace_bytes, pa_dtype dtype, cudaStream_t stream) {
  if (num_seqs > 0 && (!k_scales || !v_scales)) return PA_ERR_ARG;
  return decode_call(q, nullptr, nullptr, k_codes, v_codes, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream, false, 1.f,
                     1.f, k_scales, v_scales);
}

int pa_decode_append_int4(const void* q, const void* key_new, const void* value_new,
                          void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          float scale, void* out, void* workspace, size_t workspace_bytes,
                          pa_dtype dtype, cudaStream_t stream) {
  if (num_seqs > 0 && (!key_new || !value_new || !k_scales || !v_scales)) return PA_ERR_ARG;
  // one launch: the warp that computes a sequence's last stage quantises its newest rows
  return decode_call(q, key_new, value_new, k_codes, v_codes, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream, false, 1.f,
                     1.f, k_scales, v_scales);
}

int pa_copy_blocks_int4(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                        const int32_t* block_mapping, int num_pairs, int num_blocks,
                        int num_kv_heads, int head_dim, int block_size, cudaStream_t stream) {
  if (num_pairs < 0 || num_blocks < 1 || !shape_ok(num_kv_heads, head_dim, block_size))
    return PA_ERR_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_mapping || !int4_arrays_ok(k_codes, v_codes, k_scales, v_scales)) return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  int st = pa::copy_blocks_launch(k_codes, v_codes, block_mapping, num_pairs, num_blocks,
                                  num_kv_heads, head_dim / 2, block_size, di.err, stream);
  if (st != 0) return PA_ERR_CUDA;
  st = pa::copy_blocks_launch(k_scales, v_scales, block_mapping, num_pairs, num_blocks,
                              num_kv_heads, 4, block_size, di.err, stream);
  return st == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_swap_blocks_int4(const void* src_k, const void* src_v, const float* src_ks,
                        const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                        float* dst_vs, const int32_t* block_mapping, int num_pairs,
                        int src_num_blocks, int dst_num_blocks, int num_kv_heads, int head_dim,
                        int block_size, cudaStream_t stream) {
  if (num_pairs < 0 || src_num_blocks < 1 || dst_num_blocks < 1 ||
      !shape_ok(num_kv_heads, head_dim, block_size))
    return PA_ERR_ARG;
  if (num_pairs == 0) return PA_OK;
  const void* ptrs[9] = {src_k, src_v, src_ks, src_vs, dst_k, dst_v, dst_ks, dst_vs, block_mapping};
  void* dev[9];
  for (int i = 0; i < 9; ++i) {
    dev[i] = device_view(ptrs[i]);
    if (!dev[i]) return PA_ERR_ARG;
    if (i < 8 && !aligned16(dev[i])) return PA_ERR_ARG;
  }
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  const auto* map = static_cast<const int32_t*>(dev[8]);
  int st = pa::swap_blocks_launch(dev[0], dev[1], dev[4], dev[5], map, num_pairs, src_num_blocks,
                                  dst_num_blocks, num_kv_heads, head_dim / 2, block_size, di.err,
                                  stream);
  if (st != 0) return PA_ERR_CUDA;
  st = pa::swap_blocks_launch(dev[2], dev[3], dev[6], dev[7], map, num_pairs, src_num_blocks,
                              dst_num_blocks, num_kv_heads, 4, block_size, di.err, stream);
  return st == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* context_lens, const int32_t* query_start, int num_seqs,
               int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
               int block_size, int num_blocks, float scale, void* out, pa_dtype dtype,
               cudaStream_t stream) {
  if (num_seqs < 0 || max_query_len < 0 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      !shape_ok(num_kv_heads, head_dim, block_size) || num_q_heads < num_kv_heads ||
      num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 64 ||
      !std::isfinite(scale) || (dtype != PA_FP16 && dtype != PA_BF16) ||
      static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL ||
      static_cast<long long>(num_blocks) * num_kv_heads * block_size > 0x7fffffffLL)
    return PA_ERR_ARG;
  if (num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
    return PA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  pa::PrefillArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.out = out;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_query_len = max_query_len;
  a.scale = scale;
  a.bf16 = dtype == PA_BF16;
  a.err = di.err;
  return pa::prefill_launch(a, stream);
}

int pa_decode_append(const void* q, const void* key_new, const void* value_new, void* k_cache,
                     void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     void* out, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                     cudaStream_t stream) {
  if (num_seqs > 0 && (!key_new || !value_new)) return PA_ERR_ARG;
  return decode_call(q, key_new, value_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, out, workspace, workspace_bytes, dtype, stream);
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping, int num_pairs,
                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                   pa_dtype dtype, cudaStream_t stream) {
  if (num_pairs < 0 || num_blocks < 1 || !shape_ok(num_kv_heads, head_dim, block_size) ||
      (dtype != PA_FP16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3))
    return PA_ERR_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_mapping) return PA_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  return pa::copy_blocks_launch(k_cache, v_cache, block_mapping, num_pairs, num_blocks,
                                num_kv_heads, head_dim * (dtype == PA_FP8_E4M3 ? 1 : 2),
                                block_size, di.err, stream);
}

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int32_t* block_mapping, int num_pairs, int src_num_blocks,
                   int dst_num_blocks, int num_kv_heads, int head_dim, int block_size,
                   pa_dtype dtype, cudaStream_t stream) {
  if (num_pairs < 0 || src_num_blocks < 1 || dst_num_blocks < 1 ||
      !shape_ok(num_kv_heads, head_dim, block_size) ||
      (dtype != PA_FP16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3))
    return PA_ERR_ARG;
  if (num_pairs == 0) return PA_OK;
  const void* ptrs[5] = {src_k, src_v, dst_k, dst_v, block_mapping};
  void* dev[5];
  for (int i = 0; i < 5; ++i) {
    dev[i] = device_view(ptrs[i]);
    if (!dev[i]) return PA_ERR_ARG;
    if (i < 4 && !aligned16(dev[i])) return PA_ERR_ARG;
  }
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  return pa::swap_blocks_launch(dev[0], dev[1], dev[2], dev[3], static_cast<const int32_t*>(dev[4]),
                                num_pairs, src_num_blocks, dst_num_blocks, num_kv_heads,
                                head_dim * (dtype == PA_FP8_E4M3 ? 1 : 2), block_size, di.err,
                                stream);
}

int pa_check_block_mapping(const int32_t* host_block_mapping, int num_pairs, int num_blocks) {
  if (num_pairs < 0 || num_blocks < 1 || (num_pairs > 0 && !host_block_mapping)) return PA_ERR_ARG;
  std::set<int32_t> dsts, srcs;
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t s = host_block_mapping[2 * i], d = host_block_mapping[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PA_ERR_ARG;
    if (!dsts.insert(d).second) return PA_ERR_ARG;
    srcs.insert(s);
  }
  for (int32_t d : dsts)
    if (srcs.count(d)) return PA_ERR_ARG;
  return PA_OK;
}

int pa_get_device_error(cudaStream_t stream, uint32_t* flags_out) {
  if (!flags_out) return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, di.err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemsetAsync(di.err, 0, sizeof(v), stream) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
  *flags_out = v;
  return PA_OK;
}

}  // extern "C"
