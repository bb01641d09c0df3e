// pa_decode_fixed_scratch: paged decode for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at all: a serving process that handed
// almost all of HBM to the KV block pool up front (an allocation could fail, or stall the
// device while it waits for memory), or a host framework that owns every device buffer
// and forbids allocations made behind its back.  pa_decode asks such callers for a
// workspace they may have no way to provide.  This entry point needs none: its split-KV
// scratch is a fixed array compiled into the library, present on every GPU that loads it
// until the process exits.
//
// Usage notes for callers:
// * The scratch is shared by every call on a device and keeps whatever the last call
//   left in it.  Nothing in it has to start at zero: every decode call writes each
//   scratch entry it later reads.  Two calls whose GPU work overlaps (different streams
//   without ordering between them) race on it and give undefined output.
// * The first call on each device looks up the array's device address there (the name of
//   a __device__ array is only a host-side stand-in, not something a kernel may use).
//   Make that first call before any stream capture begins.
// * If a device needs more scratch than the fixed maximum below (very many SMs), the call
//   returns PA_ERR_WORKSPACE and launches nothing.
// * q must be device memory of the current device (the scratch address is looked up per
//   device); otherwise the call returns PA_ERR_ARG.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"

namespace {

// 32 MiB: the largest decode workspace (16 query heads per kv head, 8 or more kv heads,
// head_dim 128) of a device with up to about 250 SMs
constexpr size_t kFixedScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of g_fixed_scratch, per device

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_fixed_scratch(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, float scale, void* out,
                                       pa_dtype dtype, cudaStream_t stream) {
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  // The scratch address is the current device's: q must live there too.
  if (q) {
    int dev = 0;
    cudaPointerAttributes attr;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaPointerGetAttributes(&attr, q) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice || attr.device != dev) return PA_ERR_ARG;
  }
  // pa_decode checks every argument and rejects a scratch smaller than this device needs.
  return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                   out, scratch, kFixedScratchBytes, dtype, stream);
}
