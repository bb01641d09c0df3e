// Shared device helpers for the paged-attention kernels (sm_103a).
//
// mbarrier + cp.async.bulk (the TMA engine's 1-D bulk copy) move whole K/V block
// rows from HBM into shared memory; every wait on a barrier is bounded by a wall-clock
// limit so that a lost copy turns into an error bit instead of a hung GPU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace pa {

// Wall-clock limit of every pipeline wait.  A healthy wait lasts microseconds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Device error bits (mirrors include/pa.h).
constexpr unsigned kErrBadBlock = 0x1u;
constexpr unsigned kErrBadContext = 0x2u;
constexpr unsigned kErrBadSlot = 0x4u;
constexpr unsigned kErrBadPair = 0x8u;
constexpr unsigned kErrTimeout = 0x10u;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase of `bar` with parity `parity` has completed.  Gives up (returns
// false) when *abort becomes non-zero or after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 4-D tiled TMA load through the tensor map at `map` (a kernel parameter): x = d, y = row
// in the block, z = kv head, w = block; completion counted in bytes on `bar`.  x * the
// element size is a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, int x, int y, int z,
                                            int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (a hint: no data moves to the SM, and a
// later write by another kernel is seen by later reads).  src 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch (PDL) controls.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Packed fp32x2 fused multiply-add (sm_100+): d = a * b + c, lane-wise, RN.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Barrier over `count` threads of named barrier `id` that also ORs `pred` across them:
// every participant gets the same answer.
__device__ __forceinline__ bool bar_red_or(int id, int count, bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.s32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.s32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<int>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Two packed 16-bit values -> two floats (exact).
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  // bf16 is the top half of an fp32: shifting the bits into place is exact.
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);

template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

// One float -> one 16-bit value, round to nearest even.
template <typename T>
__device__ __forceinline__ T from_float(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_float<__half>(float v) {
  return __float2half_rn(v);
}

// FP8 (E4M3) quantisation shared by the cache-write kernel and the fused decode step, so
// that both produce the same codes: x / scale in IEEE float32, then round to nearest-even
// with magnitudes above 448 clamped (the hardware's satfinite conversion).
// Two float32 values -> two codes, `hi` in the upper byte, `lo` in the lower.
__device__ __forceinline__ uint16_t e4m3x2_of(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Sixteen 16-bit values (two 16-byte vectors, element 0 first) -> their 16 codes.
template <typename T>
__device__ __forceinline__ uint4 quantize16_e4m3(const uint4& a, const uint4& b, float scale) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x0 = unpack2<T>(w[2 * k]), x1 = unpack2<T>(w[2 * k + 1]);
    out[k] = static_cast<uint32_t>(e4m3x2_of(__fdiv_rn(x0.y, scale), __fdiv_rn(x0.x, scale))) |
             (static_cast<uint32_t>(e4m3x2_of(__fdiv_rn(x1.y, scale), __fdiv_rn(x1.x, scale)))
              << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// INT4 quantisation of one row of D values spread over a warp, lane l holding values
// (D/32) l .. (D/32) l + D/32 - 1, shared by the cache-write kernel and the fused decode
// step so that both produce the same codes: s = max |x| / 7 (IEEE float32), c = x / s
// rounded half to even and clamped to [-7, 7] (0 for an all-zero row), nibble u = c + 8,
// this lane's nibbles packed low first.  Returns the packed nibbles; s in `scale`.
template <int D>
__device__ __forceinline__ uint32_t int4_quantize_lane(const float (&x)[D / 32], float& scale) {
  constexpr int PER = D / 32;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 7.f);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const float c = amax == 0.f ? 0.f : fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(x[i], s))));
    packed |= static_cast<uint32_t>(static_cast<int>(c) + 8) << (4 * i);
  }
  scale = s;
  return packed;
}

// This lane's D/32 values of a 16-bit row at `src` (lane l: values (D/32) l ..).
template <typename T, int D>
__device__ __forceinline__ void int4_row_values(const T* src, int lane, float (&x)[D / 32]) {
  if constexpr (D / 32 == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src + 4 * lane);
    const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const float2 a = unpack2<T>(*reinterpret_cast<const uint32_t*>(src + 2 * lane));
    x[0] = a.x; x[1] = a.y;
  }
}

}  // namespace pa
