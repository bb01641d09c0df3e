// Diagnostics (pa_decode_timeline): the 16-bit decode kernel of pa_decode_kernel.cuh compiled
// once more under another name, with the phase stamps that PA_DECODE_TIMELINE turns on, for
// head_dim 128 and up to 8 query heads a pair.  The kernels that serve ordinary calls are
// compiled in the other translation units without them.
#define PA_DECODE_TIMELINE
#include "pa_decode_kernel.cuh"

namespace pa {

int decode_launch_timed(const decode::Params& p, int grid, bool bf16, cudaStream_t stream,
                        unsigned long long* timeline) {
  if (p.key_new)
    return bf16 ? decode::launch_timed<128, 1, __nv_bfloat16, decode::kKv16, true>(p, grid, stream, timeline)
                : decode::launch_timed<128, 1, __half, decode::kKv16, true>(p, grid, stream, timeline);
  return bf16 ? decode::launch_timed<128, 1, __nv_bfloat16, decode::kKv16, false>(p, grid, stream, timeline)
              : decode::launch_timed<128, 1, __half, decode::kKv16, false>(p, grid, stream, timeline);
}

}  // namespace pa
