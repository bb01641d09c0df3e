// Paged decode attention over FP8 (E4M3) K/V blocks: the FP8 instantiations of the kernel
// in pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {

int decode_launch_fp8(const decode::Params& p, int grid, int head_dim, bool bf16,
                      cudaStream_t stream) {
#define PA_DECODE_FP8_CASE(DD, NN)                                                       \
  if (head_dim == DD && (p.heads_per_pair > 8) == (NN == 2))                            \
    return bf16 ? decode::launch<DD, NN, __nv_bfloat16, decode::kKvFp8>(p, grid, stream) \
                : decode::launch<DD, NN, __half, decode::kKvFp8>(p, grid, stream);
  PA_DECODE_FP8_CASE(128, 1)
  PA_DECODE_FP8_CASE(128, 2)
  PA_DECODE_FP8_CASE(64, 1)
  PA_DECODE_FP8_CASE(64, 2)
#undef PA_DECODE_FP8_CASE
  return -1;
}

}  // namespace pa
