// The fused step over FP8 (E4M3) K/V blocks (the newest rows quantised, attended and written
// by the decode kernel): its instantiations of pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace decode {
template int launch_format<kKvFp8, true>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode
}  // namespace pa
