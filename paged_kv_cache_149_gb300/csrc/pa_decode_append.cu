// The fused step over 16-bit K/V blocks (the newest rows attended from the step's input and
// written to the cache by the decode kernel): its instantiations of pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace decode {
template int launch_format<kKv16, true>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode
}  // namespace pa
