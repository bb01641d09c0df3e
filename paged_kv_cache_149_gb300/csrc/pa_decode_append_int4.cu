// The fused step over INT4 K/V blocks (the newest rows quantised with a scale per row,
// attended and written by the decode kernel): its instantiations of pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace decode {
template int launch_format<kKvInt4, true>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode
}  // namespace pa
