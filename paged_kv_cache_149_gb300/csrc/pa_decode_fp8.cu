// Paged decode attention over FP8 (E4M3) K/V blocks (codes with one scale per cache):
// the plain-decode instantiations of the kernel in pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace decode {
template int launch_format<kKvFp8, false>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode
}  // namespace pa
