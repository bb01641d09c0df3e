// Paged decode attention over INT4 K/V blocks (codes with a float32 scale per row):
// the plain-decode instantiations of the kernel in pa_decode_kernel.cuh.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace decode {
template int launch_format<kKvInt4, false>(const Params&, int, int, bool, cudaStream_t);
}  // namespace decode
}  // namespace pa
