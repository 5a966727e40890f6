// decode_u16.cu — the decompression kernels instantiated for U16.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_u16(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_U16>(delta, a, s); }

} // namespace zc
