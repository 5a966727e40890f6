// decode_u8.cu — the decompression kernels instantiated for U8.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_u8(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_U8>(delta, a, s); }

} // namespace zc
