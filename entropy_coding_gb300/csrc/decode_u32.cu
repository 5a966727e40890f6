// decode_u32.cu — the decompression kernels instantiated for U32.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_u32(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_U32>(delta, a, s); }

} // namespace zc
