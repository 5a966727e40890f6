// decode_bf16.cu — the decompression kernels instantiated for BF16.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_bf16(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_BF16>(delta, a, s); }

} // namespace zc
