// decode_fp16.cu — the decompression kernels instantiated for FP16.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_fp16(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_FP16>(delta, a, s); }

} // namespace zc
