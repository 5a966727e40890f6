// decode_fp32.cu — the decompression kernels instantiated for FP32.
#include "decode_impl.cuh"

namespace zc {

int launch_decode_fp32(bool delta, const DecodeArgs &a, cudaStream_t s) { return launch_decode_dtype<ZC_FP32>(delta, a, s); }

} // namespace zc
