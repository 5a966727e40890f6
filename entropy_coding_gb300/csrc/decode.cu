// decode.cu — decompression entry of the library: the launch plan of format
// v2 and the dispatch to the per-dtype kernels (decode_<dtype>.cu).
#include "decode_impl.cuh"

namespace zc {

uint32_t decode_v2_pairs(uint64_t total_chunks, bool packed) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1)
        sms = 1;
    // one CTA per SM holds its chunks when they fit; else CTAs of kV2Pairs
    // (ZC_PACKED: CTAs of kV2Pairs whatever the number of chunks)
    const uint64_t per_sm = packed ? total_chunks : (total_chunks + uint64_t(sms) - 1) / uint64_t(sms);
    return uint32_t(std::max<uint64_t>(1, std::min<uint64_t>(kV2Pairs, per_sm)));
}

int launch_decode(int dtype, bool delta, const DecodeArgs &a, cudaStream_t s) {
    if (a.total_chunks == 0) return ZC_OK;
    switch (dtype) {
    case ZC_U8: return launch_decode_u8(delta, a, s);
    case ZC_U16: return launch_decode_u16(delta, a, s);
    case ZC_U32: return launch_decode_u32(delta, a, s);
    case ZC_BF16: return launch_decode_bf16(delta, a, s);
    case ZC_FP16: return launch_decode_fp16(delta, a, s);
    case ZC_FP32: return launch_decode_fp32(delta, a, s);
    default: return ZC_EINVAL;
    }
}

} // namespace zc
