// crc.cu — piecewise CRC-32 of any device buffer (cuZipNN API,
// hash_tensor_with_crc32: a zlib-compatible CRC of every checksum-chunk-sized
// piece of a tensor's bytes, computed on the GPU).
//
// Each piece is cut into work units of at most `unit` bytes; one warp takes
// one unit. CRC-32 is linear over GF(2), so the register after a whole piece
// is the XOR of each unit's register shifted by the bytes that follow it in
// the piece; the first unit starts from the preset register and also carries
// the final complement. Units add their terms into the piece's output with an
// atomic XOR (the output is zeroed on the stream first).
#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kWarps = 8;

// Raw register over an arbitrarily aligned range: bytes up to the first
// 16-byte boundary are taken one at a time, the rest by the warp.
__device__ uint32_t warp_crc_raw_any(const uint8_t *p, uint64_t len, uint32_t init, const uint32_t *T,
                                     const uint32_t (*G)[256]) {
    uint64_t head = (16 - (reinterpret_cast<uintptr_t>(p) & 15)) & 15;
    if (head > len) head = len;
    uint32_t reg = init;
    const uint32_t *row = crc_row(T);
    for (uint64_t i = 0; i < head; i++) reg = crc_rep_byte(reg, __ldg(p + i), row);
    return crc_strided<1, false>(p + head, len - head, reg, T, G, nullptr);
}

__global__ void __launch_bounds__(kWarps * 32) crc_kernel(CrcArgs a) {
    __shared__ __align__(16) uint32_t tab[kCrcRepWords];
    __shared__ uint32_t gap[4][256];
    load_crc_rep(tab);
    load_shift_smem(gap, gap_table<32>());
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint64_t u = uint64_t(blockIdx.x) * kWarps + warp; u < a.n_units; u += uint64_t(gridDim.x) * kWarps) {
        uint64_t piece = u / a.units_per_piece, k = u % a.units_per_piece;
        uint64_t p0 = piece * a.piece, p1 = min(p0 + a.piece, a.nbytes);
        uint64_t b0 = p0 + k * a.unit;
        if (b0 >= p1) continue;
        uint64_t b1 = min(b0 + a.unit, p1);
        uint32_t reg = warp_crc_raw_any(a.data + b0, b1 - b0, k == 0 ? 0xFFFFFFFFu : 0u, tab, gap);
        if (lane == 0) {
            uint32_t term = shift_bytes(reg, p1 - b1);
            if (k == 0) term ^= 0xFFFFFFFFu;
            atomicXor(&a.out[piece], term);
        }
    }
}

} // namespace

int launch_crc(const CrcArgs &a, cudaStream_t s) {
    if (a.n_units == 0) return ZC_OK;
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZC_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZC_ECUDA;
    uint64_t blocks = (a.n_units + kWarps - 1) / kWarps;
    uint64_t cap = uint64_t(sms) * 8;
    crc_kernel<<<int(blocks < cap ? blocks : cap), kWarps * 32, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

} // namespace zc
