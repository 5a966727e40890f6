// crc.cu — piecewise CRC-32 of any device buffer (cuZipNN API,
// hash_tensor_with_crc32: a zlib-compatible CRC of every checksum-chunk-sized
// piece of a tensor's bytes, computed on the GPU), and the check of a blob's
// CRCs without decoding it (cuZipNN API: verify an untrusted blob with the
// CRC-32 helpers before decompressing it).
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

// One CTA per chunk (grid-stride), and one unit more for the header: the
// header CRC runs over the header with its CRC field read as zero and over
// the chunk table (v2: and the plane tables); a chunk's over its stored
// bytes. A table entry that points outside the blob is reported as a format
// error and its bytes are not read.
constexpr int kVerifyWarps = 8;

__global__ void __launch_bounds__(kVerifyWarps * 32) verify_kernel(VerifyArgs a) {
    __shared__ __align__(16) uint32_t tab[kCrcRepWords];
    __shared__ uint32_t gap[4][256];
    __shared__ uint32_t s_reg[kVerifyWarps];
    load_crc_rep(tab);
    load_shift_smem(gap, gap_table<kVerifyWarps * 32>());
    __syncthreads();
    const uint32_t *row = crc_row(tab);
    for (uint64_t u = blockIdx.x; u <= a.n_chunks; u += gridDim.x) {
        if (u == a.n_chunks) {
            uint32_t reg = 0xFFFFFFFFu;
            for (int i = 0; i < 28; i++) reg = crc_rep_byte(reg, __ldg(a.blob + i), row);
            reg = crc_rep_word(reg, 0u, row);
            reg = crc_strided<kVerifyWarps, false>(a.blob + 32, a.table_end - 32, reg, tab, gap, s_reg);
            const uint32_t want = __ldg(reinterpret_cast<const uint32_t *>(a.blob + 28));
            if (threadIdx.x == 0 && (reg ^ 0xFFFFFFFFu) != want) status_or(a.d_status, ZC_ECRC);
            continue;
        }
        const uint4 ent = __ldg(reinterpret_cast<const uint4 *>(a.blob + ZC_HEADER_BYTES) + u);
        const uint64_t off = uint64_t(ent.x) | (uint64_t(ent.y) << 32);
        const uint64_t stored = ent.z & 0x7FFFFFFFu;
        if ((off & 15) || off < a.table_end || off > a.blob_bytes || stored > a.blob_bytes - off) {
            if (threadIdx.x == 0) status_or(a.d_status, ZC_EFORMAT);
            continue;
        }
        const uint32_t reg = crc_strided<kVerifyWarps, false>(a.blob + off, stored, 0xFFFFFFFFu, tab, gap, s_reg);
        if (threadIdx.x == 0 && (reg ^ 0xFFFFFFFFu) != ent.w) status_or(a.d_status, ZC_ECRC);
    }
}

} // namespace

int launch_verify(const VerifyArgs &a, cudaStream_t s) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZC_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZC_ECUDA;
    const uint64_t units = uint64_t(a.n_chunks) + 1;
    const uint64_t cap = uint64_t(sms) * 4;
    verify_kernel<<<int(units < cap ? units : cap), kVerifyWarps * 32, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

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
