// zc_kernels.cuh — argument blocks and launchers of the compression,
// decompression and CRC-32 kernels (host <-> device boundary inside the
// library; the public C ABI is in include/zc.h).
#pragma once

#include "zc_common.cuh"

namespace zc {

struct EncodeArgs {
    const uint8_t *src;
    uint64_t nbytes;
    uint32_t chunk_bytes;
    uint32_t n_chunks;
    double threshold;
    uint8_t *blob;
    uint64_t cap;
    uint64_t *d_blob_bytes;
    int32_t *d_status;
    uint8_t *ws_ctrl;               // u32 ticket, u32 done, u32 header-CRC accumulator
    unsigned long long *ws_status;  // per chunk: flag << 62 | padded size or prefix
    uint8_t *ws_slots;              // per-CTA staging for coded records
    uint64_t slot_bytes;
    uint32_t header[24];            // the 96-byte header, CRC field zero (final CRC if empty)
};

struct DecodeArgs {
    const uint8_t *blob;
    uint64_t blob_bytes;
    uint64_t nbytes;
    uint32_t chunk_bytes;
    uint32_t n_chunks;
    uint8_t *dst;
    uint32_t flags;
    int32_t *d_status;
};

struct CrcArgs {
    const uint8_t *data;
    uint64_t nbytes;
    uint64_t piece;          // bytes per output CRC
    uint64_t unit;           // bytes per warp work unit (divides into pieces)
    uint64_t units_per_piece;
    uint64_t n_units;
    uint32_t *out;
};

int launch_encode(int dtype, const EncodeArgs &a, int grid, cudaStream_t s);
int encode_ctas_per_sm();
int launch_decode(int dtype, const DecodeArgs &a, cudaStream_t s);
int launch_crc(const CrcArgs &a, cudaStream_t s);

} // namespace zc
