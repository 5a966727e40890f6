// zc_kernels.cuh — argument blocks and launchers of the compression,
// decompression and CRC-32 kernels (host <-> device boundary inside the
// library; the public C ABI is in include/zc.h).
#pragma once

#include "zc_common.cuh"

namespace zc {

struct EncodeArgs {
    const uint8_t *src;
    const uint8_t *base;            // delta: the base tensor (src XOR base is coded), else null
    uint64_t nbytes;
    uint32_t chunk_bytes;
    uint32_t n_chunks;
    double threshold;
    uint8_t *blob;
    uint64_t cap;
    uint64_t *d_blob_bytes;
    int32_t *d_status;
    uint8_t *ws_ctrl;               // u32 coder ticket, u32 done, u32 header-CRC accumulator
    unsigned long long *ws_status;  // per chunk: flag << 62 | padded size or prefix
    uint8_t *ws_info;               // per chunk of the wave: 32 B {CRC, W stream words}
    uint8_t *ws_ftab;               // per chunk of the wave and stream: 256 u16 table
    uint8_t *ws_cand;               // per chunk of the wave and stream: n_pad symbol bytes
    uint64_t n_pad;                 // chunk_bytes / W rounded up to whole steps of 32
    uint8_t *ws_slots;              // per coding warp: W records of rec_stride bytes
    uint64_t slot_bytes;
    uint64_t rec_stride;
    uint32_t wave_start;            // first chunk of this wave
    uint32_t wave_n;                // chunks in this wave
    uint32_t workers;               // coding warps
    uint32_t header[24];            // the 96-byte header, CRC field zero (final CRC if empty)
};

struct DecodeArgs {
    const uint8_t *blob;
    const uint8_t *base;            // delta: the output is the decoded bytes XOR base, else null
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

// Statistics and coding kernels for chunks [wave_start, wave_start + wave_n);
// the empty-tensor blob when n_chunks == 0.
int launch_encode_wave(int dtype, const EncodeArgs &a, cudaStream_t s);
int encode_warps_per_sm();
int launch_decode(int dtype, const DecodeArgs &a, cudaStream_t s);
int launch_crc(const CrcArgs &a, cudaStream_t s);

} // namespace zc
