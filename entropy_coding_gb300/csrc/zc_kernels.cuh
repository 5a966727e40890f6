// zc_kernels.cuh — argument blocks and launchers of the compression,
// decompression and CRC-32 kernels (host <-> device boundary inside the
// library; the public C ABI is in include/zc.h).
#pragma once

#include "zc_common.cuh"

namespace zc {

// One tensor of a compression call.
struct TensorDesc {
    const uint8_t *src;
    const uint8_t *base;            // delta: the base tensor (src XOR base is coded), else null
    uint8_t *blob;
    uint64_t *d_blob_bytes;
    uint64_t nbytes;
    uint64_t cap;                   // blob capacity
    uint32_t n_chunks;
    uint32_t chunk_base;            // call-wide index of its first chunk
    uint32_t header[24];            // the 96-byte header, CRC field zero (final CRC if empty)
};

struct EncodeArgs {
    TensorDesc one;                 // the tensor, when the call has one
    const TensorDesc *tensors;      // device table of the tensors, when it has more
    uint32_t n_tensors;
    uint32_t total_chunks;          // over all tensors
    uint32_t chunk_bytes;
    double threshold;
    int32_t *d_status;
    uint8_t *ws_ctrl;               // u32 coder ticket; per tensor t at 256 + 16 t: u32 done, u32 header-CRC acc.
    unsigned long long *ws_status;  // per chunk (call-wide index): flag << 62 | padded size or prefix
    uint8_t *ws_info;               // per chunk of the wave: 32 B {CRC, W stream words}
    uint8_t *ws_ftab;               // per chunk of the wave and stream: 256 u16 table
    uint8_t *ws_cand;               // per chunk of the wave and stream: n_pad symbol bytes
    uint64_t n_pad;                 // chunk_bytes / W rounded up to whole steps of 32
    uint8_t *ws_slots;              // per coding warp: W records of rec_stride bytes
    uint64_t slot_bytes;
    uint64_t rec_stride;
    uint32_t wave_start;            // first chunk of this wave (call-wide index)
    uint32_t wave_n;                // chunks in this wave
    uint32_t workers;               // coding warps
    // format v2 (shared plane tables): a wave holds whole tensors [wave_t0, wave_t1)
    uint32_t version;               // 1 or 2
    uint32_t wave_t0, wave_t1;
    unsigned long long *ws_hist;    // v2: per tensor and plane, 256 u64 counts over the tensor
    uint8_t *ws_ptab;               // v2: per tensor and plane, the 12-bit table (256 u16)
    uint32_t hooks;                 // test hooks (zc_set_test_hooks)
    uint32_t spin_limit;            // polls of one look-back wait before it gives up
    uint32_t packed;                // ZC_PACKED: coding CTAs of up to 16 warps, filling few SMs
};

// One blob of a decompression call.
struct BlobDesc {
    const uint8_t *blob;
    const uint8_t *base;            // delta: the output is the decoded bytes XOR base, else null
    uint8_t *dst;
    uint64_t blob_bytes;
    uint64_t nbytes;
    uint32_t n_chunks;
    uint32_t chunk_base;            // call-wide index of its first chunk
    uint32_t cta_base;              // v2: index of the blob's first CTA (CTAs never span blobs)
    uint32_t pad_;
};

struct DecodeArgs {
    BlobDesc one;                   // the blob, when the call has one
    const BlobDesc *blobs;          // device table of the blobs, when it has more
    uint32_t n_blobs;
    uint32_t total_chunks;
    uint32_t chunk_bytes;
    uint32_t flags;
    int32_t *d_status;
    uint32_t version;               // 1 or 2 (every blob of the call)
    uint32_t pairs;                 // v2: chunks (warp pairs) per CTA
    uint32_t n_ctas;                // v2: CTAs of the call
    uint32_t hooks;                 // test hooks (zc_set_test_hooks)
    unsigned long long wait_cycles; // clock cycles of one barrier wait before it gives up
};

// Wait limits: about a second of polling in normal calls, a short one under
// the test hooks that make a wait run out.
constexpr uint32_t kSpinLimit = 1u << 22, kSpinLimitTest = 1u << 10;
constexpr unsigned long long kWaitCycles = 1ull << 31, kWaitCyclesTest = 1ull << 20;

// zc_verify: a blob's header CRC and every chunk's CRC, without decoding.
struct VerifyArgs {
    const uint8_t *blob;
    uint64_t blob_bytes;
    uint64_t table_end;      // header + chunk table (v2: + plane tables)
    uint32_t n_chunks;
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

// Statistics and coding kernels for chunks [wave_start, wave_start + wave_n)
// (total_chunks > 0).
int launch_encode_wave(int dtype, bool delta, const EncodeArgs &a, cudaStream_t s);
// The blobs (header alone; v2: and zero plane tables) of the call's tensors
// that have no chunks.
int launch_empty_blobs(const EncodeArgs &a, cudaStream_t s);
// v2: the plane tables of the wave's tensors (after its statistics kernel).
int launch_plane_tables(int dtype, const EncodeArgs &a, cudaStream_t s);
// v2 decoding: CTAs of `pairs` chunks each, never spanning two blobs.
uint32_t decode_v2_pairs(uint64_t total_chunks, bool packed);

// The tensor (blob) of a call-wide chunk index: the last one whose first
// chunk is at or before it (binary search over the table).
template <class D>
__device__ __forceinline__ uint32_t owner_of(const D *table, uint32_t n, uint32_t g) {
    uint32_t lo = 0, hi = n;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (table[mid].chunk_base <= g) lo = mid;
        else hi = mid;
    }
    return lo;
}
int encode_warps_per_sm();
// delta: whether the blobs carry base tensors (all or none of them)
int launch_decode(int dtype, bool delta, const DecodeArgs &a, cudaStream_t s);
// the kernels of one dtype (decode_<dtype>.cu)
int launch_decode_u8(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_decode_u16(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_decode_u32(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_decode_bf16(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_decode_fp16(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_decode_fp32(bool delta, const DecodeArgs &a, cudaStream_t s);
int launch_crc(const CrcArgs &a, cudaStream_t s);
int launch_verify(const VerifyArgs &a, cudaStream_t s);

} // namespace zc
