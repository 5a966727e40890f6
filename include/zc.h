/*
 * zc.h — C ABI of the GB300 (sm_103a) lossless compressor for float model
 * tensors: exponent extraction + byte grouping, per-chunk order-0 12-bit
 * frequency tables, 32-lane interleaved rANS with raw passthrough, a chunk
 * offset prefix scan, and per-chunk CRC-32.
 *
 * Sources (web pages, cited by title and section):
 *   cuZipNN 0.1.0 (PyPI): Usage (tensor in, blob out, torch.equal round trip;
 *     the blob records dtype and shape), API (chunk_bytes, passthrough
 *     threshold, CRC-32 helpers that match zlib.crc32), Blob format (a format
 *     version that other versions reject).
 *   nucleation NOTE-241: ZipNN — Method 1-5 (exponent extraction, byte
 *     grouping, entropy-only coding, all-constant streams stored as a header,
 *     fixed chunks with a metadata map of variable compressed sizes).
 *   lmzip 1.3.0 (PyPI metadata) — "Building on lmz": the device entry point
 *     takes the caller's device pointers and stream, allocates nothing,
 *     creates no context and does not synchronise; interleaved rANS lanes.
 *
 * Conventions for every entry point:
 *   - "d_" pointers are device pointers on the current CUDA device; "h_"
 *     pointers are host pointers. The caller owns every buffer, the stream and
 *     the context. No entry point allocates device memory, creates streams, or
 *     synchronises.
 *   - Host-blob mode (cuZipNN Usage: GPU tensor to CPU blob and back). The
 *     data buffers of the compression and decompression calls (sources,
 *     bases, blobs, outputs and d_blob_bytes) may also be page-locked host
 *     memory (cudaHostAlloc, cudaHostRegister) or managed memory: the kernels
 *     then read and write host memory directly over the host link, as they
 *     code, with no separate copy. Pointers are checked with
 *     cudaPointerGetAttributes after the other argument checks; unregistered
 *     (pageable) host memory and another device's memory are refused with
 *     ZC_EINVAL before any launch. Workspaces and d_status must be device
 *     memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - The return value reports argument errors found on the host before any
 *     launch, and launch errors (ZC_ECUDA). Errors only the device can see
 *     are OR-ed into *d_status, which the caller zeroes before the call;
 *     results and *d_status are valid once the stream has been synchronised.
 *   - Blob format v1 (byte layout): 96-byte header ("ZCNN", version 1,
 *     dtype, ndim, chunk_bytes, lanes = 32, prob_bits = 12, nbytes,
 *     n_chunks, header CRC-32 over header + chunk table, shape[8]); a chunk
 *     table of 16-byte entries {u64 offset, u32 stored | raw << 31, u32
 *     CRC-32 of the chunk's `stored` payload bytes at `offset`}; then the
 *     chunk payloads, each zero-padded to 16 bytes. All integers
 *     little-endian. The chunk CRCs are over pieces of the blob (cuZipNN API:
 *     CRC-32 helpers over checksum-sized pieces, used to check an untrusted
 *     blob before decompressing it), so zc_verify can check a blob without
 *     decoding it.
 */
#ifndef ZC_H
#define ZC_H

#include <stdint.h>

#if defined(__GNUC__)
#define ZC_API __attribute__((visibility("default")))
#else
#define ZC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the tensor. The float types get exponent extraction
 * (exponent byte first, then sign, then mantissa); the integer types are
 * byte-grouped as they are. */
enum zc_dtype { ZC_U8 = 1, ZC_U16 = 2, ZC_U32 = 3, ZC_BF16 = 4, ZC_FP16 = 5, ZC_FP32 = 6 };

/* Status bits; several may be OR-ed together. */
enum zc_status {
    ZC_OK = 0,
    ZC_EINVAL = 1,     /* bad argument (host) */
    ZC_EFORMAT = 2,    /* not a v1 blob, or a malformed header/table */
    ZC_ECRC = 4,       /* a CRC-32 did not match */
    ZC_ECORRUPT = 8,   /* payload structure or rANS stream invalid */
    ZC_ETIMEOUT = 16,  /* a bounded device wait gave up */
    ZC_ECAPACITY = 32, /* an output or workspace buffer is too small */
    ZC_ECUDA = 64      /* a CUDA launch or memset failed */
};

/* zc_decompress flag: skip the per-chunk CRC-32 check. */
#define ZC_NO_VERIFY 1u
/* compression flag: blob format v2 (one 12-bit table per byte plane of the
 * tensor, shared by all its chunks; lmzip "Building on lmz") */
#define ZC_SHARED_TABLES 2u
/* compression flag: blob format v3 (v1 with a word list per rANS lane in
 * every coded record; lmzip "On a GPU": the decoder is bound by the lanes'
 * dependent chains). Not combinable with ZC_SHARED_TABLES. */
#define ZC_LANE_WORDS 4u
/* flag of the compression and decompression calls (the pages have no
 * counterpart; a launch-shape choice that changes no byte of any blob): pack
 * the call's chunks into as few SMs as they fill, up to 16 coding warps or 16
 * decoding warp pairs per SM, instead of spreading them over every SM. Meant
 * for calls issued on several streams at once (one call per tensor of a
 * model): the SMs a call leaves free run the other streams' calls, and every
 * SM holds more rANS chains. A call alone on the GPU is faster without it. */
#define ZC_PACKED 8u

/* Parameter limits of format v1. */
#define ZC_MIN_CHUNK 64u
#define ZC_MAX_CHUNK 131072u   /* chunk_bytes: a multiple of 64 in [64, 131072] */
#define ZC_HEADER_BYTES 96u
#define ZC_ENTRY_BYTES 16u

/* What a blob header and chunk table say (filled by zc_blob_info). */
typedef struct {
    int32_t dtype;
    int32_t ndim;
    int64_t shape[8];
    uint64_t nbytes;      /* original tensor bytes */
    uint64_t blob_bytes;  /* total blob length */
    uint32_t n_chunks;
    uint32_t chunk_bytes;
    uint32_t version;     /* blob format: 1 (a table per coded stream) or 2 (shared plane tables) */
    uint32_t reserved;
} zc_info;

/* Worst-case blob length for compressing nbytes of dtype with these
 * parameters (cuZipNN API: a chunk is kept coded only if it shrinks below
 * threshold x its size, so for threshold <= 1 no chunk grows beyond its raw
 * size; threshold > 1, a test setting that forces coding, allows growth).
 * Returns 0 if the parameters are invalid. Host only, no CUDA call. */
ZC_API uint64_t zc_blob_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold);

/* Device workspace zc_compress needs for these parameters on the current
 * device: chunk status words for the offset scan; per chunk of a wave (at
 * most 512 MiB of it) the statistics pass's results and the bytes of the
 * streams it chose to code; per coding warp room for a chunk's coded
 * records. With at least this much, any threshold works; thresholds above 1
 * may run fewer coding warps. Returns 0 for invalid parameters. Queries the
 * device's SM count; no allocation, no synchronisation. */
ZC_API uint64_t zc_workspace_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes);

/* Parse and check a blob's header and chunk table from a host copy of its
 * first `avail` bytes (at least 96 + 16 * n_chunks). Checks magic, version,
 * field ranges, the header CRC-32 and that the table describes the packed
 * layout exactly. Returns ZC_OK, ZC_EFORMAT or ZC_ECRC. Host only. */
ZC_API int zc_blob_info(const void *h_blob_prefix, uint64_t avail, zc_info *out);

/* Check a blob without decoding it (cuZipNN API: verify an untrusted blob
 * with the CRC-32 helpers before decompress_tensor). On the device, over the
 * blob as it is in memory: the header CRC-32 (header with its CRC field read
 * as zero, chunk table, and for format v2 the plane tables) and each chunk's
 * CRC-32 over its stored bytes; a table entry that points outside
 * info->blob_bytes is reported as ZC_EFORMAT and not read.
 *   d_blob     the blob (device or page-locked host memory, 16-byte aligned)
 *   info       from zc_blob_info on a host copy of the blob's prefix
 *   d_status   device int32, OR-ed with ZC_ECRC / ZC_EFORMAT
 * Returns ZC_EINVAL for inconsistent info or unusable pointers (nothing
 * launched), ZC_ECUDA for a launch error, else ZC_OK. One launch, no
 * allocation, no synchronisation. A blob that passes decodes with
 * zc_decompress without a CRC error. */
ZC_API int zc_verify(const void *d_blob, const zc_info *info, int32_t *d_status, void *stream);

/* Compress a contiguous row-major tensor (cuZipNN Usage: tensor in,
 * self-describing blob out).
 *   d_src        nbytes of input, aligned to the element size
 *   dtype, ndim, shape[ndim]  recorded in the header; prod(shape) * element
 *                size must equal nbytes; 0 <= ndim <= 8
 *   chunk_bytes  multiple of 64 in [64, 131072] (ZipNN Method 5 chunks;
 *                cuZipNN default 131072)
 *   threshold    > 0 (cuZipNN passthrough_threshold; 0.95 by default)
 *   d_blob       output, blob_capacity >= zc_blob_size(...)
 *   d_blob_bytes receives the blob length (device u64)
 *   d_ws         workspace of ws_bytes >= zc_workspace_size(...); its
 *                contents are scratch and need no initialisation
 *   d_status     device int32, OR-ed with ZC_ETIMEOUT / ZC_ECAPACITY
 * The output is byte-identical to the format's CPU definition. */
ZC_API int zc_compress(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                uint32_t chunk_bytes, double threshold,
                void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream);

/* Decompress a device-resident blob whose header was read with zc_blob_info
 * into `info` (cuZipNN API decompress_tensor: decoding runs on the GPU).
 *   d_blob       the blob (info->blob_bytes bytes)
 *   d_dst        output, dst_capacity >= info->nbytes, aligned to the
 *                element size
 *   flags        0, or ZC_NO_VERIFY (skip the per-chunk CRC check) and/or
 *                ZC_PACKED (the launch shape for calls on several streams)
 *   d_status     device int32, OR-ed with ZC_ECRC / ZC_ECORRUPT / ZC_EFORMAT
 * With the check, each chunk's CRC-32 is taken over its stored bytes in the
 * same pass that reads them for decoding, and compared at the end of the
 * chunk. The output bytes of a chunk that fails a check are unspecified; any
 * nonzero status means the tensor must not be used. Every device read is
 * bounds-checked against the blob, so a damaged blob is never read or
 * written out of bounds; writes stay within the first info->nbytes bytes of
 * d_dst. To reject an untrusted blob before any output is written, call
 * zc_verify first. */
ZC_API int zc_decompress(const void *d_blob, const zc_info *info, void *d_dst, uint64_t dst_capacity,
                  uint32_t flags, int32_t *d_status, void *stream);

/* Compress the XOR of two same-layout tensors (ZipNN note, Method 6 and
 * Deltas: XOR a checkpoint against a base, then code the byte groups), fused:
 * the difference is formed as the input is read and never stored. The blob
 * is exactly the blob zc_compress makes of (base XOR new) with the same
 * parameters, so zc_decompress of it gives that difference back and
 * zc_decompress_delta gives `new`.
 *   d_base, d_new  device tensors of nbytes bytes each, 16-byte aligned
 *   dtype          ZC_U8, ZC_U16 or ZC_U32: the word size the difference is
 *                  grouped by (ZC_U16 for BF16/FP16 checkpoints, ZC_U32 for
 *                  FP32); float dtypes are rejected (ZC_EINVAL)
 *   everything else as zc_compress (same workspace size).
 * Returns ZC_EINVAL for a non-integer dtype or misaligned inputs, else what
 * zc_compress returns. */
ZC_API int zc_compress_delta(const void *d_base, const void *d_new, uint64_t nbytes, int dtype, int ndim,
                      const int64_t *h_shape, uint32_t chunk_bytes, double threshold,
                      void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                      void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream);

/* Decompress a blob made by zc_compress_delta (or by zc_compress of a
 * difference) and XOR it with the base in the same pass: d_dst receives
 * base XOR decoded. The per-chunk CRC is checked over the stored bytes, as
 * in zc_decompress, unless flags has ZC_NO_VERIFY; ZC_PACKED as there.
 *   info           from zc_blob_info; its dtype must be ZC_U8/U16/U32
 *   d_base, d_dst  device buffers of info->nbytes bytes, 16-byte aligned;
 *                  d_dst may not overlap d_base or the blob
 * Errors as zc_decompress, plus ZC_EINVAL for a float dtype or misaligned
 * buffers. */
ZC_API int zc_decompress_delta(const void *d_blob, const zc_info *info, const void *d_base, void *d_dst,
                        uint64_t dst_capacity, uint32_t flags, int32_t *d_status, void *stream);

/* Batched compression: n tensors of one dtype and chunk size in one call,
 * each to its own blob, byte-identical to zc_compress (or, with d_bases,
 * zc_compress_delta) of that tensor alone. The chunks of all the tensors
 * form one grid, so a model's many small tensors (ZipNN note, Table II
 * models; lmzip README, safetensors shards compressed tensor by tensor) keep
 * every SM busy where a call per tensor would leave most of them idle.
 *   n                  number of tensors; 0 is a no-op
 *   d_srcs[t]          device tensor t (host array of n device pointers)
 *   d_bases            NULL, or n device base tensors: tensor t is then coded
 *                      as d_srcs[t] XOR d_bases[t] as in zc_compress_delta
 *                      (dtype ZC_U8/U16/U32, both 16-byte aligned)
 *   nbytes[t]          host array: bytes of tensor t (0 allowed)
 *   ndims[t], shapes   host arrays: rank of tensor t and its shape in
 *                      shapes[8 t .. 8 t + ndims[t])
 *   d_blobs[t], blob_capacities[t]
 *                      blob t (16-byte aligned) and its capacity, as in
 *                      zc_compress
 *   flags              0 (format v1), ZC_SHARED_TABLES (format v2, below) or
 *                      ZC_LANE_WORDS (format v3), each with ZC_PACKED or not
 *   d_blob_bytes       DEVICE array of n uint64: entry t receives blob t's size
 *   d_ws, ws_bytes     ws_bytes >= zc_workspace_size_batch(nbytes, n, ...)
 *   d_status           one device int32 for the whole call
 * The descriptor table travels with the launches: the host arrays may be
 * reused or freed when the call returns. Blobs must not overlap one another
 * or any input. Returns ZC_EINVAL (with nothing launched) when any tensor's
 * arguments are invalid, and zc_compress's other codes. */
ZC_API int zc_compress_batch(uint32_t n, const void *const *d_srcs, const void *const *d_bases,
                             const uint64_t *nbytes, int dtype, const int32_t *ndims, const int64_t *shapes,
                             uint32_t chunk_bytes, double threshold, uint32_t flags, void *const *d_blobs,
                             const uint64_t *blob_capacities, uint64_t *d_blob_bytes, void *d_ws,
                             uint64_t ws_bytes, int32_t *d_status, void *stream);

/* Workspace bytes for zc_compress_batch of n tensors of the given sizes and
 * flags (0 if a size or the parameters are invalid). Host only. */
ZC_API uint64_t zc_workspace_size_batch(const uint64_t *nbytes, uint32_t n, int dtype, uint32_t chunk_bytes,
                                        uint32_t flags);

/* Batched decompression of n blobs of one dtype and chunk size in one grid,
 * each output byte-identical to zc_decompress (or, with d_bases,
 * zc_decompress_delta) of that blob alone.
 *   d_blobs[t], infos[t]   blob t (device, 16-byte aligned) and its
 *                          zc_blob_info; every info has the same dtype and
 *                          chunk_bytes (else ZC_EINVAL)
 *   d_bases                NULL, or n device base tensors (delta blobs)
 *   d_dsts[t], dst_capacities[t]  output t, as in zc_decompress
 *   flags                  as in zc_decompress (ZC_NO_VERIFY, ZC_PACKED)
 *   d_ws, ws_bytes         ws_bytes >= zc_decompress_workspace_size_batch(n)
 *                          (0 for n <= 1, when d_ws may be NULL)
 *   d_status               one device int32 for the whole call
 * Host arrays may be reused or freed when the call returns. */
ZC_API int zc_decompress_batch(uint32_t n, const void *const *d_blobs, const zc_info *infos,
                               const void *const *d_bases, void *const *d_dsts, const uint64_t *dst_capacities,
                               uint32_t flags, void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream);

/* Workspace bytes for zc_decompress_batch of n blobs (the descriptor table). */
ZC_API uint64_t zc_decompress_workspace_size_batch(uint32_t n);

/* Format v2: shared plane tables (lmzip "Building on lmz": one frequency
 * table per plane kind for many chunks). With flags = ZC_SHARED_TABLES the
 * compressor writes blob version 2: the W plane tables (256 u16 each: the
 * 12-bit table of stream j over the whole tensor, zeros for a plane with
 * fewer than two symbols) follow the chunk table and are covered by the
 * header CRC, and rANS records hold only the lane states and the words.
 * Every other rule (grouping, CONST/RAW/RANS choice per stream, the chunk
 * threshold, CRCs) is that of v1. zc_decompress, zc_decompress_delta and
 * zc_decompress_batch read both versions (zc_info.version); a batch must
 * not mix them. The decoder builds each plane's one-level table once per
 * CTA and shares it among the CTA's chunks.
 *   zc_compress_ex        zc_compress with flags: 0, ZC_SHARED_TABLES or
 *                         ZC_LANE_WORDS (the format), each with ZC_PACKED
 *                         or not (the launch shape)
 *   zc_workspace_size_ex  its workspace (v2 holds a whole tensor's
 *                         statistics in one wave)
 *   zc_blob_size_ex       worst-case blob bytes (v2 adds 512 W) */
ZC_API int zc_compress_ex(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                          uint32_t chunk_bytes, double threshold, uint32_t flags,
                          void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                          void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream);
ZC_API uint64_t zc_workspace_size_ex(uint64_t nbytes, int dtype, uint32_t chunk_bytes, uint32_t flags);
ZC_API uint64_t zc_blob_size_ex(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold, uint32_t flags);

/* zlib-compatible CRC-32 of each piece_bytes-byte piece of a device buffer,
 * the last piece possibly shorter (cuZipNN API hash_tensor_with_crc32,
 * checksum_chunk_bytes). piece_bytes = 0 means one CRC of the whole buffer.
 * d_out receives ceil(nbytes / piece_bytes) uint32 values (1 for
 * piece_bytes = 0; none for nbytes = 0 with pieces); it is zeroed on the
 * stream by this call before the kernel runs. */
ZC_API int zc_crc32(const void *d_data, uint64_t nbytes, uint64_t piece_bytes, uint32_t *d_out, void *stream);

/* Test hooks, for the library's own tests of its bounded waits (not for
 * use in production). Every device wait of the library gives up after a
 * limit and reports ZC_ETIMEOUT instead of hanging; these hooks make a wait
 * run out on purpose, with a short limit (about a millisecond), so that a
 * test can check that the kernel then returns and reports it.
 *   ZC_HOOK_LOOKBACK_STALL  compression: the first chunk of each tensor
 *                           never publishes its offset, so the other chunks'
 *                           offset-scan (look-back) waits run out; those
 *                           chunks are not written
 *   ZC_HOOK_PRODUCER_STALL  decompression: the warp that runs a chunk's rANS
 *                           lanes stops before it signals anything, so the
 *                           partner warp's barrier wait runs out
 * zc_set_test_hooks sets the hooks (0 = none, the default) for the calls
 * that the process makes afterwards, from any thread. */
#define ZC_HOOK_LOOKBACK_STALL 1u
#define ZC_HOOK_PRODUCER_STALL 2u
ZC_API void zc_set_test_hooks(uint32_t hooks);

/* Compression without any device allocation: the same work and the same
 * output as zc_compress, but the workspace comes from a fixed 64 MiB scratch
 * array that the library keeps in device memory (none of the source pages
 * has a counterpart to this entry point). It is for callers that cannot
 * allocate device memory, such as a service whose memory is all owned by
 * another allocator, or a runtime that forbids allocations after start-up;
 * the caller still provides the input, the blob, d_blob_bytes and d_status
 * exactly as for zc_compress.
 *   Limit: at most 1,048,576 chunks (nbytes <= 2^20 * chunk_bytes);
 *   larger tensors are rejected with ZC_ECAPACITY before any launch.
 *   The scratch array occupies 64 MiB on every device where this part of the
 *   library is loaded, until the process exits.
 *   All calls share the array: calls that may overlap on the GPU (different
 *   streams, or unordered host threads) race and must be ordered by the
 *   caller.
 *   The first call on a device looks up the array's address on that device;
 *   make that first call before starting any stream capture. Under CUDA's
 *   lazy module loading (the default) that first call also loads this part
 *   of the library and so commits the 64 MiB: a caller whose memory pool
 *   reserves all free device memory at start-up should make it before the
 *   pool does. The address is kept for the rest of the process; after
 *   cudaDeviceReset this entry point must not be used on that device again.
 *   Arguments are checked as in zc_compress first (ZC_EINVAL), then the
 *   chunk limit (ZC_ECAPACITY). The 64 MiB holds the offset-scan words and
 *   a wave of per-chunk statistics with a coding warp per chunk (about 250
 *   chunks of 128 KiB FP32); a larger tensor is compressed in several waves
 *   on the stream. */
ZC_API int zc_compress_noalloc(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                               uint32_t chunk_bytes, double threshold,
                               void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                               int32_t *d_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif
