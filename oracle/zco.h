/*
 * zco — the CPU oracle for byte-grouped, per-chunk order-0 rANS compression
 * of float model tensors.
 *
 * TEST INFRASTRUCTURE ONLY. This plain, single-threaded, scalar C program
 * defines the blob format and the exact bytes a compressor must produce.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it. The GPU library shares no code, header, table or constant
 * with it, and it never calls the GPU library.
 *
 * Sources (web pages; cited by title and section):
 *   [ZipNN]  "nucleation NOTE-241: ZipNN" — Method steps 1-5 (exponent
 *            extraction, byte grouping, entropy-only coding, chunking with a
 *            metadata map), Key insight (order-0 statistics), Table II.
 *   [cuZipNN] "cuZipNN 0.1.0" (PyPI) — API section: chunk_bytes,
 *            passthrough_threshold, CRC-32 helpers matching zlib.crc32;
 *            Usage/Blob format sections: blob records dtype, shape, version.
 *   [lmz]    "lmzip 1.3.0" (PyPI metadata) — "On a GPU" / "Building on lmz":
 *            interleaved rANS states per stream, a frequency table per stream.
 * The pages give no byte layout and no rANS parameters; every such choice is
 * a reading, stated where it is made in zco.c.
 */
#ifndef ZCO_H
#define ZCO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes stored in the blob header */
enum { ZCO_U8 = 1, ZCO_U16 = 2, ZCO_U32 = 3, ZCO_BF16 = 4, ZCO_FP16 = 5, ZCO_FP32 = 6 };

/* status bits (OR-ed) */
enum {
    ZCO_OK = 0, ZCO_EINVAL = 1, ZCO_EFORMAT = 2, ZCO_ECRC = 4,
    ZCO_ECORRUPT = 8, ZCO_ECAPACITY = 32
};

/* decode flag: skip the per-chunk CRC check */
enum { ZCO_NO_VERIFY = 1 };

/* Stream modes in a grouped chunk's directory. */
enum { ZCO_MODE_RAW = 0, ZCO_MODE_RANS = 1, ZCO_MODE_CONST = 2 };

/* Bytes per element for a dtype code, or 0 if the code is unknown. */
int zco_word_bytes(int dtype);

/* zlib CRC-32 (reflected 0xEDB88320, init and final xor 0xFFFFFFFF),
 * computed bit by bit. */
uint32_t zco_crc32(const uint8_t *p, uint64_t n);

/* Exponent extraction + byte grouping of n_elem words (little-endian in
 * src) into W streams of n_elem bytes each: streams[j*n_elem + i] is byte j
 * (counted from the most significant byte) of the permuted word i. */
void zco_group_split(const uint8_t *src, uint64_t n_elem, int dtype, uint8_t *streams);
/* Inverse of zco_group_split. */
void zco_group_merge(const uint8_t *streams, uint64_t n_elem, int dtype, uint8_t *dst);

/* 12-bit quantised frequency table from a 256-bin histogram of n symbols
 * (at least two distinct symbols). Writes f[256]; returns 0 or ZCO_EINVAL. */
int zco_normalize(const uint32_t counts[256], uint32_t n, uint32_t f[256]);

/* Encode one stream of n symbols into an rANS record (states, table, words).
 * Returns the record's unpadded byte count, or 0 if rec_cap is too small or
 * the stream has fewer than two distinct symbols. */
uint64_t zco_rans_record(const uint8_t *sym, uint32_t n, uint8_t *rec, uint64_t rec_cap);
/* Decode an rANS record of rec_bytes bytes into n symbols. Returns status. */
int zco_rans_decode(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, uint8_t *sym);

/* Encode one chunk (len bytes, a multiple of the word size) into its stored
 * payload. *mode_raw is set to 1 for a RAW chunk. Returns the stored byte
 * count (unpadded), or 0 on error (cap too small). */
uint64_t zco_encode_chunk(const uint8_t *src, uint32_t len, int dtype, double threshold,
                          uint8_t *out, uint64_t cap, int *mode_raw);

/* Worst-case blob size for these parameters. */
uint64_t zco_blob_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold);

/* Compress a tensor. Returns status; *blob_bytes receives the blob length. */
int zco_compress(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                 uint32_t chunk_bytes, double threshold,
                 uint8_t *blob, uint64_t cap, uint64_t *blob_bytes);

/* Parse and check a blob header and chunk table (format v1 or v2; for v2
 * also the plane tables). Fills the optional out fields. Returns status. */
int zco_blob_info(const uint8_t *blob, uint64_t avail, int *dtype, int *ndim, int64_t shape[8],
                  uint64_t *nbytes, uint32_t *n_chunks, uint32_t *chunk_bytes, uint64_t *blob_bytes);

/* Format v2 (shared plane tables). 12-bit table from 64-bit counts, by the
 * zco_normalize rule. */
int zco_normalize64(const uint64_t counts[256], uint64_t n, uint32_t f[256]);
/* The W plane tables of a tensor (planes[256 j + s]); zeros for a plane
 * with fewer than two distinct symbols. */
int zco_plane_tables(const uint8_t *src, uint64_t nbytes, int dtype, uint32_t chunk_bytes, uint32_t *planes);
/* v2 record (32 states + words) of n symbols with table f; 0 on error. */
uint64_t zco_rans_record_shared(const uint8_t *sym, uint32_t n, const uint32_t f[256], uint8_t *rec,
                                uint64_t rec_cap);
/* Inverse of zco_rans_record_shared. Returns status. */
int zco_rans_decode_shared(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, const uint32_t f[256],
                           uint8_t *sym);
/* One chunk in format v2 (coded streams use the plane tables). */
uint64_t zco_encode_chunk_shared(const uint8_t *src, uint32_t len, int dtype, double threshold,
                                 const uint32_t *planes, uint8_t *out, uint64_t cap, int *mode_raw);
/* Format v3 (a word list per lane): the record of zco_rans_record's steps
 * with each lane's words in a list of its own (counts, then the lists, each
 * padded to 8 words), and its inverse. */
uint64_t zco_rans_record_lanes(const uint8_t *sym, uint32_t n, uint8_t *rec, uint64_t rec_cap);
int zco_rans_decode_lanes(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, uint8_t *sym);
uint64_t zco_encode_chunk_lanes(const uint8_t *src, uint32_t len, int dtype, double threshold,
                                uint8_t *out, uint64_t cap, int *mode_raw);
/* Worst-case blob size of format version 1, 2 or 3. */
uint64_t zco_blob_size_v(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold, int version);
/* Compress a tensor in format version 1, 2 or 3. */
int zco_compress_v(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                   uint32_t chunk_bytes, double threshold, int version,
                   uint8_t *blob, uint64_t cap, uint64_t *blob_bytes);
/* Decompress a blob into dst (capacity cap). Unless flags has
 * ZCO_NO_VERIFY, each chunk's CRC-32 over its stored bytes is checked before
 * the chunk is decoded; a chunk that fails is reported (ZCO_ECRC) and not
 * decoded. Returns status. */
int zco_decompress(const uint8_t *blob, uint64_t blob_len, uint8_t *dst, uint64_t cap, uint32_t flags);
/* Check a blob's header, table and every chunk CRC without decoding it.
 * Returns status (ZCO_OK, ZCO_EFORMAT or ZCO_ECRC bits). */
int zco_verify(const uint8_t *blob, uint64_t blob_len);

#ifdef __cplusplus
}
#endif
#endif
