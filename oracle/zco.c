/*
 * zco.c — CPU oracle (TEST INFRASTRUCTURE ONLY; see zco.h).
 *
 * Plain single-threaded scalar C. Every step follows the pages in the order
 * they give it; no blocking, fusion or reordering. The GPU library
 * (entropy_coding_gb300/csrc) shares nothing with this file.
 *
 * Blob format v1 (all integers little-endian; the pages give no layout, so
 * this whole layout is a reading — cuZipNN "Blob format" only fixes that a
 * blob carries dtype, shape and a format version that other versions reject):
 *
 *   off  size  field
 *   0    4     magic "ZCNN"
 *   4    2     version = 1
 *   6    1     dtype code
 *   7    1     ndim (0..8)
 *   8    4     chunk_bytes
 *   12   1     lanes = 32
 *   13   1     prob_bits = 12
 *   14   2     reserved = 0
 *   16   8     nbytes (original)
 *   24   4     n_chunks = ceil(nbytes / chunk_bytes)
 *   28   4     header_crc: CRC-32 of bytes [0, 96 + 16*n_chunks) with this
 *              field read as zero
 *   32   64    shape[8] as int64, unused dims zero
 *   96   16*n  chunk table: u64 offset, u32 stored | raw_flag << 31,
 *              u32 CRC-32 of the chunk's stored payload bytes (the
 *              `stored` bytes at `offset`, without the padding after them)
 *   then each chunk's payload in chunk order, zero-padded to 16 bytes;
 *   offset_0 = 96 + 16n, offset_{c+1} = offset_c + pad16(stored_c).
 *
 *   RAW chunk payload: the chunk's original bytes.
 *   GROUPED chunk payload: W x u32 directory entries (mode << 30 | v),
 *   zero-padded to 16, then for each stream in order its record padded to 16:
 *     mode RAW   (0): v = n, record = the stream's n bytes
 *     mode RANS  (1): v = unpadded record bytes
 *     mode CONST (2): v = the symbol, no record
 *   RANS record: 32 x u32 final encoder states (lane 0 first); 32-byte
 *   presence bitmap (bit s at byte s>>3, bit s&7); k x u16 frequencies of the
 *   present symbols in ascending order; zero pad to 16; then the 16-bit
 *   renormalisation words in the order the encoder emitted them (a decoder
 *   consumes them from the last one backwards).
 *
 * Blob format v3 (a word list per lane) differs from v1 in the RANS record
 * only: after v1's head (32 final states, presence bitmap, frequencies, zero
 * pad to 16) come 32 x u16 word counts c_0 .. c_31, then for lane 0 .. 31
 * the c_l words that lane emitted, in the order it emitted them (a decoder
 * consumes each list from its end backwards), each list zero-padded to a
 * multiple of 8 words (16 bytes, so that a lane reads its list in aligned
 * 16-byte blocks). Record bytes = head + 64 + 2 * sum pad8(c_l).
 *
 * Blob format v2 (shared tables; lmz "Building on lmz": one table per plane
 * kind for many chunks) differs from v1 in three places only:
 *   - version = 2;
 *   - after the chunk table come W plane tables of 256 x u16 (512 bytes
 *     each): plane j's 12-bit table, or all zeros when stream j has fewer
 *     than two distinct symbols over the whole tensor; the header CRC covers
 *     bytes [0, 96 + 16*n_chunks + 512*W) and offset_0 = 96 + 16n + 512W;
 *   - a RANS record is the 32 final states followed by the words (no bitmap,
 *     no frequencies): the stream is coded with its plane's table.
 */
#include "zco.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ZCO_HEADER 96u
#define ZCO_ENTRY 16u
#define ZCO_LANES 32u
#define ZCO_PROB_BITS 12u
#define ZCO_M (1u << ZCO_PROB_BITS) /* 4096 */
#define ZCO_L (1u << 16)            /* lower bound of the rANS state */
#define ZCO_REC_HEAD 160u           /* 32 states + 32-byte bitmap */

static uint64_t pad16(uint64_t x) { return (x + 15u) & ~(uint64_t)15u; }

static void put16(uint8_t *p, uint32_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put32(uint8_t *p, uint32_t v) {
    for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static void put64(uint8_t *p, uint64_t v) {
    for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get16(const uint8_t *p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t get32(const uint8_t *p) {
    uint32_t v = 0;
    for (int i = 3; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}
static uint64_t get64(const uint8_t *p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}

int zco_word_bytes(int dtype) {
    switch (dtype) {
    case ZCO_U8: return 1;
    case ZCO_U16: case ZCO_BF16: case ZCO_FP16: return 2;
    case ZCO_U32: case ZCO_FP32: return 4;
    default: return 0;
    }
}

/* Exponent width of the float dtypes; 0 means plain byte grouping. */
static int exp_bits(int dtype) {
    switch (dtype) {
    case ZCO_BF16: case ZCO_FP32: return 8;
    case ZCO_FP16: return 5;
    default: return 0;
    }
}

/* ---------------------------------------------------------------- CRC-32 */

/* cuZipNN, API "compress_tensor_with_crc32": checksums match zlib.crc32.
 * That is CRC-32 with the reflected polynomial 0xEDB88320, register preset
 * to all ones and complemented at the end; done here one bit at a time. */
uint32_t zco_crc32(const uint8_t *p, uint64_t n) {
    uint32_t c = 0xFFFFFFFFu;
    for (uint64_t i = 0; i < n; i++) {
        c ^= p[i];
        for (int b = 0; b < 8; b++) c = (c & 1u) ? (c >> 1) ^ 0xEDB88320u : (c >> 1);
    }
    return c ^ 0xFFFFFFFFu;
}

/* ------------------------------------------- exponent extraction + grouping */

/* ZipNN, Method 1 "Exponent extraction": move every exponent into its own
 * byte stream; Method 2 "Byte grouping": one stream per byte position.
 * Reading (the bit-layout figures are not reproduced on the page): the
 * exponent goes to the top of the word, the sign directly below it, the
 * mantissa stays in place. For BF16 and FP32 the exponent then fills the most
 * significant byte on its own; Table II's clean-FP32 rows (last group 0.0%)
 * need the low mantissa bytes untouched, which this layout keeps. */
static uint32_t permute_word(uint32_t w, int dtype) {
    int E = exp_bits(dtype);
    if (E == 0) return w;
    int B = 8 * zco_word_bytes(dtype);
    uint32_t s = (w >> (B - 1)) & 1u;
    uint32_t e = (w >> (B - 1 - E)) & ((1u << E) - 1u);
    uint32_t m = w & ((1u << (B - 1 - E)) - 1u);
    return (e << (B - E)) | (s << (B - E - 1)) | m;
}

static uint32_t unpermute_word(uint32_t p, int dtype) {
    int E = exp_bits(dtype);
    if (E == 0) return p;
    int B = 8 * zco_word_bytes(dtype);
    uint32_t e = (p >> (B - E)) & ((1u << E) - 1u);
    uint32_t s = (p >> (B - E - 1)) & 1u;
    uint32_t m = p & ((1u << (B - 1 - E)) - 1u);
    return (s << (B - 1)) | (e << (B - 1 - E)) | m;
}

static uint32_t load_word(const uint8_t *p, int W) {
    uint32_t w = 0;
    for (int b = W - 1; b >= 0; b--) w = (w << 8) | p[b];
    return w;
}

static void store_word(uint8_t *p, int W, uint32_t w) {
    for (int b = 0; b < W; b++) p[b] = (uint8_t)(w >> (8 * b));
}

void zco_group_split(const uint8_t *src, uint64_t n_elem, int dtype, uint8_t *streams) {
    int W = zco_word_bytes(dtype);
    for (uint64_t i = 0; i < n_elem; i++) {
        uint32_t p = permute_word(load_word(src + (uint64_t)W * i, W), dtype);
        for (int j = 0; j < W; j++) /* stream j = byte j counted from the MSB */
            streams[(uint64_t)j * n_elem + i] = (uint8_t)(p >> (8 * (W - 1 - j)));
    }
}

void zco_group_merge(const uint8_t *streams, uint64_t n_elem, int dtype, uint8_t *dst) {
    int W = zco_word_bytes(dtype);
    for (uint64_t i = 0; i < n_elem; i++) {
        uint32_t p = 0;
        for (int j = 0; j < W; j++) p = (p << 8) | streams[(uint64_t)j * n_elem + i];
        store_word(dst + (uint64_t)W * i, W, unpermute_word(p, dtype));
    }
}

/* ------------------------------------------------ frequency normalisation */

/* A 12-bit quantised table (frequencies sum to 4096) from order-0 counts.
 * ZipNN Key insight: the gain is all order-0, single-symbol statistics; lmz
 * "Building on lmz": each rANS stream carries its own frequency table. The
 * pages do not give a quantisation rule; the one used (a reading) is:
 *   1. f_s = 0 for an absent symbol, else max(1, floor(c_s * 4096 / n));
 *   2. any shortfall 4096 - sum goes to the most frequent symbol (lowest s
 *      on ties);
 *   3. while the sum is above 4096, take one from the largest f_s among
 *      those above 1 (lowest s on ties). */
int zco_normalize(const uint32_t counts[256], uint32_t n, uint32_t f[256]) {
    uint64_t total = 0;
    int present = 0;
    for (int s = 0; s < 256; s++) {
        total += counts[s];
        if (counts[s]) present++;
    }
    if (total != n || present < 2) return ZCO_EINVAL;

    int64_t sum = 0;
    for (int s = 0; s < 256; s++) {
        if (counts[s] == 0) {
            f[s] = 0;
        } else {
            uint64_t q = (uint64_t)counts[s] * ZCO_M / n;
            f[s] = q < 1 ? 1u : (uint32_t)q;
        }
        sum += f[s];
    }
    if (sum < (int64_t)ZCO_M) {
        int best = 0;
        for (int s = 1; s < 256; s++)
            if (counts[s] > counts[best]) best = s;
        f[best] += (uint32_t)((int64_t)ZCO_M - sum);
        sum = ZCO_M;
    }
    while (sum > (int64_t)ZCO_M) {
        int best = -1;
        for (int s = 0; s < 256; s++)
            if (f[s] > 1 && (best < 0 || f[s] > f[best])) best = s;
        f[best] -= 1;
        sum -= 1;
    }
    return ZCO_OK;
}

/* --------------------------------------------------------------- rANS */

/* Interleaved rANS (lmz "On a GPU": one stream is several interleaved rANS
 * states, each a lane of work). Parameters, a reading since the pages name
 * none: 32 lanes, symbol i on lane i mod 32; 32-bit state kept in
 * [2^16, 2^32); 12-bit probabilities; 16-bit renormalisation words, at most
 * one per symbol.
 *
 * Encoding walks the symbols from last to first (steps T-1 .. 0, lanes
 * 31 .. 0 within a step). Before coding symbol s a lane whose state has
 * reached f_s * 2^20 writes its low 16 bits out and shifts them away; then
 * x <- floor(x / f_s) * 4096 + (x mod f_s) + cum_s. */
uint64_t zco_rans_record(const uint8_t *sym, uint32_t n, uint8_t *rec, uint64_t rec_cap) {
    uint32_t counts[256] = {0}, f[256], cum[257];
    for (uint32_t i = 0; i < n; i++) counts[sym[i]]++;
    if (zco_normalize(counts, n, f) != ZCO_OK) return 0;
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];

    uint32_t k = 0;
    for (int s = 0; s < 256; s++) k += f[s] ? 1u : 0u;
    uint64_t words_at = ZCO_REC_HEAD + pad16(2u * (uint64_t)k);
    if (rec_cap < words_at) return 0;
    memset(rec, 0, (size_t)words_at);

    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) x[l] = ZCO_L;
    uint64_t nwords = 0;
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;
    for (uint32_t t = T; t-- > 0;) {
        for (uint32_t l = ZCO_LANES; l-- > 0;) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t s = sym[i];
            if (x[l] >= (f[s] << 20)) {
                if (words_at + 2 * (nwords + 1) > rec_cap) return 0;
                put16(rec + words_at + 2 * nwords, x[l] & 0xFFFFu);
                nwords++;
                x[l] >>= 16;
            }
            x[l] = ((x[l] / f[s]) << ZCO_PROB_BITS) + (x[l] % f[s]) + cum[s];
        }
    }

    for (uint32_t l = 0; l < ZCO_LANES; l++) put32(rec + 4 * l, x[l]);
    uint8_t *bitmap = rec + 4 * ZCO_LANES;
    uint8_t *freqs = bitmap + 32;
    uint32_t j = 0;
    for (int s = 0; s < 256; s++) {
        if (!f[s]) continue;
        bitmap[s >> 3] |= (uint8_t)(1u << (s & 7));
        put16(freqs + 2 * j, f[s]);
        j++;
    }
    return words_at + 2 * nwords;
}

/* Decoding runs the steps forward (steps 0 .. T-1, lanes 0 .. 31): the slot
 * x mod 4096 names the symbol s with cum_s <= slot < cum_s + f_s; then
 * x <- f_s * (x >> 12) + slot - cum_s, and a state that fell below 2^16 takes
 * in the next word, read from the end of the word list backwards. A valid
 * record ends with every state at 2^16 and every word consumed. */
int zco_rans_decode(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, uint8_t *sym) {
    if (rec_bytes < ZCO_REC_HEAD) return ZCO_ECORRUPT;
    const uint8_t *bitmap = rec + 4 * ZCO_LANES;
    const uint8_t *freqs = bitmap + 32;
    uint32_t f[256], cum[257];
    uint32_t k = 0;
    for (int s = 0; s < 256; s++) k += (bitmap[s >> 3] >> (s & 7)) & 1u;
    uint64_t words_at = ZCO_REC_HEAD + pad16(2u * (uint64_t)k);
    if (k < 2 || rec_bytes < words_at || ((rec_bytes - words_at) & 1u)) return ZCO_ECORRUPT;
    for (uint64_t b = ZCO_REC_HEAD + 2u * k; b < words_at; b++)
        if (rec[b]) return ZCO_ECORRUPT;
    uint32_t j = 0;
    for (int s = 0; s < 256; s++) {
        f[s] = 0;
        if ((bitmap[s >> 3] >> (s & 7)) & 1u) {
            f[s] = get16(freqs + 2 * j);
            j++;
            if (f[s] == 0 || f[s] >= ZCO_M) return ZCO_ECORRUPT;
        }
    }
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];
    if (cum[256] != ZCO_M) return ZCO_ECORRUPT;

    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) {
        x[l] = get32(rec + 4 * l);
        if (x[l] < ZCO_L) return ZCO_ECORRUPT;
    }
    const uint8_t *words = rec + words_at;
    uint64_t ptr = (rec_bytes - words_at) / 2; /* words left to consume */
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;
    for (uint32_t t = 0; t < T; t++) {
        for (uint32_t l = 0; l < ZCO_LANES; l++) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t slot = x[l] & (ZCO_M - 1);
            uint32_t s = 0;
            while (!(cum[s] <= slot && slot < cum[s + 1])) s++;
            x[l] = f[s] * (x[l] >> ZCO_PROB_BITS) + slot - cum[s];
            if (x[l] < ZCO_L) {
                if (ptr == 0) return ZCO_ECORRUPT;
                ptr--;
                x[l] = (x[l] << 16) | get16(words + 2 * ptr);
            }
            sym[i] = (uint8_t)s;
        }
    }
    for (uint32_t l = 0; l < ZCO_LANES; l++)
        if (x[l] != ZCO_L) return ZCO_ECORRUPT;
    if (ptr != 0) return ZCO_ECORRUPT;
    return ZCO_OK;
}

/* ------------------------------------------ format v3: a word list per lane */

/* lmz "On a GPU": a GPU rANS decoder is bound by the dependent chain of each
 * lane's steps. With one word list for all lanes (v1), where a lane's next
 * word lies depends on how many words the lanes before it took in the same
 * step, so every step of every lane also waits on the other lanes. A v3
 * record gives each lane its own list (see the top of this file); the coding
 * steps are exactly zco_rans_record's, only the place a word is written
 * differs. */
static uint64_t pad8w(uint64_t words) { return (words + 7u) & ~(uint64_t)7u; }

uint64_t zco_rans_record_lanes(const uint8_t *sym, uint32_t n, uint8_t *rec, uint64_t rec_cap) {
    uint32_t counts[256] = {0}, f[256], cum[257];
    for (uint32_t i = 0; i < n; i++) counts[sym[i]]++;
    if (zco_normalize(counts, n, f) != ZCO_OK) return 0;
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];

    uint32_t k = 0;
    for (int s = 0; s < 256; s++) k += f[s] ? 1u : 0u;
    const uint64_t head = ZCO_REC_HEAD + pad16(2u * (uint64_t)k);
    const uint64_t lists_at = head + 2u * ZCO_LANES;
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;

    /* each lane's words in the order it emits them */
    uint16_t *lw = (uint16_t *)malloc(((size_t)ZCO_LANES * T + 1) * sizeof(uint16_t));
    if (!lw) return 0;
    uint32_t c[ZCO_LANES] = {0};
    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) x[l] = ZCO_L;
    for (uint32_t t = T; t-- > 0;) {
        for (uint32_t l = ZCO_LANES; l-- > 0;) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t s = sym[i];
            if (x[l] >= (f[s] << 20)) {
                lw[(uint64_t)l * T + c[l]] = (uint16_t)(x[l] & 0xFFFFu);
                c[l]++;
                x[l] >>= 16;
            }
            x[l] = ((x[l] / f[s]) << ZCO_PROB_BITS) + (x[l] % f[s]) + cum[s];
        }
    }

    uint64_t size = lists_at;
    for (uint32_t l = 0; l < ZCO_LANES; l++) size += 2u * pad8w(c[l]);
    if (size > rec_cap) {
        free(lw);
        return 0;
    }
    memset(rec, 0, (size_t)size);
    for (uint32_t l = 0; l < ZCO_LANES; l++) put32(rec + 4 * l, x[l]);
    uint8_t *bitmap = rec + 4 * ZCO_LANES;
    uint8_t *freqs = bitmap + 32;
    uint32_t j = 0;
    for (int s = 0; s < 256; s++) {
        if (!f[s]) continue;
        bitmap[s >> 3] |= (uint8_t)(1u << (s & 7));
        put16(freqs + 2 * j, f[s]);
        j++;
    }
    uint64_t off = lists_at;
    for (uint32_t l = 0; l < ZCO_LANES; l++) {
        put16(rec + head + 2 * l, c[l]);
        for (uint32_t q = 0; q < c[l]; q++) put16(rec + off + 2u * q, lw[(uint64_t)l * T + q]);
        off += 2u * pad8w(c[l]);
    }
    free(lw);
    return size;
}

/* Inverse of zco_rans_record_lanes: zco_rans_decode's steps, with lane l
 * taking its words from the end of its own list backwards. The counts must
 * describe the record exactly and the padding must be zero. */
int zco_rans_decode_lanes(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, uint8_t *sym) {
    if (rec_bytes < ZCO_REC_HEAD) return ZCO_ECORRUPT;
    const uint8_t *bitmap = rec + 4 * ZCO_LANES;
    const uint8_t *freqs = bitmap + 32;
    uint32_t f[256], cum[257];
    uint32_t k = 0;
    for (int s = 0; s < 256; s++) k += (bitmap[s >> 3] >> (s & 7)) & 1u;
    const uint64_t head = ZCO_REC_HEAD + pad16(2u * (uint64_t)k);
    const uint64_t lists_at = head + 2u * ZCO_LANES;
    if (k < 2 || rec_bytes < lists_at) return ZCO_ECORRUPT;
    for (uint64_t b = ZCO_REC_HEAD + 2u * k; b < head; b++)
        if (rec[b]) return ZCO_ECORRUPT;
    uint32_t j = 0;
    for (int s = 0; s < 256; s++) {
        f[s] = 0;
        if ((bitmap[s >> 3] >> (s & 7)) & 1u) {
            f[s] = get16(freqs + 2 * j);
            j++;
            if (f[s] == 0 || f[s] >= ZCO_M) return ZCO_ECORRUPT;
        }
    }
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];
    if (cum[256] != ZCO_M) return ZCO_ECORRUPT;

    uint64_t base[ZCO_LANES], left[ZCO_LANES];
    uint64_t off = lists_at;
    for (uint32_t l = 0; l < ZCO_LANES; l++) {
        uint32_t c = get16(rec + head + 2 * l);
        base[l] = off;
        left[l] = c;
        off += 2u * pad8w(c);
        if (off > rec_bytes) return ZCO_ECORRUPT;
        for (uint64_t q = c; q < pad8w(c); q++)
            if (get16(rec + base[l] + 2u * q)) return ZCO_ECORRUPT;
    }
    if (off != rec_bytes) return ZCO_ECORRUPT;

    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) {
        x[l] = get32(rec + 4 * l);
        if (x[l] < ZCO_L) return ZCO_ECORRUPT;
    }
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;
    for (uint32_t t = 0; t < T; t++) {
        for (uint32_t l = 0; l < ZCO_LANES; l++) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t slot = x[l] & (ZCO_M - 1);
            uint32_t s = 0;
            while (!(cum[s] <= slot && slot < cum[s + 1])) s++;
            x[l] = f[s] * (x[l] >> ZCO_PROB_BITS) + slot - cum[s];
            if (x[l] < ZCO_L) {
                if (left[l] == 0) return ZCO_ECORRUPT;
                left[l]--;
                x[l] = (x[l] << 16) | get16(rec + base[l] + 2u * left[l]);
            }
            sym[i] = (uint8_t)s;
        }
    }
    for (uint32_t l = 0; l < ZCO_LANES; l++)
        if (x[l] != ZCO_L || left[l] != 0) return ZCO_ECORRUPT;
    return ZCO_OK;
}

/* ---------------------------------------------------------------- chunks */

/* ZipNN Method 3: all-zero streams are truncated to a header (generalised
 * here to any constant stream); cuZipNN API passthrough_threshold: data is
 * kept coded only if it shrinks below threshold x its raw size, otherwise it
 * is stored raw. Reading: the rule is applied per stream (Table II shows
 * incompressible groups at 100% beside a coded exponent) and again per chunk
 * (an incompressible chunk then decodes as a copy); "below" is strict and the
 * comparison is in IEEE double. */
static uint64_t encode_chunk_v(const uint8_t *src, uint32_t len, int dtype, double threshold,
                               uint8_t *out, uint64_t cap, int *mode_raw, int lanes);

uint64_t zco_encode_chunk(const uint8_t *src, uint32_t len, int dtype, double threshold,
                          uint8_t *out, uint64_t cap, int *mode_raw) {
    return encode_chunk_v(src, len, dtype, threshold, out, cap, mode_raw, 0);
}

/* One chunk in format v3 (a word list per lane in every RANS record). */
uint64_t zco_encode_chunk_lanes(const uint8_t *src, uint32_t len, int dtype, double threshold,
                                uint8_t *out, uint64_t cap, int *mode_raw) {
    return encode_chunk_v(src, len, dtype, threshold, out, cap, mode_raw, 1);
}

static uint64_t encode_chunk_v(const uint8_t *src, uint32_t len, int dtype, double threshold,
                               uint8_t *out, uint64_t cap, int *mode_raw, int lanes) {
    int W = zco_word_bytes(dtype);
    uint32_t n = len / (uint32_t)W;
    uint8_t *streams = (uint8_t *)malloc(len ? len : 1);
    /* v1: head + table + one word per symbol at most; v3 adds the counts and
     * the padding of each list to 8 words */
    uint64_t rec_cap = ZCO_REC_HEAD + 512u + 2u * (uint64_t)n + (lanes ? 64u + 16u * ZCO_LANES : 0u);
    uint8_t *rec = (uint8_t *)malloc((size_t)rec_cap);
    uint8_t *grouped = (uint8_t *)malloc((size_t)(16 + (uint64_t)W * pad16(rec_cap)));
    uint64_t result = 0;
    if (!streams || !rec || !grouped) goto done;

    zco_group_split(src, n, dtype, streams);

    uint64_t g = pad16(4u * (uint64_t)W);
    memset(grouped, 0, (size_t)g);
    for (int j = 0; j < W; j++) {
        const uint8_t *sj = streams + (uint64_t)j * n;
        uint32_t counts[256] = {0};
        for (uint32_t i = 0; i < n; i++) counts[sj[i]]++;
        int present = 0, only = 0;
        for (int s = 0; s < 256; s++)
            if (counts[s]) { present++; only = s; }

        uint32_t entry;
        if (present == 1) {
            entry = ((uint32_t)ZCO_MODE_CONST << 30) | (uint32_t)only;
        } else {
            uint64_t r = lanes ? zco_rans_record_lanes(sj, n, rec, rec_cap) : zco_rans_record(sj, n, rec, rec_cap);
            if (r == 0) goto done;
            if ((double)r < threshold * (double)n) {
                entry = ((uint32_t)ZCO_MODE_RANS << 30) | (uint32_t)r;
                memcpy(grouped + g, rec, (size_t)r);
                memset(grouped + g + r, 0, (size_t)(pad16(r) - r));
                g += pad16(r);
            } else {
                entry = ((uint32_t)ZCO_MODE_RAW << 30) | n;
                memcpy(grouped + g, sj, n);
                memset(grouped + g + n, 0, (size_t)(pad16(n) - n));
                g += pad16(n);
            }
        }
        put32(grouped + 4 * j, entry);
    }

    if ((double)g < threshold * (double)len) {
        if (g > cap) goto done;
        memcpy(out, grouped, (size_t)g);
        *mode_raw = 0;
        result = g;
    } else {
        if (len > cap) goto done;
        memcpy(out, src, len);
        *mode_raw = 1;
        result = len;
    }
done:
    free(streams);
    free(rec);
    free(grouped);
    return result;
}

/* ------------------------------------------ format v2: shared plane tables */

/* lmz "Building on lmz": a table per plane kind shared by many chunks (the
 * chunk records then carry none). Reading: plane j's table is the 12-bit
 * table of the histogram of stream j over every element of the tensor,
 * quantised by the same rule as zco_normalize (written out again here for
 * 64-bit counts, since a tensor may hold more than 2^32 elements). */
int zco_normalize64(const uint64_t counts[256], uint64_t n, uint32_t f[256]) {
    uint64_t total = 0;
    int present = 0;
    for (int s = 0; s < 256; s++) {
        total += counts[s];
        if (counts[s]) present++;
    }
    if (total != n || present < 2 || n > (1ull << 50)) return ZCO_EINVAL;

    int64_t sum = 0;
    for (int s = 0; s < 256; s++) {
        if (counts[s] == 0) {
            f[s] = 0;
        } else {
            uint64_t q = counts[s] * ZCO_M / n;
            f[s] = q < 1 ? 1u : (uint32_t)q;
        }
        sum += f[s];
    }
    if (sum < (int64_t)ZCO_M) {
        int best = 0;
        for (int s = 1; s < 256; s++)
            if (counts[s] > counts[best]) best = s;
        f[best] += (uint32_t)((int64_t)ZCO_M - sum);
        sum = ZCO_M;
    }
    while (sum > (int64_t)ZCO_M) {
        int best = -1;
        for (int s = 0; s < 256; s++)
            if (f[s] > 1 && (best < 0 || f[s] > f[best])) best = s;
        f[best] -= 1;
        sum -= 1;
    }
    return ZCO_OK;
}

/* The W plane tables of a tensor (planes[j*256 + s]), from the streams of
 * every chunk; all zeros for a plane with fewer than two distinct symbols. */
int zco_plane_tables(const uint8_t *src, uint64_t nbytes, int dtype, uint32_t chunk_bytes, uint32_t *planes) {
    int W = zco_word_bytes(dtype);
    if (W == 0 || chunk_bytes == 0 || nbytes % (uint64_t)W) return ZCO_EINVAL;
    uint64_t *counts = (uint64_t *)calloc(256u * (size_t)W, sizeof(uint64_t));
    uint8_t *streams = (uint8_t *)malloc(chunk_bytes);
    if (!counts || !streams) {
        free(counts);
        free(streams);
        return ZCO_EINVAL;
    }
    for (uint64_t off = 0; off < nbytes; off += chunk_bytes) {
        uint32_t len = (uint32_t)(nbytes - off < chunk_bytes ? nbytes - off : chunk_bytes);
        uint32_t n = len / (uint32_t)W;
        zco_group_split(src + off, n, dtype, streams);
        for (int j = 0; j < W; j++)
            for (uint32_t i = 0; i < n; i++) counts[256u * j + streams[(uint64_t)j * n + i]]++;
    }
    int st = ZCO_OK;
    for (int j = 0; j < W; j++) {
        uint32_t *f = planes + 256u * j;
        if (zco_normalize64(counts + 256u * j, nbytes / (uint64_t)W, f) != ZCO_OK)
            memset(f, 0, 256 * sizeof(uint32_t));  /* fewer than two symbols (or an empty tensor) */
    }
    free(counts);
    free(streams);
    return st;
}

/* v2 record: the same rANS steps as zco_rans_record with the plane's table
 * f; the record is the 32 final states and the words. Returns the record's
 * byte count, or 0 if rec_cap is too small or a symbol has no frequency. */
uint64_t zco_rans_record_shared(const uint8_t *sym, uint32_t n, const uint32_t f[256], uint8_t *rec,
                                uint64_t rec_cap) {
    uint32_t cum[257];
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];
    if (cum[256] != ZCO_M) return 0;
    const uint64_t words_at = 4u * ZCO_LANES;
    if (rec_cap < words_at) return 0;

    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) x[l] = ZCO_L;
    uint64_t nwords = 0;
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;
    for (uint32_t t = T; t-- > 0;) {
        for (uint32_t l = ZCO_LANES; l-- > 0;) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t s = sym[i];
            if (f[s] == 0) return 0;
            if (x[l] >= (f[s] << 20)) {
                if (words_at + 2 * (nwords + 1) > rec_cap) return 0;
                put16(rec + words_at + 2 * nwords, x[l] & 0xFFFFu);
                nwords++;
                x[l] >>= 16;
            }
            x[l] = ((x[l] / f[s]) << ZCO_PROB_BITS) + (x[l] % f[s]) + cum[s];
        }
    }
    for (uint32_t l = 0; l < ZCO_LANES; l++) put32(rec + 4 * l, x[l]);
    return words_at + 2 * nwords;
}

/* Inverse of zco_rans_record_shared (the steps of zco_rans_decode). */
int zco_rans_decode_shared(const uint8_t *rec, uint64_t rec_bytes, uint32_t n, const uint32_t f[256],
                           uint8_t *sym) {
    const uint64_t words_at = 4u * ZCO_LANES;
    uint32_t cum[257];
    cum[0] = 0;
    for (int s = 0; s < 256; s++) cum[s + 1] = cum[s] + f[s];
    if (cum[256] != ZCO_M) return ZCO_ECORRUPT;
    if (rec_bytes < words_at || ((rec_bytes - words_at) & 1u)) return ZCO_ECORRUPT;
    uint32_t x[ZCO_LANES];
    for (uint32_t l = 0; l < ZCO_LANES; l++) {
        x[l] = get32(rec + 4 * l);
        if (x[l] < ZCO_L) return ZCO_ECORRUPT;
    }
    const uint8_t *words = rec + words_at;
    uint64_t ptr = (rec_bytes - words_at) / 2;
    uint32_t T = (n + ZCO_LANES - 1) / ZCO_LANES;
    for (uint32_t t = 0; t < T; t++) {
        for (uint32_t l = 0; l < ZCO_LANES; l++) {
            uint64_t i = (uint64_t)t * ZCO_LANES + l;
            if (i >= n) continue;
            uint32_t slot = x[l] & (ZCO_M - 1);
            uint32_t s = 0;
            while (!(cum[s] <= slot && slot < cum[s + 1])) s++;
            x[l] = f[s] * (x[l] >> ZCO_PROB_BITS) + slot - cum[s];
            if (x[l] < ZCO_L) {
                if (ptr == 0) return ZCO_ECORRUPT;
                ptr--;
                x[l] = (x[l] << 16) | get16(words + 2 * ptr);
            }
            sym[i] = (uint8_t)s;
        }
    }
    for (uint32_t l = 0; l < ZCO_LANES; l++)
        if (x[l] != ZCO_L) return ZCO_ECORRUPT;
    if (ptr != 0) return ZCO_ECORRUPT;
    return ZCO_OK;
}

/* One chunk in format v2: the per-stream and per-chunk rules of
 * zco_encode_chunk, with coded streams using their plane's table. */
uint64_t zco_encode_chunk_shared(const uint8_t *src, uint32_t len, int dtype, double threshold,
                                 const uint32_t *planes, uint8_t *out, uint64_t cap, int *mode_raw) {
    int W = zco_word_bytes(dtype);
    uint32_t n = len / (uint32_t)W;
    uint8_t *streams = (uint8_t *)malloc(len ? len : 1);
    uint64_t rec_cap = 4u * ZCO_LANES + 2u * (uint64_t)n;
    uint8_t *rec = (uint8_t *)malloc((size_t)rec_cap);
    uint8_t *grouped = (uint8_t *)malloc((size_t)(16 + (uint64_t)W * pad16(rec_cap)));
    uint64_t result = 0;
    if (!streams || !rec || !grouped) goto done;

    zco_group_split(src, n, dtype, streams);

    uint64_t g = pad16(4u * (uint64_t)W);
    memset(grouped, 0, (size_t)g);
    for (int j = 0; j < W; j++) {
        const uint8_t *sj = streams + (uint64_t)j * n;
        uint32_t counts[256] = {0};
        for (uint32_t i = 0; i < n; i++) counts[sj[i]]++;
        int present = 0, only = 0;
        for (int s = 0; s < 256; s++)
            if (counts[s]) { present++; only = s; }

        uint32_t entry;
        if (present == 1) {
            entry = ((uint32_t)ZCO_MODE_CONST << 30) | (uint32_t)only;
        } else {
            uint64_t r = zco_rans_record_shared(sj, n, planes + 256u * j, rec, rec_cap);
            if (r == 0) goto done;
            if ((double)r < threshold * (double)n) {
                entry = ((uint32_t)ZCO_MODE_RANS << 30) | (uint32_t)r;
                memcpy(grouped + g, rec, (size_t)r);
                memset(grouped + g + r, 0, (size_t)(pad16(r) - r));
                g += pad16(r);
            } else {
                entry = ((uint32_t)ZCO_MODE_RAW << 30) | n;
                memcpy(grouped + g, sj, n);
                memset(grouped + g + n, 0, (size_t)(pad16(n) - n));
                g += pad16(n);
            }
        }
        put32(grouped + 4 * j, entry);
    }

    if ((double)g < threshold * (double)len) {
        if (g > cap) goto done;
        memcpy(out, grouped, (size_t)g);
        *mode_raw = 0;
        result = g;
    } else {
        if (len > cap) goto done;
        memcpy(out, src, len);
        *mode_raw = 1;
        result = len;
    }
done:
    free(streams);
    free(rec);
    free(grouped);
    return result;
}

/* --------------------------------------------------------------- blobs */

static int valid_params(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold) {
    int W = zco_word_bytes(dtype);
    if (W == 0) return 0;
    if (nbytes % (uint64_t)W) return 0;
    if (chunk_bytes < 64 || chunk_bytes > 131072 || chunk_bytes % 64) return 0;
    if (!(threshold > 0.0) || !(threshold <= 1e9)) return 0;
    if ((nbytes + chunk_bytes - 1) / chunk_bytes > 0xFFFFFFFFull) return 0;
    return 1;
}

/* Largest possible grouped payload for a chunk of len bytes; v3 records
 * also hold the word counts and up to 3 padding words per lane. */
static uint64_t max_grouped_v(uint64_t len, int W, int version) {
    uint64_t n = len / (uint64_t)W;
    uint64_t extra = version == 3 ? 64u + 14u * ZCO_LANES : 0u;
    return pad16(4u * (uint64_t)W) + (uint64_t)W * pad16(ZCO_REC_HEAD + 512u + 2u * n + extra);
}

static uint64_t blob_size_of(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold, int version) {
    if (!valid_params(nbytes, dtype, chunk_bytes, threshold)) return 0;
    int W = zco_word_bytes(dtype);
    uint64_t nc = (nbytes + chunk_bytes - 1) / chunk_bytes;
    uint64_t total = ZCO_HEADER + ZCO_ENTRY * nc;
    for (uint64_t c = 0; c < nc; c++) {
        uint64_t len = (c + 1 < nc) ? chunk_bytes : nbytes - c * chunk_bytes;
        uint64_t worst = pad16(len);
        uint64_t g = max_grouped_v(len, W, version);
        if (threshold > 1.0 && g > worst) worst = g;
        total += worst;
    }
    return total;
}

uint64_t zco_blob_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold) {
    return blob_size_of(nbytes, dtype, chunk_bytes, threshold, 1);
}

/* Worst case of any format: v2 adds the W plane tables; v3 records may be
 * longer (only reachable with threshold > 1). */
uint64_t zco_blob_size_v(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold, int version) {
    if (version < 1 || version > 3) return 0;
    uint64_t b = blob_size_of(nbytes, dtype, chunk_bytes, threshold, version);
    if (b == 0) return 0;
    return version == 2 ? b + 512u * (uint64_t)zco_word_bytes(dtype) : b;
}

/* Format v2 compression (see the top of this file). */
static int compress_shared(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                           uint32_t chunk_bytes, double threshold, uint8_t *blob, uint64_t cap,
                           uint64_t *blob_bytes) {
    int W = zco_word_bytes(dtype);
    uint64_t nc = (nbytes + chunk_bytes - 1) / chunk_bytes;
    uint64_t table_end = ZCO_HEADER + ZCO_ENTRY * nc;
    uint64_t planes_end = table_end + 512u * (uint64_t)W;
    if (cap < planes_end) return ZCO_ECAPACITY;
    uint32_t planes[4 * 256];
    if (zco_plane_tables(src, nbytes, dtype, chunk_bytes, planes) != ZCO_OK) return ZCO_EINVAL;
    memset(blob, 0, (size_t)planes_end);

    memcpy(blob, "ZCNN", 4);
    put16(blob + 4, 2);
    blob[6] = (uint8_t)dtype;
    blob[7] = (uint8_t)ndim;
    put32(blob + 8, chunk_bytes);
    blob[12] = (uint8_t)ZCO_LANES;
    blob[13] = (uint8_t)ZCO_PROB_BITS;
    put64(blob + 16, nbytes);
    put32(blob + 24, (uint32_t)nc);
    for (int d = 0; d < ndim; d++) put64(blob + 32 + 8 * d, (uint64_t)shape[d]);
    for (int j = 0; j < W; j++)
        for (int v = 0; v < 256; v++) put16(blob + table_end + 512u * j + 2u * v, planes[256 * j + v]);

    uint64_t off = planes_end;
    for (uint64_t c = 0; c < nc; c++) {
        uint32_t len = (uint32_t)((c + 1 < nc) ? chunk_bytes : nbytes - c * chunk_bytes);
        int raw = 0;
        uint64_t room = cap > off ? cap - off : 0;
        uint64_t stored = zco_encode_chunk_shared(src + c * (uint64_t)chunk_bytes, len, dtype, threshold, planes,
                                                  blob + off, room, &raw);
        if (stored == 0 || pad16(stored) > room) return ZCO_ECAPACITY;
        memset(blob + off + stored, 0, (size_t)(pad16(stored) - stored));
        uint8_t *e = blob + ZCO_HEADER + ZCO_ENTRY * c;
        put64(e, off);
        put32(e + 8, (uint32_t)stored | ((uint32_t)raw << 31));
        put32(e + 12, zco_crc32(blob + off, stored));
        off += pad16(stored);
    }
    put32(blob + 28, zco_crc32(blob, planes_end));
    *blob_bytes = off;
    return ZCO_OK;
}

static int compress_v13(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                        uint32_t chunk_bytes, double threshold, int version,
                        uint8_t *blob, uint64_t cap, uint64_t *blob_bytes);

int zco_compress_v(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                   uint32_t chunk_bytes, double threshold, int version,
                   uint8_t *blob, uint64_t cap, uint64_t *blob_bytes) {
    if (version == 1 || version == 3)
        return compress_v13(src, nbytes, dtype, ndim, shape, chunk_bytes, threshold, version, blob, cap, blob_bytes);
    if (version != 2) return ZCO_EINVAL;
    if (!valid_params(nbytes, dtype, chunk_bytes, threshold)) return ZCO_EINVAL;
    if (ndim < 0 || ndim > 8) return ZCO_EINVAL;
    int W = zco_word_bytes(dtype);
    uint64_t elems = 1;
    for (int d = 0; d < ndim; d++) {
        if (shape[d] < 0) return ZCO_EINVAL;
        elems *= (uint64_t)shape[d];
    }
    if (elems * (uint64_t)W != nbytes) return ZCO_EINVAL;
    return compress_shared(src, nbytes, dtype, ndim, shape, chunk_bytes, threshold, blob, cap, blob_bytes);
}

int zco_compress(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                 uint32_t chunk_bytes, double threshold,
                 uint8_t *blob, uint64_t cap, uint64_t *blob_bytes) {
    return compress_v13(src, nbytes, dtype, ndim, shape, chunk_bytes, threshold, 1, blob, cap, blob_bytes);
}

/* Formats v1 and v3 (they differ in the RANS records only). */
static int compress_v13(const uint8_t *src, uint64_t nbytes, int dtype, int ndim, const int64_t *shape,
                        uint32_t chunk_bytes, double threshold, int version,
                        uint8_t *blob, uint64_t cap, uint64_t *blob_bytes) {
    if (!valid_params(nbytes, dtype, chunk_bytes, threshold)) return ZCO_EINVAL;
    if (ndim < 0 || ndim > 8) return ZCO_EINVAL;
    int W = zco_word_bytes(dtype);
    uint64_t elems = 1;
    for (int d = 0; d < ndim; d++) {
        if (shape[d] < 0) return ZCO_EINVAL;
        elems *= (uint64_t)shape[d];
    }
    if (elems * (uint64_t)W != nbytes) return ZCO_EINVAL;

    uint64_t nc = (nbytes + chunk_bytes - 1) / chunk_bytes;
    uint64_t table_end = ZCO_HEADER + ZCO_ENTRY * nc;
    if (cap < table_end) return ZCO_ECAPACITY;
    memset(blob, 0, (size_t)table_end);

    memcpy(blob, "ZCNN", 4);
    put16(blob + 4, (uint32_t)version);
    blob[6] = (uint8_t)dtype;
    blob[7] = (uint8_t)ndim;
    put32(blob + 8, chunk_bytes);
    blob[12] = (uint8_t)ZCO_LANES;
    blob[13] = (uint8_t)ZCO_PROB_BITS;
    put64(blob + 16, nbytes);
    put32(blob + 24, (uint32_t)nc);
    for (int d = 0; d < ndim; d++) put64(blob + 32 + 8 * d, (uint64_t)shape[d]);

    /* ZipNN Method 5: fixed-size chunks; a metadata map records each
     * chunk's variable compressed size so chunks decode independently. The
     * map here holds offsets, which are the running sum of the padded sizes
     * of the chunks before. Each entry also carries the zlib CRC-32 of the
     * chunk's stored payload (cuZipNN API: checksums match zlib.crc32 and
     * are taken over pieces of the blob, so that an untrusted blob can be
     * checked before it is decoded). */
    uint64_t off = table_end;
    for (uint64_t c = 0; c < nc; c++) {
        uint32_t len = (uint32_t)((c + 1 < nc) ? chunk_bytes : nbytes - c * chunk_bytes);
        int raw = 0;
        uint64_t room = cap > off ? cap - off : 0;
        uint64_t stored = version == 3 ? zco_encode_chunk_lanes(src + c * (uint64_t)chunk_bytes, len, dtype,
                                                                threshold, blob + off, room, &raw)
                                       : zco_encode_chunk(src + c * (uint64_t)chunk_bytes, len, dtype, threshold,
                                                          blob + off, room, &raw);
        if (stored == 0 || pad16(stored) > room) return ZCO_ECAPACITY;
        memset(blob + off + stored, 0, (size_t)(pad16(stored) - stored));
        uint8_t *e = blob + ZCO_HEADER + ZCO_ENTRY * c;
        put64(e, off);
        put32(e + 8, (uint32_t)stored | ((uint32_t)raw << 31));
        put32(e + 12, zco_crc32(blob + off, stored));
        off += pad16(stored);
    }
    put32(blob + 28, zco_crc32(blob, table_end));
    *blob_bytes = off;
    return ZCO_OK;
}

int zco_blob_info(const uint8_t *blob, uint64_t avail, int *dtype_out, int *ndim_out,
                  int64_t shape_out[8], uint64_t *nbytes_out, uint32_t *n_chunks_out,
                  uint32_t *chunk_bytes_out, uint64_t *blob_bytes_out) {
    if (avail < ZCO_HEADER) return ZCO_EFORMAT;
    int version = (int)get16(blob + 4);
    if (memcmp(blob, "ZCNN", 4) != 0 || version < 1 || version > 3) return ZCO_EFORMAT;
    int dtype = blob[6], ndim = blob[7];
    uint32_t chunk_bytes = get32(blob + 8);
    uint64_t nbytes = get64(blob + 16);
    uint32_t nc = get32(blob + 24);
    int W = zco_word_bytes(dtype);
    if (W == 0 || ndim > 8 || blob[12] != ZCO_LANES || blob[13] != ZCO_PROB_BITS ||
        get16(blob + 14) != 0)
        return ZCO_EFORMAT;
    if (!valid_params(nbytes, dtype, chunk_bytes, 1.0)) return ZCO_EFORMAT;
    if ((uint64_t)nc != (nbytes + chunk_bytes - 1) / chunk_bytes) return ZCO_EFORMAT;
    uint64_t elems = 1;
    for (int d = 0; d < 8; d++) {
        int64_t v = (int64_t)get64(blob + 32 + 8 * d);
        if (d >= ndim) {
            if (v != 0) return ZCO_EFORMAT;
            continue;
        }
        if (v < 0) return ZCO_EFORMAT;
        elems *= (uint64_t)v;
    }
    if (elems * (uint64_t)W != nbytes) return ZCO_EFORMAT;
    uint64_t table_end = ZCO_HEADER + ZCO_ENTRY * (uint64_t)nc;
    if (version == 2) table_end += 512u * (uint64_t)W; /* the plane tables */
    if (avail < table_end) return ZCO_EFORMAT;
    if (version == 2) {
        /* each plane table is all zeros or a 12-bit table of at least two symbols */
        for (int j = 0; j < W; j++) {
            const uint8_t *t = blob + table_end - 512u * (uint64_t)(W - j);
            uint32_t sum = 0, nz = 0;
            for (int v = 0; v < 256; v++) {
                uint32_t f = get16(t + 2 * v);
                sum += f;
                nz += f ? 1u : 0u;
            }
            if (!(sum == 0 || (sum == ZCO_M && nz >= 2))) return ZCO_EFORMAT;
        }
    }

    /* header CRC with its own field read as zero */
    uint8_t *copy = (uint8_t *)malloc((size_t)table_end);
    if (!copy) return ZCO_EINVAL;
    memcpy(copy, blob, (size_t)table_end);
    put32(copy + 28, 0);
    uint32_t hcrc = zco_crc32(copy, table_end);
    free(copy);
    if (hcrc != get32(blob + 28)) return ZCO_ECRC;

    /* the table must describe exactly the packed layout */
    uint64_t off = table_end;
    for (uint32_t c = 0; c < nc; c++) {
        const uint8_t *e = blob + ZCO_HEADER + ZCO_ENTRY * (uint64_t)c;
        uint64_t len = (c + 1 < nc) ? chunk_bytes : nbytes - (uint64_t)c * chunk_bytes;
        uint32_t sm = get32(e + 8);
        uint32_t stored = sm & 0x7FFFFFFFu;
        int raw = (int)(sm >> 31);
        if (get64(e) != off) return ZCO_EFORMAT;
        if (raw && stored != len) return ZCO_EFORMAT;
        if (!raw && (stored % 16 || stored > max_grouped_v(len, W, version))) return ZCO_EFORMAT;
        off += pad16(stored);
    }
    if (dtype_out) *dtype_out = dtype;
    if (ndim_out) *ndim_out = ndim;
    if (shape_out)
        for (int d = 0; d < 8; d++) shape_out[d] = (int64_t)get64(blob + 32 + 8 * d);
    if (nbytes_out) *nbytes_out = nbytes;
    if (n_chunks_out) *n_chunks_out = nc;
    if (chunk_bytes_out) *chunk_bytes_out = chunk_bytes;
    if (blob_bytes_out) *blob_bytes_out = off;
    return ZCO_OK;
}

/* Inverse of one grouped chunk payload; planes is NULL for v1, else the
 * v2 plane tables (a RANS stream then uses its plane's table). */
static int decode_grouped(const uint8_t *p, uint32_t stored, uint32_t len, int dtype, const uint32_t *planes,
                          int lanes, uint8_t *dst) {
    int W = zco_word_bytes(dtype);
    uint32_t n = len / (uint32_t)W;
    uint64_t g = pad16(4u * (uint64_t)W);
    if (stored < g) return ZCO_ECORRUPT;
    for (uint64_t b = 4u * (uint64_t)W; b < g; b++)
        if (p[b]) return ZCO_ECORRUPT;
    uint8_t *streams = (uint8_t *)malloc(len ? len : 1);
    if (!streams) return ZCO_EINVAL;
    int st = ZCO_OK;
    for (int j = 0; j < W && st == ZCO_OK; j++) {
        uint32_t entry = get32(p + 4 * j);
        uint32_t mode = entry >> 30, v = entry & 0x3FFFFFFFu;
        uint8_t *sj = streams + (uint64_t)j * n;
        if (mode == ZCO_MODE_CONST) {
            if (v > 255) st = ZCO_ECORRUPT;
            else memset(sj, (int)v, n);
        } else if (mode == ZCO_MODE_RAW || mode == ZCO_MODE_RANS) {
            if (mode == ZCO_MODE_RAW && v != n) { st = ZCO_ECORRUPT; break; }
            if (g + pad16(v) > stored) { st = ZCO_ECORRUPT; break; }
            for (uint64_t b = g + v; b < g + pad16(v); b++)
                if (p[b]) st = ZCO_ECORRUPT;
            if (st != ZCO_OK) break;
            if (mode == ZCO_MODE_RAW) memcpy(sj, p + g, n);
            else if (planes) st = zco_rans_decode_shared(p + g, v, n, planes + 256u * j, sj);
            else if (lanes) st = zco_rans_decode_lanes(p + g, v, n, sj);
            else st = zco_rans_decode(p + g, v, n, sj);
            g += pad16(v);
        } else {
            st = ZCO_ECORRUPT;
        }
    }
    if (st == ZCO_OK && g != stored) st = ZCO_ECORRUPT;
    if (st == ZCO_OK) zco_group_merge(streams, n, dtype, dst);
    free(streams);
    return st;
}

int zco_decompress(const uint8_t *blob, uint64_t blob_len, uint8_t *dst, uint64_t cap, uint32_t flags) {
    int dtype, ndim;
    uint64_t nbytes, total;
    uint32_t nc, chunk_bytes;
    int st = zco_blob_info(blob, blob_len, &dtype, &ndim, NULL, &nbytes, &nc, &chunk_bytes, &total);
    if (st != ZCO_OK) return st;
    if (total > blob_len) return ZCO_EFORMAT;
    if (cap < nbytes) return ZCO_ECAPACITY;
    uint32_t planes[4 * 256];
    const int shared = get16(blob + 4) == 2;
    if (shared) {
        int W = zco_word_bytes(dtype);
        const uint8_t *t = blob + ZCO_HEADER + ZCO_ENTRY * (uint64_t)nc;
        for (int j = 0; j < W; j++)
            for (int v = 0; v < 256; v++) planes[256 * j + v] = get16(t + 512u * j + 2u * v);
    }
    int status = ZCO_OK;
    for (uint32_t c = 0; c < nc; c++) {
        const uint8_t *e = blob + ZCO_HEADER + ZCO_ENTRY * (uint64_t)c;
        uint64_t off = get64(e);
        uint32_t sm = get32(e + 8);
        uint32_t stored = sm & 0x7FFFFFFFu;
        uint32_t len = (uint32_t)((c + 1 < nc) ? chunk_bytes : nbytes - (uint64_t)c * chunk_bytes);
        uint8_t *out = dst + (uint64_t)c * chunk_bytes;
        /* the chunk CRC covers the stored payload: a chunk that fails it is
         * reported and not decoded (its output bytes are left as they were) */
        if (!(flags & ZCO_NO_VERIFY) && zco_crc32(blob + off, stored) != get32(e + 12)) {
            status |= ZCO_ECRC;
            continue;
        }
        if (sm >> 31) memcpy(out, blob + off, len);
        else status |= decode_grouped(blob + off, stored, len, dtype, shared ? planes : NULL, get16(blob + 4) == 3,
                                      out);
    }
    return status;
}

/* Check a blob without decoding it (cuZipNN API: verify an untrusted blob
 * with the CRC-32 helpers before decompressing it): the header and chunk
 * table as zco_blob_info checks them, that the payloads lie within blob_len,
 * then every chunk's CRC over its stored bytes. Returns status. */
int zco_verify(const uint8_t *blob, uint64_t blob_len) {
    uint64_t total;
    uint32_t nc;
    int st = zco_blob_info(blob, blob_len, NULL, NULL, NULL, NULL, &nc, NULL, &total);
    if (st != ZCO_OK) return st;
    if (total > blob_len) return ZCO_EFORMAT;
    int status = ZCO_OK;
    for (uint32_t c = 0; c < nc; c++) {
        const uint8_t *e = blob + ZCO_HEADER + ZCO_ENTRY * (uint64_t)c;
        if (zco_crc32(blob + get64(e), get32(e + 8) & 0x7FFFFFFFu) != get32(e + 12)) status |= ZCO_ECRC;
    }
    return status;
}
