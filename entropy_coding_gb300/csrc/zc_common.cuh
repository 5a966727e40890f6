// zc_common.cuh — device-side constants and helpers shared by the kernels:
// format constants, exponent extraction, CRC-32 tables and the GF(2)
// arithmetic that combines CRCs of adjacent byte ranges.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "zc.h"  // from include/ (on the -I path)

namespace zc {

constexpr uint32_t kLanes = 32;          // interleaved rANS states per stream
constexpr uint32_t kProbBits = 12;       // frequency tables sum to 4096
constexpr uint32_t kM = 1u << kProbBits;
constexpr uint32_t kRansL = 1u << 16;    // rANS state lives in [2^16, 2^32)
constexpr uint32_t kRecHead = 160;       // 32 u32 states + 32-byte bitmap
constexpr uint32_t kMaxTable = 512;      // 256 u16 frequencies
constexpr uint32_t kModeRaw = 0, kModeRans = 1, kModeConst = 2;
constexpr unsigned kFull = 0xFFFFFFFFu;

__host__ __device__ inline uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }
__host__ __device__ inline uint64_t pad16(uint64_t x) { return (x + 15) & ~uint64_t(15); }

__host__ __device__ inline int word_bytes(int dtype) {
    switch (dtype) {
    case ZC_U8: return 1;
    case ZC_U16: case ZC_BF16: case ZC_FP16: return 2;
    case ZC_U32: case ZC_FP32: return 4;
    default: return 0;
    }
}

// Largest grouped payload of a chunk of n symbols per stream and W streams:
// the directory plus W records of at most 160 + 512 + 2n bytes each (format
// v3: and 64 bytes of word counts and up to 7 padding words per lane).
__host__ __device__ inline uint64_t max_grouped(uint64_t len, int W, uint32_t version = 1) {
    uint64_t n = len / uint64_t(W);
    const uint64_t extra = version == 3 ? 64 + 14 * kLanes : 0;
    return pad16(4ull * W) + uint64_t(W) * pad16(kRecHead + kMaxTable + 2 * n + extra);
}

// ---------------------------------------------------------------------------
// Exponent extraction (ZipNN note, Method 1): the exponent moves to the top of
// the word, the sign directly below it, the mantissa stays where it is. Byte
// grouping (Method 2) then takes byte j from the most significant end as
// stream j. Integer dtypes are grouped without the permutation.
template <int DT> struct Perm;
// fwd2 and inv2 apply fwd and inv to two 16-bit words packed in one 32-bit
// register.
template <> struct Perm<ZC_U8>  { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } };
template <> struct Perm<ZC_U16> { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } static __device__ __forceinline__ uint32_t fwd2(uint32_t v) { return v; } static __device__ __forceinline__ uint32_t inv2(uint32_t v) { return v; } };
template <> struct Perm<ZC_U32> { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } };
// BF16: s e8 m7 -> e8 s m7
template <> struct Perm<ZC_BF16> {
    static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return ((w << 1) & 0xFF00u) | ((w >> 8) & 0x80u) | (w & 0x7Fu); }
    static __device__ __forceinline__ uint32_t inv(uint32_t p) { return ((p & 0x80u) << 8) | ((p >> 1) & 0x7F80u) | (p & 0x7Fu); }
    static __device__ __forceinline__ uint32_t fwd2(uint32_t v) { return ((v << 1) & 0xFF00FF00u) | ((v >> 8) & 0x00800080u) | (v & 0x007F007Fu); }
    static __device__ __forceinline__ uint32_t inv2(uint32_t v) { return ((v & 0x00800080u) << 8) | ((v >> 1) & 0x7F807F80u) | (v & 0x007F007Fu); }
};
// FP16: s e5 m10 -> e5 s m10
template <> struct Perm<ZC_FP16> {
    static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return ((w << 1) & 0xF800u) | ((w >> 5) & 0x400u) | (w & 0x3FFu); }
    static __device__ __forceinline__ uint32_t inv(uint32_t p) { return ((p & 0x400u) << 5) | ((p >> 1) & 0x7C00u) | (p & 0x3FFu); }
    static __device__ __forceinline__ uint32_t fwd2(uint32_t v) { return ((v << 1) & 0xF800F800u) | ((v >> 5) & 0x04000400u) | (v & 0x03FF03FFu); }
    static __device__ __forceinline__ uint32_t inv2(uint32_t v) { return ((v & 0x04000400u) << 5) | ((v >> 1) & 0x7C007C00u) | (v & 0x03FF03FFu); }
};
// FP32: s e8 m23 -> e8 s m23
template <> struct Perm<ZC_FP32> {
    static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return ((w << 1) & 0xFF000000u) | ((w >> 8) & 0x800000u) | (w & 0x7FFFFFu); }
    static __device__ __forceinline__ uint32_t inv(uint32_t p) { return ((p & 0x800000u) << 8) | ((p >> 1) & 0x7F800000u) | (p & 0x7FFFFFu); }
};
template <int DT> struct WordOf { static constexpr int W = (DT == ZC_U8) ? 1 : (DT == ZC_U32 || DT == ZC_FP32) ? 4 : 2; };

// ---------------------------------------------------------------------------
// CRC-32 as zlib computes it (cuZipNN API: checksums match zlib.crc32):
// reflected polynomial 0xEDB88320, register preset to ones, final complement.
// In the reflected register, bit 31 holds the coefficient of x^0 and bit 0
// that of x^31; multiplying by x is a right shift, folding x^32 back in as the
// polynomial.
constexpr uint32_t kPoly = 0xEDB88320u;

__host__ __device__ constexpr uint32_t gf2_mul_x(uint32_t a) { return (a & 1u) ? (a >> 1) ^ kPoly : (a >> 1); }

// a * b mod P in the reflected representation.
__host__ __device__ constexpr uint32_t gf2_mulmod(uint32_t a, uint32_t b) {
    uint32_t r = 0;
    for (int i = 0; i < 32; i++) {          // coefficient of x^i of a is bit 31-i
        if ((a >> (31 - i)) & 1u) r ^= b;
        b = gf2_mul_x(b);
    }
    return r;
}

struct CrcTables {
    uint32_t t[8][256];   // t[k][b]: register contribution of byte b followed by k zero bytes
};

constexpr CrcTables make_crc_tables() {
    CrcTables c{};
    for (uint32_t b = 0; b < 256; b++) {
        uint32_t r = b;
        for (int k = 0; k < 8; k++) r = gf2_mul_x(r);
        c.t[0][b] = r;
    }
    for (int k = 1; k < 8; k++)
        for (uint32_t b = 0; b < 256; b++) c.t[k][b] = (c.t[k - 1][b] >> 8) ^ c.t[0][c.t[k - 1][b] & 0xFFu];
    return c;
}

__device__ constexpr CrcTables kCrc = make_crc_tables();

// Register update over a little-endian 32-bit word from the global tables
// (slicing by four: byte i of the word is followed by 3 - i more bytes).
__device__ __forceinline__ uint32_t crc_word_global(uint32_t c, uint32_t w) {
    const uint32_t u = c ^ w;
    return __ldg(&kCrc.t[3][u & 0xFFu]) ^ __ldg(&kCrc.t[2][(u >> 8) & 0xFFu]) ^ __ldg(&kCrc.t[1][(u >> 16) & 0xFFu]) ^
           __ldg(&kCrc.t[0][u >> 24]);
}

// Multiplying a CRC register by a fixed x^(8n) mod P ("appending n zero
// bytes") is linear in the register, so it is four table lookups, one per
// register byte. Tables: kShPow + j shifts by 2^j bytes (j = 0..39), then the
// stride gaps 248, 496, 992, 2032, 4080, 8176 and 16352 bytes used by the
// strided CRCs (a round of NT threads x P-byte pieces leaves a gap of
// (NT - 1) P).
constexpr int kShPow = 0, kShPowCount = 40, kSh248 = 40, kSh496 = 41, kSh992 = 42, kSh2032 = 43, kSh4080 = 44,
              kSh8176 = 45, kSh16352 = 46, kShCount = 47;

struct ShiftTables {
    uint32_t t[kShCount][4][256];
};

constexpr ShiftTables make_shift_tables() {
    ShiftTables s{};
    uint32_t pw[kShPowCount] = {};
    uint32_t x8 = 0x80000000u;  // x^0
    for (int k = 0; k < 8; k++) x8 = gf2_mul_x(x8);
    pw[0] = x8;
    for (int j = 1; j < kShPowCount; j++) pw[j] = gf2_mulmod(pw[j - 1], pw[j - 1]);
    auto xpow8 = [&](uint32_t n) {
        uint32_t r = 0x80000000u;
        for (int j = 0; n; j++, n >>= 1)
            if (n & 1u) r = gf2_mulmod(r, pw[j]);
        return r;
    };
    uint32_t K[kShCount] = {};
    for (int j = 0; j < kShPowCount; j++) K[kShPow + j] = pw[j];
    K[kSh248] = xpow8(248);
    K[kSh496] = xpow8(496);
    K[kSh992] = xpow8(992);
    K[kSh2032] = xpow8(2032);
    K[kSh4080] = xpow8(4080);
    K[kSh8176] = xpow8(8176);
    K[kSh16352] = xpow8(16352);
    for (int c = 0; c < kShCount; c++) {
        // register bit m is the coefficient of x^(31-m); its image is K x^(31-m)
        uint32_t basis[32] = {};
        uint32_t v = K[c];
        for (int m = 31; m >= 0; m--) {
            basis[m] = v;
            v = gf2_mul_x(v);
        }
        for (int i = 0; i < 4; i++) {
            s.t[c][i][0] = 0;
            for (uint32_t b = 1; b < 256; b++) {
                int low = 0;
                while (!((b >> low) & 1u)) low++;
                s.t[c][i][b] = s.t[c][i][b & (b - 1)] ^ basis[8 * i + low];
            }
        }
    }
    return s;
}

__device__ constexpr ShiftTables kShift = make_shift_tables();

__device__ __forceinline__ uint32_t shift_by(uint32_t c, int table) {
    const uint32_t(*t)[256] = kShift.t[table];
    return __ldg(&t[0][c & 0xFF]) ^ __ldg(&t[1][(c >> 8) & 0xFF]) ^ __ldg(&t[2][(c >> 16) & 0xFF]) ^
           __ldg(&t[3][c >> 24]);
}

__device__ __forceinline__ uint32_t shift_smem(uint32_t c, const uint32_t (*t)[256]) {
    return t[0][c & 0xFF] ^ t[1][(c >> 8) & 0xFF] ^ t[2][(c >> 16) & 0xFF] ^ t[3][c >> 24];
}

// Shared-memory copy of one shift table (4 KB), filled once per CTA.
__device__ inline void load_shift_smem(uint32_t (*dst)[256], int table) {
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) dst[i >> 8][i & 255] = kShift.t[table][i >> 8][i & 255];
}

template <int NT>
constexpr int gap_table() { return NT == 32 ? kSh496 : NT == 128 ? kSh2032 : NT == 256 ? kSh4080 : kSh8176; }

// Register shifted by n bytes (n < 2^40): one table multiply per set bit.
__device__ inline uint32_t shift_bytes(uint32_t c, uint64_t n) {
    for (int j = 0; n; j++, n >>= 1)
        if (n & 1u) c = shift_by(c, kShPow + j);
    return c;
}

// The CRC tables in shared memory for slicing by four (Kounavis and Berry,
// 2005): table k holds the register contribution of byte b followed by k zero
// bytes (kCrc.t[k]), so a 32-bit word is four independent lookups instead of a
// chain of four. C copies interleaved word by word: entry (k, b) of copy r is
// word (256 k + b) * C + r and lane l reads copy l % C, so a lookup
// instruction meets at most 32 / C lanes per bank. 4 C KB per CTA (C = 8:
// 32 KB; the decoders that run one CTA per SM take 16 copies, 64 KB, which
// halves the lanes that can collide on a bank).
template <int C = 8>
constexpr uint32_t crc_rep_words() { return 4u * 256u * C; }
constexpr uint32_t kCrcRepWords = crc_rep_words<8>();

// Fill the copies: each of the 1024 table entries is read once and written
// as C consecutive words (16-byte stores; t 16-byte aligned), so a CTA reads
// 4 KB of tables whatever C is.
template <int C = 8>
__device__ inline void load_crc_rep(uint32_t *t) {
    static_assert(C == 4 || C == 8 || C == 16, "4, 8 or 16 table copies");
    for (uint32_t e = threadIdx.x; e < 4 * 256; e += blockDim.x) {
        const uint32_t v = kCrc.t[e >> 8][e & 0xFFu];
        uint4 *d = reinterpret_cast<uint4 *>(t + e * C);
#pragma unroll
        for (int q = 0; q < C / 4; q++) d[q] = make_uint4(v, v, v, v);
    }
}

// This lane's copy of the tables.
template <int C = 8>
__device__ __forceinline__ const uint32_t *crc_row(const uint32_t *t) { return t + (threadIdx.x & (C - 1)); }

// Sarwate's byte step (table 0); row = crc_row(table)
template <int C = 8>
__device__ __forceinline__ uint32_t crc_rep_byte(uint32_t c, uint32_t byte, const uint32_t *row) {
    return row[((c ^ byte) & 0xFFu) * C] ^ (c >> 8);
}

// Register update over a little-endian 32-bit word: with u = c ^ w, byte i of
// u is followed by 3 - i more bytes of the word.
template <int C = 8>
__device__ __forceinline__ uint32_t crc_rep_word(uint32_t c, uint32_t w, const uint32_t *row) {
    const uint32_t u = c ^ w;
    constexpr uint32_t S = 256u * C;  // one slice table
    return row[3 * S + (u & 0xFFu) * C] ^ row[2 * S + ((u >> 8) & 0xFFu) * C] ^
           row[1 * S + ((u >> 16) & 0xFFu) * C] ^ row[(u >> 24) * C];
}

template <int C = 8>
__device__ __forceinline__ uint32_t crc_rep16(uint32_t c, uint4 v, const uint32_t *row) {
    c = crc_rep_word<C>(c, v.x, row);
    c = crc_rep_word<C>(c, v.y, row);
    c = crc_rep_word<C>(c, v.z, row);
    return crc_rep_word<C>(c, v.w, row);
}

template <bool kLdcg>
__device__ __forceinline__ uint4 load16(const uint8_t *p) {
    return kLdcg ? __ldcg(reinterpret_cast<const uint4 *>(p)) : __ldg(reinterpret_cast<const uint4 *>(p));
}

// Piece assignment of the strided CRC: NT threads take the 16-byte pieces of
// a range round-robin, aligned to the END of the range (only the first round
// can be short). Thread t's piece in round r is NT r + t - v0.
struct Strided {
    uint64_t pieces, rounds, v0;
    __device__ Strided(uint64_t len16, int NT) {
        pieces = len16 / 16;
        rounds = (pieces + NT - 1) / NT;
        v0 = rounds * NT - pieces;
    }
};

// Multiplying a register by a FIXED x^(8 2^J) mod P with no table: the
// product is linear in the register, so it is the XOR of the images of the
// register's set bits, 32 constants worked out at compile time (register
// bit m is the coefficient of x^(31-m); its image is K x^(31-m)). About 64
// integer instructions and no memory access, where a table lookup that
// misses L1 costs an L2 round trip on the dependency chain.
__host__ __device__ constexpr uint32_t x8pow2(int J) {  // x^(8 * 2^J) mod P
    uint32_t k = 0x80000000u;                            // x^0
    for (int i = 0; i < 8; i++) k = gf2_mul_x(k);
    for (int i = 0; i < J; i++) k = gf2_mulmod(k, k);
    return k;
}

// Column m: the image of register bit m under multiplication by K, i.e.
// K x^(31-m) mod P.
__host__ __device__ constexpr uint32_t mul_column(uint32_t K, int m) {
    uint32_t v = K;
    for (int i = 0; i < 31 - m; i++) v = gf2_mul_x(v);
    return v;
}

template <int J, int M>
__device__ __forceinline__ uint32_t mul_bits(uint32_t r) {
    if constexpr (M == 32) {
        return 0u;
    } else {
        constexpr uint32_t c = mul_column(x8pow2(J), M);
        return ((0u - ((r >> M) & 1u)) & c) ^ mul_bits<J, M + 1>(r);
    }
}

// Register shifted by 2^J bytes, in registers.
template <int J>
__device__ __forceinline__ uint32_t shift_pow2(uint32_t r) { return mul_bits<J, 0>(r); }

template <int J, int END>
__device__ __forceinline__ uint32_t shift_bits(uint32_t c, uint32_t n) {
    if constexpr (J == END) {
        return c;
    } else {
        if ((n >> J) & 1u) c = shift_pow2<J>(c);
        return shift_bits<J + 1, END>(c, n);
    }
}

// Register shifted by n < 2^20 bytes (a chunk's parts), in registers: one
// constant multiply per set bit of n.
static __device__ __noinline__ uint32_t shift_bytes_small(uint32_t c, uint32_t n) { return shift_bits<0, 20>(c, n); }

// Register over A followed by B, from the register over A (any preset) and
// the register over B taken from zero, B being len < 2^20 bytes (linearity).
__device__ __forceinline__ uint32_t crc_append_small(uint32_t reg_a, uint32_t reg_b0, uint32_t len) {
    return shift_bytes_small(reg_a, len) ^ reg_b0;
}

// Levels K .. KEND-1 of a fold tree over lanes: at level k a lane's register
// moves over 2^(L2 + k) bytes and takes in the register of the lane 2^k
// above it.
template <int L2, int K, int KEND>
__device__ __forceinline__ uint32_t fold_levels(uint32_t R) {
    if constexpr (K == KEND) {
        return R;
    } else {
        const uint32_t right = __shfl_down_sync(kFull, R, 1 << K);
        return fold_levels<L2, K + 1, KEND>(shift_pow2<L2 + K>(R) ^ right);
    }
}

// Fold the per-thread registers of a strided CRC into the range's register.
// Each thread holds the register of its own pieces with all other bytes
// taken as zero, ending at its last piece; CRC-32 is linear, so the range's
// register is the XOR of those registers, each shifted by the bytes after
// its thread's last piece: a tree over threads with shifts of piece, 2
// pieces, ... (piece = 2^L2 bytes). NW > 1 uses s_reg[NW] and
// __syncthreads (every thread of the CTA must call it). Returns the result
// in every thread.
template <int NW, int L2>
__device__ inline uint32_t crc_fold(uint32_t R, uint32_t *s_reg) {
    const int lane = threadIdx.x & 31;
    R = fold_levels<L2, 0, 5>(R);
    if constexpr (NW > 1) {
        constexpr int kLevels = NW >= 16 ? 4 : NW >= 8 ? 3 : NW >= 4 ? 2 : 1;
        static_assert((1 << kLevels) == NW, "NW is a power of two up to 16");
        const int warp = threadIdx.x >> 5;
        if (lane == 0) s_reg[warp] = R;
        __syncthreads();
        if (warp == 0) {
            R = lane < NW ? s_reg[lane] : 0u;
            R = fold_levels<L2 + 5, 0, kLevels>(R);
            if (lane == 0) s_reg[0] = R;
        }
        __syncthreads();
        R = s_reg[0];
        __syncthreads();
        return R;
    } else {
        return __shfl_sync(kFull, R, 0);
    }
}

// Raw CRC register (no final complement) over [p, p + len) from register
// `init`, by NT = 32 NW threads with coalesced 16-byte loads (see Strided and
// crc_fold); each thread shifts its register over the other threads' pieces
// with the gap table G = gap_table<NT>() in shared memory, T is the
// replicated byte table. The last len % 16 bytes are added by every thread.
// p must be 16-byte aligned. Every thread of the group calls it.
template <int NW, bool kLdcg, int C = 8>
__device__ inline uint32_t crc_strided(const uint8_t *p, uint64_t len, uint32_t init, const uint32_t *T,
                                       const uint32_t (*G)[256], uint32_t *s_reg) {
    constexpr int NT = 32 * NW;
    static_assert(NT == 32 || NT == 128 || NT == 256 || NT == 512, "strided CRC runs on 1, 4, 8 or 16 warps");
    const int tid = NW == 1 ? int(threadIdx.x & 31) : int(threadIdx.x);
    const uint32_t *row = crc_row<C>(T);
    const uint64_t main = len & ~uint64_t(15);
    const Strided sp(main, NT);
    uint32_t reg = init;
    if (sp.pieces) {
        uint32_t R = 0;
        int64_t pidx = int64_t(tid) - int64_t(sp.v0);
        uint4 cur = pidx >= 0 ? load16<kLdcg>(p + 16 * pidx) : make_uint4(0, 0, 0, 0);
        for (uint64_t r = 0; r < sp.rounds; r++) {
            uint4 nxt = make_uint4(0, 0, 0, 0);
            if (r + 1 < sp.rounds) nxt = load16<kLdcg>(p + 16 * (pidx + NT));
            uint32_t c = r == 0 ? (pidx == 0 ? init : 0u) : shift_smem(R, G);
            if (pidx >= 0) c = crc_rep16<C>(c, cur, row);
            R = c;
            cur = nxt;
            pidx += NT;
        }
        reg = crc_fold<NW, 4>(R, s_reg);
    }
    for (uint64_t i = main; i < len; i++) reg = crc_rep_byte<C>(reg, kLdcg ? __ldcg(p + i) : __ldg(p + i), row);
    return reg;
}

// CRC register, taken from zero, of len bytes (a multiple of 16) at p
// (16-byte aligned), by one warp: 16-byte pieces taken round-robin, aligned
// to the end of the range (only the first round can be short), with U
// loads in flight per lane, so that a short range costs about one memory
// latency per U rounds instead of one per round.
template <int C, bool kLdcg, int U = 8>
__device__ inline uint32_t warp_crc16(const uint8_t *p, uint32_t len, const uint32_t *T, const uint32_t (*G)[256]) {
    const int lane = threadIdx.x & 31;
    const uint32_t *row = crc_row<C>(T);
    const uint32_t pieces = len / 16;
    const uint32_t rounds = (pieces + 31) / 32, v0 = rounds * 32 - pieces;
    uint32_t R = 0;
    for (uint32_t r0 = 0; r0 < rounds; r0 += U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t v = int64_t(32) * (r0 + u) + lane - v0;
            t[u] = (r0 + u < rounds && v >= 0) ? load16<kLdcg>(p + 16 * v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const uint32_t r = r0 + u;
            if (r >= rounds) break;
            if (r > 0) R = shift_smem(R, G);
            if (int64_t(32) * r + lane >= v0) R = crc_rep16<C>(R, t[u], row);
        }
    }
    return rounds ? crc_fold<1, 4>(R, nullptr) : 0u;
}

// As crc_strided, for a range that need not be 16-byte aligned: the bytes up
// to the first 16-byte boundary are taken one at a time first.
template <int NW, bool kLdcg, int C = 8>
__device__ inline uint32_t crc_any(const uint8_t *p, uint64_t len, uint32_t init, const uint32_t *T,
                                   const uint32_t (*G)[256], uint32_t *s_reg) {
    uint64_t head = (16 - (reinterpret_cast<uintptr_t>(p) & 15)) & 15;
    if (head > len) head = len;
    const uint32_t *row = crc_row<C>(T);
    uint32_t reg = init;
    for (uint64_t i = 0; i < head; i++) reg = crc_rep_byte<C>(reg, kLdcg ? __ldcg(p + i) : __ldg(p + i), row);
    return crc_strided<NW, kLdcg, C>(p + head, len - head, reg, T, G, s_reg);
}

// One 32-byte read-only global load (p 32-byte aligned) as two 16-byte halves.
__device__ __forceinline__ void ldg32(const void *p, uint4 &lo, uint4 &hi) {
    asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
}

// 16-byte asynchronous global -> shared copies (both addresses 16-aligned).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = uint32_t(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// bring the 128-byte line at p into L2 (no register result, no wait)
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t lanemask_lt() { uint32_t m; asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m)); return m; }
__device__ __forceinline__ uint32_t lanemask_gt() { uint32_t m; asm("mov.u32 %0, %%lanemask_gt;" : "=r"(m)); return m; }

__device__ __forceinline__ void status_or(int32_t *d_status, int32_t bits) {
    if (bits) atomicOr(d_status, bits);
}

} // namespace zc
