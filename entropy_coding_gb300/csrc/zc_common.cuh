// zc_common.cuh — device-side constants and helpers shared by the kernels:
// format constants, exponent extraction, CRC-32 tables and the GF(2)
// arithmetic that combines CRCs of adjacent byte ranges.
#pragma once

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
// the directory plus W records of at most 160 + 512 + 2n bytes each.
__host__ __device__ inline uint64_t max_grouped(uint64_t len, int W) {
    uint64_t n = len / uint64_t(W);
    return pad16(4ull * W) + uint64_t(W) * pad16(kRecHead + kMaxTable + 2 * n);
}

// ---------------------------------------------------------------------------
// Exponent extraction (ZipNN note, Method 1): the exponent moves to the top of
// the word, the sign directly below it, the mantissa stays where it is. Byte
// grouping (Method 2) then takes byte j from the most significant end as
// stream j. Integer dtypes are grouped without the permutation.
template <int DT> struct Perm;
// inv2 applies inv to two 16-bit words packed in one 32-bit register.
template <> struct Perm<ZC_U8>  { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } };
template <> struct Perm<ZC_U16> { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } static __device__ __forceinline__ uint32_t inv2(uint32_t v) { return v; } };
template <> struct Perm<ZC_U32> { static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return w; } static __device__ __forceinline__ uint32_t inv(uint32_t p) { return p; } };
// BF16: s e8 m7 -> e8 s m7
template <> struct Perm<ZC_BF16> {
    static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return ((w << 1) & 0xFF00u) | ((w >> 8) & 0x80u) | (w & 0x7Fu); }
    static __device__ __forceinline__ uint32_t inv(uint32_t p) { return ((p & 0x80u) << 8) | ((p >> 1) & 0x7F80u) | (p & 0x7Fu); }
    static __device__ __forceinline__ uint32_t inv2(uint32_t v) { return ((v & 0x00800080u) << 8) | ((v >> 1) & 0x7F807F80u) | (v & 0x007F007Fu); }
};
// FP16: s e5 m10 -> e5 s m10
template <> struct Perm<ZC_FP16> {
    static __device__ __forceinline__ uint32_t fwd(uint32_t w) { return ((w << 1) & 0xF800u) | ((w >> 5) & 0x400u) | (w & 0x3FFu); }
    static __device__ __forceinline__ uint32_t inv(uint32_t p) { return ((p & 0x400u) << 5) | ((p >> 1) & 0x7C00u) | (p & 0x3FFu); }
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
    uint32_t pow2[64];    // x^(8 * 2^j) mod P: shifting a register by 2^j bytes
    uint32_t seg16[1025]; // x^(8 * 16 * m) mod P for m = 0..1024
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
    uint32_t x8 = 0x80000000u;                 // x^0
    for (int k = 0; k < 8; k++) x8 = gf2_mul_x(x8);  // x^8
    c.pow2[0] = x8;
    for (int j = 1; j < 64; j++) c.pow2[j] = gf2_mulmod(c.pow2[j - 1], c.pow2[j - 1]);
    c.seg16[0] = 0x80000000u;
    for (int m = 1; m <= 1024; m++) c.seg16[m] = gf2_mulmod(c.seg16[m - 1], c.pow2[4]);
    return c;
}

__device__ constexpr CrcTables kCrc = make_crc_tables();

// x^(8n) mod P by square-and-multiply over the bits of n.
__device__ inline uint32_t gf2_xpow8(uint64_t n) {
    uint32_t r = 0x80000000u;
    for (int j = 0; n; j++, n >>= 1)
        if (n & 1u) r = gf2_mulmod(r, kCrc.pow2[j]);
    return r;
}

// Shared-memory copy of the slicing tables (8 KB), filled once per CTA.
__device__ inline void load_crc_smem(uint32_t (*tab)[256]) {
    for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) tab[i >> 8][i & 255] = kCrc.t[i >> 8][i & 255];
}

// Register update over 8 bytes given as two little-endian words (slicing by 8).
__device__ __forceinline__ uint32_t crc_step8(uint32_t c, uint32_t lo, uint32_t hi, const uint32_t (*T)[256]) {
    uint32_t v = c ^ lo;
    return T[7][v & 0xFF] ^ T[6][(v >> 8) & 0xFF] ^ T[5][(v >> 16) & 0xFF] ^ T[4][v >> 24] ^
           T[3][hi & 0xFF] ^ T[2][(hi >> 8) & 0xFF] ^ T[1][(hi >> 16) & 0xFF] ^ T[0][hi >> 24];
}

__device__ __forceinline__ uint32_t crc_step1(uint32_t c, uint32_t byte, const uint32_t (*T)[256]) {
    return T[0][(c ^ byte) & 0xFF] ^ (c >> 8);
}

// Raw CRC register over [p, p + len) starting from register `init`, computed
// by the whole warp: each lane takes an equal run of 16-byte blocks (the runs
// are aligned to the end of the range, so the first lane's run may start
// before p and only its real bytes are read), then the lanes' registers are
// combined pairwise with shifts of 1, 2, 4, 8, 16 runs. The < 16-byte tail is
// finished by one lane. p must be 16-byte aligned. Returns the register (no
// final complement) on every lane. `ldcg` reads through L2 only.
template <bool kLdcg>
__device__ inline uint32_t warp_crc_raw(const uint8_t *p, uint64_t len, uint32_t init, const uint32_t (*T)[256]) {
    const int lane = threadIdx.x & 31;
    uint64_t main = len & ~uint64_t(15);
    uint32_t reg = init;
    if (main) {
        uint64_t seg = ((main / 16 + 31) / 32) * 16;  // bytes per lane
        int64_t s = int64_t(main) - int64_t(32 - lane) * int64_t(seg);
        int64_t e = s + int64_t(seg);
        uint32_t c = (s <= 0 && e > 0) ? init : 0u;
        if (s < 0) s = 0;
        int64_t off = s;
        for (; off + 64 <= e; off += 64) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; u++)
                v[u] = kLdcg ? __ldcg(reinterpret_cast<const uint4 *>(p + off) + u)
                             : __ldg(reinterpret_cast<const uint4 *>(p + off) + u);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                c = crc_step8(c, v[u].x, v[u].y, T);
                c = crc_step8(c, v[u].z, v[u].w, T);
            }
        }
        for (; off < e; off += 16) {
            uint4 v = kLdcg ? __ldcg(reinterpret_cast<const uint4 *>(p + off))
                            : __ldg(reinterpret_cast<const uint4 *>(p + off));
            c = crc_step8(c, v.x, v.y, T);
            c = crc_step8(c, v.z, v.w, T);
        }
        uint32_t K = (seg / 16 <= 1024) ? kCrc.seg16[seg / 16] : gf2_xpow8(seg);
#pragma unroll
        for (int k = 0; k < 5; k++) {
            uint32_t right = __shfl_down_sync(kFull, c, 1 << k);
            c = gf2_mulmod(c, K) ^ right;
            K = gf2_mulmod(K, K);
        }
        reg = __shfl_sync(kFull, c, 0);
    }
    for (uint64_t i = main; i < len; i++) reg = crc_step1(reg, kLdcg ? __ldcg(p + i) : p[i], T);
    return reg;
}

// Raw CRC register over [p, p + len) computed by a whole CTA of NW warps, the
// same way as warp_crc_raw but with 32 * NW runs: each warp folds its 32
// lanes, then warp 0 folds the NW warp registers (through s_reg[NW] in shared
// memory). Every thread of the CTA must call it; the result is valid in all
// threads. p must be 16-byte aligned; reads go through L2 only.
template <int NW>
__device__ inline uint32_t block_crc_raw(const uint8_t *p, uint64_t len, uint32_t init, const uint32_t (*T)[256],
                                         uint32_t *s_reg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kRuns = 32 * NW;
    const uint64_t main = len & ~uint64_t(15);
    uint32_t reg = init;
    if (main) {
        const uint64_t seg = ((main / 16 + kRuns - 1) / kRuns) * 16;
        int64_t s = int64_t(main) - int64_t(kRuns - tid) * int64_t(seg);
        const int64_t e = s + int64_t(seg);
        uint32_t c = (s <= 0 && e > 0) ? init : 0u;
        if (s < 0) s = 0;
        int64_t off = s;
        for (; off + 32 <= e; off += 32) {
            uint4 v0 = __ldcg(reinterpret_cast<const uint4 *>(p + off));
            uint4 v1 = __ldcg(reinterpret_cast<const uint4 *>(p + off + 16));
            c = crc_step8(c, v0.x, v0.y, T);
            c = crc_step8(c, v0.z, v0.w, T);
            c = crc_step8(c, v1.x, v1.y, T);
            c = crc_step8(c, v1.z, v1.w, T);
        }
        if (off < e) {
            uint4 v = __ldcg(reinterpret_cast<const uint4 *>(p + off));
            c = crc_step8(c, v.x, v.y, T);
            c = crc_step8(c, v.z, v.w, T);
        }
        uint32_t K = (seg / 16 <= 1024) ? kCrc.seg16[seg / 16] : gf2_xpow8(seg);
#pragma unroll
        for (int k = 0; k < 5; k++) {
            uint32_t right = __shfl_down_sync(kFull, c, 1 << k);
            c = gf2_mulmod(c, K) ^ right;
            K = gf2_mulmod(K, K);
        }
        if (lane == 0) s_reg[warp] = c;
        __syncthreads();
        if (warp == 0) {
            c = lane < NW ? s_reg[lane] : 0u;
#pragma unroll
            for (int k = 1; k < NW; k <<= 1) {
                uint32_t right = __shfl_down_sync(kFull, c, k);
                c = gf2_mulmod(c, K) ^ right;
                K = gf2_mulmod(K, K);
            }
            if (lane == 0) s_reg[0] = c;
        }
        __syncthreads();
        reg = s_reg[0];
        __syncthreads();
    }
    for (uint64_t i = main; i < len; i++) reg = crc_step1(reg, __ldcg(p + i), T);
    return reg;
}

__device__ __forceinline__ uint32_t lanemask_lt() { uint32_t m; asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m)); return m; }
__device__ __forceinline__ uint32_t lanemask_gt() { uint32_t m; asm("mov.u32 %0, %%lanemask_gt;" : "=r"(m)); return m; }

__device__ __forceinline__ void status_or(int32_t *d_status, int32_t bits) {
    if (bits) atomicOr(d_status, bits);
}

} // namespace zc
