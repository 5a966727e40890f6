// encode.cu — compression: a statistics kernel and a coding kernel per wave
// of chunks (ZipNN note, Method 5: fixed-size chunks coded independently).
//
// stats_kernel, one CTA per chunk (persistent CTAs, grid-stride over the
// wave): one pass over the chunk's bytes builds the 256-bin histogram of
// every byte stream of the exponent-extracted words (order-0 statistics,
// ZipNN note Key insight). Then
// warp j takes stream j: a stream with one symbol is CONST; otherwise its
// histogram is quantised to the 12-bit table, and the stream is RAW if its
// coded size provably cannot come below the threshold, else a candidate
// whose table goes to the workspace.
//
// code_kernel, one warp per chunk (persistent warps taking chunk tickets in
// order): rANS-codes the candidate streams (32 interleaved lanes) into the
// warp's workspace slot, applies the passthrough rule per stream and per
// chunk (cuZipNN API, passthrough_threshold), finds the chunk's blob offset
// with a decoupled look-back over the chunks before it (an exclusive prefix
// scan of the metadata map, ZipNN note Method 5), and writes the payload,
// taking the CRC-32 of the stored bytes as it writes them (cuZipNN API: the
// CRCs are over pieces of the blob), and the chunk table entry. The last
// warp to finish writes the header and its CRC.
//
// The serial part of rANS coding (each lane's state runs through the whole
// stream) stays on single warps that never wait at a CTA barrier, so an SM
// keeps many such chains in flight, while the histogram pass, which is bound
// by shared-memory traffic, runs on whole CTAs with per-lane counter copies.
#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kStatWarps = 16;
constexpr int kStatThreads = 32 * kStatWarps;
constexpr uint32_t kPiece = 32;  // bytes per thread per round of the statistics pass
constexpr int kCodeWarps = 16;    // coding warps per SM (and at most per CTA)
constexpr int kCodeThreads = 32 * kCodeWarps;
constexpr uint32_t kModeCand = 3;  // statistics -> coder only: a stream to rANS-code
constexpr uint32_t kAborted = 0xFFFFFFFFu;
constexpr uint32_t kCodeWarpSmem = 4096 + 4096 + 4096;  // per coding warp: rANS table, symbol ring, 2 word stages
constexpr uint64_t kFlagAgg = 1ull << 62, kFlagPre = 2ull << 62, kValMask = (1ull << 62) - 1;

// Exact division by a table frequency f in [1, 4095] for every dividend the
// encoder can see (x < 2^20 f, since larger states are renormalised first):
// floor(x / f) = (x * m + a) >> k with a 32-bit m and a in {0, m}. This is
// the round-up reciprocal (a = 0, m = ceil(2^k / f)) or the round-down one
// with increment (a = m, m = floor(2^k / f)) of Granlund & Montgomery (1994)
// and Robison (2005); for each f the first k >= 32 whose error term e
// satisfies e (2^20 f - 1) < 2^k (round-up) or e 2^20 f <= 2^k (round-down)
// is taken. Built at compile time.
struct Recip {
    uint32_t m[4096];
    uint32_t ka[4096];  // k | round-down flag << 8
};

constexpr Recip make_recip() {
    Recip r{};
    using u128 = unsigned __int128;
    const u128 X = u128(1) << 20;
    for (uint32_t f = 1; f < 4096; f++) {
        for (uint32_t k = 32; k < 64; k++) {
            const u128 p = u128(1) << k;
            const u128 mu = (p + f - 1) / f;
            if (mu < (u128(1) << 32) && (mu * f - p) * (X * f - 1) < p) {
                r.m[f] = uint32_t(mu);
                r.ka[f] = k;
                break;
            }
            u128 md = p / f;
            if (md > 0xFFFFFFFFu) md = 0xFFFFFFFFu;
            if ((p - md * f) * X * f <= p) {
                r.m[f] = uint32_t(md);
                r.ka[f] = k | 0x100u;
                break;
            }
        }
    }
    return r;
}

__device__ constexpr Recip kRecip = make_recip();

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

template <int W>
__device__ __forceinline__ uint32_t load_word(const uint8_t *p) {
    if (W == 4) return *reinterpret_cast<const uint32_t *>(p);
    if (W == 2) return *reinterpret_cast<const uint16_t *>(p);
    return *p;
}

template <int W>
__device__ __forceinline__ uint32_t stream_byte(uint32_t perm, int j) {
    return (perm >> (8 * (W - 1 - j))) & 0xFFu;
}

// The bytes a compression kernel reads: a tensor, or for a checkpoint delta
// (ZipNN note, Method 6: XOR against a base) the XOR of two tensors of the
// same layout, formed as it is read (kDelta), so that the difference never
// goes through memory.
template <bool kDelta>
struct Source {
    const uint8_t *p;  // the tensor (for a delta, the new one)
    const uint8_t *x;  // the base tensor (kDelta only)
    __device__ __forceinline__ Source at(uint64_t o) const { return Source{p + o, kDelta ? x + o : nullptr}; }
    // bits that must be clear for an access of that alignment
    __device__ __forceinline__ uintptr_t addr_bits() const {
        return reinterpret_cast<uintptr_t>(p) | (kDelta ? reinterpret_cast<uintptr_t>(x) : 0);
    }
    __device__ __forceinline__ uint4 vec(uint64_t o) const {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(p + o));
        if constexpr (kDelta) {
            const uint4 b = __ldg(reinterpret_cast<const uint4 *>(x + o));
            v.x ^= b.x; v.y ^= b.y; v.z ^= b.z; v.w ^= b.w;
        }
        return v;
    }
    __device__ __forceinline__ uint4 vec_last(uint64_t o) const {  // last use: evict first
        uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p + o));
        if constexpr (kDelta) {
            const uint4 b = __ldcs(reinterpret_cast<const uint4 *>(x + o));
            v.x ^= b.x; v.y ^= b.y; v.z ^= b.z; v.w ^= b.w;
        }
        return v;
    }
    __device__ __forceinline__ void vec32(uint64_t o, uint4 &lo, uint4 &hi) const {
        ldg32(p + o, lo, hi);
        if constexpr (kDelta) {
            uint4 a, b;
            ldg32(x + o, a, b);
            lo.x ^= a.x; lo.y ^= a.y; lo.z ^= a.z; lo.w ^= a.w;
            hi.x ^= b.x; hi.y ^= b.y; hi.z ^= b.z; hi.w ^= b.w;
        }
    }
    __device__ __forceinline__ uint32_t byte(uint64_t i) const {
        return kDelta ? uint32_t(__ldg(p + i) ^ __ldg(x + i)) : uint32_t(__ldg(p + i));
    }
    template <int W>
    __device__ __forceinline__ uint32_t word(uint64_t i) const {  // element i
        const uint32_t w = load_word<W>(p + i * W);
        return kDelta ? w ^ load_word<W>(x + i * W) : w;
    }
};

// The tensor a call-wide chunk index belongs to (fields read once per chunk).
struct TView {
    const uint8_t *src, *base;
    uint8_t *blob;
    uint64_t nbytes, cap;
    uint32_t n_chunks, chunk_base, t;
};

__device__ __forceinline__ TView tensor_view(const EncodeArgs &a, uint32_t g) {
    TView v;
    if (a.n_tensors == 1) {
        v.src = a.one.src;
        v.base = a.one.base;
        v.blob = a.one.blob;
        v.nbytes = a.one.nbytes;
        v.cap = a.one.cap;
        v.n_chunks = a.one.n_chunks;
        v.chunk_base = 0;
        v.t = 0;
    } else {
        v.t = owner_of(a.tensors, a.n_tensors, g);
        const TensorDesc &d = a.tensors[v.t];
        v.src = d.src;
        v.base = d.base;
        v.blob = d.blob;
        v.nbytes = d.nbytes;
        v.cap = d.cap;
        v.n_chunks = d.n_chunks;
        v.chunk_base = d.chunk_base;
    }
    return v;
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
    for (int o = 16; o; o >>= 1) v += __shfl_down_sync(kFull, v, o);
    return __shfl_sync(kFull, v, 0);
}
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
    for (int o = 16; o; o >>= 1) v += __shfl_down_sync(kFull, v, o);
    return __shfl_sync(kFull, v, 0);
}
__device__ __forceinline__ float warp_sum_f32(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_down_sync(kFull, v, o);
    return __shfl_sync(kFull, v, 0);
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
    uint32_t inc = v;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += t;
    }
    return inc - v;
}

// 12-bit table from counts held as 8 bins per lane (symbol 8*lane + k).
// Same rule as the format's definition: floor share with a floor of 1,
// shortfall to the most frequent symbol, excess taken from the largest
// frequencies (lowest symbol on ties); runs of decrements on a unique maximum
// are taken at once, which gives the same result as one at a time.
__device__ void normalize_warp(const uint32_t cnt[8], uint32_t n, uint32_t f[8]) {
    const int lane = threadIdx.x & 31;
    uint32_t local = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        f[k] = cnt[k] ? max(1u, (cnt[k] * kM) / n) : 0u;
        local += f[k];
    }
    uint32_t sum = warp_sum_u32(local);
    if (sum < kM) {
        uint32_t key = 0;
#pragma unroll
        for (int k = 0; k < 8; k++) key = max(key, (cnt[k] << 8) | (255u - (8 * lane + k)));
        key = warp_max_u32(key);
        uint32_t sb = 255u - (key & 0xFFu);
        if ((sb >> 3) == uint32_t(lane)) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (k == int(sb & 7)) f[k] += kM - sum;
        }
    }
    while (sum > kM) {
        uint32_t key = 0;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (f[k] > 1) key = max(key, (f[k] << 8) | (255u - (8 * lane + k)));
        key = warp_max_u32(key);
        uint32_t f1 = key >> 8, s1 = 255u - (key & 0xFFu);
        uint32_t key2 = 0;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (f[k] > 1 && 8 * lane + k != s1) key2 = max(key2, f[k]);
        uint32_t m2 = max(warp_max_u32(key2), 1u);
        uint32_t dec = (f1 > m2) ? min(sum - kM, f1 - m2) : 1u;
        if ((s1 >> 3) == uint32_t(lane)) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (k == int(s1 & 7)) f[k] -= dec;
        }
        sum -= dec;
    }
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(kFull, v, o);
        v = t > v ? t : v;
    }
    return v;
}

// The same quantisation rule as normalize_warp for a plane's counts over a
// whole tensor (shared tables; lmzip "Building on lmz": one table per plane
// kind), which may exceed 32 bits: 64-bit counts and keys in the first two
// steps; the third works on the frequencies alone.
__device__ void normalize_plane_warp(const unsigned long long cnt[8], unsigned long long n, uint32_t f[8]) {
    const int lane = threadIdx.x & 31;
    uint32_t local = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const unsigned long long q = cnt[k] * kM / n;
        f[k] = cnt[k] ? (q < 1 ? 1u : uint32_t(q)) : 0u;
        local += f[k];
    }
    uint32_t sum = warp_sum_u32(local);
    if (sum < kM) {
        unsigned long long key = 0;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const unsigned long long kk = (cnt[k] << 8) | (255u - (8 * lane + k));
            key = kk > key ? kk : key;
        }
        key = warp_max_u64(key);
        const uint32_t sb = 255u - uint32_t(key & 0xFFu);
        if ((sb >> 3) == uint32_t(lane)) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (k == int(sb & 7)) f[k] += kM - sum;
        }
    }
    while (sum > kM) {
        uint32_t key = 0;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (f[k] > 1) key = max(key, (f[k] << 8) | (255u - (8 * lane + k)));
        key = warp_max_u32(key);
        uint32_t f1 = key >> 8, s1 = 255u - (key & 0xFFu);
        uint32_t key2 = 0;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (f[k] > 1 && 8 * lane + k != s1) key2 = max(key2, f[k]);
        uint32_t m2 = max(warp_max_u32(key2), 1u);
        uint32_t dec = (f1 > m2) ? min(sum - kM, f1 - m2) : 1u;
        if ((s1 >> 3) == uint32_t(lane)) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (k == int(s1 & 7)) f[k] -= dec;
        }
        sum -= dec;
    }
}

// Exclusive prefix of this chunk's padded size over the chunks before it
// (decoupled look-back, one warp). Every wait is bounded (spin_limit polls);
// a timeout sets ZC_ETIMEOUT and the chunk is not placed. With the test hook
// ZC_HOOK_LOOKBACK_STALL the first chunk never publishes its prefix, so the
// waits of the others run out.
__device__ uint64_t lookback(unsigned long long *st, uint32_t c, uint64_t agg, int32_t *d_status, bool *timed,
                             uint32_t spin_limit, uint32_t hooks) {
    const int lane = threadIdx.x & 31;
    *timed = false;
    if (c == 0) {
        if (lane == 0 && !(hooks & ZC_HOOK_LOOKBACK_STALL)) st_release(&st[0], kFlagPre | agg);
        return 0;
    }
    if (lane == 0) st_release(&st[c], kFlagAgg | agg);
    uint64_t excl = 0;
    int64_t j = int64_t(c) - 1;
    for (;;) {
        int64_t idx = j - lane;
        unsigned long long v = kFlagPre;  // before chunk 0: prefix 0
        bool timed_out = false;
        if (idx >= 0) {
            uint32_t spins = 0;
            v = ld_acquire(&st[idx]);
            while ((v >> 62) == 0) {
                if (++spins > spin_limit) {
                    timed_out = true;
                    break;
                }
                __nanosleep(64);
                v = ld_acquire(&st[idx]);
            }
        }
        if (__any_sync(kFull, timed_out)) {
            if (lane == 0) status_or(d_status, ZC_ETIMEOUT);
            *timed = true;
            return excl;
        }
        uint32_t pre = __ballot_sync(kFull, (v >> 62) == 2);
        int first = pre ? __ffs(pre) - 1 : 31;
        excl += warp_sum_u64(lane <= first ? (v & kValMask) : 0ull);
        if (pre) break;
        j -= 32;
    }
    if (lane == 0) st_release(&st[c], kFlagPre | (excl + agg));
    return excl;
}

// ---------------------------------------------------------------- statistics

// Shared memory of a statistics CTA. The histogram of stream j keeps one copy
// per lane index, so the 32 lanes of a warp always add into 32 different
// banks. For W <= 2 word b * 32 + lane holds the 32-bit count of bin b (32 KB
// per stream); for W = 4, where that would not leave room for two CTAs per
// SM, word (b >> 1) * 32 + lane holds the 16-bit counts of bins b & ~1 (low
// half) and b | 1 (high half): a copy sees at most about n / 32 counts of one
// stream (each thread's pieces hold at most 1/512 of the chunk plus one
// piece, 16 threads share a copy), far below 2^16.
template <int W>
struct StatsSmem {
    static constexpr int kWords = W <= 2 ? 256 : 128;  // counter words per stream and lane
    uint32_t hist[W][kWords * 32];
    uint32_t cnt[W][256];            // merged counts
    uint32_t plane[W][256];          // v2: counts of this CTA's recent chunks of one tensor, per plane
};

// Count one element into the histograms; hrow = &h[0][lane]. For the byte b
// of stream j at bit sh of the permuted word, the counter word is b * 32 +
// lane of stream j (W <= 2), or (b >> 1) * 32 + lane with the half b & 1.
template <int DT>
__device__ __forceinline__ void count_elem(uint32_t w, uint32_t *hrow) {
    constexpr int W = WordOf<DT>::W;
    const uint32_t p = Perm<DT>::fwd(w);
#pragma unroll
    for (int j = 0; j < W; j++) {
        const int sh = 8 * (W - 1 - j);
        if constexpr (W <= 2) {
            atomicAdd(hrow + j * (256 * 32) + ((p >> sh) & 0xFFu) * 32, 1u);
        } else {
            const uint32_t half = (p >> (sh + 1)) & 0x7Fu;
            const uint32_t inc = (p & (1u << sh)) ? 0x10000u : 1u;
            atomicAdd(hrow + j * (128 * 32) + half * 32, inc);
        }
    }
}

template <int DT>
__device__ __forceinline__ void count_vec(const uint4 &q, uint32_t *hrow) {
    constexpr int W = WordOf<DT>::W;
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; k++)
#pragma unroll
        for (int e = 0; e < 4 / W; e++)
            count_elem<DT>(W == 4 ? u[k] : (u[k] >> (8 * W * e)) & ((1u << (8 * W)) - 1u), hrow);
}

// 2-byte words: count the 8 elements of a 16-byte vector and return the
// bytes of stream 0 (the top byte of each permuted element) in o[0..1], in
// element order; the permutation runs on two elements per register.
template <int DT>
__device__ __forceinline__ void count_vec2(const uint4 &q, uint32_t *hrow, uint32_t o[2]) {
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
    uint32_t p[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        p[k] = Perm<DT>::fwd2(u[k]);
#pragma unroll
        for (int e = 0; e < 2; e++) {
            atomicAdd(hrow + ((p[k] >> (16 * e + 8)) & 0xFFu) * 32, 1u);              // stream 0
            atomicAdd(hrow + 256 * 32 + ((p[k] >> (16 * e)) & 0xFFu) * 32, 1u);        // stream 1
        }
    }
    o[0] = __byte_perm(p[0], p[1], 0x7531);
    o[1] = __byte_perm(p[2], p[3], 0x7531);
}

// Bytes of stream 0 (the top byte of each permuted element) of a 16-byte
// vector: 16 / W of them, in element order, in the low bytes of o.
template <int DT>
__device__ __forceinline__ void stream0_bytes(const uint4 &q, uint32_t o[4]) {
    constexpr int W = WordOf<DT>::W;
    if constexpr (W == 1) {
        o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w;
    } else if constexpr (W == 2) {
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
        uint32_t t[4];
#pragma unroll
        for (int k = 0; k < 4; k++)
            t[k] = __byte_perm(Perm<DT>::fwd(u[k] & 0xFFFFu), Perm<DT>::fwd(u[k] >> 16), 0x0051);  // [e0, e1]
        o[0] = __byte_perm(t[0], t[1], 0x5410);
        o[1] = __byte_perm(t[2], t[3], 0x5410);
    } else {
        const uint32_t a = __byte_perm(Perm<DT>::fwd(q.x), Perm<DT>::fwd(q.y), 0x0073);
        const uint32_t b = __byte_perm(Perm<DT>::fwd(q.z), Perm<DT>::fwd(q.w), 0x0073);
        o[0] = __byte_perm(a, b, 0x5410);
    }
}

// Histograms of the chunk's W byte streams by the CTA from one pass, and
// stream 0's bytes for the coder. Aligned input: the threads take 32-byte
// pieces round-robin (the next round's piece is loaded while this round's is
// counted); a piece is one 32-byte load when the chunk is 32-byte aligned (a
// warp then reads 1 KiB contiguously), else two 16-byte loads.
template <int DT, bool kDelta>
__device__ void chunk_stats(Source<kDelta> src, uint32_t len, StatsSmem<WordOf<DT>::W> &sm, uint8_t *cand0) {
    constexpr int W = WordOf<DT>::W;
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t *hrow = &sm.hist[0][lane];
    uint32_t done = 0;  // elements counted by the vector pass
    if (kDelta || (src.addr_bits() & 15) == 0) {  // delta inputs are 16-byte aligned
        const uint32_t pieces = len / kPiece;
        const bool wide = (src.addr_bits() & 31) == 0;
        auto load_piece = [&](uint32_t pi, uint4 &lo, uint4 &hi) {
            const uint64_t o = uint64_t(pi) * kPiece;
            if (wide) {
                src.vec32(o, lo, hi);
            } else {
                lo = src.vec(o);
                hi = src.vec(o + 16);
            }
        };
        uint32_t pidx = tid;
        uint4 n0 = make_uint4(0, 0, 0, 0), n1 = n0;
        if (pidx < pieces) load_piece(pidx, n0, n1);
        for (; pidx < pieces; pidx += kStatThreads) {
            const uint4 q0 = n0, q1 = n1;
            if (pidx + kStatThreads < pieces) load_piece(pidx + kStatThreads, n0, n1);
            // stream 0's bytes of the piece, for the coder in case the
            // stream is a candidate
            uint8_t *d = cand0 + uint64_t(pidx) * (kPiece / W);
            uint32_t o0[4], o1[4];
            if constexpr (W == 2) {
                count_vec2<DT>(q0, hrow, o0);
                count_vec2<DT>(q1, hrow, o1);
            } else {
                count_vec<DT>(q0, hrow);
                count_vec<DT>(q1, hrow);
                stream0_bytes<DT>(q0, o0);
                stream0_bytes<DT>(q1, o1);
            }
            if constexpr (W == 4) {
                *reinterpret_cast<uint2 *>(d) = make_uint2(o0[0], o1[0]);
            } else if constexpr (W == 2) {
                *reinterpret_cast<uint4 *>(d) = make_uint4(o0[0], o0[1], o1[0], o1[1]);
            } else {
                reinterpret_cast<uint4 *>(d)[0] = q0;
                reinterpret_cast<uint4 *>(d)[1] = q1;
            }
        }
        done = pieces * (kPiece / W);
    }
    // the rest (or, for input aligned to its element size only, all of it):
    // one word at a time
    for (uint32_t i = done + tid; i < len / W; i += kStatThreads) {
        const uint32_t w = src.template word<W>(i);
        count_elem<DT>(w, hrow);
        cand0[i] = uint8_t(stream_byte<W>(Perm<DT>::fwd(w), 0));
    }
}

// Sum the 32 counter copies of every stream into cnt[j][b] (and zero them
// for the next chunk), by all warps of the CTA.
template <int W>
__device__ void merge_counts(StatsSmem<W> &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int K = StatsSmem<W>::kWords;
#pragma unroll 4
    for (int w = warp; w < W * K; w += kStatWarps) {
        uint32_t *cell = &sm.hist[w / K][(w % K) * 32 + lane];
        const uint32_t v = *cell;
        *cell = 0;
        if constexpr (K == 256) {
            const uint32_t c = __reduce_add_sync(kFull, v);
            if (lane == 0) sm.cnt[w / K][w % K] = c;
        } else {
            const uint32_t lo = __reduce_add_sync(kFull, v & 0xFFFFu);
            const uint32_t hi = __reduce_add_sync(kFull, v >> 16);
            if (lane == 0) {
                sm.cnt[w / K][2 * (w % K)] = lo;
                sm.cnt[w / K][2 * (w % K) + 1] = hi;
            }
        }
    }
}

// Stream j's decision after the histogram pass, by one warp, from its merged
// counts (8 bins per lane: symbol 8 lane + k): CONST / RAW / candidate. A
// candidate's 12-bit table goes to ftab (256 u16).
template <int W>
__device__ bool plan_stats(const EncodeArgs &a, uint32_t n, const uint32_t *counts, uint32_t *sv, uint8_t *ftab,
                           uint32_t *plane) {
    const int lane = threadIdx.x & 31;
    uint32_t cnt[8];
    const uint4 c0 = reinterpret_cast<const uint4 *>(counts)[2 * lane];
    const uint4 c1 = reinterpret_cast<const uint4 *>(counts)[2 * lane + 1];
    cnt[0] = c0.x; cnt[1] = c0.y; cnt[2] = c0.z; cnt[3] = c0.w;
    cnt[4] = c1.x; cnt[5] = c1.y; cnt[6] = c1.z; cnt[7] = c1.w;
    uint32_t pres = 0, only = 0;
#pragma unroll
    for (int k = 0; k < 8; k++)
        if (cnt[k]) {
            pres++;
            only = 8 * lane + k;
            // v2: the chunk's counts join the CTA's count of the plane
            if (plane) plane[8 * lane + k] += cnt[k];
        }
    const uint32_t k_total = warp_sum_u32(pres);
    uint32_t mode, val;
    if (k_total == 1) {
        const uint32_t who = __ballot_sync(kFull, pres != 0);
        mode = kModeConst;
        val = __shfl_sync(kFull, only, __ffs(who) - 1);
    } else if (plane) {
        // v2: the table is the tensor's, not known yet. Its cost is at least
        // the chunk's own order-0 information n H (Gibbs' inequality: no
        // table codes the chunk below its empirical entropy), so the bound
        // below, with the v2 record head (32 states, no table), holds for
        // whatever table the tensor gets.
        const float lg_n = __log2f(float(n));
        float info = 0.f;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (cnt[k]) info += float(cnt[k]) * (lg_n - __log2f(float(cnt[k])));
        info = warp_sum_f32(info);
        const float words_lb = (info * (1.0f - 1.0f / 1024) - 0.0932f * float(n) - 512.0f - 64.0f) / 16.1f;
        const uint64_t rec_lb = 128 + 2ull * uint64_t(words_lb > 0.f ? words_lb : 0.f);
        mode = double(rec_lb) < a.threshold * double(n) ? kModeCand : kModeRaw;
        val = mode == kModeRaw ? n : 0;
    } else {
        uint32_t f[8];
        normalize_warp(cnt, n, f);
        // Lower bound on the coded size from the table's information content:
        // every coded symbol adds at least log2(4096/f_s) + log2(15/16) bits
        // to its lane's state, every word removes at most 16.1 bits, and 32
        // states of at most 32 bits remain. A stream whose bound already
        // reaches threshold x n cannot be kept coded, so it is not coded.
        float info = 0.f;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (cnt[k]) info += float(cnt[k]) * (12.0f - __log2f(float(f[k])));
        info = warp_sum_f32(info);
        const float words_lb = (info * (1.0f - 1.0f / 1024) - 0.0932f * float(n) - 512.0f - 64.0f) / 16.1f;
        const uint64_t rec_lb = kRecHead + pad16(2 * k_total) + 2ull * uint64_t(words_lb > 0.f ? words_lb : 0.f);
        mode = kModeRaw;
        val = n;
        if (double(rec_lb) < a.threshold * double(n)) {
            mode = kModeCand;
            val = 0;
            uint4 v;
            v.x = f[0] | f[1] << 16;
            v.y = f[2] | f[3] << 16;
            v.z = f[4] | f[5] << 16;
            v.w = f[6] | f[7] << 16;
            reinterpret_cast<uint4 *>(ftab)[lane] = v;
        }
    }
    if (lane == 0) *sv = (mode << 30) | val;
    return mode == kModeCand;
}

// The bytes of stream j of the chunk, in element order, into out: a second
// pass over the chunk (now in L2) by one warp, 16-byte vectors with eight in
// flight per lane; byte j (from the top) of four elements is gathered into a
// word with two byte permutes and a merge.
template <int DT, bool kDelta>
__device__ void warp_write_cand(Source<kDelta> src, uint32_t len, int j, uint8_t *out) {
    constexpr int W = WordOf<DT>::W;
    constexpr int E = 16 / W;  // elements per vector
    constexpr int U = 8;
    const int lane = threadIdx.x & 31;
    const uint32_t n = len / W;
    const uint32_t bj = uint32_t(W - 1 - j);
    const uint32_t sel = bj | (4 + bj) << 4;
    uint32_t done = 0;
    if ((src.addr_bits() & 15) == 0) {
        const uint32_t nvec = len / 16;
        for (uint32_t v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; u++)
                q[u] = v0 + 32 * u < nvec ? src.vec(16ull * (v0 + 32 * u)) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; u++) {
                const uint32_t v = v0 + 32 * u;
                if (v >= nvec) break;
                const uint32_t w4[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                uint32_t p[E];
#pragma unroll
                for (int k = 0; k < 4; k++)
#pragma unroll
                    for (int e = 0; e < 4 / W; e++)
                        p[k * (4 / W) + e] = Perm<DT>::fwd(W == 4 ? w4[k] : (w4[k] >> (8 * W * e)) & ((1u << (8 * W)) - 1u));
                uint32_t o[E / 4];
#pragma unroll
                for (int h = 0; h < E / 4; h++)
                    o[h] = __byte_perm(__byte_perm(p[4 * h], p[4 * h + 1], sel), __byte_perm(p[4 * h + 2], p[4 * h + 3], sel),
                                       0x5410);
                if constexpr (E == 4) *reinterpret_cast<uint32_t *>(out + 4ull * v) = o[0];
                else if constexpr (E == 8) *reinterpret_cast<uint2 *>(out + 8ull * v) = make_uint2(o[0], o[1]);
                else *reinterpret_cast<uint4 *>(out + 16ull * v) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        done = nvec * E;
    }
    for (uint32_t i = done + lane; i < n; i += 32) {
        const uint32_t p = Perm<DT>::fwd(src.template word<W>(i));
        uint32_t b = 0;
#pragma unroll
        for (int k = 0; k < W; k++)
            if (k == j) b = stream_byte<W>(p, k);
        out[i] = uint8_t(b);
    }
}

// One CTA per chunk of the wave (grid-stride). Writes per chunk 32 bytes of
// info {unused word, W stream words mode << 30 | value}, the tables of the
// candidate streams and their bytes.
template <int DT, bool kDelta>
__global__ void __launch_bounds__(kStatThreads, 2) stats_kernel(EncodeArgs a) {
    constexpr int W = WordOf<DT>::W;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    StatsSmem<W> &sm = *reinterpret_cast<StatsSmem<W> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    // the coding kernel's chunk ticket starts from zero in every wave (the
    // previous wave's coding kernel has finished: same stream)
    if (blockIdx.x == 0 && tid == 0) reinterpret_cast<uint32_t *>(a.ws_ctrl)[0] = 0;
    for (int i = tid; i < W * StatsSmem<W>::kWords * 32; i += kStatThreads) (&sm.hist[0][0])[i] = 0;
    for (int i = tid; i < W * 256; i += kStatThreads) (&sm.plane[0][0])[i] = 0;
    // v2: warp j < W adds stream j's counts into sm.plane[j] for tensor cur_t
    // and moves them to the tensor's plane histogram in global memory when
    // the tensor changes, every 4096 chunks (32-bit counters) and at the end
    uint32_t cur_t = 0xFFFFFFFFu, since = 0;
    auto flush = [&](uint32_t t) {
        unsigned long long *h = a.ws_hist + (uint64_t(t) * W + warp) * 256;
        uint32_t *row = sm.plane[warp];
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const uint32_t v = row[8 * (tid & 31) + k];
            if (v) atomicAdd(h + 8 * (tid & 31) + k, (unsigned long long)v);
            row[8 * (tid & 31) + k] = 0;
        }
    };
    __syncthreads();
    for (uint32_t cl = blockIdx.x; cl < a.wave_n; cl += gridDim.x) {
        const uint32_t g = a.wave_start + cl;
        const TView tv = tensor_view(a, g);
        const uint64_t c = g - tv.chunk_base;
        const Source<kDelta> src = Source<kDelta>{tv.src, tv.base}.at(c * a.chunk_bytes);
        const uint32_t len = uint32_t(umin64(a.chunk_bytes, tv.nbytes - c * a.chunk_bytes));
        uint8_t *cand = a.ws_cand + uint64_t(cl) * W * a.n_pad;
        chunk_stats<DT, kDelta>(src, len, sm, cand);
        __syncthreads();
        merge_counts<W>(sm);
        __syncthreads();
        uint32_t *info = reinterpret_cast<uint32_t *>(a.ws_info + 32ull * cl);
        // warp j decides stream j (and, when stream j >= 1 is a candidate,
        // writes its bytes for the coder; stream 0's are already there) while
        // the other warps go on to the next chunk: the counters were zeroed by
        // the merge, and the next merge comes after the next barrier
        if (warp < W) {
            if (a.version == 2 && (tv.t != cur_t || since == 4096)) {
                if (cur_t != 0xFFFFFFFFu) flush(cur_t);
                cur_t = tv.t;
                since = 0;
            }
            since++;
            const bool cand_j = plan_stats<W>(a, len / W, sm.cnt[warp], info + 1 + warp,
                                              a.ws_ftab + (uint64_t(cl) * W + warp) * 512,
                                              a.version == 2 ? sm.plane[warp] : nullptr);
            if (warp > 0 && cand_j) warp_write_cand<DT, kDelta>(src, len, warp, cand + uint64_t(warp) * a.n_pad);
        }
    }
    if (warp < W && cur_t != 0xFFFFFFFFu) flush(cur_t);  // v2 only: cur_t is set only there
}

// ---------------------------------------------------------------- coding

// Code one stream of the chunk into rec (the warp's slot), one warp, with the
// 12-bit table f (8 entries per lane) and the stream's bytes in cand (element
// order, padded to whole steps). Per symbol the table keeps 16 bytes,
// {m, a, 2^20 f, (4096 - f) | cum << 13 | (k-32) << 25} (bits 29-31 zero;
// a = 0 or m), so that a step is:
// renormalise if x >= 2^20 f, q = (x m + a) >> k, x += q (4096 - f) + cum.
// The steps run in blocks of 32 (the last steps of the stream first); the
// symbols of the next three blocks are in flight into a shared-memory ring
// (row s of a block = the 32 symbols of its step s), and each step's table
// entry is read two steps ahead. Returns the record's unpadded size, or
// kAborted once the record has reached lim bytes (it can then no longer be
// kept: the stream is stored raw).
//
// One word list (v1, v2): a step stages the low 16 bits of its state in
// shared memory and keeps one flag bit; the words of the emitting lanes of a
// block are written out step by step (lanes 31..0 within a step) while the
// next block is coded, which keeps the word stores off the state's
// dependency chain.
//
// kLanes (format v3, a word list per lane): no lane depends on another, so
// a step appends its word to the lane's 8-byte block in registers at once,
// without a branch, and each full block (4 words) goes to the lane's own
// list; lane l's list is staged at a stride of pad8(T) words after the 32
// counts (the record's size counts each list padded to 8 words), and
// warp_copy_crc_lanes gathers the lists into place in the blob.
template <bool kLanes>
__device__ uint32_t rans_encode_stream(const uint8_t *cand, uint32_t n, const uint32_t f[8], uint4 *etab,
                                       uint8_t *ring, uint16_t *stage_base, uint8_t *rec, uint64_t lim,
                                       bool shared) {
    const int lane = threadIdx.x & 31;
    uint16_t *stage = stage_base + lane;  // step s of a block: stage[32 s]
    const int T = int((n + 31) / 32);
    const int nb = (T + 31) / 32;
    // block b holds steps t = T-1-32b-s (s = 0..31); lane l fetches row l
    auto issue = [&](int b) {
        if (b < nb) {
            const int t = T - 1 - 32 * b - lane;
            if (t >= 0) {
                uint8_t *d = ring + (b & 3) * 1024 + lane * 32;
                cp_async16(d, cand + uint64_t(t) * 32);
                cp_async16(d + 16, cand + uint64_t(t) * 32 + 16);
            }
        }
        cp_async_commit();
    };
    issue(0);
    issue(1);
    issue(2);

    uint32_t present = 0, fsum = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        present += f[k] ? 1u : 0u;
        fsum += f[k];
    }
    uint32_t rank = warp_excl_scan(present);
    uint32_t cum = warp_excl_scan(fsum);
    const uint32_t k_total = __shfl_sync(kFull, rank + present, 31);
    uint32_t bits = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint32_t s = 8 * lane + k, fs = f[k];
        if (fs) {
            bits |= 1u << k;
            if (!shared) reinterpret_cast<uint16_t *>(rec + kRecHead)[rank] = uint16_t(fs);
            rank++;
            const uint32_t ka = kRecip.ka[fs], m = kRecip.m[fs];
            etab[s] = make_uint4(m, (ka >> 8) ? m : 0u, fs << 20, (kM - fs) | (cum << 13) | (((ka & 0xFFu) - 32) << 25));
        }
        cum += fs;
    }
    // v1 record: states | presence bitmap | frequencies | pad | words; v2
    // (shared plane tables): states | words
    uint32_t words_at = 128;
    if (!shared) {
        rec[128 + lane] = uint8_t(bits);
        words_at = kRecHead + uint32_t(pad16(2 * k_total));
        for (uint32_t b = kRecHead + 2 * k_total + lane; b < words_at; b += 32) rec[b] = 0;
    }

    // v3: the lists follow the 32 counts; lane l stages its words at
    // lists_at + 2 l Ts, Ts = pad8(T), in 8-byte blocks collected in acc
    const uint32_t lists_at = words_at + 64;
    const uint32_t Ts = (uint32_t(T) + 7) & ~7u;
    uint16_t *wout = reinterpret_cast<uint16_t *>(rec + (kLanes ? lists_at : words_at));
    uint2 *lw2 = reinterpret_cast<uint2 *>(wout + uint32_t(lane) * Ts);
    uint2 acc = make_uint2(0, 0);
    // append a word to the lane's block (words in emission order, the first
    // at the lowest address); a full block (4 words) goes to the lane's list
    auto push = [&](uint32_t w, uint32_t &count) {
        acc.x = __funnelshift_r(acc.x, acc.y, 16);
        acc.y = (acc.y >> 16) | (w << 16);
        if ((++count & 3u) == 0) lw2[(count >> 2) - 1] = acc;
    };
    // the same for a lane that may or may not emit, without a branch on em
    // (the shifted block is selected; only a full block's store branches)
    auto push_if = [&](bool em, uint32_t w, uint32_t &count) {
        const uint2 sh = make_uint2(__funnelshift_r(acc.x, acc.y, 16), (acc.y >> 16) | (w << 16));
        acc.x = em ? sh.x : acc.x;
        acc.y = em ? sh.y : acc.y;
        count += em ? 1u : 0u;
        if (em && (count & 3u) == 0) lw2[(count >> 2) - 1] = acc;
    };
    const uint32_t gt = lanemask_gt();
    uint32_t x = kRansL;
    uint32_t wc = 0;  // v1/v2: words of the warp; v3: words of this lane
    const bool first_active = uint32_t(T - 1) * 32 + lane < n;
    // one coding step with table entry ec; returns whether it renormalised
    // (emitting the low 16 bits of the state before it)
    auto code_step = [&](const uint4 ec) -> bool {
        const bool emit = x >= ec.z;
        if constexpr (kLanes) push_if(emit, x & 0xFFFFu, wc);
        x = emit ? x >> 16 : x;
        const uint32_t q = uint32_t((uint64_t(x) * ec.x + ec.y) >> 32) >> (ec.w >> 25);
        x = x + q * (ec.w & 0x1FFFu) + ((ec.w >> 13) & 0xFFFu);
        return emit;
    };
    // step T-1, the only one that may be partial; no lane emits a word there
    // (x = 2^16 is below every 2^20 f)
    auto first_step = [&](const uint4 ec) {
        const uint32_t q = uint32_t((uint64_t(x) * ec.x + ec.y) >> 32) >> (ec.w >> 25);
        if (first_active) x = x + q * (ec.w & 0x1FFFu) + ((ec.w >> 13) & 0xFFFu);
    };
    // write out the words of one staged block (steps 0..cnt-1, emitting lanes
    // 31..0 within a step)
    auto flush = [&](const uint16_t *st, uint32_t flags, int cnt) {
#pragma unroll 4
        for (int s = 0; s < cnt; s++) {
            const bool em = (flags >> s) & 1u;
            const uint32_t B = __ballot_sync(kFull, em);
            if (em) wout[wc + __popc(B & gt)] = st[s * 32];
            wc += __popc(B);
        }
    };
    // the record's size if it ended with the words written so far
    auto size_now = [&]() -> uint64_t {
        if constexpr (kLanes) return lists_at + 2ull * warp_sum_u32((wc + 7) & ~7u);
        else return words_at + 2ull * wc;
    };
    uint32_t flags_prev = 0;
    bool aborted = false;
    for (int b = 0; b < nb; b++) {
        issue(b + 3);
        cp_async_wait<3>();
        __syncwarp();
        // rows past the block read the next ring slot (or the stage after the
        // last slot): harmless values that are never used
        const uint8_t *blk = ring + (b & 3) * 1024 + lane;
        const int cnt = min(32, T - 32 * b);
        if constexpr (kLanes) {
            int s = 0;
            if (b == 0) {
                first_step(etab[blk[0]]);
                s = 1;
            }
            uint32_t sym_n = blk[(s + 2) * 32];
            uint4 e = etab[blk[s * 32]], e2 = etab[blk[(s + 1) * 32]];
            if (cnt == 32 && s == 0) {
#pragma unroll 8
                for (int k = 0; k < 32; k++) {
                    const uint4 ec = e;
                    e = e2;
                    e2 = etab[sym_n];
                    sym_n = blk[(k + 3) * 32];
                    code_step(ec);
                }
            } else {
#pragma unroll 4
                for (; s < cnt; s++) {
                    const uint4 ec = e;
                    e = e2;
                    e2 = etab[sym_n];
                    sym_n = blk[(s + 3) * 32];
                    code_step(ec);
                }
            }
        } else {
            uint16_t *st_cur = stage + (b & 1) * 1024;
            const uint16_t *st_prev = stage + ((b + 1) & 1) * 1024;
            uint32_t flags = 0;
            if (b > 0 && cnt == 32) {
                // a full block, interleaved with the write-out of the previous
                // one (always full): one straight-line body, so the two
                // chains overlap
                uint32_t sym_n = blk[64];
                uint4 e = etab[blk[0]], e2 = etab[blk[32]];
                uint32_t fp = flags_prev;
#pragma unroll 8
                for (int s = 0; s < 32; s++) {
                    const uint4 ec = e;
                    e = e2;
                    e2 = etab[sym_n];
                    sym_n = blk[(s + 3) * 32];
                    st_cur[s * 32] = uint16_t(x);
                    flags |= code_step(ec) ? (1u << s) : 0u;

                    const bool em = fp & 1u;
                    fp >>= 1;
                    const uint32_t B = __ballot_sync(kFull, em);
                    if (em) wout[wc + __popc(B & gt)] = st_prev[s * 32];
                    wc += __popc(B);
                }
            } else {
                if (b > 0) flush(st_prev, flags_prev, 32);
                int s = 0;
                if (b == 0) {
                    first_step(etab[blk[0]]);
                    s = 1;
                }
                uint32_t sym_n = blk[(s + 2) * 32];
                uint4 e = etab[blk[s * 32]], e2 = etab[blk[(s + 1) * 32]];
#pragma unroll 4
                for (; s < cnt; s++) {
                    const uint4 ec = e;
                    e = e2;
                    e2 = etab[sym_n];
                    sym_n = blk[(s + 3) * 32];
                    st_cur[s * 32] = uint16_t(x);
                    if (code_step(ec)) flags |= 1u << s;
                }
            }
            flags_prev = flags;
        }
        __syncwarp();
        // v1/v2: the words written so far belong to the blocks before this one
        if (size_now() >= lim) {
            aborted = true;
            break;
        }
    }
    if (!kLanes && !aborted) {
        flush(stage + ((nb - 1) & 1) * 1024, flags_prev, T - 32 * (nb - 1));
        __syncwarp();
        aborted = size_now() >= lim;
    }
    cp_async_wait_all();  // the ring is reused by the next stream
    __syncwarp();
    if (aborted) return kAborted;
    reinterpret_cast<uint32_t *>(rec)[lane] = x;
    uint32_t rec_bytes = words_at + 2 * wc;
    if constexpr (kLanes) {
        // the lane's last, partial blocks: zero words pushed in behind its
        // words move them to the bottom, up to a whole 8 words
        if (wc & 7u) {
            uint32_t c = wc;
            while (c & 7u) push(0u, c);
        }
        __syncwarp();
        // the counts; the lists stay at their staging places, and the copy
        // into the blob gathers them to lists_at + 2 off_l (off_l = the
        // padded counts of the lanes below)
        const uint32_t padded = (wc + 7) & ~7u;
        reinterpret_cast<uint16_t *>(rec + words_at)[lane] = uint16_t(wc);
        rec_bytes = lists_at + 2 * warp_sum_u32(padded);
    }
    for (uint32_t b = rec_bytes + lane; b < pad16(rec_bytes); b += 32) rec[b] = 0;
    __syncwarp();
    return rec_bytes;
}

// The coder's CRC tables in shared memory: 4 copies of the slicing tables
// (16 KB) and the register shift over the 31 other lanes' 16-byte pieces
// (496 bytes) of the strided CRCs below.
constexpr int kCodeCrcCopies = 4;
constexpr uint32_t kCodeCrcBytes = crc_rep_words<kCodeCrcCopies>() * 4 + 4 * 256 * 4;

struct CrcSmem {
    const uint32_t *rep;              // crc_rep_words<kCodeCrcCopies>() words
    const uint32_t (*gap496)[256];
};

// Pieces of a region of `pieces` 16-byte pieces taken by the warp's lanes
// round-robin, aligned to the END of the region (only the first round can be
// short): lane l's piece in round r is 32 r + l - v0. Each lane's CRC
// register then ends 16 (31 - l) bytes before the region's end, which
// crc_fold undoes.
struct EndAligned {
    uint32_t rounds, v0;
    __device__ explicit EndAligned(uint32_t pieces) {
        rounds = (pieces + 31) / 32;
        v0 = rounds * 32 - pieces;
    }
};

// All raw streams of a grouped chunk in one pass over the input, by the
// warp: a lane takes 16 consecutive elements at a time (G groups, 8 vectors
// in flight) and writes 16 bytes to every raw stream, gathering byte j (from
// the top) of four elements into a word with two byte permutes and a merge.
// Returns in reg[j] the CRC register, taken from zero, of raw stream j's
// stored bytes (its n bytes and the zero padding to 16), which are exactly
// the vectors written.
template <int DT, bool kDelta>
__device__ void warp_raw_streams(Source<kDelta> src, uint32_t n, const uint32_t mode[4], const uint32_t roff[4],
                                 uint8_t *out, const CrcSmem &cs, uint32_t reg[4]) {
    constexpr int W = WordOf<DT>::W;
    constexpr int G = 8 / W;
    const int lane = threadIdx.x & 31;
    const uint32_t *row = crc_row<kCodeCrcCopies>(cs.rep);
#pragma unroll
    for (int j = 0; j < W; j++) reg[j] = 0;
    bool any = false;
#pragma unroll
    for (int j = 0; j < W; j++) any |= mode[j] == kModeRaw;
    if (!any) return;
    const uint32_t groups = (n + 15) / 16;
    const EndAligned ea(groups);
    const bool vec = (src.addr_bits() & 15) == 0;
    for (uint32_t r0 = 0; r0 < ea.rounds; r0 += G) {
        uint4 qv[G][W];
#pragma unroll
        for (int gi = 0; gi < G; gi++) {
            const int64_t g = int64_t(32) * (r0 + gi) + lane - ea.v0;
#pragma unroll
            for (int v = 0; v < W; v++)
                qv[gi][v] = (vec && r0 + gi < ea.rounds && g >= 0 && 16 * (g + 1) <= n)
                                ? src.vec_last(uint64_t(g) * 16 * W + 16 * v)
                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int gi = 0; gi < G; gi++) {
            const uint32_t r = r0 + gi;
            if (r >= ea.rounds) break;
            const int64_t gs = int64_t(32) * r + lane - ea.v0;
            // the register moves over the other lanes' pieces of this round
            if (r > 0) {
#pragma unroll
                for (int j = 0; j < W; j++)
                    if (mode[j] == kModeRaw) reg[j] = shift_smem(reg[j], cs.gap496);
            }
            if (gs < 0) continue;  // first round only
            const uint32_t g = uint32_t(gs);
            // the 16 elements permuted: W = 2 two to a register (wd[k] holds
            // elements 2k and 2k + 1), else one to a register
            constexpr int NR = W == 2 ? 8 : 16;
            uint32_t wd[NR];
            if (vec && 16 * (g + 1) <= n) {
#pragma unroll
                for (int v = 0; v < W; v++) {
                    const uint32_t u[4] = {qv[gi][v].x, qv[gi][v].y, qv[gi][v].z, qv[gi][v].w};
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        if constexpr (W == 2) {
                            wd[4 * v + k] = u[k];
                        } else {
#pragma unroll
                            for (int e = 0; e < 4 / W; e++)
                                wd[(v * 4 + k) * (4 / W) + e] =
                                    (W == 4) ? u[k] : (u[k] >> (8 * W * e)) & ((1u << (8 * W)) - 1u);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < 16; k++) {
                    const uint32_t i = g * 16 + k;
                    const uint32_t w = i < n ? src.template word<W>(i) : 0u;
                    if constexpr (W == 2) {
                        if (k & 1) wd[k >> 1] |= w << 16;
                        else wd[k >> 1] = w;
                    } else {
                        wd[k] = w;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < NR; k++) {
                if constexpr (W == 2) wd[k] = Perm<DT>::fwd2(wd[k]);
                else wd[k] = Perm<DT>::fwd(wd[k]);
            }
#pragma unroll
            for (int j = 0; j < W; j++) {
                if (mode[j] != kModeRaw) continue;
                const uint32_t bj = uint32_t(W - 1 - j);        // byte of stream j in a permuted element
                uint32_t o[4];
                if constexpr (W == 2) {
                    // [e0.bj, e1.bj, e2.bj, e3.bj] from two registers of two elements
                    const uint32_t sel = bj | (2 + bj) << 4 | (4 + bj) << 8 | (6 + bj) << 12;
#pragma unroll
                    for (int q = 0; q < 4; q++) o[q] = __byte_perm(wd[2 * q], wd[2 * q + 1], sel);
                } else {
                    const uint32_t sel = bj | (4 + bj) << 4;         // [x.bj, y.bj, -, -]
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t lo = __byte_perm(wd[4 * q], wd[4 * q + 1], sel);
                        const uint32_t hi = __byte_perm(wd[4 * q + 2], wd[4 * q + 3], sel);
                        o[q] = __byte_perm(lo, hi, 0x5410);
                    }
                }
                // elements past n contribute zero bytes
                if (16 * (g + 1) > n) {
#pragma unroll
                    for (int q = 0; q < 4; q++)
#pragma unroll
                        for (int b = 0; b < 4; b++)
                            if (g * 16 + 4 * q + b >= n) o[q] &= ~(0xFFu << (8 * b));
                }
                const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
                reinterpret_cast<uint4 *>(out + roff[j])[g] = ov;
                reg[j] = crc_rep16<kCodeCrcCopies>(reg[j], ov, row);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < W; j++)
        if (mode[j] == kModeRaw) reg[j] = crc_fold<1, 4>(reg[j], nullptr);
}

// Copy len bytes (a multiple of 16) from a 16-byte aligned source by the
// warp, 8 vectors in flight per lane, and return the CRC register of the
// copied bytes taken from zero; dst is 16-aligned.
__device__ uint32_t warp_copy_crc(const uint8_t *src, uint64_t len, uint8_t *dst, const CrcSmem &cs) {
    const int lane = threadIdx.x & 31;
    const uint32_t *row = crc_row<kCodeCrcCopies>(cs.rep);
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    const EndAligned ea(uint32_t(len / 16));
    constexpr int U = 8;
    uint32_t R = 0;
    for (uint32_t r0 = 0; r0 < ea.rounds; r0 += U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t v = int64_t(32) * (r0 + u) + lane - ea.v0;
            t[u] = (r0 + u < ea.rounds && v >= 0) ? __ldcs(s4 + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const uint32_t r = r0 + u;
            if (r >= ea.rounds) break;
            const int64_t v = int64_t(32) * r + lane - ea.v0;
            if (r > 0) R = shift_smem(R, cs.gap496);
            if (v >= 0) {
                d4[v] = t[u];
                R = crc_rep16<kCodeCrcCopies>(R, t[u], row);
            }
        }
    }
    return ea.rounds ? crc_fold<1, 4>(R, nullptr) : 0u;
}

// Format v3: copy a record staged by rans_encode_stream<true> into the blob
// (len bytes, a multiple of 16) and return its CRC register taken from
// zero: the head and the counts (lists_at bytes) as they are, then output
// block ob of the lists from lane l's staged list, l the lane with
// boff_l <= ob < boff_l + the lane's padded count / 8 (boff_l = the blocks
// of the lanes below). The pieces go round-robin as in warp_copy_crc.
__device__ uint32_t warp_copy_crc_lanes(const uint8_t *rec, uint32_t len, uint32_t lists_at, uint32_t Ts,
                                        uint8_t *dst, const CrcSmem &cs) {
    const int lane = threadIdx.x & 31;
    const uint32_t *row = crc_row<kCodeCrcCopies>(cs.rep);
    const uint32_t cnt = reinterpret_cast<const uint16_t *>(rec + lists_at - 64)[lane];
    const uint32_t blocks = (cnt + 7) / 8;
    const uint32_t boff = warp_excl_scan(blocks);
    const uint32_t head = lists_at / 16;
    // every lane runs the whole search (its shuffles need all 32 lanes),
    // whichever part of the record its piece is in
    auto src_of = [&](uint32_t v) -> const uint4 * {
        const uint32_t ob = v < head ? 0u : v - head;
        uint32_t lo = 0, hi = 32;  // the last lane whose first block is at or before ob
#pragma unroll
        for (int it = 0; it < 5; it++) {
            const uint32_t mid = (lo + hi) >> 1;
            if (__shfl_sync(kFull, boff, mid) <= ob) lo = mid;
            else hi = mid;
        }
        const uint32_t base = __shfl_sync(kFull, boff, lo);
        const uint4 *list = reinterpret_cast<const uint4 *>(rec + lists_at + 2ull * lo * Ts) + (ob - base);
        return v < head ? reinterpret_cast<const uint4 *>(rec) + v : list;
    };
    const EndAligned ea(len / 16);
    constexpr int U = 8;
    uint32_t R = 0;
    for (uint32_t r0 = 0; r0 < ea.rounds; r0 += U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t v = int64_t(32) * (r0 + u) + lane - ea.v0;
            const uint32_t vv = v < 0 ? 0u : uint32_t(v);
            const uint4 *sp = src_of(vv);  // every lane takes part in the search's shuffles
            t[u] = (r0 + u < ea.rounds && v >= 0) ? __ldcs(sp) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const uint32_t r = r0 + u;
            if (r >= ea.rounds) break;
            const int64_t v = int64_t(32) * r + lane - ea.v0;
            if (r > 0) R = shift_smem(R, cs.gap496);
            if (v >= 0) {
                reinterpret_cast<uint4 *>(dst)[v] = t[u];
                R = crc_rep16<kCodeCrcCopies>(R, t[u], row);
            }
        }
    }
    return ea.rounds ? crc_fold<1, 4>(R, nullptr) : 0u;
}

// Copy the len bytes of a source (zero-padded to 16) by the warp, 8 vectors
// in flight per lane; dst is 16-aligned.
template <bool kDelta>
__device__ void warp_copy_src(Source<kDelta> src, uint64_t len, uint8_t *dst) {
    const int lane = threadIdx.x & 31;
    const uint64_t nvec = (src.addr_bits() & 15) ? 0 : len / 16;
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    constexpr int U = 8;
    for (uint64_t v0 = lane; v0 < nvec; v0 += 32 * U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; u++)
            if (v0 + 32 * u < nvec) t[u] = src.vec_last(16 * (v0 + 32 * u));
#pragma unroll
        for (int u = 0; u < U; u++)
            if (v0 + 32 * u < nvec) d4[v0 + 32 * u] = t[u];
    }
    for (uint64_t i = nvec * 16 + lane; i < pad16(len); i += 32) dst[i] = i < len ? uint8_t(src.byte(i)) : 0;
}

template <int DT, int J>
__device__ __forceinline__ void code_stream(const EncodeArgs &a, uint32_t cl, uint32_t t, uint32_t n, uint64_t lim,
                                            uint4 *etab, uint8_t *ring, uint8_t *slot, uint32_t mode[4],
                                            uint32_t val[4]) {
    constexpr int W = WordOf<DT>::W;
    if (mode[J] != kModeCand) return;
    const int lane = threadIdx.x & 31;
    // v1: the chunk's own table; v2: its tensor's plane table
    const uint8_t *ftab = a.version == 2 ? a.ws_ptab + (uint64_t(t) * W + J) * 512
                                         : a.ws_ftab + (uint64_t(cl) * W + J) * 512;
    const uint4 fv = reinterpret_cast<const uint4 *>(ftab)[lane];
    const uint32_t f[8] = {fv.x & 0xFFFFu, fv.x >> 16, fv.y & 0xFFFFu, fv.y >> 16,
                           fv.z & 0xFFFFu, fv.z >> 16, fv.w & 0xFFFFu, fv.w >> 16};
    const uint8_t *cand = a.ws_cand + (uint64_t(cl) * W + J) * a.n_pad;
    uint16_t *stage = reinterpret_cast<uint16_t *>(ring + 4096);
    uint8_t *rec = slot + uint64_t(J) * a.rec_stride;
    const uint32_t rb = a.version == 3 ? rans_encode_stream<true>(cand, n, f, etab, ring, stage, rec, lim, false)
                                       : rans_encode_stream<false>(cand, n, f, etab, ring, stage, rec, lim,
                                                                   a.version == 2);
    if (rb != kAborted && rb < lim) {
        mode[J] = kModeRans;
        val[J] = rb;
    } else {
        mode[J] = kModeRaw;
        val[J] = n;
    }
}

template <int DT, bool kDelta>
__global__ void __launch_bounds__(kCodeThreads, 1) code_kernel(EncodeArgs a) {
    constexpr int W = WordOf<DT>::W;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t gw = blockIdx.x * (blockDim.x >> 5) + warp;
    // the CTA's CRC tables, then 12 KB per warp
    uint32_t *crc_rep = reinterpret_cast<uint32_t *>(smem_raw);
    uint32_t(*gap496)[256] = reinterpret_cast<uint32_t(*)[256]>(smem_raw + crc_rep_words<kCodeCrcCopies>() * 4);
    load_crc_rep<kCodeCrcCopies>(crc_rep);
    load_shift_smem(gap496, kSh496);
    __syncthreads();
    if (gw >= a.workers) return;
    const CrcSmem cs{crc_rep, gap496};
    uint8_t *warp_smem = smem_raw + kCodeCrcBytes + kCodeWarpSmem * warp;
    uint4 *etab = reinterpret_cast<uint4 *>(warp_smem);
    uint8_t *ring = warp_smem + 4096;
    uint8_t *slot = a.ws_slots + uint64_t(gw) * a.slot_bytes;
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws_ctrl);

    for (;;) {
        uint32_t cl = 0;
        if (lane == 0) cl = atomicAdd(&ctrl[0], 1u);
        cl = __shfl_sync(kFull, cl, 0);
        if (cl >= a.wave_n) break;
        const uint32_t g = a.wave_start + cl;
        const TView tv = tensor_view(a, g);
        const uint32_t c = g - tv.chunk_base;  // chunk of its tensor
        // the tensor's done counter, header-CRC accumulator and (v2) plane-table CRC
        uint32_t *tctrl = ctrl + 64 + 4 * tv.t;
        // payloads start after the chunk table (v2: and the W plane tables)
        const uint64_t table_end = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * tv.n_chunks +
                                   (a.version == 2 ? 512ull * W : 0ull);
        const Source<kDelta> src = Source<kDelta>{tv.src, tv.base}.at(uint64_t(c) * a.chunk_bytes);
        const uint32_t len = uint32_t(umin64(a.chunk_bytes, tv.nbytes - uint64_t(c) * a.chunk_bytes));
        const uint32_t n = len / W;
        const uint32_t *info = reinterpret_cast<const uint32_t *>(a.ws_info + 32ull * cl);
        uint32_t mode[4] = {0, 0, 0, 0}, val[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < W; j++) {
            const uint32_t sv = info[1 + j];
            mode[j] = sv >> 30;
            val[j] = sv & 0x3FFFFFFFu;
        }
        // a record is kept iff its size is below threshold x n, i.e. below lim
        const uint64_t lim = uint64_t(ceil(a.threshold * double(n)));
        code_stream<DT, 0>(a, cl, tv.t, n, lim, etab, ring, slot, mode, val);
        if constexpr (W > 1) code_stream<DT, 1>(a, cl, tv.t, n, lim, etab, ring, slot, mode, val);
        if constexpr (W > 2) {
            code_stream<DT, 2>(a, cl, tv.t, n, lim, etab, ring, slot, mode, val);
            code_stream<DT, 3>(a, cl, tv.t, n, lim, etab, ring, slot, mode, val);
        }

        uint64_t grouped = 16;  // pad16(4W) for W <= 4
        uint32_t roff[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < W; j++) {
            roff[j] = uint32_t(grouped);
            if (mode[j] != kModeConst) grouped += pad16(val[j]);
        }
        const bool raw_chunk = !(double(grouped) < a.threshold * double(len));
        const uint64_t stored = raw_chunk ? len : grouped;
        bool timed;
        const uint64_t off = table_end + lookback(a.ws_status + tv.chunk_base, c, pad16(stored), a.d_status, &timed,
                                                 a.spin_limit, a.hooks);
        const bool fits = off + pad16(stored) <= tv.cap;
        if (!fits && lane == 0) status_or(a.d_status, ZC_ECAPACITY);

        if (fits && !timed) {
            uint8_t *out = tv.blob + off;
            // CRC-32 of the stored bytes, taken as they are written: the
            // register of each part taken from zero, appended in payload order
            uint32_t reg;
            if (raw_chunk) {
                // a copy of the chunk; its CRC from the written bytes (L2)
                warp_copy_src(src, len, out);
                __syncwarp();
                reg = crc_strided<1, true, kCodeCrcCopies>(out, len, 0xFFFFFFFFu, crc_rep, gap496, nullptr);
            } else {
                // directory: W words mode << 30 | value, zero-padded to 16 bytes
                uint32_t e[4] = {0, 0, 0, 0};
#pragma unroll
                for (int j = 0; j < W; j++) e[j] = (mode[j] << 30) | val[j];
                if (lane == 0) reinterpret_cast<uint4 *>(out)[0] = make_uint4(e[0], e[1], e[2], e[3]);
                reg = crc_rep16<kCodeCrcCopies>(0xFFFFFFFFu, make_uint4(e[0], e[1], e[2], e[3]),
                                                crc_row<kCodeCrcCopies>(crc_rep));
                uint32_t part[4];
                warp_raw_streams<DT, kDelta>(src, n, mode, roff, out, cs, part);
#pragma unroll
                for (int j = 0; j < W; j++) {
                    if (mode[j] != kModeRans) continue;
                    const uint8_t *rec = slot + uint64_t(j) * a.rec_stride;
                    if (a.version == 3) {
                        // v3: the lists follow the table and the counts
                        const uint32_t k = warp_sum_u32(__popc(rec[128 + lane]));
                        const uint32_t lists_at = kRecHead + uint32_t(pad16(2 * k)) + 64;
                        const uint32_t Ts = ((n + 31) / 32 + 7) & ~7u;
                        part[j] = warp_copy_crc_lanes(rec, val[j], lists_at, Ts, out + roff[j], cs);
                    } else {
                        part[j] = warp_copy_crc(rec, pad16(val[j]), out + roff[j], cs);
                    }
                }
#pragma unroll
                for (int j = 0; j < W; j++) {
                    if (mode[j] == kModeConst) continue;
                    reg = crc_append_small(reg, part[j], uint32_t(mode[j] == kModeRaw ? pad16(n) : pad16(val[j])));
                }
            }
            const uint32_t crc = reg ^ 0xFFFFFFFFu;
            if (lane == 0) {
                uint4 ent;
                ent.x = uint32_t(off);
                ent.y = uint32_t(off >> 32);
                ent.z = uint32_t(stored) | (raw_chunk ? 0x80000000u : 0u);
                ent.w = crc;
                reinterpret_cast<uint4 *>(tv.blob + ZC_HEADER_BYTES)[c] = ent;
                // header CRC = shift(crc(header), 16 n) ^ XOR_c shift(crc(entry_c), 16 (n-1-c))
                uint32_t ec = 0xFFFFFFFFu;
                ec = crc_word_global(ec, ent.x);
                ec = crc_word_global(ec, ent.y);
                ec = crc_word_global(ec, ent.z);
                ec = crc_word_global(ec, ent.w) ^ 0xFFFFFFFFu;
                atomicXor(&tctrl[1], shift_bytes(ec, 16ull * (tv.n_chunks - 1 - c)));
            }
        }
        if (lane == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(&tctrl[0], 1u);
            if (done == tv.n_chunks - 1) {
                // the tensor's last chunk: its header and blob length
                __threadfence();
                const uint32_t acc = atomicXor(&tctrl[1], 0u);
                const unsigned long long last = ld_acquire(&a.ws_status[tv.chunk_base + tv.n_chunks - 1]);
                const uint64_t total = table_end + (last & kValMask);
                const uint32_t *header = a.n_tensors == 1 ? a.one.header : a.tensors[tv.t].header;
                uint64_t *d_blob_bytes = a.n_tensors == 1 ? a.one.d_blob_bytes : a.tensors[tv.t].d_blob_bytes;
                uint32_t hc = 0xFFFFFFFFu;
                for (int q = 0; q < 24; q++) hc = crc_word_global(hc, header[q]);
                hc ^= 0xFFFFFFFFu;
                uint32_t hcrc = shift_bytes(hc, 16ull * tv.n_chunks) ^ acc;
                // v2: the CRC runs on over the plane tables that follow
                if (a.version == 2) hcrc = shift_bytes(hcrc, 512ull * W) ^ atomicXor(&tctrl[2], 0u);
                uint32_t *hdr = reinterpret_cast<uint32_t *>(tv.blob);
                for (int q = 0; q < 24; q++) hdr[q] = (q == 7) ? hcrc : header[q];
                *d_blob_bytes = total;
            }
        }
        __syncwarp();
    }
}

// A blob of an empty tensor is its header alone (v2: and W zero plane
// tables); its CRC is made on the host.
__global__ void empty_blob_kernel(EncodeArgs a) {
    for (uint32_t t = blockIdx.x; t < a.n_tensors; t += gridDim.x) {
        const TensorDesc &d = a.n_tensors == 1 ? a.one : a.tensors[t];
        if (d.n_chunks != 0) continue;
        uint32_t *b = reinterpret_cast<uint32_t *>(d.blob);
        if (threadIdx.x < 24) b[threadIdx.x] = d.header[threadIdx.x];
        const int W = word_bytes(int(d.header[1] >> 16) & 0xFF);
        const uint32_t plane_words = a.version == 2 ? 128u * W : 0u;
        for (uint32_t i = threadIdx.x; i < plane_words; i += blockDim.x) b[24 + i] = 0;
        if (threadIdx.x == 0) *d.d_blob_bytes = ZC_HEADER_BYTES + 4ull * plane_words;
    }
}

// v2: the plane tables of the wave's tensors, one warp per tensor and plane.
// The plane's counts over the whole tensor (every chunk's statistics have
// been added) give its 12-bit table, or zeros for fewer than two symbols.
// The table goes to the blob (after the chunk table) and to the workspace
// for the coder; the CRC of the W tables (512 bytes each, in plane order)
// is accumulated into the tensor's control word for the header CRC.
template <int W>
__global__ void plane_kernel(EncodeArgs a) {
    const int lane = threadIdx.x & 31;
    const uint32_t gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const uint32_t t = a.wave_t0 + gw / W, j = gw % W;
    if (t >= a.wave_t1) return;
    const TensorDesc &d = a.n_tensors == 1 ? a.one : a.tensors[t];
    if (d.n_chunks == 0) return;  // written whole by empty_blob_kernel
    const unsigned long long *h = a.ws_hist + (uint64_t(t) * W + j) * 256;
    unsigned long long cnt[8];
    uint32_t pres = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        cnt[k] = h[8 * lane + k];
        pres += cnt[k] ? 1u : 0u;
    }
    uint32_t f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (warp_sum_u32(pres) >= 2) normalize_plane_warp(cnt, d.nbytes / W, f);
    uint4 v;
    v.x = f[0] | f[1] << 16;
    v.y = f[2] | f[3] << 16;
    v.z = f[4] | f[5] << 16;
    v.w = f[6] | f[7] << 16;
    const uint64_t at = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * d.n_chunks + 512ull * j;
    reinterpret_cast<uint4 *>(d.blob + at)[lane] = v;
    reinterpret_cast<uint4 *>(a.ws_ptab + (uint64_t(t) * W + j) * 512)[lane] = v;
    // CRC(P_0 .. P_{W-1}) = XOR over the 16-byte pieces of shift(CRC(piece),
    // bytes after it), by linearity
    uint32_t c = 0xFFFFFFFFu;
    c = crc_word_global(c, v.x);
    c = crc_word_global(c, v.y);
    c = crc_word_global(c, v.z);
    c = crc_word_global(c, v.w) ^ 0xFFFFFFFFu;
    c = shift_bytes(c, 16ull * (31 - lane) + 512ull * (W - 1 - j));
    c = __reduce_xor_sync(kFull, c);
    if (lane == 0) atomicXor(reinterpret_cast<uint32_t *>(a.ws_ctrl) + 64 + 4 * t + 2, c);
}

int sms_of_device() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

template <int DT, bool kDelta>
int launch_wave_t(const EncodeArgs &a, cudaStream_t s) {
    constexpr int W = WordOf<DT>::W;
    const size_t ssm = sizeof(StatsSmem<W>);
    const size_t csm = kCodeCrcBytes + size_t(kCodeWarps) * kCodeWarpSmem;
    if (cudaFuncSetAttribute(stats_kernel<DT, kDelta>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(ssm)) != cudaSuccess)
        return ZC_ECUDA;
    if (cudaFuncSetAttribute(code_kernel<DT, kDelta>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(csm)) != cudaSuccess)
        return ZC_ECUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stats_kernel<DT, kDelta>, kStatThreads, ssm) != cudaSuccess)
        return ZC_ECUDA;
    const uint64_t most = uint64_t(per_sm < 1 ? 1 : per_sm) * uint64_t(sms_of_device() < 1 ? 1 : sms_of_device());
    const int sgrid = int(a.wave_n < most ? a.wave_n : most);
    stats_kernel<DT, kDelta><<<sgrid, kStatThreads, ssm, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return ZC_ECUDA;
    if (a.version == 2) {  // the wave holds whole tensors: their plane tables are complete now
        const int st = launch_plane_tables(DT, a, s);
        if (st != ZC_OK) return st;
    }
    // the warps spread evenly over the SMs: CTAs of just enough warps for one
    // CTA per SM (the block scheduler then gives every SM the same share);
    // ZC_PACKED: CTAs of up to kCodeWarps warps, on as few SMs as they fill
    const int sms = sms_of_device() < 1 ? 1 : sms_of_device();
    const uint32_t wpc = a.packed ? std::min<uint32_t>(kCodeWarps, a.workers)
                                  : std::min<uint32_t>(kCodeWarps, (a.workers + sms - 1) / sms);
    const int cgrid = int((a.workers + wpc - 1) / wpc);
    code_kernel<DT, kDelta><<<cgrid, 32 * wpc, kCodeCrcBytes + size_t(wpc) * kCodeWarpSmem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

} // namespace

int launch_empty_blobs(const EncodeArgs &a, cudaStream_t s) {
    empty_blob_kernel<<<std::min<uint32_t>(a.n_tensors, 1024), 32, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

int launch_plane_tables(int dtype, const EncodeArgs &a, cudaStream_t s) {
    const int W = word_bytes(dtype);
    const uint32_t warps = (a.wave_t1 - a.wave_t0) * uint32_t(W);
    if (warps == 0) return ZC_OK;
    const uint32_t grid = (warps + 3) / 4;
    switch (W) {
    case 1: plane_kernel<1><<<grid, 128, 0, s>>>(a); break;
    case 2: plane_kernel<2><<<grid, 128, 0, s>>>(a); break;
    case 4: plane_kernel<4><<<grid, 128, 0, s>>>(a); break;
    default: return ZC_EINVAL;
    }
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

int launch_encode_wave(int dtype, bool delta, const EncodeArgs &a, cudaStream_t s) {
    if (a.total_chunks == 0) return ZC_EINVAL;
    switch (dtype) {
    case ZC_U8: return delta ? launch_wave_t<ZC_U8, true>(a, s) : launch_wave_t<ZC_U8, false>(a, s);
    case ZC_U16: return delta ? launch_wave_t<ZC_U16, true>(a, s) : launch_wave_t<ZC_U16, false>(a, s);
    case ZC_U32: return delta ? launch_wave_t<ZC_U32, true>(a, s) : launch_wave_t<ZC_U32, false>(a, s);
    // deltas are compressed as unsigned words only
    case ZC_BF16: return delta ? ZC_EINVAL : launch_wave_t<ZC_BF16, false>(a, s);
    case ZC_FP16: return delta ? ZC_EINVAL : launch_wave_t<ZC_FP16, false>(a, s);
    case ZC_FP32: return delta ? ZC_EINVAL : launch_wave_t<ZC_FP32, false>(a, s);
    default: return ZC_EINVAL;
    }
}

int encode_warps_per_sm() { return kCodeWarps; }

} // namespace zc
