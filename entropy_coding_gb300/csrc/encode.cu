// encode.cu — single-pass compression kernel.
//
// One CTA compresses one chunk at a time (ZipNN note, Method 5: fixed-size
// chunks coded independently); CTAs are persistent and take chunk indices
// from a global ticket counter, so every chunk below a CTA's chunk is already
// owned by a running CTA. Per chunk:
//   1. all warps build one 256-bin histogram per byte stream (order-0
//      statistics, ZipNN note Key insight) of the exponent-extracted words;
//   2. warp j takes stream j: a constant stream needs no record; otherwise it
//      quantises the histogram to a 12-bit table, skips the stream if it
//      provably cannot shrink below the threshold, and else rANS-codes it
//      (32 interleaved lanes) into the CTA's workspace slot;
//   3. warp 0 applies the passthrough rule per stream and per chunk (cuZipNN
//      API, passthrough_threshold), publishes the chunk's padded size and
//      finds its blob offset with a decoupled look-back over the chunks
//      before it (an exclusive prefix scan of the metadata map, ZipNN note
//      Method 5);
//   4. all warps write the payload: the directory, the raw streams (one pass
//      over the input for all of them), the coded records; then compute its
//      CRC-32 together and write the chunk table entry.
// The last CTA to finish writes the header and its CRC.
#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kCtasPerSM = 3;
constexpr uint64_t kFlagAgg = 1ull << 62, kFlagPre = 2ull << 62, kValMask = (1ull << 62) - 1;
constexpr uint32_t kSpinLimit = 1u << 22;

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

// Histogram of the W byte streams of one chunk into h[W][256], by the CTA,
// and the raw CRC register of the chunk's bytes (the chunk table's check of
// the original data) from the same loads: the 16-byte pieces are dealt to
// the threads as in crc_strided, so each thread's register only needs the
// gap shift between its pieces. Returns the raw register in every thread.
template <int DT>
__device__ uint32_t chunk_stats(const uint8_t *src, uint32_t len, uint32_t (*h)[256], const uint32_t *crc_rep,
                                const uint32_t (*gap)[256], uint32_t *s_reg) {
    constexpr int W = WordOf<DT>::W;
    const int tid = threadIdx.x;
    const uint32_t *row = crc_rep + (tid & 31);
    for (int i = tid; i < W * 256; i += kThreads) h[i >> 8][i & 255] = 0;
    __syncthreads();
    auto count = [&](uint32_t w) {
        const uint32_t p = Perm<DT>::fwd(w);
#pragma unroll
        for (int j = 0; j < W; j++) atomicAdd(&h[j][stream_byte<W>(p, j)], 1u);
    };
    uint32_t reg;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const uint32_t main = len & ~15u;
        const Strided sp(main, kThreads);
        uint32_t R = 0;
        int64_t pidx = int64_t(tid) - int64_t(sp.v0);
        constexpr int U = 4;  // pieces in flight per thread
        for (uint64_t r0 = 0; r0 < sp.rounds; r0 += U) {
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t pi = pidx + int64_t(u) * kThreads;
                q[u] = (r0 + u < sp.rounds && pi >= 0) ? __ldg(reinterpret_cast<const uint4 *>(src) + pi)
                                                      : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                if (r0 + u >= sp.rounds) break;
                const int64_t pi = pidx + int64_t(u) * kThreads;
                uint32_t c = (r0 + u == 0) ? (pi == 0 ? 0xFFFFFFFFu : 0u) : shift_smem(R, gap);
                if (pi >= 0) {
                    c = crc_rep16(c, q[u], row);
                    const uint32_t uu[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                    for (int k = 0; k < 4; k++)
#pragma unroll
                        for (int e = 0; e < 4 / W; e++)
                            count(W == 4 ? uu[k] : (uu[k] >> (8 * W * e)) & ((1u << (8 * W)) - 1u));
                }
                R = c;
            }
            pidx += int64_t(U) * kThreads;
        }
        reg = sp.pieces ? crc_fold<kWarps>(R, 4, s_reg) : 0xFFFFFFFFu;
        for (uint32_t i = main; i < len; i++) reg = crc_rep_byte(reg, __ldg(src + i), row);
        for (uint32_t i = main / W + tid; i < len / W; i += kThreads) count(load_word<W>(src + uint64_t(i) * W));
    } else {
        // unaligned input: words one at a time; the CRC takes the bytes up to
        // the first 16-byte boundary one by one, then the aligned rest
        for (uint32_t i = tid; i < len / W; i += kThreads) count(load_word<W>(src + uint64_t(i) * W));
        uint32_t head = uint32_t((16 - (reinterpret_cast<uintptr_t>(src) & 15)) & 15);
        if (head > len) head = len;
        uint32_t c = 0xFFFFFFFFu;
        for (uint32_t i = 0; i < head; i++) c = crc_rep_byte(c, __ldg(src + i), row);
        reg = crc_strided<kWarps, false>(src + head, len - head, c, crc_rep, gap, s_reg);
    }
    __syncthreads();
    return reg;
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

// Exclusive prefix of this chunk's padded size over the chunks before it
// (decoupled look-back, one warp). Every wait is bounded; a timeout sets
// ZC_ETIMEOUT and the chunk is not placed.
__device__ uint64_t lookback(unsigned long long *st, uint32_t c, uint64_t agg, int32_t *d_status, bool *timed) {
    const int lane = threadIdx.x & 31;
    *timed = false;
    if (c == 0) {
        if (lane == 0) st_release(&st[0], kFlagPre | agg);
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
                if (++spins > kSpinLimit) {
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

// Code stream J of the chunk into rec (the workspace record area), one warp.
// Returns the record's unpadded size. f holds the lane's 8 table entries.
// Per symbol the table keeps {m, a, 2^20 f, (4096 - f) | cum << 13 | (k-32) << 25}
// so that a step is: renormalise if x >= 2^20 f, q = (x m + a) >> k,
// x += q (4096 - f) + cum.
template <int DT, int J>
__device__ uint32_t rans_encode_stream(const uint8_t *src, uint32_t n, const uint32_t f[8], uint4 *etab, uint8_t *rec) {
    constexpr int W = WordOf<DT>::W;
    const int lane = threadIdx.x & 31;
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
            reinterpret_cast<uint16_t *>(rec + kRecHead)[rank++] = uint16_t(fs);
            const uint32_t ka = kRecip.ka[fs], m = kRecip.m[fs];
            etab[s] = make_uint4(m, (ka >> 8) ? m : 0u, fs << 20, (kM - fs) | (cum << 13) | (((ka & 0xFFu) - 32) << 25));
        }
        cum += fs;
    }
    rec[128 + lane] = uint8_t(bits);
    const uint32_t words_at = kRecHead + uint32_t(pad16(2 * k_total));
    for (uint32_t b = kRecHead + 2 * k_total + lane; b < words_at; b += 32) rec[b] = 0;
    __syncwarp();

    uint16_t *wout = reinterpret_cast<uint16_t *>(rec + words_at);
    const uint32_t gt = lanemask_gt();
    uint32_t x = kRansL;
    uint32_t wc = 0;
    const int T = int((n + 31) / 32);

    auto sym_of = [&](uint32_t word) { return stream_byte<W>(Perm<DT>::fwd(word), J); };
    auto step = [&](const uint4 &e, bool active) {
        const bool emit = active && x >= e.z;
        const uint32_t bal = __ballot_sync(kFull, emit);
        // the store reads its own copy of x, so updating x need not wait for it
        uint32_t wv;
        asm volatile("mov.b32 %0, %1;" : "=r"(wv) : "r"(x));
        const uint32_t pos = wc + __popc(bal & gt);
        if (emit) wout[pos] = uint16_t(wv);
        x = emit ? x >> 16 : x;
        wc += __popc(bal);
        const uint32_t q = uint32_t((uint64_t(x) * e.x + e.y) >> 32) >> ((e.w >> 25) & 0xFu);
        const uint32_t xn = x + q * (e.w & 0x1FFFu) + ((e.w >> 13) & 0xFFFu);
        if (active) x = xn;
    };

    // the last step first (the only one that may be partial)
    {
        const uint32_t i = uint32_t(T - 1) * 32 + lane;
        const bool active = i < n;
        step(etab[sym_of(active ? load_word<W>(src + uint64_t(i) * W) : 0u)], active);
    }
    // then the full steps T-2 .. 0, 16 at a time with the next 16 words in
    // flight; each step's table entry is read one step ahead
    constexpr int B = 16;
    uint32_t buf[B];
#pragma unroll
    for (int k = 0; k < B; k++) {
        const int t = T - 2 - k;
        buf[k] = t >= 0 ? load_word<W>(src + (uint64_t(t) * 32 + lane) * W) : 0u;
    }
    uint4 e_next = etab[sym_of(buf[0])];
    for (int t0 = T - 2; t0 >= 0; t0 -= B) {
        uint32_t nxt[B];
#pragma unroll
        for (int k = 0; k < B; k++) {
            const int t = t0 - B - k;
            nxt[k] = t >= 0 ? load_word<W>(src + (uint64_t(t) * 32 + lane) * W) : 0u;
        }
        const bool full = t0 >= B - 1;
#pragma unroll
        for (int k = 0; k < B; k++) {
            const uint4 e = e_next;
            e_next = etab[sym_of(k + 1 < B ? buf[k + 1] : nxt[0])];
            if (full || t0 - k >= 0) step(e, true);
        }
#pragma unroll
        for (int k = 0; k < B; k++) buf[k] = nxt[k];
    }
    reinterpret_cast<uint32_t *>(rec)[lane] = x;
    const uint32_t rec_bytes = words_at + 2 * wc;
    for (uint32_t b = rec_bytes + lane; b < pad16(rec_bytes); b += 32) rec[b] = 0;
    __syncwarp();
    return rec_bytes;
}

struct Plan {
    uint32_t mode[4];
    uint32_t val[4];   // RAW: n, RANS: record bytes, CONST: symbol
    uint32_t roff[4];  // record offset within the payload
    uint64_t off;      // payload offset in the blob
    uint64_t stored;
    uint32_t raw_chunk;
    uint32_t write;    // 0 when the chunk is not placed (capacity or timeout)
    uint32_t c;
    uint32_t crc;      // CRC-32 of the chunk's original bytes
    uint32_t crc_reg[kWarps];
};

// Per-stream decision, by warp j for stream j.
template <int DT, int J>
__device__ void plan_stream(const EncodeArgs &a, const uint8_t *src, uint32_t n, const uint32_t (*h)[256],
                            uint4 *etab, uint8_t *rec, Plan &pl) {
    constexpr int j = J;
    const int lane = threadIdx.x & 31;
    uint32_t cnt[8];
#pragma unroll
    for (int k = 0; k < 8; k++) cnt[k] = h[j][8 * lane + k];
    uint32_t pres = 0, only = 0;
#pragma unroll
    for (int k = 0; k < 8; k++)
        if (cnt[k]) {
            pres++;
            only = 8 * lane + k;
        }
    const uint32_t k_total = warp_sum_u32(pres);
    uint32_t mode, val;
    if (k_total == 1) {
        const uint32_t who = __ballot_sync(kFull, pres != 0);
        mode = kModeConst;
        val = __shfl_sync(kFull, only, __ffs(who) - 1);
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
            const uint32_t rb = rans_encode_stream<DT, J>(src, n, f, etab, rec);
            if (double(rb) < a.threshold * double(n)) {
                mode = kModeRans;
                val = rb;
            }
        }
    }
    if (lane == 0) {
        pl.mode[j] = mode;
        pl.val[j] = val;
    }
}

// All raw streams of a grouped chunk in one pass over the input: each thread
// takes 16 consecutive elements and writes 16 bytes to every raw stream.
template <int DT>
__device__ void write_raw_streams(const uint8_t *src, uint32_t n, const Plan &pl, uint8_t *out) {
    constexpr int W = WordOf<DT>::W;
    bool any = false;
#pragma unroll
    for (int j = 0; j < W; j++) any |= pl.mode[j] == kModeRaw;
    if (!any) return;
    const uint32_t groups = (n + 15) / 16;
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    for (uint32_t g = threadIdx.x; g < groups; g += kThreads) {
        uint32_t wd[16];
        if (vec && 16 * (g + 1) <= n) {
#pragma unroll
            for (int v = 0; v < W; v++) {
                uint4 q = __ldcs(reinterpret_cast<const uint4 *>(src + uint64_t(g) * 16 * W) + v);
                uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; k++)
#pragma unroll
                    for (int e = 0; e < 4 / W; e++)
                        wd[(v * 4 + k) * (4 / W) + e] =
                            (W == 4) ? u[k] : (u[k] >> (8 * W * e)) & ((1u << (8 * W)) - 1u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; k++) {
                uint32_t i = g * 16 + k;
                wd[k] = i < n ? load_word<W>(src + uint64_t(i) * W) : 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < 16; k++) wd[k] = Perm<DT>::fwd(wd[k]);
#pragma unroll
        for (int j = 0; j < W; j++) {
            if (pl.mode[j] != kModeRaw) continue;
            uint32_t b[16];
#pragma unroll
            for (int k = 0; k < 16; k++) b[k] = (g * 16 + k < n) ? stream_byte<W>(wd[k], j) : 0u;
            uint4 v;
            v.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            v.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
            v.z = b[8] | (b[9] << 8) | (b[10] << 16) | (b[11] << 24);
            v.w = b[12] | (b[13] << 8) | (b[14] << 16) | (b[15] << 24);
            reinterpret_cast<uint4 *>(out + pl.roff[j])[g] = v;
        }
    }
}

// Copy len bytes (zero-padded to 16) by the CTA; dst is 16-aligned.
__device__ void block_copy(const uint8_t *src, uint64_t len, uint8_t *dst) {
    const uint64_t nvec = (reinterpret_cast<uintptr_t>(src) & 15) ? 0 : len / 16;
    for (uint64_t v = threadIdx.x; v < nvec; v += kThreads)
        reinterpret_cast<uint4 *>(dst)[v] = __ldcs(reinterpret_cast<const uint4 *>(src) + v);
    for (uint64_t i = nvec * 16 + threadIdx.x; i < pad16(len); i += kThreads) dst[i] = i < len ? src[i] : 0;
}

// Dynamic shared memory of the compression CTA.
template <int W>
struct EncodeSmem {
    uint32_t crc_rep[kCrcRepWords];  // replicated CRC byte table (32 KB)
    uint32_t gap[4][256];            // register shift over the other threads' pieces
    uint32_t hist[W][256];
    uint4 etab[W][256];
    Plan pl;
};

template <int DT>
__global__ void __launch_bounds__(kThreads, kCtasPerSM) encode_kernel(EncodeArgs a) {
    constexpr int W = WordOf<DT>::W;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    EncodeSmem<W> &sm = *reinterpret_cast<EncodeSmem<W> *>(smem_raw);
    Plan &pl = sm.pl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    load_crc_rep(sm.crc_rep);
    load_shift_smem(sm.gap, gap_table<kThreads>());
    const uint32_t *row = sm.crc_rep + lane;

    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws_ctrl);
    uint8_t *slot = a.ws_slots + uint64_t(blockIdx.x) * a.slot_bytes;
    const uint64_t table_end = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * a.n_chunks;
    const uint64_t rec_stride = pad16(kRecHead + kMaxTable + 2ull * (a.chunk_bytes / W));

    for (;;) {
        if (tid == 0) pl.c = atomicAdd(&ctrl[0], 1u);
        __syncthreads();
        const uint32_t c = pl.c;
        if (c >= a.n_chunks) break;
        const uint8_t *src = a.src + uint64_t(c) * a.chunk_bytes;
        const uint32_t len = uint32_t(umin64(a.chunk_bytes, a.nbytes - uint64_t(c) * a.chunk_bytes));
        const uint32_t n = len / W;

        const uint32_t crc = chunk_stats<DT>(src, len, sm.hist, sm.crc_rep, sm.gap, pl.crc_reg) ^ 0xFFFFFFFFu;

        if (warp == 0) plan_stream<DT, 0>(a, src, n, sm.hist, sm.etab[0], slot, pl);
        if constexpr (W > 1) {
            if (warp == 1) plan_stream<DT, 1>(a, src, n, sm.hist, sm.etab[1], slot + rec_stride, pl);
        }
        if constexpr (W > 2) {
            if (warp == 2) plan_stream<DT, 2>(a, src, n, sm.hist, sm.etab[2], slot + 2 * rec_stride, pl);
            if (warp == 3) plan_stream<DT, 3>(a, src, n, sm.hist, sm.etab[3], slot + 3 * rec_stride, pl);
        }
        __syncthreads();

        if (warp == 0) {
            uint64_t grouped = 16;  // pad16(4W) for W <= 4
            uint32_t roff[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < W; j++) {
                roff[j] = uint32_t(grouped);
                if (pl.mode[j] != kModeConst) grouped += pad16(pl.val[j]);
            }
            const bool raw_chunk = !(double(grouped) < a.threshold * double(len));
            const uint64_t stored = raw_chunk ? len : grouped;
            bool timed;
            const uint64_t off = table_end + lookback(a.ws_status, c, pad16(stored), a.d_status, &timed);
            const bool fits = off + pad16(stored) <= a.cap;
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < W; j++) pl.roff[j] = roff[j];
                pl.off = off;
                pl.stored = stored;
                pl.raw_chunk = raw_chunk;
                pl.write = fits && !timed;
                if (!fits) status_or(a.d_status, ZC_ECAPACITY);
            }
        }
        __syncthreads();

        if (pl.write) {
            uint8_t *out = a.blob + pl.off;
            if (pl.raw_chunk) {
                block_copy(src, len, out);
            } else {
                if (tid < 4) {
                    uint32_t e = 0;
#pragma unroll
                    for (int j = 0; j < W; j++)
                        if (tid == j) e = (pl.mode[j] << 30) | pl.val[j];
                    reinterpret_cast<uint32_t *>(out)[tid] = e;
                }
                write_raw_streams<DT>(src, n, pl, out);
#pragma unroll
                for (int j = 0; j < W; j++)
                    if (pl.mode[j] == kModeRans)
                        block_copy(slot + uint64_t(j) * rec_stride, pad16(pl.val[j]), out + pl.roff[j]);
            }
            if (tid == 0) {
                uint4 ent;
                ent.x = uint32_t(pl.off);
                ent.y = uint32_t(pl.off >> 32);
                ent.z = uint32_t(pl.stored) | (pl.raw_chunk ? 0x80000000u : 0u);
                ent.w = crc;
                reinterpret_cast<uint4 *>(a.blob + ZC_HEADER_BYTES)[c] = ent;
                // header CRC = shift(crc(header), 16 n) ^ XOR_c shift(crc(entry_c), 16 (n-1-c))
                const uint32_t ec = crc_rep16(0xFFFFFFFFu, ent, row) ^ 0xFFFFFFFFu;
                atomicXor(&ctrl[2], shift_bytes(ec, 16ull * (a.n_chunks - 1 - c)));
            }
        }
        if (tid == 0) {
            __threadfence();
            const uint32_t done = atomicAdd(&ctrl[1], 1u);
            if (done == a.n_chunks - 1) {
                __threadfence();
                const uint32_t acc = atomicXor(&ctrl[2], 0u);
                const unsigned long long last = ld_acquire(&a.ws_status[a.n_chunks - 1]);
                const uint64_t total = table_end + (last & kValMask);
                uint32_t hc = 0xFFFFFFFFu;
                for (int q = 0; q < 24; q++) hc = crc_rep_word(hc, a.header[q], row);
                hc ^= 0xFFFFFFFFu;
                const uint32_t hcrc = shift_bytes(hc, 16ull * a.n_chunks) ^ acc;
                uint32_t *hdr = reinterpret_cast<uint32_t *>(a.blob);
                for (int q = 0; q < 24; q++) hdr[q] = (q == 7) ? hcrc : a.header[q];
                *a.d_blob_bytes = total;
            }
        }
        __syncthreads();
    }
}

// A blob of an empty tensor is its header alone (its CRC made on the host).
__global__ void empty_blob_kernel(EncodeArgs a) {
    if (threadIdx.x < 24) reinterpret_cast<uint32_t *>(a.blob)[threadIdx.x] = a.header[threadIdx.x];
    if (threadIdx.x == 0) *a.d_blob_bytes = ZC_HEADER_BYTES;
}

template <int DT>
int launch_encode_t(const EncodeArgs &a, int grid, cudaStream_t s) {
    const size_t smem = sizeof(EncodeSmem<WordOf<DT>::W>);
    if (cudaFuncSetAttribute(encode_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return ZC_ECUDA;
    encode_kernel<DT><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

} // namespace

int launch_encode(int dtype, const EncodeArgs &a, int grid, cudaStream_t s) {
    if (a.n_chunks == 0) {
        empty_blob_kernel<<<1, 32, 0, s>>>(a);
        return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
    }
    switch (dtype) {
    case ZC_U8: return launch_encode_t<ZC_U8>(a, grid, s);
    case ZC_U16: return launch_encode_t<ZC_U16>(a, grid, s);
    case ZC_U32: return launch_encode_t<ZC_U32>(a, grid, s);
    case ZC_BF16: return launch_encode_t<ZC_BF16>(a, grid, s);
    case ZC_FP16: return launch_encode_t<ZC_FP16>(a, grid, s);
    case ZC_FP32: return launch_encode_t<ZC_FP32>(a, grid, s);
    default: return ZC_EINVAL;
    }
}

int encode_ctas_per_sm() { return kCtasPerSM; }

} // namespace zc
