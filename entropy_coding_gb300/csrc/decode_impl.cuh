// decode_impl.cuh — the decompression kernels (included by one translation
// unit per dtype, decode_<dtype>.cu, which instantiate them for that dtype
// only, so that the kernels compile in parallel).
//
// Chunks are independent (ZipNN note, Method 5: the metadata map lets chunks
// decode in parallel); each one is restored by a pair of warps:
//   - both warps read and bounds-check the chunk table entry and the grouped
//     chunk's directory;
//   - the producer warp parses the frequency table of the chunk's first rANS
//     stream into a slot -> symbol lookup table in shared memory and runs the
//     32 interleaved rANS lanes, eight steps (256 elements) at a time, into a
//     queue of four 256-byte stage buffers;
//   - the consumer warp takes each group of symbols, gathers the bytes of 8
//     consecutive elements per lane from every stream (coded, raw or
//     constant), transposes them into words, undoes the exponent extraction
//     and stores them with vector stores. Unless the caller asked not to, it
//     also takes the CRC-32 of the chunk's stored bytes (cuZipNN API: the
//     CRCs are over pieces of the blob): the raw streams' bytes as it reads
//     them, the directory and the coded records at the end, and checks it
//     against the chunk table; a RAW chunk is a copy done by the consumer.
// So the serial chain of rANS states is the only work on the producer's
// critical path. The queue is guarded by shared-memory mbarriers; every wait
// gives up after about a second (ZC_ETIMEOUT) so that a fault in one warp
// cannot hang its partner.
// Renormalisation words are consumed from the end of each record backwards
// and staged in a four-block shared-memory ring filled by cp.async, topped up
// once per group so that a decoding step has no branch. Chunks with more than
// one coded stream first have the producer decode the other ones into the
// tail of their own output range (one byte per element and stream,
// interleaved); the consumer reads them from there, group by group, before
// any of its stores can reach them (the write front advances W bytes per
// element, the read front q < W bytes per element from (W - q) n onward, and
// they meet only at the end).
#pragma once

#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kPairs = 16;                // chunks per CTA at most, one warp pair each (one CTA per SM)
constexpr int kThreads = 64 * kPairs;
constexpr uint64_t kBigPairs = 7;        // pairs per CTA at most with one-level tables (one CTA per SM)
constexpr int kStages = 4;                // symbol groups in flight within a pair
constexpr uint32_t kLutBytes = 4096, kSymBytes = 1024, kRingWords = 1024;
// CRC slicing tables (C copies) + shift tables: one group's bytes of a
// stream (256) and the 496-byte gap
template <int C>
constexpr uint32_t crc_smem() { return crc_rep_words<C>() * 4 + 2 * 4 * 256 * 4; }
constexpr uint32_t kV2Pairs = 16;             // v2: chunks per CTA at most (one CTA per SM)
constexpr int kV2Threads = 64 * kV2Pairs;

// Shared memory of one warp pair. With kBig (few pairs per SM) the decoding
// step reads a one-level table slot -> symbol | f << 8 | (slot - cum) << 20
// instead of the two-level slot -> symbol -> (f, cum), one dependent load
// fewer per step.
template <bool kBig>
struct PairSmem {
    uint8_t lut[kLutBytes];          // slot -> symbol
    uint32_t sym[256];               // symbol -> f | cum << 12
    uint16_t ring[kRingWords];       // renormalisation words
    uint32_t big[kBig ? kM : 1];     // one-level table (kBig)
    alignas(16) uint8_t stage[kStages][256];  // decoded symbols, row k = step k of a group (read as uint2)
    unsigned long long full[kStages], empty[kStages], start;
    unsigned long long crc_bar;      // kBig: the second CRC warp's half is in crc_part
    uint32_t flag;                   // producer -> consumer: 1 when the main stream is ready
    uint32_t crc_part;
};

// Shared memory of one warp pair in format v2: the decoding tables are the
// CTA's (one per plane, shared by all its pairs), so a pair keeps only its
// word ring, its stage queue and their barriers.
struct PairSmemV2 {
    uint16_t ring[kRingWords];
    alignas(16) uint8_t stage[kStages][256];
    unsigned long long full[kStages], empty[kStages], start;
    uint32_t flag;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return uint32_t(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mbar_init(unsigned long long *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    // the thread may be suspended until the phase completes (at most 0.1 ms
    // per call), so a waiting warp takes no issue slots
    asm volatile(
        "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n\tselp.b32 %0, 1, 0, P;\n}"
        : "=r"(done)
        : "r"(smem_u32(b)), "r"(parity), "r"(100000u)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_done(unsigned long long *b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\tmbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\tselp.b32 %0, 1, 0, P;\n}"
        : "=r"(done)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait (the whole warp) until the phase of the given parity has completed;
// false after `limit` clock cycles (about a second in normal calls). A
// phase that has already completed costs one test and no clock read.
__device__ bool mbar_wait(unsigned long long *b, uint32_t parity, unsigned long long limit) {
    if (__all_sync(kFull, mbar_done(b, parity))) return true;
    const long long t0 = clock64();
    for (;;) {
        if (__all_sync(kFull, mbar_test(b, parity))) return true;
        if ((unsigned long long)(clock64() - t0) > limit) return false;
    }
}

template <int W>
__device__ __forceinline__ uint32_t load_word_any(const uint8_t *p) {
    if (W == 4) return *reinterpret_cast<const uint32_t *>(p);
    if (W == 2) return *reinterpret_cast<const uint16_t *>(p);
    return *p;
}

struct Rans {
    uint32_t x;          // this lane's state
    int32_t ptr;         // one list: words left to consume (warp-uniform); lane lists: this lane's next word (-1: none)
    int32_t lo;          // lowest 256-word block fetched so far (warp-uniform)
    const uint8_t *wbase;  // one list: the word area; lane lists: this lane's list
    uint32_t padded;     // pad16(2 * nwords)
    const uint8_t *lut;
    const uint32_t *sym;
    const uint32_t *big;
    uint16_t *ring;
    int32_t filled;      // lane lists: the lowest block of this lane's list requested into its ring
};

// Lane lists (format v3): each lane keeps the 4 blocks of 8 words of its
// list that hold its next words in shared memory, in its own 32 ring words,
// filled by asynchronous copies, so that no register waits on a global
// load. A step reads its word with one shared load whose address is known
// before the step starts. Lanes 2r and 2r + 1 share the 128-byte row r of
// the ring, one half each (swapped for r & 4), and word p of a lane's list
// is word (p & 31) ^ 8 ((r & 3)) of its half: lanes that read the same word
// of their lists (they start together and drift apart slowly) then meet 4
// to a bank instead of 16, and each 16-byte block stays whole and aligned.
__device__ __forceinline__ uint32_t lane_ring_base() {  // in words
    const uint32_t l = threadIdx.x & 31u;
    return 64u * (l >> 1) + 32u * ((l ^ (l >> 3)) & 1u);
}
__device__ __forceinline__ uint32_t lane_ring_xor() { return ((threadIdx.x >> 1) & 3u) << 3; }
__device__ __forceinline__ uint16_t *lane_slot(uint16_t *ring, int32_t b) {
    return ring + lane_ring_base() + ((8u * (uint32_t(b) & 3u)) ^ lane_ring_xor());
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Request this lane's blocks down to `lowest` (none below block 0) and
// commit them as one group.
__device__ __forceinline__ void lane_fill(Rans &r, int32_t lowest) {
    for (; r.filled > lowest && r.filled > 0;) {
        r.filled--;
        cp_async16(lane_slot(r.ring, r.filled), r.wbase + 16 * r.filled);
    }
    cp_async_commit();
}

// After every 8 steps: a lane keeps its current block and the three below
// it in its ring. A lane takes at most 8 words in 8 steps, so it crosses at
// most one block boundary between two calls and at most one block is
// requested per call; the copy for a block is requested 3 blocks before it
// is entered and waited for 3 calls later (wait_group 2: every lane commits
// one group per call).
__device__ __forceinline__ void lane_refill(Rans &r) {
    const int32_t want = (r.ptr >> 3) - 3;
    if (r.filled > want && r.filled > 0) {
        r.filled--;
        cp_async16(lane_slot(r.ring, r.filled), r.wbase + 16 * r.filled);
    }
    cp_async_commit();
    cp_async_wait<2>();
}

// Fetch 256-word block b of a record's word area into its ring slot.
__device__ __forceinline__ void fetch_block(const Rans &r, int b) {
    const int lane = threadIdx.x & 31;
    uint32_t byte = uint32_t(b) * 512u + 16u * lane;
    if (byte < r.padded) cp_async16(reinterpret_cast<uint8_t *>(r.ring) + (b & 3) * 512 + 16 * lane, r.wbase + byte);
}

// Keep the ring ahead of the words still to be consumed: blocks down to
// b - 3 requested and blocks b - 1 .. b complete, b being the block of the
// next word. Block k goes to ring slot k & 3, whose previous block (k + 4)
// lies wholly above the next word. One commit group per block, empty past the
// record's first block, so the two newest groups are always the two lowest
// blocks. Between two calls at most 256 words may be consumed.
__device__ __forceinline__ void ring_refill(Rans &r) {
    const int b = (r.ptr - 1) >> 8;
    const int target = max(b - 3, -4);
    if (r.lo > target) {
        do {
            r.lo--;
            if (r.lo >= 0) fetch_block(r, r.lo);
            cp_async_commit();
        } while (r.lo > target);
        cp_async_wait<2>();
        __syncwarp();
    }
}

// Parse a rANS record (val bytes) into lookup tables in `slot` (and the
// one-level table `big` when kBig) and load the lane states and the first
// word blocks. Returns false if malformed.
// kLanes (format v3): after the table come 32 u16 word counts and the
// lanes' lists (each padded to 8 words); each lane's next blocks go into
// its ring (lane_slot), the whole lists being prefetched into L2 first.
template <bool kBig, bool kLanes = false>
__device__ bool rans_setup(const uint8_t *rec, uint32_t val, uint8_t *slot, uint32_t *big, Rans &r) {
    const int lane = threadIdx.x & 31;
    uint8_t *lut = slot;
    uint32_t *sym = reinterpret_cast<uint32_t *>(slot + kLutBytes);
    uint32_t bits = rec[128 + lane];
    uint32_t present = __popc(bits);
    uint32_t k = __reduce_add_sync(kFull, present);
    uint32_t inc = present;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += t;
    }
    uint32_t rank = inc - present;
    const uint32_t words_at = kRecHead + uint32_t(pad16(2 * k));
    bool bad = k < 2 || val < words_at + (kLanes ? 64u : 0u) || ((val - words_at) & (kLanes ? 15u : 1u));
    const uint16_t *freqs = reinterpret_cast<const uint16_t *>(rec + kRecHead);
    uint32_t f8[8], fsum = 0;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        f8[q] = 0;
        if (!bad && ((bits >> q) & 1u)) {
            f8[q] = freqs[rank++];
            bad |= f8[q] == 0 || f8[q] >= kM;
        }
        fsum += f8[q];
    }
    for (uint32_t b = kRecHead + 2 * k + lane; !bad && b < words_at; b += 32) bad |= rec[b] != 0;
    inc = fsum;
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += t;
    }
    uint32_t cum = inc - fsum;
    bad |= __shfl_sync(kFull, inc, 31) != kM;
    r.x = reinterpret_cast<const uint32_t *>(rec)[lane];
    bad |= r.x < kRansL;
    uint32_t lane_off = 0, lane_cnt = 0;
    if constexpr (kLanes) {
        // the counts must describe the record exactly
        if (!__any_sync(kFull, bad)) {
            lane_cnt = reinterpret_cast<const uint16_t *>(rec + words_at)[lane];
            const uint32_t padded = (lane_cnt + 7) & ~7u;
            uint32_t incl = padded;
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += t;
            }
            lane_off = incl - padded;
            bad |= words_at + 64 + 2 * __shfl_sync(kFull, incl, 31) != val;
        }
    }
    if (__any_sync(kFull, bad)) return false;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        uint32_t s = 8 * lane + q;
        if (f8[q]) {
            sym[s] = f8[q] | (cum << 12);
            uint32_t a = cum, e = cum + f8[q];
            for (; a < e && (a & 3); a++) lut[a] = uint8_t(s);
            for (; a + 4 <= e; a += 4) *reinterpret_cast<uint32_t *>(lut + a) = s * 0x01010101u;
            for (; a < e; a++) lut[a] = uint8_t(s);
        }
        cum += f8[q];
    }
    r.lut = lut;
    r.sym = sym;
    r.big = big;
    r.ring = reinterpret_cast<uint16_t *>(slot + kLutBytes + kSymBytes);
    if constexpr (kBig) {
        __syncwarp();
        for (uint32_t sl = lane; sl < kM; sl += 32) {
            const uint32_t sy = lut[sl], e = sym[sy];
            big[sl] = sy | (e & 0xFFFu) << 8 | (sl - (e >> 12)) << 20;
        }
    }
    if constexpr (kLanes) {
        const uint8_t *lists = rec + words_at + 64;
        for (uint32_t o = 128 * lane; o < val - words_at - 64; o += 32 * 128) prefetch_l2(lists + o);
        r.wbase = lists + 2 * lane_off;
        r.ptr = int32_t(lane_cnt) - 1;
        r.ring = reinterpret_cast<uint16_t *>(slot + kLutBytes + kSymBytes);
        // the current block and the three below it; all of them in place
        r.filled = (r.ptr >> 3) + 1;
        lane_fill(r, (r.ptr >> 3) - 3);
        cp_async_commit();
        cp_async_commit();
        cp_async_wait<0>();
        // the padding after the lane's last word is zero
        const uint32_t used = lane_cnt & 7u;
        bool pad_bad = false;
        if (used != 0) {
            const uint16_t *blk = lane_slot(r.ring, r.ptr >> 3);
            for (uint32_t h = used; h < 8; h++) pad_bad |= blk[h] != 0;
        }
        r.lo = 0;
        __syncwarp();
        return !__any_sync(kFull, pad_bad);
    } else {
        const uint32_t nwords = (val - words_at) / 2;
        r.ptr = int32_t(nwords);
        r.wbase = rec + words_at;
        r.padded = uint32_t(pad16(2 * nwords));
        r.lo = nwords ? int((nwords - 1) >> 8) + 1 : 0;
        __syncwarp();
        ring_refill(r);
        return true;
    }
}

// Format v2 record: the 32 lane states, then the words; the table is the
// plane's one-level table `big` built by the CTA (null when the blob's plane
// table is not a valid 12-bit table). Returns false if malformed.
__device__ bool rans_setup_shared(const uint8_t *rec, uint32_t val, const uint32_t *big, uint16_t *ring, Rans &r) {
    const int lane = threadIdx.x & 31;
    bool bad = big == nullptr || val < 128 || ((val - 128) & 1u);
    r.x = bad ? kRansL : reinterpret_cast<const uint32_t *>(rec)[lane];
    bad |= r.x < kRansL;
    if (__any_sync(kFull, bad)) return false;
    const uint32_t nwords = (val - 128) / 2;
    r.ptr = int32_t(nwords);
    r.wbase = rec + 128;
    r.padded = uint32_t(pad16(2 * nwords));
    r.lut = nullptr;
    r.sym = nullptr;
    r.big = big;
    r.ring = ring;
    r.lo = nwords ? int((nwords - 1) >> 8) + 1 : 0;
    __syncwarp();
    ring_refill(r);
    return true;
}

// One rANS decode step of the warp with a word list per lane (format v3):
// the lane's next word is read from its ring before the table is, so the
// step's dependent chain is the table read and the state update alone;
// blocks are refilled every 8 steps (lane_refill), outside the steps.
template <bool kBig>
__device__ __forceinline__ uint32_t rans_step_lanes(Rans &r, bool active) {
    // this lane's next word, from its ring (a lane that has no word left
    // reads a slot it will not use)
    const uint32_t w = r.ring[lane_ring_base() + ((uint32_t(r.ptr) & 31u) ^ lane_ring_xor())];
    const uint32_t slot = r.x & (kM - 1);
    uint32_t s, xn;
    if constexpr (kBig) {
        const uint32_t e = r.big[slot];
        s = e & 0xFFu;
        xn = ((e >> 8) & 0xFFFu) * (r.x >> kProbBits) + (e >> 20);
    } else {
        s = r.lut[slot];
        const uint32_t e = r.sym[s];
        xn = (e & 0xFFFu) * (r.x >> kProbBits) + slot - (e >> 12);
    }
    const bool need = active && xn < kRansL;
    xn = need ? ((xn << 16) | w) : xn;
    if (active) r.x = xn;
    r.ptr -= need ? 1 : 0;
    return s;
}

// One rANS decode step of the warp: returns this lane's symbol.
template <bool kBig>
__device__ __forceinline__ uint32_t rans_step(Rans &r, bool active, uint32_t lt) {
    // lane l's candidate is the (l + 1)-th word from the top, read before the
    // table so that the load is off the state's chain; the lane with p
    // emitting lanes below it takes lane p's (the range read is the same
    // ring range as a direct read of the word: blocks b - 1 .. b)
    const uint32_t wl = r.ring[uint32_t(r.ptr - 1 - int32_t(threadIdx.x & 31)) & (kRingWords - 1)];
    const uint32_t slot = r.x & (kM - 1);
    uint32_t s, xn;
    if constexpr (kBig) {
        const uint32_t e = r.big[slot];
        s = e & 0xFFu;
        xn = ((e >> 8) & 0xFFFu) * (r.x >> kProbBits) + (e >> 20);
    } else {
        s = r.lut[slot];
        const uint32_t e = r.sym[s];
        xn = (e & 0xFFFu) * (r.x >> kProbBits) + slot - (e >> 12);
    }
    const bool need = active && xn < kRansL;
    const uint32_t bal = __ballot_sync(kFull, need);
    const uint32_t w = __shfl_sync(kFull, wl, __popc(bal & lt));
    xn = need ? ((xn << 16) | w) : xn;
    if (active) r.x = xn;
    r.ptr -= int32_t(__popc(bal));
    return s;
}

template <bool kLanes = false>
__device__ __forceinline__ bool rans_final_ok(const Rans &r) {
    return !__any_sync(kFull, r.x != kRansL || r.ptr != (kLanes ? -1 : 0));
}


// 8 consecutive elements' bytes of stream j packed in two words (element e
// of the eight in byte e of the pair), from each kind of stream.
struct Col8 {
    uint32_t lo, hi;
};

// Stream kinds.
constexpr uint32_t kKConst = 0, kKRaw = 1, kKMain = 2, kKStaged = 3;

// What both warps of a pair know about a grouped chunk.
struct ChunkCtx {
    const uint8_t *p;      // payload
    uint8_t *out;          // output range
    uint8_t *tail;         // staged bytes of the coded streams after the first
    const uint8_t *base;   // delta: the base tensor's bytes of this chunk (the output is decoded XOR base)
    uint32_t n, len, q, groups, T, stored;
    bool have_main;
    uint32_t kind[4], val[4], roff[4], sub[4];
};

// Parse a grouped chunk's directory. Returns false if malformed.
template <int W, bool kV2>
__device__ bool parse_directory(const uint8_t *p, uint32_t stored, uint32_t n, ChunkCtx &cx) {
    const int lane = threadIdx.x & 31;
    // W entries of mode << 30 | value, zero-padded to 16 bytes
    const uint32_t dir = lane < 4 ? reinterpret_cast<const uint32_t *>(p)[lane] : 0u;
    bool bad = __any_sync(kFull, lane >= W && lane < 4 && dir != 0);
    uint32_t pos = 16, coded = 0;
    cx.have_main = false;
#pragma unroll
    for (int j = 0; j < W; j++) {
        const uint32_t e = __shfl_sync(kFull, dir, j);
        const uint32_t mode = e >> 30;
        cx.val[j] = e & 0x3FFFFFFFu;
        cx.roff[j] = pos;
        cx.sub[j] = 0;
        if (mode == kModeConst) {
            cx.kind[j] = kKConst;
            bad |= cx.val[j] > 255;
        } else if (mode == kModeRaw) {
            cx.kind[j] = kKRaw;
            bad |= cx.val[j] != n;
            pos += uint32_t(pad16(n));
        } else if (mode == kModeRans) {
            cx.kind[j] = coded == 0 ? kKMain : kKStaged;
            cx.sub[j] = coded == 0 ? 0 : coded - 1;
            cx.have_main = true;
            coded++;
            bad |= cx.val[j] < (kV2 ? 128u : kRecHead) || cx.val[j] > stored;
            pos += uint32_t(pad16(cx.val[j]));
        } else {
            cx.kind[j] = kKConst;
            bad = true;
        }
        if (pos > stored) bad = true;
    }
    cx.q = coded > 1 ? coded - 1 : 0;
    return !bad && pos == stored;
}

// Producer warp: staged streams into the output tail, then the main stream's
// symbols group by group into the stage queue (the last group may be
// partial: steps past the stream leave the states alone).
template <int DT, bool kBig, bool kV2, bool kLanes, class PS>
__device__ void produce(const DecodeArgs &a, const ChunkCtx &cx, PS &ps, const uint32_t *const *pbig) {
    constexpr int W = WordOf<DT>::W;
    const int lane = threadIdx.x & 31;
    // test hook: the producer stops before its first signal (nothing in
    // flight), so the consumer's wait runs out
    if (a.hooks & ZC_HOOK_PRODUCER_STALL) return;
    const uint32_t lt = lanemask_lt();
    // v1: the record's own table, built into the pair's tables; v2: the
    // CTA's table of the stream's plane
    auto setup = [&](int j, Rans &r) -> bool {
        if constexpr (kV2) {
            return rans_setup_shared(cx.p + cx.roff[j], cx.val[j], pbig[j], ps.ring, r);
        } else {
            return rans_setup<kBig, kLanes>(cx.p + cx.roff[j], cx.val[j], ps.lut, ps.big, r);
        }
    };
    auto step = [&](Rans &r, bool active) -> uint32_t {
        if constexpr (kLanes) return rans_step_lanes<kBig>(r, active);
        else return rans_step<kBig>(r, active, lt);
    };
    bool bad = false;
    if (cx.q) {
#pragma unroll
        for (int j = 0; j < W; j++) {
            if (cx.kind[j] != kKStaged) continue;
            Rans r;
            if (!setup(j, r)) bad = true;
            if (!bad) {
                for (uint32_t t = 0; t < cx.T; t++) {
                    const uint32_t i = t * 32 + lane;
                    const bool active = i < cx.n;
                    if constexpr (!kLanes) ring_refill(r);
                    else if ((t & 7u) == 0) lane_refill(r);
                    const uint32_t s = step(r, active);
                    if (active) cx.tail[uint64_t(i) * cx.q + cx.sub[j]] = uint8_t(s);
                }
                bad |= !rans_final_ok<kLanes>(r);
            }
            cp_async_wait_all();  // the ring is reused by the next stream
            __syncwarp();
            if (bad) break;
        }
    }
    Rans rs;
#pragma unroll
    for (int j = 0; j < W; j++)
        if (!bad && cx.kind[j] == kKMain && !setup(j, rs)) bad = true;
    if (lane == 0) ps.flag = bad ? 0u : 1u;
    __syncwarp();
    mbar_arrive(&ps.start);
    if (bad) {
        cp_async_wait_all();
        if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
        return;
    }
    const uint32_t ng = (cx.T + 7) / 8;  // groups including a partial last one
    for (uint32_t g = 0; g < ng; g++) {
        const uint32_t k = g % kStages;
        // the consumer frees the stages in order: at an even group, wait for
        // the stage of the next group too (one wait for two groups)
        if ((g & 1u) == 0) {
            const uint32_t gw = g + 1 < ng ? g + 1 : g, kw = gw % kStages, rw = gw / kStages;
            if (rw > 0 && !mbar_wait(&ps.empty[kw], (rw - 1) & 1u, a.wait_cycles)) {
                if (lane == 0) status_or(a.d_status, ZC_ETIMEOUT);
                cp_async_wait_all();
                return;
            }
        }
        if constexpr (!kLanes) ring_refill(rs);
        else lane_refill(rs);
        uint8_t *st = ps.stage[k];
        if constexpr (kLanes && kBig) {
            if (8 * g + 8 <= cx.n / 32) {
                // a group of 8 steps in which every lane has a symbol: the
                // step reduced to its dependent chain (32-bit shared
                // addresses; renormalisation by one byte permute)
                const uint32_t ring_lane = smem_u32(rs.ring) + 2u * lane_ring_base(), big_base = smem_u32(rs.big);
                const uint32_t rx = lane_ring_xor();
                uint32_t x = rs.x;
                int32_t ptr = rs.ptr;
#pragma unroll
                for (int s = 0; s < 8; s++) {
                    const uint32_t w = lds_u16(ring_lane + (((uint32_t(ptr) & 31u) ^ rx) << 1));
                    const uint32_t e = lds_u32(big_base + ((x & (kM - 1)) << 2));
                    const uint32_t xn = ((e >> 8) & 0xFFFu) * (x >> kProbBits) + (e >> 20);
                    const bool need = xn < kRansL;
                    x = need ? __byte_perm(w, xn, 0x5410) : xn;
                    ptr -= need ? 1 : 0;
                    st[32 * s + lane] = uint8_t(e);
                }
                rs.x = x;
                rs.ptr = ptr;
                mbar_arrive(&ps.full[k]);
                continue;
            }
        }
        if constexpr (kLanes && !kBig && !kV2) {
            if (8 * g + 8 <= cx.n / 32) {
                // the same with the two-level table: slot -> symbol, then
                // symbol -> f | cum << 12
                const uint32_t ring_lane = smem_u32(rs.ring) + 2u * lane_ring_base();
                const uint32_t lut_base = smem_u32(rs.lut), sym_base = smem_u32(rs.sym);
                const uint32_t rx = lane_ring_xor();
                uint32_t x = rs.x;
                int32_t ptr = rs.ptr;
#pragma unroll
                for (int s = 0; s < 8; s++) {
                    const uint32_t w = lds_u16(ring_lane + (((uint32_t(ptr) & 31u) ^ rx) << 1));
                    const uint32_t slot = x & (kM - 1);
                    const uint32_t sy = lds_u8(lut_base + slot);
                    const uint32_t e = lds_u32(sym_base + (sy << 2));
                    const uint32_t xn = (e & 0xFFFu) * (x >> kProbBits) + slot - (e >> 12);
                    const bool need = xn < kRansL;
                    x = need ? __byte_perm(w, xn, 0x5410) : xn;
                    ptr -= need ? 1 : 0;
                    st[32 * s + lane] = uint8_t(sy);
                }
                rs.x = x;
                rs.ptr = ptr;
                mbar_arrive(&ps.full[k]);
                continue;
            }
        }
#pragma unroll
        for (int s = 0; s < 8; s++) {
            const uint32_t t = 8 * g + s;
            const bool active = t < cx.T && t * 32 + lane < cx.n;
            st[32 * s + lane] = uint8_t(step(rs, active));
        }
        mbar_arrive(&ps.full[k]);
    }
    if (!rans_final_ok<kLanes>(rs) && lane == 0) status_or(a.d_status, ZC_ECORRUPT);
    cp_async_wait_all();
}

// Consumer warp: the chunk's output and the CRC of its stored bytes. For a
// raw stream the lane register follows the lane's pieces: with 4-byte words
// group g of the stream is its bytes [256 g, 256 g + 256) and lane l takes
// bytes 8 l .. 8 l + 7 of it (the bytes it reads for the output), so after
// group g the register is shift(register after g - 1, 256 bytes) XOR the
// register of the new piece taken from zero (linearity); with words of up to
// 2 bytes the lane takes bytes 32 l .. 32 l + 31 of every 4 groups (1024
// bytes), read again, coalesced, two groups before they are used: fewer
// lookups per byte (one shift per 32 bytes instead of per 8). The lanes are
// folded at the end (crc_fold) and the stream's bytes after its last whole
// piece round (and its padding) are added from the blob. The directory and the coded records are taken from the blob at the
// end, and the parts are appended in payload order. (Taking each lane's CRC
// over a contiguous slice of the stream instead needs no shift, but its
// loads, 32 lines per instruction, cost more than the shift saves.)
// The consumer's shift table (gshift): the stride of a lane's raw-stream
// pieces, 1024 bytes for words of up to 2 bytes, else 256.
template <int W>
constexpr int consume_shift_table() { return kShPow + (W <= 2 ? 10 : 8); }

template <int DT, bool kVerify, bool kDelta, int C, class PS>
__device__ void consume(const DecodeArgs &a, const ChunkCtx &cx, PS &ps, uint32_t expect_crc,
                        const uint32_t *crc_rep, const uint32_t (*gshift)[256], const uint32_t (*gap496)[256]) {
    constexpr int W = WordOf<DT>::W;
    constexpr bool kBlk = W <= 2;  // 32-byte pieces every 4 groups
    const int lane = threadIdx.x & 31;
    const uint32_t *row = crc_row<C>(crc_rep);
    const uint32_t groups = cx.groups;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(cx.out) & 15) == 0;
    if (cx.have_main) {
        if (!mbar_wait(&ps.start, 0, a.wait_cycles)) {
            if (lane == 0) status_or(a.d_status, ZC_ETIMEOUT);
            return;
        }
        if (ps.flag == 0) {  // the producer has reported the chunk: is the payload the stored one?
            if constexpr (kVerify) {
                const uint32_t reg = crc_strided<1, false, C>(cx.p, cx.stored, 0xFFFFFFFFu, crc_rep, gap496, nullptr);
                if ((reg ^ 0xFFFFFFFFu) != expect_crc && lane == 0) status_or(a.d_status, ZC_ECRC);
            }
            return;
        }
    }
    uint32_t Rraw[W];  // CRC registers of the raw streams (kVerify)
    uint4 cb0[W], cb1[W];  // kBlk: the lane's next 32-byte piece of each raw stream
    const uint32_t blocks = kBlk ? groups / 4 : 0;
#pragma unroll
    for (int j = 0; j < W; j++) {
        Rraw[j] = 0;
        cb0[j] = cb1[j] = make_uint4(0, 0, 0, 0);
    }
    // The raw streams are read 8 bytes per lane and group, two groups ahead,
    // too few bytes in flight to cover a DRAM access: their lines are
    // prefetched into L2 kAhead groups ahead (a group of a stream is 256
    // bytes, two lines), the first kAhead groups now.
    constexpr uint32_t kAhead = 16;
#pragma unroll
    for (int j = 0; j < W; j++) {
        if (cx.kind[j] != kKRaw) continue;
        const uint32_t upto = 256 * min(groups, kAhead);
        for (uint32_t o = 128 * lane; o < upto; o += 32 * 128) prefetch_l2(cx.p + cx.roff[j] + o);
    }
    uint2 rn1[W], rn2[W];  // raw columns of the next two groups
#pragma unroll
    for (int j = 0; j < W; j++) {
        const uint2 *src = reinterpret_cast<const uint2 *>(cx.p + cx.roff[j]) + lane;
        rn1[j] = (cx.kind[j] == kKRaw && groups > 0) ? __ldg(src) : make_uint2(0, 0);
        rn2[j] = (cx.kind[j] == kKRaw && groups > 1) ? __ldg(src + 32) : make_uint2(0, 0);
    }
    for (uint32_t g = 0; g < groups; g++) {
        const uint32_t k = g % kStages, r = g / kStages;
        // delta: the base bytes this group's output is XOR-ed with, loaded
        // before they are needed (delta buffers are 16-byte aligned)
        uint4 bv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if constexpr (kDelta) {
            const uint64_t b0 = uint64_t(W) * (256 * g + 8 * lane);
            if constexpr (W == 4) {
                bv[0] = __ldcs(reinterpret_cast<const uint4 *>(cx.base + b0));
                bv[1] = __ldcs(reinterpret_cast<const uint4 *>(cx.base + b0) + 1);
            } else if constexpr (W == 2) {
                bv[0] = __ldcs(reinterpret_cast<const uint4 *>(cx.base + b0));
            } else {
                const uint2 t = __ldcs(reinterpret_cast<const uint2 *>(cx.base + b0));
                bv[0] = make_uint4(t.x, t.y, 0, 0);
            }
        }
        auto xb = [](uint4 v, const uint4 &b) { return make_uint4(v.x ^ b.x, v.y ^ b.y, v.z ^ b.z, v.w ^ b.w); };
        if (lane < 2 && g + kAhead < groups) {
#pragma unroll
            for (int j = 0; j < W; j++)
                if (cx.kind[j] == kKRaw) prefetch_l2(cx.p + cx.roff[j] + 256 * (g + kAhead) + 128 * lane);
        }
        Col8 col[W];
#pragma unroll
        for (int j = 0; j < W; j++) {
            col[j].lo = rn1[j].x;
            col[j].hi = rn1[j].y;
            rn1[j] = rn2[j];
            if (cx.kind[j] == kKRaw && g + 2 < groups)
                rn2[j] = __ldg(reinterpret_cast<const uint2 *>(cx.p + cx.roff[j] + 256 * (g + 2)) + lane);
            if constexpr (kVerify && kBlk) {
                const uint32_t k = g >> 2;
                if (cx.kind[j] == kKRaw && k < blocks) {
                    if ((g & 3u) == 1u) {
                        const uint4 *q = reinterpret_cast<const uint4 *>(cx.p + cx.roff[j] + 1024ull * k) + 2 * lane;
                        cb0[j] = __ldg(q);
                        cb1[j] = __ldg(q + 1);
                    } else if ((g & 3u) == 3u) {
                        Rraw[j] = (k ? shift_smem(Rraw[j], gshift) : 0u) ^
                                  crc_rep16<C>(crc_rep16<C>(0u, cb0[j], row), cb1[j], row);
                    }
                }
            } else if constexpr (kVerify) {
                if (cx.kind[j] == kKRaw)
                    Rraw[j] = (g ? shift_smem(Rraw[j], gshift) : 0u) ^
                              crc_rep_word<C>(crc_rep_word<C>(0u, col[j].lo, row), col[j].hi, row);
            }
        }
        uint2 mv = make_uint2(0, 0);
        if (cx.have_main) {
            if (!mbar_wait(&ps.full[k], r & 1u, a.wait_cycles)) {
                if (lane == 0) status_or(a.d_status, ZC_ETIMEOUT);
                return;
            }
            mv = *reinterpret_cast<const uint2 *>(ps.stage[k] + 8 * lane);
            mbar_arrive(&ps.empty[k]);
        }
        const uint32_t e0 = 256 * g + 8 * lane;
#pragma unroll
        for (int j = 0; j < W; j++) {
            const uint32_t cv = cx.val[j] * 0x01010101u;
            col[j].lo = cx.kind[j] == kKConst ? cv : cx.kind[j] == kKMain ? mv.x : col[j].lo;
            col[j].hi = cx.kind[j] == kKConst ? cv : cx.kind[j] == kKMain ? mv.y : col[j].hi;
            if (cx.kind[j] == kKStaged) {
                uint32_t v[2] = {0, 0};
                for (int e = 0; e < 8; e++)
                    v[e >> 2] |= uint32_t(__ldcg(cx.tail + uint64_t(e0 + e) * cx.q + cx.sub[j])) << (8 * (e & 3));
                col[j].lo = v[0];
                col[j].hi = v[1];
            }
        }
        if constexpr (W == 4) {
            uint4 v[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t c0 = h ? col[0].hi : col[0].lo, c1 = h ? col[1].hi : col[1].lo;
                const uint32_t c2 = h ? col[2].hi : col[2].lo, c3 = h ? col[3].hi : col[3].lo;
                const uint32_t lo32 = __byte_perm(c3, c2, 0x5140), hi32 = __byte_perm(c3, c2, 0x7362);
                const uint32_t lo10 = __byte_perm(c1, c0, 0x5140), hi10 = __byte_perm(c1, c0, 0x7362);
                v[h].x = Perm<DT>::inv(__byte_perm(lo32, lo10, 0x5410));
                v[h].y = Perm<DT>::inv(__byte_perm(lo32, lo10, 0x7632));
                v[h].z = Perm<DT>::inv(__byte_perm(hi32, hi10, 0x5410));
                v[h].w = Perm<DT>::inv(__byte_perm(hi32, hi10, 0x7632));
            }
            if constexpr (kDelta) {
                v[0] = xb(v[0], bv[0]);
                v[1] = xb(v[1], bv[1]);
            }
            if (vec_ok) {
                uint4 *o = reinterpret_cast<uint4 *>(cx.out + 4ull * e0);
                o[0] = v[0];
                o[1] = v[1];
            } else {
                uint32_t *o = reinterpret_cast<uint32_t *>(cx.out) + e0;
                o[0] = v[0].x; o[1] = v[0].y; o[2] = v[0].z; o[3] = v[0].w;
                o[4] = v[1].x; o[5] = v[1].y; o[6] = v[1].z; o[7] = v[1].w;
            }
        } else if constexpr (W == 2) {
            uint4 v;
            v.x = Perm<DT>::inv2(__byte_perm(col[1].lo, col[0].lo, 0x5140));
            v.y = Perm<DT>::inv2(__byte_perm(col[1].lo, col[0].lo, 0x7362));
            v.z = Perm<DT>::inv2(__byte_perm(col[1].hi, col[0].hi, 0x5140));
            v.w = Perm<DT>::inv2(__byte_perm(col[1].hi, col[0].hi, 0x7362));
            if constexpr (kDelta) v = xb(v, bv[0]);
            if (vec_ok) {
                *reinterpret_cast<uint4 *>(cx.out + 2ull * e0) = v;
            } else {
                uint16_t *o = reinterpret_cast<uint16_t *>(cx.out) + e0;
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                for (int e = 0; e < 4; e++) {
                    o[2 * e] = uint16_t(w4[e]);
                    o[2 * e + 1] = uint16_t(w4[e] >> 16);
                }
            }
        } else {
            if constexpr (kDelta) {
                col[0].lo ^= bv[0].x;
                col[0].hi ^= bv[0].y;
            }
            if ((reinterpret_cast<uintptr_t>(cx.out) & 7) == 0) {
                *reinterpret_cast<uint2 *>(cx.out + e0) = make_uint2(col[0].lo, col[0].hi);
            } else {
                for (int e = 0; e < 8; e++)
                    cx.out[e0 + e] = uint8_t((e < 4 ? col[0].lo : col[0].hi) >> (8 * (e & 3)));
            }
        }
    }
    // the last < 256 elements: the producer's partial group, step by step
    if (cx.T > 8 * groups) {
        const uint32_t k = groups % kStages, r = groups / kStages;
        if (cx.have_main && !mbar_wait(&ps.full[k], r & 1u, a.wait_cycles)) {
            if (lane == 0) status_or(a.d_status, ZC_ETIMEOUT);
            return;
        }
        for (uint32_t t = groups * 8; t < cx.T; t++) {
            const uint32_t i = t * 32 + lane;
            if (i >= cx.n) continue;
            const uint32_t sm = cx.have_main ? ps.stage[k][32 * (t - groups * 8) + lane] : 0u;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < W; j++) {
                uint32_t b;
                if (cx.kind[j] == kKConst) b = cx.val[j];
                else if (cx.kind[j] == kKRaw) b = __ldg(cx.p + cx.roff[j] + i);
                else if (cx.kind[j] == kKMain) b = sm;
                else b = __ldcg(cx.tail + uint64_t(i) * cx.q + cx.sub[j]);
                word = (word << 8) | b;
            }
            uint32_t w = Perm<DT>::inv(word);
            if constexpr (kDelta) w ^= load_word_any<W>(cx.base + uint64_t(i) * W);
            if (W == 4) reinterpret_cast<uint32_t *>(cx.out)[i] = w;
            else if (W == 2) reinterpret_cast<uint16_t *>(cx.out)[i] = uint16_t(w);
            else cx.out[i] = uint8_t(w);
        }
        __syncwarp();
    }
    if constexpr (kVerify) {
        // the directory (16 bytes) from the preset register
        uint32_t reg = crc_rep16<C>(0xFFFFFFFFu, __ldg(reinterpret_cast<const uint4 *>(cx.p)), row);
#pragma unroll
        for (int j = 0; j < W; j++) {
            if (cx.kind[j] == kKConst) continue;
            const uint8_t *seg = cx.p + cx.roff[j];
            uint64_t seg_len;
            uint32_t part;
            if (cx.kind[j] == kKRaw) {
                seg_len = pad16(cx.n);
                uint32_t done;
                if constexpr (kBlk) {
                    part = blocks ? crc_fold<1, 5>(Rraw[j], nullptr) : 0u;
                    done = 1024 * blocks;
                } else {
                    part = groups ? crc_fold<1, 3>(Rraw[j], nullptr) : 0u;
                    done = 256 * groups;
                }
                part = crc_strided<1, false, C>(seg + done, seg_len - done, part, crc_rep, gap496, nullptr);
            } else {
                seg_len = pad16(cx.val[j]);
                part = warp_crc16<C, true, 4>(seg, uint32_t(seg_len), crc_rep, gap496);
            }
            reg = crc_append_small(reg, part, uint32_t(seg_len));
        }
        if ((reg ^ 0xFFFFFFFFu) != expect_crc && lane == 0) status_or(a.d_status, ZC_ECRC);
    }
}

// Chunk c of blob bd, by one warp pair (kV2: format v2, with the CTA's
// plane tables pbig).
// role: 0 the producer (rANS lanes), 1 the consumer (output), 2 the CRC
// warp (kCrcWarp: the chunk's CRC over its stored bytes is checked by a
// warp of its own, in parallel with the decoding; else the consumer takes
// it as it reads the payload).
template <int DT, bool kBig, bool kDelta, bool kV2, int C, bool kLanes, bool kCrcWarp, class PS>
__device__ void decode_chunk(const DecodeArgs &a, const BlobDesc &bd, uint32_t c, int role, PS &ps,
                             const uint32_t *crc_rep, const uint32_t (*gshift)[256], const uint32_t (*gap496)[256],
                             const uint32_t *const *pbig) {
    constexpr int W = WordOf<DT>::W;
    const int lane = threadIdx.x & 31;
    const bool producer = role == 0;
    const uint8_t *const blob = bd.blob;
    const uint64_t blob_bytes = bd.blob_bytes, nbytes = bd.nbytes;
    const uint32_t n_chunks = bd.n_chunks;
    uint8_t *const dst = bd.dst;
    const uint8_t *const base = bd.base;
    // payloads follow the chunk table (v2: and the W plane tables)
    const uint64_t table_end =
        ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * n_chunks + (kV2 ? 512ull * W : 0ull);

    uint4 ent = make_uint4(0, 0, 0, 0);
    if (lane == 0) ent = reinterpret_cast<const uint4 *>(blob + ZC_HEADER_BYTES)[c];
    ent.x = __shfl_sync(kFull, ent.x, 0);
    ent.y = __shfl_sync(kFull, ent.y, 0);
    ent.z = __shfl_sync(kFull, ent.z, 0);
    ent.w = __shfl_sync(kFull, ent.w, 0);
    const uint64_t off = uint64_t(ent.x) | (uint64_t(ent.y) << 32);
    const uint32_t stored = ent.z & 0x7FFFFFFFu;
    const bool raw = ent.z >> 31;
    const uint32_t len = uint32_t(umin64(a.chunk_bytes, nbytes - uint64_t(c) * a.chunk_bytes));
    const uint32_t n = len / W;

    bool ok = (off & 15) == 0 && off >= table_end && off <= blob_bytes && stored <= blob_bytes - off;
    ok = ok && (raw ? stored == len : (stored % 16 == 0 && stored >= 16 && stored <= max_grouped(len, W, a.version)));
    if (!ok) {
        if (!producer && lane == 0) status_or(a.d_status, ZC_EFORMAT);
        return;
    }
    const uint8_t *p = blob + off;
    const bool verify = !(a.flags & ZC_NO_VERIFY);
    if (role >= 2) {
        // the two CRC warps: the stored bytes' first and second half of the
        // 16-byte pieces (8 in flight per lane), each register taken from
        // zero; the second warp hands its register over through shared
        // memory, the first appends it (linearity) and the last stored % 16
        // bytes one at a time
        if (!verify) return;
        const uint32_t main = stored & ~15u, half = kCrcWarp ? (main >> 5) << 4 : main;
        if constexpr (kCrcWarp) {
            if (role == 3) {
                const uint32_t r1 = warp_crc16<C, false, 8>(p + half, main - half, crc_rep, gap496);
                if (lane == 0) ps.crc_part = r1;
                __syncwarp();
                mbar_arrive(&ps.crc_bar);
                return;
            }
        }
        uint32_t reg = warp_crc16<C, false, 8>(p, half, crc_rep, gap496);
        if constexpr (kCrcWarp) {
            if (!mbar_wait(&ps.crc_bar, 0, a.wait_cycles)) {
                if (lane == 0) status_or(a.d_status, ZC_ETIMEOUT);
                return;
            }
            reg = shift_bytes_small(reg, main - half) ^ ps.crc_part;
        }
        reg ^= shift_bytes_small(0xFFFFFFFFu, main);
        const uint32_t *row = crc_row<C>(crc_rep);
        for (uint32_t i = main; i < stored; i++) reg = crc_rep_byte<C>(reg, __ldg(p + i), row);
        if ((reg ^ 0xFFFFFFFFu) != ent.w && lane == 0) status_or(a.d_status, ZC_ECRC);
        return;
    }
    uint8_t *out = dst + uint64_t(c) * a.chunk_bytes;
    const uint8_t *basec = kDelta ? base + uint64_t(c) * a.chunk_bytes : nullptr;
    if (raw) {
        if (producer) return;
        uint32_t nvec = (reinterpret_cast<uintptr_t>(out) & 15) ? 0 : len / 16;
        for (uint32_t v = lane; v < nvec; v += 32) {
            uint4 t = __ldg(reinterpret_cast<const uint4 *>(p) + v);
            if constexpr (kDelta) {
                const uint4 b = __ldcs(reinterpret_cast<const uint4 *>(basec) + v);
                t.x ^= b.x; t.y ^= b.y; t.z ^= b.z; t.w ^= b.w;
            }
            reinterpret_cast<uint4 *>(out)[v] = t;
        }
        for (uint32_t i = nvec * 16 + lane; i < len; i += 32) out[i] = kDelta ? uint8_t(p[i] ^ basec[i]) : p[i];
        // a RAW chunk stores the original bytes, so its CRC is the payload's
        if (!kCrcWarp && verify &&
            (crc_strided<1, false, C>(p, len, 0xFFFFFFFFu, crc_rep, gap496, nullptr) ^ 0xFFFFFFFFu) != ent.w &&
            lane == 0)
            status_or(a.d_status, ZC_ECRC);
        return;
    }

    ChunkCtx cx;
    if (!parse_directory<W, kV2>(p, stored, n, cx)) {
        if (!producer) {
            if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
            // a changed payload is reported as such (the check the caller asked for)
            if (!kCrcWarp && verify &&
                (crc_strided<1, false, C>(p, stored, 0xFFFFFFFFu, crc_rep, gap496, nullptr) ^ 0xFFFFFFFFu) !=
                    ent.w && lane == 0)
                status_or(a.d_status, ZC_ECRC);
        }
        return;
    }
    cx.p = p;
    cx.stored = stored;
    cx.out = out;
    cx.n = n;
    cx.len = len;
    cx.T = (n + 31) / 32;
    cx.groups = n / 256;
    cx.tail = out + (len - cx.q * n);
    cx.base = basec;
    if (producer) {
        if (cx.have_main) produce<DT, kBig, kV2, kLanes>(a, cx, ps, pbig);
    } else if (verify && !kCrcWarp) {
        consume<DT, true, kDelta, C>(a, cx, ps, ent.w, crc_rep, gshift, gap496);
    } else {
        consume<DT, false, kDelta, C>(a, cx, ps, ent.w, crc_rep, gshift, gap496);
    }
}

// One CTA per SM. With one-level tables (kBig: few chunks per SM, 16 KB of
// table per pair) the CRC tables have 8 copies; with two-level tables (up
// to 16 pairs) they have 16, so fewer lanes meet on a bank.
// Warps per chunk: with one-level tables (few chunks per SM, so the pair's
// chains are latency-bound) two more warps check the chunk's CRC, half of
// the stored bytes each; with up to 16 pairs per CTA there is no room for
// them and the consumer takes the CRC.
template <bool kBig>
constexpr int warps_per_chunk() { return kBig ? 4 : 2; }

template <int DT, bool kBig, bool kDelta, bool kLanes>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int C = kBig ? 8 : 16;
    uint32_t *crc_rep = reinterpret_cast<uint32_t *>(smem);
    uint32_t(*gshift)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + crc_rep_words<C>() * 4);
    uint32_t(*gap496)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + crc_rep_words<C>() * 4 + 4 * 256 * 4);
    PairSmem<kBig> *pairs = reinterpret_cast<PairSmem<kBig> *>(smem + crc_smem<C>());
    const int warp = threadIdx.x >> 5;
    if (!(a.flags & ZC_NO_VERIFY)) {
        load_crc_rep<C>(crc_rep);
        load_shift_smem(gshift, consume_shift_table<WordOf<DT>::W>());
        load_shift_smem(gap496, kSh496);
    }
    constexpr int kWpc = warps_per_chunk<kBig>();
    const uint32_t pairs_per_cta = blockDim.x / (32 * kWpc);
    if (threadIdx.x < pairs_per_cta) {
        PairSmem<kBig> &ps = pairs[threadIdx.x];
        for (int k = 0; k < kStages; k++) {
            mbar_init(&ps.full[k], 32);
            mbar_init(&ps.empty[k], 32);
        }
        mbar_init(&ps.start, 32);
        mbar_init(&ps.crc_bar, 32);
    }
    __syncthreads();
    // warp w has role w / pairs_per_cta for chunk slot w % pairs_per_cta: the
    // warps of one role are consecutive, so they spread over the SM's four
    // schedulers (warp w issues from scheduler w % 4) instead of piling one
    // role onto one of them
    const uint32_t slot = uint32_t(warp) % pairs_per_cta;
    const int role = int(uint32_t(warp) / pairs_per_cta);
    const uint32_t g = blockIdx.x * pairs_per_cta + slot;
    if (g >= a.total_chunks) return;
    // the blob of this call-wide chunk index
    const BlobDesc bd = a.n_blobs == 1 ? a.one : a.blobs[owner_of(a.blobs, a.n_blobs, g)];
    decode_chunk<DT, kBig, kDelta, false, C, kLanes, kBig>(a, bd, g - bd.chunk_base, role, pairs[slot], crc_rep,
                                                           gshift, gap496, nullptr);
}

// Format v2 (shared plane tables): a CTA decodes up to a.pairs consecutive
// chunks of one blob (CTAs never span blobs). It first checks the blob's W
// plane tables and builds the one-level table of each valid one
// (slot -> symbol | f << 8 | (slot - cum) << 20, as the v1 big tables),
// which all its warp pairs then share: every decoding step is a single
// table read, whatever the number of chunks per SM, and no chunk builds a
// table of its own.
template <int DT, bool kDelta>
__global__ void __launch_bounds__(kV2Threads, 1) decode_v2_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int W = WordOf<DT>::W;
    constexpr int C = 16;  // CRC table copies
    uint32_t *crc_rep = reinterpret_cast<uint32_t *>(smem);
    uint32_t(*gshift)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + crc_rep_words<C>() * 4);
    uint32_t(*gap496)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + crc_rep_words<C>() * 4 + 4 * 256 * 4);
    uint32_t *big = reinterpret_cast<uint32_t *>(smem + crc_smem<C>());  // W x 4096
    uint32_t *symcum = big + W * kM;                                  // W x 256: f | cum << 12
    uint32_t *pvalid = symcum + W * 256;                              // W flags (padded to 16 bytes)
    uint8_t *luts = reinterpret_cast<uint8_t *>(pvalid + 4);           // W x 4096: slot -> symbol, scratch
    PairSmemV2 *pairs = reinterpret_cast<PairSmemV2 *>(luts + W * kM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the blob: the last one whose first CTA is at or before this one
    uint32_t bi = 0;
    if (a.n_blobs > 1) {
        uint32_t lo = 0, hi = a.n_blobs;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (a.blobs[mid].cta_base <= blockIdx.x) lo = mid;
            else hi = mid;
        }
        bi = lo;
    }
    const BlobDesc bd = a.n_blobs == 1 ? a.one : a.blobs[bi];
    const uint32_t first = (blockIdx.x - bd.cta_base) * a.pairs;

    if (!(a.flags & ZC_NO_VERIFY)) {
        load_crc_rep<C>(crc_rep);
        load_shift_smem(gshift, consume_shift_table<W>());
        load_shift_smem(gap496, kSh496);
    }
    const uint32_t pairs_per_cta = blockDim.x >> 6;
    if (threadIdx.x < pairs_per_cta) {
        PairSmemV2 &ps = pairs[threadIdx.x];
        for (int k = 0; k < kStages; k++) {
            mbar_init(&ps.full[k], 32);
            mbar_init(&ps.empty[k], 32);
        }
        mbar_init(&ps.start, 32);
    }
    // the warps check the plane tables in turn (256 u16 each after the chunk
    // table; the host checked that the blob holds them) and lay out
    // f | cum << 12 (a CTA may have fewer warps than planes)
    for (int j = warp; j < W; j += int(blockDim.x >> 5)) {
        const uint8_t *pt = bd.blob + ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * bd.n_chunks + 512ull * j;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(pt) + lane);
        const uint32_t f[8] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16,
                               v.z & 0xFFFFu, v.z >> 16, v.w & 0xFFFFu, v.w >> 16};
        uint32_t fsum = 0, nz = 0;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            fsum += f[k];
            nz += f[k] ? 1u : 0u;
        }
        uint32_t cum = fsum;
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, cum, o);
            if (lane >= o) cum += t;
        }
        const bool ok = __shfl_sync(kFull, cum, 31) == kM && __reduce_add_sync(kFull, nz) >= 2;
        cum -= fsum;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            symcum[j * 256 + 8 * lane + k] = f[k] | cum << 12;
            cum += f[k];
        }
        if (lane == 0) pvalid[j] = ok ? 1u : 0u;
    }
    __syncthreads();
    // slot -> symbol bytes, laid out by runs (a thread per plane and symbol,
    // whole words where a run covers them), then each slot's entry from its
    // symbol: two independent reads per slot. A valid table's runs tile
    // [0, 4096) exactly.
    for (uint32_t i = threadIdx.x; i < uint32_t(W) * 256; i += blockDim.x) {
        const uint32_t j = i >> 8, sy = i & 255;
        if (!pvalid[j]) continue;
        const uint32_t e = symcum[i];
        uint8_t *lut = luts + j * kM;
        uint32_t s = e >> 12;
        const uint32_t end = s + (e & 0xFFFu);
        for (; s < end && (s & 3); s++) lut[s] = uint8_t(sy);
        for (; s + 4 <= end; s += 4) *reinterpret_cast<uint32_t *>(lut + s) = sy * 0x01010101u;
        for (; s < end; s++) lut[s] = uint8_t(sy);
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < uint32_t(W) * kM; i += blockDim.x) {
        const uint32_t j = i / kM, slot = i % kM;
        if (!pvalid[j]) continue;
        const uint32_t sy = luts[i];
        const uint32_t e = symcum[j * 256 + sy];
        big[i] = sy | (e & 0xFFFu) << 8 | (slot - (e >> 12)) << 20;
    }
    __syncthreads();
    // warp w: role w / pairs_per_cta for pair w % pairs_per_cta (the roles
    // spread over the SM's schedulers)
    const uint32_t pair = uint32_t(warp) % pairs_per_cta;
    if (first + pair >= bd.n_chunks) return;
    const uint32_t *pbig[4] = {nullptr, nullptr, nullptr, nullptr};
#pragma unroll
    for (int j = 0; j < W; j++) pbig[j] = pvalid[j] ? big + j * kM : nullptr;
    decode_chunk<DT, true, kDelta, true, C, false, false>(a, bd, first + pair, int(uint32_t(warp) / pairs_per_cta),
                                                          pairs[pair], crc_rep, gshift, gap496, pbig);
}

template <int DT, bool kBig, bool kDelta, bool kLanes>
int launch_decode_mode(const DecodeArgs &a, uint32_t pc, cudaStream_t s) {
    constexpr int C = kBig ? 8 : 16;
    constexpr size_t most = kBig ? kBigPairs : kPairs;
    const size_t smem = crc_smem<C>() + size_t(pc) * sizeof(PairSmem<kBig>);
    const size_t smem_max = crc_smem<C>() + most * sizeof(PairSmem<kBig>);
    if (cudaFuncSetAttribute(decode_kernel<DT, kBig, kDelta, kLanes>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(std::min<size_t>(smem_max, 227 * 1024))) != cudaSuccess)
        return ZC_ECUDA;
    const int grid = int((a.total_chunks + pc - 1) / pc);
    decode_kernel<DT, kBig, kDelta, kLanes><<<grid, 32 * warps_per_chunk<kBig>() * pc, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

template <int DT, bool kDelta, bool kLanes>
int launch_decode_lt(const DecodeArgs &a, cudaStream_t s) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZC_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZC_ECUDA;
    // One CTA per SM holding the SM's share of the chunks. Few chunks per SM
    // (the rANS chains are then the critical path): one-level tables. Many:
    // the smaller two-level tables, up to kPairs chunks per CTA. Either way
    // the chunks spread evenly over the SMs.
    const uint64_t per_sm = (a.total_chunks + sms - 1) / uint64_t(sms);
    // ZC_PACKED: CTAs of up to kPairs chunks, on as few SMs as they fill
    if (a.flags & ZC_PACKED)
        return launch_decode_mode<DT, false, kDelta, kLanes>(
            a, uint32_t(std::max<uint64_t>(1, std::min<uint64_t>(kPairs, a.total_chunks))), s);
    if (per_sm <= kBigPairs)
        return launch_decode_mode<DT, true, kDelta, kLanes>(a, uint32_t(std::max<uint64_t>(per_sm, 1)), s);
    return launch_decode_mode<DT, false, kDelta, kLanes>(a, uint32_t(std::min<uint64_t>(kPairs, per_sm)), s);
}

// format v1 (one word list per record) or v3 (a word list per lane)
template <int DT, bool kDelta>
int launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
    return a.version == 3 ? launch_decode_lt<DT, kDelta, true>(a, s) : launch_decode_lt<DT, kDelta, false>(a, s);
}

template <int DT, bool kDelta>
int launch_decode_v2_t(const DecodeArgs &a, cudaStream_t s) {
    constexpr int W = WordOf<DT>::W;
    if (a.pairs == 0 || a.pairs > kV2Pairs || a.n_ctas == 0) return ZC_EINVAL;
    const size_t fixed = crc_smem<16>() + size_t(W) * (kM * 4 + 256 * 4) + 16 + size_t(W) * kM;
    const size_t smem = fixed + size_t(a.pairs) * sizeof(PairSmemV2);
    const size_t smem_max = fixed + size_t(kV2Pairs) * sizeof(PairSmemV2);
    if (cudaFuncSetAttribute(decode_v2_kernel<DT, kDelta>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem_max)) != cudaSuccess)
        return ZC_ECUDA;
    decode_v2_kernel<DT, kDelta><<<a.n_ctas, 64 * a.pairs, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

// The decompression launch of one dtype: format v2 (shared plane tables) or
// v1/v3; the XOR-delta variants exist for the integer dtypes only.
template <int DT>
int launch_decode_dtype(bool delta, const DecodeArgs &a, cudaStream_t s) {
    constexpr bool kInt = DT == ZC_U8 || DT == ZC_U16 || DT == ZC_U32;
    if constexpr (kInt) {
        if (a.version == 2) return delta ? launch_decode_v2_t<DT, true>(a, s) : launch_decode_v2_t<DT, false>(a, s);
        return delta ? launch_decode_t<DT, true>(a, s) : launch_decode_t<DT, false>(a, s);
    } else {
        if (delta) return ZC_EINVAL;  // deltas are coded as unsigned words only
        return a.version == 2 ? launch_decode_v2_t<DT, false>(a, s) : launch_decode_t<DT, false>(a, s);
    }
}

} // namespace

} // namespace zc
