// decode.cu — decompression kernel.
//
// One warp restores one chunk (chunks are independent: ZipNN note, Method 5,
// the metadata map lets chunks decode in parallel). Per chunk a warp:
//   1. reads and bounds-checks the chunk table entry;
//   2. checks the CRC-32 of the stored bytes (cuZipNN: verify a blob before
//      decoding it), unless the caller asked not to;
//   3. copies a RAW chunk, or parses a grouped chunk's directory and the
//      frequency table of its first rANS stream into a slot -> symbol lookup
//      table in shared memory;
//   4. runs the 32 interleaved rANS lanes forward eight steps at a time,
//      staging the decoded symbols of the 256 elements of those steps in
//      shared memory, then lets each lane gather the bytes of 8 consecutive
//      elements from every stream (coded, raw or constant), transpose them
//      into words, undo the exponent extraction and store them with vector
//      stores.
// Renormalisation words are consumed from the end of each record backwards
// and staged in a two-block shared-memory ring filled by cp.async. Chunks
// with more than one coded stream first decode the other ones into the
// tail of their own output range (one byte per element and stream,
// interleaved); the main pass reads them from there before any store can
// reach them (the write front advances W bytes per element, the read front
// q < W bytes per element from (W - q) n onward, and they meet only at the
// end).
#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kWarps = 8;
constexpr uint32_t kLutBytes = 4096, kSymBytes = 1024, kRingWords = 512, kRingBytes = 2 * kRingWords,
                   kStageBytes = 256;
constexpr uint32_t kSlotSmem = kLutBytes + kSymBytes + kRingBytes + kStageBytes;
// replicated CRC byte table + the gap table of the output pieces + the 496-byte gap table
constexpr uint32_t kCrcSmem = kCrcRepWords * 4 + 2 * 4 * 256 * 4;


struct Rans {
    uint32_t x;          // this lane's state
    int32_t ptr;         // words left to consume (warp-uniform)
    int32_t next_block;  // next 256-word block to fetch, < 0 when all fetched
    const uint8_t *wbase;
    uint32_t padded;     // pad16(2 * nwords)
    const uint8_t *lut;
    const uint32_t *sym;
    uint16_t *ring;
    uint8_t *stage;
};

// Fetch 256-word block b of a record's word area into its ring slot.
__device__ __forceinline__ void fetch_block(const Rans &r, int b) {
    const int lane = threadIdx.x & 31;
    uint32_t byte = uint32_t(b) * 512u + 16u * lane;
    if (byte < r.padded) cp_async16(reinterpret_cast<uint8_t *>(r.ring) + (b & 1) * 512 + 16 * lane, r.wbase + byte);
}

// Parse a rANS record (val bytes) into lookup tables in `slot` and load the
// lane states and the last two word blocks. Returns false if malformed.
__device__ bool rans_setup(const uint8_t *rec, uint32_t val, uint8_t *slot, Rans &r) {
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
    bool bad = k < 2 || val < words_at || ((val - words_at) & 1u);
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
    const uint32_t nwords = (val - words_at) / 2;
    r.ptr = int32_t(nwords);
    r.wbase = rec + words_at;
    r.padded = uint32_t(pad16(2 * nwords));
    r.lut = lut;
    r.sym = sym;
    r.ring = reinterpret_cast<uint16_t *>(slot + kLutBytes + kSymBytes);
    r.stage = slot + kLutBytes + kSymBytes + kRingBytes;
    int top = nwords ? int((nwords - 1) >> 8) : -1;
    if (top >= 0) fetch_block(r, top);
    if (top >= 1) fetch_block(r, top - 1);
    r.next_block = top - 2;
    cp_async_commit();
    return true;
}

// One rANS decode step of the warp: returns this lane's symbol.
__device__ __forceinline__ uint32_t rans_step(Rans &r, bool active, uint32_t lt) {
    uint32_t slot = r.x & (kM - 1);
    uint32_t s = r.lut[slot];
    uint32_t e = r.sym[s];
    uint32_t xn = (e & 0xFFFu) * (r.x >> kProbBits) + slot - (e >> 12);
    const bool need = active && xn < kRansL;
    const uint32_t bal = __ballot_sync(kFull, need);
    // every lane reads its candidate word (in bounds of the ring), so no branch
    const int32_t idx = r.ptr - 1 - int32_t(__popc(bal & lt));
    const uint32_t w = r.ring[uint32_t(idx) & (kRingWords - 1)];
    xn = need ? ((xn << 16) | w) : xn;
    if (active) r.x = xn;
    r.ptr -= int32_t(__popc(bal));
    if (r.next_block >= 0 && r.ptr <= 256 * (r.next_block + 2)) {
        __syncwarp();
        fetch_block(r, r.next_block);
        cp_async_commit();
        r.next_block--;
        if (r.next_block < 0) cp_async_wait_all();
        else cp_async_wait<1>();
        __syncwarp();
    }
    return s;
}

__device__ __forceinline__ bool rans_final_ok(const Rans &r) {
    return !__any_sync(kFull, r.x != kRansL || r.ptr != 0);
}

// Stream kinds in the main pass.
constexpr uint32_t kKConst = 0, kKRaw = 1, kKMain = 2, kKStaged = 3;

// 8 consecutive elements' bytes of stream j packed in two words (element e
// of the eight in byte e of the pair), from each kind of stream.
struct Col8 {
    uint32_t lo, hi;
};

template <int DT>
__device__ void decode_chunk(const DecodeArgs &a, uint32_t c, uint8_t *wsm, const uint32_t *crc_rep,
                             const uint32_t (*gap_out)[256], const uint32_t (*gap496)[256]) {
    constexpr int W = WordOf<DT>::W;
    const int lane = threadIdx.x & 31;
    const uint64_t table_end = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * a.n_chunks;

    uint4 ent = make_uint4(0, 0, 0, 0);
    if (lane == 0) ent = reinterpret_cast<const uint4 *>(a.blob + ZC_HEADER_BYTES)[c];
    ent.x = __shfl_sync(kFull, ent.x, 0);
    ent.y = __shfl_sync(kFull, ent.y, 0);
    ent.z = __shfl_sync(kFull, ent.z, 0);
    ent.w = __shfl_sync(kFull, ent.w, 0);
    const uint64_t off = uint64_t(ent.x) | (uint64_t(ent.y) << 32);
    const uint32_t stored = ent.z & 0x7FFFFFFFu;
    const bool raw = ent.z >> 31;
    const uint32_t len = uint32_t(umin64(a.chunk_bytes, a.nbytes - uint64_t(c) * a.chunk_bytes));
    const uint32_t n = len / W;

    bool ok = (off & 15) == 0 && off >= table_end && off <= a.blob_bytes && stored <= a.blob_bytes - off;
    ok = ok && (raw ? stored == len : (stored % 16 == 0 && stored >= 16 && stored <= max_grouped(len, W)));
    if (!ok) {
        if (lane == 0) status_or(a.d_status, ZC_EFORMAT);
        return;
    }
    const uint8_t *p = a.blob + off;
    const bool verify = !(a.flags & ZC_NO_VERIFY);
    const uint32_t *row = crc_rep + lane;
    uint8_t *out = a.dst + uint64_t(c) * a.chunk_bytes;
    if (raw) {
        uint32_t nvec = (reinterpret_cast<uintptr_t>(out) & 15) ? 0 : len / 16;
        for (uint32_t v = lane; v < nvec; v += 32)
            reinterpret_cast<uint4 *>(out)[v] = __ldg(reinterpret_cast<const uint4 *>(p) + v);
        for (uint32_t i = nvec * 16 + lane; i < len; i += 32) out[i] = p[i];
        // a RAW chunk stores the original bytes, so its CRC is the payload's
        if (verify && (crc_strided<1, false>(p, len, 0xFFFFFFFFu, crc_rep, gap496, nullptr) ^ 0xFFFFFFFFu) != ent.w &&
            lane == 0)
            status_or(a.d_status, ZC_ECRC);
        return;
    }

    // directory: W entries of mode << 30 | value, zero-padded to 16 bytes
    uint32_t dir = lane < 4 ? reinterpret_cast<const uint32_t *>(p)[lane] : 0u;
    bool bad = __any_sync(kFull, lane >= W && lane < 4 && dir != 0);
    uint32_t kind[W], val[W], roff[W], sub[W];
    uint32_t pos = 16, coded = 0;
#pragma unroll
    for (int j = 0; j < W; j++) {
        uint32_t e = __shfl_sync(kFull, dir, j);
        uint32_t mode = e >> 30;
        val[j] = e & 0x3FFFFFFFu;
        roff[j] = pos;
        sub[j] = 0;
        if (mode == kModeConst) {
            kind[j] = kKConst;
            bad |= val[j] > 255;
        } else if (mode == kModeRaw) {
            kind[j] = kKRaw;
            bad |= val[j] != n;
            pos += uint32_t(pad16(n));
        } else if (mode == kModeRans) {
            kind[j] = coded == 0 ? kKMain : kKStaged;
            sub[j] = coded == 0 ? 0 : coded - 1;
            coded++;
            bad |= val[j] < kRecHead || val[j] > stored;
            pos += uint32_t(pad16(val[j]));
        } else {
            kind[j] = kKConst;
            bad = true;
        }
        if (pos > stored) bad = true;
    }
    if (bad || pos != stored) {
        if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
        return;
    }
    const uint32_t lt = lanemask_lt();
    const uint32_t T = (n + 31) / 32;

    // coded streams after the first: decode into the output tail first, q
    // bytes per element
    const uint32_t q = coded > 1 ? coded - 1 : 0;
    uint8_t *tail = out + (len - q * n);
    if (q) {
#pragma unroll
        for (int j = 0; j < W; j++) {
            if (kind[j] != kKStaged) continue;
            Rans r;
            if (!rans_setup(p + roff[j], val[j], wsm, r)) bad = true;
            cp_async_wait_all();
            __syncwarp();
            if (bad) break;
            for (uint32_t t = 0; t < T; t++) {
                uint32_t i = t * 32 + lane;
                bool active = i < n;
                uint32_t s = rans_step(r, active, lt);
                if (active) tail[uint64_t(i) * q + sub[j]] = uint8_t(s);
            }
            bad |= !rans_final_ok(r);
            __syncwarp();
        }
        __syncwarp();
        if (bad) {
            if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
            return;
        }
    }

    Rans rs;
    bool have_main = false;
#pragma unroll
    for (int j = 0; j < W; j++) {
        if (kind[j] != kKMain) continue;
        have_main = true;
        if (!rans_setup(p + roff[j], val[j], wsm, rs)) bad = true;
    }
    cp_async_wait_all();
    __syncwarp();
    if (bad) {
        if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
        return;
    }

    // groups of 8 steps = 256 elements; each lane then owns 8 consecutive
    // elements 256 g + 8 lane .. + 7
    const uint32_t groups = n / 256;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    // CRC of the decoded bytes: lane l's 8 elements of each group form one
    // 8W-byte piece; pieces of a group are consecutive, so each lane keeps the
    // register of its own pieces and shifts it over the others' (256 W - 8 W
    // bytes) between groups, then the lanes are folded (crc_fold).
    uint32_t Rl = 0;
    uint2 rn1[W], rn2[W];  // raw columns of the next two groups
#pragma unroll
    for (int j = 0; j < W; j++) {
        const uint2 *src = reinterpret_cast<const uint2 *>(p + roff[j]) + lane;
        rn1[j] = (kind[j] == kKRaw && groups > 0) ? __ldg(src) : make_uint2(0, 0);
        rn2[j] = (kind[j] == kKRaw && groups > 1) ? __ldg(src + 32) : make_uint2(0, 0);
    }
    for (uint32_t g = 0; g < groups; g++) {
        Col8 col[W];
#pragma unroll
        for (int j = 0; j < W; j++) {
            col[j].lo = rn1[j].x;
            col[j].hi = rn1[j].y;
            rn1[j] = rn2[j];
            if (kind[j] == kKRaw && g + 2 < groups)
                rn2[j] = __ldg(reinterpret_cast<const uint2 *>(p + roff[j] + 256 * (g + 2)) + lane);
        }
        if (have_main) {
#pragma unroll
            for (int k = 0; k < 8; k++) rs.stage[32 * k + lane] = uint8_t(rans_step(rs, true, lt));
            __syncwarp();
        }
        const uint32_t e0 = 256 * g + 8 * lane;
#pragma unroll
        for (int j = 0; j < W; j++) {
            if (kind[j] == kKConst) {
                col[j].lo = col[j].hi = val[j] * 0x01010101u;
            } else if (kind[j] == kKMain) {
                const uint2 v = *reinterpret_cast<const uint2 *>(rs.stage + 8 * lane);
                col[j].lo = v.x;
                col[j].hi = v.y;
            } else if (kind[j] == kKStaged) {
                uint32_t v[2] = {0, 0};
                for (int e = 0; e < 8; e++)
                    v[e >> 2] |= uint32_t(__ldcg(tail + uint64_t(e0 + e) * q + sub[j])) << (8 * (e & 3));
                col[j].lo = v[0];
                col[j].hi = v[1];
            }
        }
        __syncwarp();
        const uint32_t cin = g == 0 ? (lane == 0 ? 0xFFFFFFFFu : 0u) : shift_smem(Rl, gap_out);
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
            if (verify) Rl = crc_rep16(crc_rep16(cin, v[0], row), v[1], row);
            if (vec_ok) {
                uint4 *o = reinterpret_cast<uint4 *>(out + 4ull * e0);
                o[0] = v[0];
                o[1] = v[1];
            } else {
                uint32_t *o = reinterpret_cast<uint32_t *>(out) + e0;
                o[0] = v[0].x; o[1] = v[0].y; o[2] = v[0].z; o[3] = v[0].w;
                o[4] = v[1].x; o[5] = v[1].y; o[6] = v[1].z; o[7] = v[1].w;
            }
        } else if constexpr (W == 2) {
            uint4 v;
            v.x = Perm<DT>::inv2(__byte_perm(col[1].lo, col[0].lo, 0x5140));
            v.y = Perm<DT>::inv2(__byte_perm(col[1].lo, col[0].lo, 0x7362));
            v.z = Perm<DT>::inv2(__byte_perm(col[1].hi, col[0].hi, 0x5140));
            v.w = Perm<DT>::inv2(__byte_perm(col[1].hi, col[0].hi, 0x7362));
            if (verify) Rl = crc_rep16(cin, v, row);
            if (vec_ok) {
                *reinterpret_cast<uint4 *>(out + 2ull * e0) = v;
            } else {
                uint16_t *o = reinterpret_cast<uint16_t *>(out) + e0;
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                for (int e = 0; e < 4; e++) {
                    o[2 * e] = uint16_t(w4[e]);
                    o[2 * e + 1] = uint16_t(w4[e] >> 16);
                }
            }
        } else {
            if (verify) Rl = crc_rep_word(crc_rep_word(cin, col[0].lo, row), col[0].hi, row);
            if ((reinterpret_cast<uintptr_t>(out) & 7) == 0) {
                *reinterpret_cast<uint2 *>(out + e0) = make_uint2(col[0].lo, col[0].hi);
            } else {
                for (int e = 0; e < 8; e++) out[e0 + e] = uint8_t((e < 4 ? col[0].lo : col[0].hi) >> (8 * (e & 3)));
            }
        }
    }
    // the last < 256 elements, one step at a time
    for (uint32_t t = groups * 8; t < T; t++) {
        const uint32_t i = t * 32 + lane;
        const bool active = i < n;
        const uint32_t sm = have_main ? rans_step(rs, active, lt) : 0u;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < W; j++) {
            uint32_t b = 0;
            if (active) {
                if (kind[j] == kKConst) b = val[j];
                else if (kind[j] == kKRaw) b = __ldg(p + roff[j] + i);
                else if (kind[j] == kKMain) b = sm;
                else b = __ldcg(tail + uint64_t(i) * q + sub[j]);
            }
            word = (word << 8) | b;
        }
        __syncwarp();
        if (active) {
            uint32_t w = Perm<DT>::inv(word);
            if (W == 4) reinterpret_cast<uint32_t *>(out)[i] = w;
            else if (W == 2) reinterpret_cast<uint16_t *>(out)[i] = uint16_t(w);
            else out[i] = uint8_t(w);
        }
    }
    bool bad_end = have_main && !rans_final_ok(rs);
    if (verify) {
        constexpr int kLogPiece = W == 4 ? 5 : W == 2 ? 4 : 3;
        uint32_t reg = groups ? crc_fold<1>(Rl, kLogPiece, nullptr) : 0xFFFFFFFFu;
        __syncwarp();
        const uint32_t done = groups * 256 * W;
        reg = crc_any<1, true>(out + done, len - done, reg, crc_rep, gap496, nullptr);
        if ((reg ^ 0xFFFFFFFFu) != ent.w && lane == 0) status_or(a.d_status, ZC_ECRC);
    }
    if (bad_end && lane == 0) status_or(a.d_status, ZC_ECORRUPT);
}

template <int DT>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int W = WordOf<DT>::W;
    uint32_t *crc_rep = reinterpret_cast<uint32_t *>(smem);
    uint32_t(*gap_out)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + kCrcRepWords * 4);
    uint32_t(*gap496)[256] = reinterpret_cast<uint32_t(*)[256]>(smem + kCrcRepWords * 4 + 4 * 256 * 4);
    const int warp = threadIdx.x >> 5;
    if (!(a.flags & ZC_NO_VERIFY)) {
        load_crc_rep(crc_rep);
        load_shift_smem(gap_out, W == 4 ? kSh992 : W == 2 ? kSh496 : kSh248);
        load_shift_smem(gap496, kSh496);
    }
    __syncthreads();
    uint32_t c = blockIdx.x * kWarps + warp;
    if (c >= a.n_chunks) return;
    decode_chunk<DT>(a, c, smem + kCrcSmem + warp * kSlotSmem, crc_rep, gap_out, gap496);
}

template <int DT>
int launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
    const size_t smem = kCrcSmem + size_t(kWarps) * kSlotSmem;
    if (cudaFuncSetAttribute(decode_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return ZC_ECUDA;
    const int grid = int((a.n_chunks + kWarps - 1) / kWarps);
    decode_kernel<DT><<<grid, kWarps * 32, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZC_OK : ZC_ECUDA;
}

} // namespace

int launch_decode(int dtype, const DecodeArgs &a, cudaStream_t s) {
    if (a.n_chunks == 0) return ZC_OK;
    switch (dtype) {
    case ZC_U8: return launch_decode_t<ZC_U8>(a, s);
    case ZC_U16: return launch_decode_t<ZC_U16>(a, s);
    case ZC_U32: return launch_decode_t<ZC_U32>(a, s);
    case ZC_BF16: return launch_decode_t<ZC_BF16>(a, s);
    case ZC_FP16: return launch_decode_t<ZC_FP16>(a, s);
    case ZC_FP32: return launch_decode_t<ZC_FP32>(a, s);
    default: return ZC_EINVAL;
    }
}

} // namespace zc
