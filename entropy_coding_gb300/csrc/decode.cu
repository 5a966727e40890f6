// decode.cu — decompression kernel.
//
// One warp restores one chunk (chunks are independent: ZipNN note, Method 5,
// the metadata map lets chunks decode in parallel). Per chunk a warp:
//   1. reads and bounds-checks the chunk table entry;
//   2. checks the CRC-32 of the stored bytes (cuZipNN: verify a blob before
//      decoding it), unless the caller asked not to;
//   3. copies a RAW chunk, or parses a grouped chunk's directory and, for
//      every rANS stream, its frequency table into a slot -> symbol lookup
//      table in shared memory;
//   4. runs the 32 interleaved rANS lanes of all coded streams forward in
//      step with the raw and constant streams, merges the W stream bytes of
//      each element back into its word (inverse exponent extraction) and
//      stores the 32 consecutive words of each step with one coalesced store.
// Renormalisation words are consumed from the end of each record backwards;
// they are staged in a 4-block shared-memory ring filled by cp.async.
#include "zc_kernels.cuh"

namespace zc {

namespace {

constexpr int kWarps = 4;
constexpr uint32_t kLutBytes = 4096, kSymBytes = 1024, kRingWords = 1024, kRingBytes = 2 * kRingWords;
constexpr uint32_t kStreamSmem = kLutBytes + kSymBytes + kRingBytes;  // 7 KB per coded stream
constexpr uint32_t kCrcSmem = 8 * 256 * 4;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = uint32_t(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Fetch 256-word block b of a record's word area into its ring slot.
__device__ __forceinline__ void fetch_block(uint16_t *ring, const uint8_t *wbase, uint32_t padded_bytes, int b) {
    const int lane = threadIdx.x & 31;
    uint32_t byte = uint32_t(b) * 512u + 16u * lane;
    if (byte < padded_bytes) cp_async16(reinterpret_cast<uint8_t *>(ring) + (b & 3) * 512 + 16 * lane, wbase + byte);
}

struct RansStream {
    uint32_t x;          // this lane's state
    int32_t ptr;         // words left (warp-uniform)
    int32_t next_block;  // next 256-word block to fetch, < 0 when done
    const uint8_t *wbase;
    uint32_t padded;     // pad16(2 * nwords)
    const uint8_t *lut;
    const uint32_t *sym;
    uint16_t *ring;
};

template <int DT>
__device__ void decode_chunk(const DecodeArgs &a, uint32_t c, uint8_t *wsm, const uint32_t (*crc_tab)[256]) {
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
    if (!(a.flags & ZC_NO_VERIFY)) {
        uint32_t crc = warp_crc_raw<false>(p, stored, 0xFFFFFFFFu, crc_tab) ^ 0xFFFFFFFFu;
        if (crc != ent.w) {
            if (lane == 0) status_or(a.d_status, ZC_ECRC);
            return;
        }
    }
    uint8_t *out = a.dst + uint64_t(c) * a.chunk_bytes;
    if (raw) {
        uint32_t nvec = (reinterpret_cast<uintptr_t>(out) & 15) ? 0 : len / 16;
        for (uint32_t v = lane; v < nvec; v += 32)
            reinterpret_cast<uint4 *>(out)[v] = __ldg(reinterpret_cast<const uint4 *>(p) + v);
        for (uint32_t i = nvec * 16 + lane; i < len; i += 32) out[i] = p[i];
        return;
    }

    // directory: W entries of mode << 30 | value, zero-padded to 16 bytes
    uint32_t dir = lane < 4 ? reinterpret_cast<const uint32_t *>(p)[lane] : 0u;
    bool bad = __any_sync(kFull, lane >= W && lane < 4 && dir != 0);
    uint32_t mode[W], val[W], roff[W];
    uint32_t pos = 16;
#pragma unroll
    for (int j = 0; j < W; j++) {
        uint32_t e = __shfl_sync(kFull, dir, j);
        mode[j] = e >> 30;
        val[j] = e & 0x3FFFFFFFu;
        roff[j] = pos;
        if (mode[j] == kModeConst) {
            bad |= val[j] > 255;
        } else if (mode[j] == kModeRaw) {
            bad |= val[j] != n;
            pos += uint32_t(pad16(n));
        } else if (mode[j] == kModeRans) {
            bad |= val[j] < kRecHead || val[j] > stored;
            pos += uint32_t(pad16(val[j]));
        } else {
            bad = true;
        }
        if (pos > stored) bad = true;
    }
    if (bad || pos != stored) {
        if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
        return;
    }

    // tables of the coded streams
    RansStream rs[W];
    bool tbad = false;
#pragma unroll
    for (int j = 0; j < W; j++) {
        if (mode[j] != kModeRans) continue;
        const uint8_t *rec = p + roff[j];
        uint8_t *lut = wsm + j * kStreamSmem;
        uint32_t *sym = reinterpret_cast<uint32_t *>(lut + kLutBytes);
        uint16_t *ring = reinterpret_cast<uint16_t *>(lut + kLutBytes + kSymBytes);
        uint32_t bits = rec[128 + lane];
        uint32_t present = __popc(bits);
        uint32_t k = __reduce_add_sync(kFull, present);
        uint32_t rank = 0;
        {   // exclusive prefix of present symbols over lanes
            uint32_t inc = present;
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t t = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += t;
            }
            rank = inc - present;
        }
        const uint32_t words_at = kRecHead + uint32_t(pad16(2 * k));
        bool lbad = k < 2 || val[j] < words_at || ((val[j] - words_at) & 1u);
        const uint16_t *freqs = reinterpret_cast<const uint16_t *>(rec + kRecHead);
        uint32_t f8[8], fsum = 0;
#pragma unroll
        for (int q = 0; q < 8; q++) {
            f8[q] = 0;
            if (!lbad && ((bits >> q) & 1u)) {
                f8[q] = freqs[rank++];
                lbad |= f8[q] == 0 || f8[q] >= kM;
            }
            fsum += f8[q];
        }
        for (uint32_t b = kRecHead + 2 * k + lane; !lbad && b < words_at; b += 32) lbad |= rec[b] != 0;
        uint32_t cum;
        {
            uint32_t inc = fsum;
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t t = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += t;
            }
            cum = inc - fsum;
            lbad |= __shfl_sync(kFull, inc, 31) != kM;
        }
        if (__any_sync(kFull, lbad)) {
            tbad = true;
            break;
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            uint32_t s = 8 * lane + q;
            if (f8[q]) {
                sym[s] = f8[q] | (cum << 12);
                for (uint32_t sl = cum; sl < cum + f8[q]; sl++) lut[sl] = uint8_t(s);
            }
            cum += f8[q];
        }
        rs[j].x = reinterpret_cast<const uint32_t *>(rec)[lane];
        const uint32_t nwords = (val[j] - words_at) / 2;
        rs[j].ptr = int32_t(nwords);
        rs[j].wbase = rec + words_at;
        rs[j].padded = uint32_t(pad16(2 * nwords));
        rs[j].lut = lut;
        rs[j].sym = sym;
        rs[j].ring = ring;
        int top = nwords ? int((nwords - 1) >> 8) : -1;
        for (int b = top; b >= 0 && b > top - 4; b--) fetch_block(ring, rs[j].wbase, rs[j].padded, b);
        rs[j].next_block = top - 4;
        if (__any_sync(kFull, rs[j].x < kRansL)) {
            tbad = true;
            break;
        }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    if (tbad) {
        if (lane == 0) status_or(a.d_status, ZC_ECORRUPT);
        return;
    }

    const uint32_t lt = lanemask_lt();
    const uint32_t T = (n + 31) / 32;
    for (uint32_t t = 0; t < T; t++) {
        const uint32_t i = t * 32 + lane;
        const bool active = i < n;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < W; j++) {
            uint32_t b;
            if (mode[j] == kModeConst) {
                b = val[j];
            } else if (mode[j] == kModeRaw) {
                b = active ? __ldg(p + roff[j] + i) : 0u;
            } else {
                RansStream &r = rs[j];
                uint32_t slot = r.x & (kM - 1);
                b = r.lut[slot];
                uint32_t e = r.sym[b];
                uint32_t xn = (e & 0xFFFu) * (r.x >> kProbBits) + slot - (e >> 12);
                bool need = active && xn < kRansL;
                uint32_t bal = __ballot_sync(kFull, need);
                if (need) {
                    int32_t idx = r.ptr - 1 - int32_t(__popc(bal & lt));
                    xn = (xn << 16) | r.ring[uint32_t(idx) & (kRingWords - 1)];
                }
                if (active) r.x = xn;
                r.ptr -= int32_t(__popc(bal));
                if (r.next_block >= 0 && r.ptr <= 256 * (r.next_block + 4)) {
                    __syncwarp();
                    fetch_block(r.ring, r.wbase, r.padded, r.next_block);
                    cp_async_commit();
                    r.next_block--;
                    if (r.next_block < 0) cp_async_wait_all();
                    else cp_async_wait2();
                    __syncwarp();
                }
            }
            word = (word << 8) | b;
        }
        if (active) {
            uint32_t w = Perm<DT>::inv(word);
            if (W == 4) reinterpret_cast<uint32_t *>(out)[i] = w;
            else if (W == 2) reinterpret_cast<uint16_t *>(out)[i] = uint16_t(w);
            else out[i] = uint8_t(w);
        }
    }
    bool fin_bad = false;
#pragma unroll
    for (int j = 0; j < W; j++)
        if (mode[j] == kModeRans) fin_bad |= rs[j].x != kRansL || rs[j].ptr != 0;
    if (__any_sync(kFull, fin_bad) && lane == 0) status_or(a.d_status, ZC_ECORRUPT);
}

template <int DT>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(DecodeArgs a) {
    constexpr int W = WordOf<DT>::W;
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t(*crc_tab)[256] = reinterpret_cast<uint32_t(*)[256]>(smem);
    const int warp = threadIdx.x >> 5;
    if (!(a.flags & ZC_NO_VERIFY)) load_crc_smem(crc_tab);
    __syncthreads();
    uint32_t c = blockIdx.x * kWarps + warp;
    if (c >= a.n_chunks) return;
    decode_chunk<DT>(a, c, smem + kCrcSmem + warp * W * kStreamSmem, crc_tab);
}

template <int DT>
int launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
    constexpr int W = WordOf<DT>::W;
    const size_t smem = kCrcSmem + size_t(kWarps) * W * kStreamSmem;
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
