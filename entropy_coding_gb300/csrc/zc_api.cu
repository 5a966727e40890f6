// zc_api.cu — the C ABI (include/zc.h): argument checks, workspace layout,
// header construction and kernel launches. No entry point allocates device
// memory or synchronises; device-side errors are reported through *d_status.
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "zc_kernels.cuh"

namespace {

using namespace zc;

constexpr uint64_t kCtrlBytes = 256;    // coder ticket; then per tensor: done counter, header CRC accumulator
constexpr uint64_t kCrcUnit = 32768;    // bytes per warp in zc_crc32

uint64_t pad256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

bool valid_params(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold) {
    int W = word_bytes(dtype);
    if (W == 0 || nbytes % uint64_t(W)) return false;
    if (chunk_bytes < ZC_MIN_CHUNK || chunk_bytes > ZC_MAX_CHUNK || chunk_bytes % 64) return false;
    if (!(threshold > 0.0) || !(threshold <= 1e9)) return false;
    if ((nbytes + chunk_bytes - 1) / chunk_bytes > 0xFFFFFFFFull) return false;
    return true;
}

uint64_t chunks_of(uint64_t nbytes, uint32_t chunk_bytes) { return (nbytes + chunk_bytes - 1) / chunk_bytes; }

constexpr uint64_t kInfoBytes = 32;          // per chunk of a wave: CRC + W stream words
constexpr uint64_t kTableBytes = 512;        // per chunk of a wave and stream: 256 u16 table
constexpr uint64_t kWaveBytes = 2048ull << 20;  // workspace of one statistics + coding wave, at most

// Room for one coded record of a stream in a coding warp's slot. A record is
// kept only while it is below lim = ceil(threshold x n) bytes, and the coder
// gives a stream up once its record has reached lim, after at most one more
// batch of 32 steps x 32 words (2048 bytes); a record can never exceed the
// header, the table and one word per symbol.
uint64_t rec_stride(uint32_t chunk_bytes, int W, double threshold, uint32_t version = 1) {
    const uint64_t n = chunk_bytes / W;
    if (version == 3) {
        // a word list per lane: each lane's words are staged at a stride of
        // pad8(T) words (T = steps) after the counts, whatever the threshold
        const uint64_t Ts = ((n + 31) / 32 + 7) & ~uint64_t(7);
        return pad16(kRecHead + kMaxTable + 64 + 2 * 32 * Ts) + 16;
    }
    const uint64_t full = kRecHead + kMaxTable + 2 * n;
    const double lim = std::ceil(threshold * double(n));
    uint64_t cap = full;
    if (lim + double(kRecHead + kMaxTable + 2048) < double(full)) cap = uint64_t(lim) + kRecHead + kMaxTable + 2048;
    return pad16(cap) + 16;
}

uint64_t slot_bytes(uint32_t chunk_bytes, int W, double threshold, uint32_t version = 1) {
    return pad256(uint64_t(W) * rec_stride(chunk_bytes, W, threshold, version));
}

// Workspace after the control block and the chunk status words: the wave's
// info and tables, then the coding warps' slots.
uint64_t n_pad(uint32_t chunk_bytes, int W) { return (uint64_t(chunk_bytes / W) + 31) / 32 * 32; }

// Chunks per wave: all of them, unless their statistics and candidate bytes
// would take more than kWaveBytes.
uint64_t wave_chunks(uint64_t nc, uint32_t chunk_bytes, int W) {
    const uint64_t per_chunk = kInfoBytes + (kTableBytes + n_pad(chunk_bytes, W)) * uint64_t(W);
    const uint64_t most = kWaveBytes / per_chunk;
    return nc < most ? nc : most;
}

struct WaveLayout {
    uint64_t info, ftab, cand, slots;  // offsets from the start of the wave area
};
WaveLayout wave_layout(uint64_t wave, int W, uint32_t chunk_bytes) {
    WaveLayout l;
    l.info = 0;
    l.ftab = pad256(kInfoBytes * wave);
    l.cand = l.ftab + pad256(kTableBytes * uint64_t(W) * wave);
    l.slots = l.cand + pad256(n_pad(chunk_bytes, W) * uint64_t(W) * wave);
    return l;
}

uint32_t host_crc_table[256];
bool host_crc_ready = false;

uint32_t host_crc32(const uint8_t *p, uint64_t n, uint32_t reg = 0xFFFFFFFFu) {
    if (!host_crc_ready) {  // idempotent; a race only recomputes the same values
        for (uint32_t b = 0; b < 256; b++) {
            uint32_t r = b;
            for (int k = 0; k < 8; k++) r = gf2_mul_x(r);
            host_crc_table[b] = r;
        }
        host_crc_ready = true;
    }
    for (uint64_t i = 0; i < n; i++) reg = host_crc_table[(reg ^ p[i]) & 0xFF] ^ (reg >> 8);
    return reg;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Coding warps that can run at once (one chunk in flight each).
uint64_t max_workers(uint64_t n_chunks) {
    uint64_t most = uint64_t(sm_count()) * uint64_t(encode_warps_per_sm());
    if (most < 1) most = 1;
    return n_chunks < most ? n_chunks : most;
}

uint32_t get32(const uint8_t *p) { return uint32_t(p[0]) | uint32_t(p[1]) << 8 | uint32_t(p[2]) << 16 | uint32_t(p[3]) << 24; }
uint64_t get64(const uint8_t *p) { return uint64_t(get32(p)) | uint64_t(get32(p + 4)) << 32; }
void put32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = uint8_t(v >> (8 * i)); }
void put64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = uint8_t(v >> (8 * i)); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::atomic<uint32_t> g_hooks{0};

// The wait limits of a call: short ones when a test hook makes a wait run out.
void set_waits(EncodeArgs &a) {
    a.hooks = g_hooks.load(std::memory_order_relaxed);
    a.spin_limit = (a.hooks & ZC_HOOK_LOOKBACK_STALL) ? kSpinLimitTest : kSpinLimit;
}
void set_waits(DecodeArgs &a) {
    a.hooks = g_hooks.load(std::memory_order_relaxed);
    a.wait_cycles = (a.hooks & ZC_HOOK_PRODUCER_STALL) ? kWaitCyclesTest : kWaitCycles;
}

} // namespace

extern "C" void zc_set_test_hooks(uint32_t hooks) {
    g_hooks.store(hooks & (ZC_HOOK_LOOKBACK_STALL | ZC_HOOK_PRODUCER_STALL), std::memory_order_relaxed);
}

extern "C" uint64_t zc_blob_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold) {
    if (!valid_params(nbytes, dtype, chunk_bytes, threshold)) return 0;
    const int W = word_bytes(dtype);
    const uint64_t nc = chunks_of(nbytes, chunk_bytes);
    uint64_t total = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * nc;
    if (nc == 0) return total;
    const uint64_t full = nc - 1, last = nbytes - full * chunk_bytes;
    auto worst = [&](uint64_t len) {
        uint64_t w = pad16(len);
        if (threshold > 1.0 && max_grouped(len, W) > w) w = max_grouped(len, W);
        return w;
    };
    return total + full * worst(chunk_bytes) + worst(last);
}

extern "C" int zc_blob_info(const void *h_blob_prefix, uint64_t avail, zc_info *out) {
    const uint8_t *b = static_cast<const uint8_t *>(h_blob_prefix);
    if (!b || !out || avail < ZC_HEADER_BYTES) return ZC_EFORMAT;
    const uint32_t version = uint32_t(b[4] | b[5] << 8);
    if (std::memcmp(b, "ZCNN", 4) != 0 || version < 1 || version > 3) return ZC_EFORMAT;
    const int dtype = b[6], ndim = b[7];
    const uint32_t chunk_bytes = get32(b + 8);
    const uint64_t nbytes = get64(b + 16);
    const uint32_t nc = get32(b + 24);
    const int W = word_bytes(dtype);
    if (W == 0 || ndim > 8 || b[12] != kLanes || b[13] != kProbBits || b[14] || b[15]) return ZC_EFORMAT;
    if (!valid_params(nbytes, dtype, chunk_bytes, 0.95) || chunks_of(nbytes, chunk_bytes) != nc) return ZC_EFORMAT;
    uint64_t elems = 1;
    for (int d = 0; d < 8; d++) {
        int64_t v = int64_t(get64(b + 32 + 8 * d));
        if (d >= ndim) {
            if (v != 0) return ZC_EFORMAT;
            continue;
        }
        if (v < 0) return ZC_EFORMAT;
        if (v && elems > UINT64_MAX / uint64_t(v)) return ZC_EFORMAT;
        elems *= uint64_t(v);
    }
    if (elems * uint64_t(W) != nbytes) return ZC_EFORMAT;
    // v2: W plane tables of 256 u16 follow the chunk table, each all zeros or
    // a 12-bit table of at least two symbols
    const uint64_t table_end = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * nc + (version == 2 ? 512ull * W : 0);
    if (avail < table_end) return ZC_EFORMAT;
    if (version == 2) {
        for (int j = 0; j < W; j++) {
            const uint8_t *t = b + table_end - 512ull * (W - j);
            uint32_t sum = 0, nz = 0;
            for (int v = 0; v < 256; v++) {
                const uint32_t f = uint32_t(t[2 * v]) | uint32_t(t[2 * v + 1]) << 8;
                sum += f;
                nz += f ? 1u : 0u;
            }
            if (!(sum == 0 || (sum == kM && nz >= 2))) return ZC_EFORMAT;
        }
    }
    uint8_t head[ZC_HEADER_BYTES];
    std::memcpy(head, b, ZC_HEADER_BYTES);
    put32(head + 28, 0);
    uint32_t reg = host_crc32(head, ZC_HEADER_BYTES);
    reg = host_crc32(b + ZC_HEADER_BYTES, table_end - ZC_HEADER_BYTES, reg);
    if ((reg ^ 0xFFFFFFFFu) != get32(b + 28)) return ZC_ECRC;
    uint64_t off = table_end;
    for (uint32_t c = 0; c < nc; c++) {
        const uint8_t *e = b + ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * c;
        const uint64_t len = (c + 1 < nc) ? chunk_bytes : nbytes - uint64_t(c) * chunk_bytes;
        const uint32_t sm = get32(e + 8), stored = sm & 0x7FFFFFFFu;
        if (get64(e) != off) return ZC_EFORMAT;
        if ((sm >> 31) ? stored != len : (stored % 16 || stored > max_grouped(len, W, version))) return ZC_EFORMAT;
        off += pad16(stored);
    }
    out->dtype = dtype;
    out->ndim = ndim;
    for (int d = 0; d < 8; d++) out->shape[d] = int64_t(get64(b + 32 + 8 * d));
    out->nbytes = nbytes;
    out->blob_bytes = off;
    out->n_chunks = nc;
    out->chunk_bytes = chunk_bytes;
    out->version = version;
    out->reserved = 0;
    return ZC_OK;
}

namespace {

// Check one tensor of a compression call and describe it for the kernels
// (chunk_base is set by the caller).
int make_tensor(const void *d_src, const void *d_base, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                uint32_t chunk_bytes, double threshold, void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                uint32_t version, TensorDesc &d) {
    if (!valid_params(nbytes, dtype, chunk_bytes, threshold)) return ZC_EINVAL;
    if (ndim < 0 || ndim > 8 || (ndim > 0 && !h_shape)) return ZC_EINVAL;
    const int W = word_bytes(dtype);
    uint64_t elems = 1;
    for (int dd = 0; dd < ndim; dd++) {
        if (h_shape[dd] < 0) return ZC_EINVAL;
        if (h_shape[dd] && elems > UINT64_MAX / uint64_t(h_shape[dd])) return ZC_EINVAL;
        elems *= uint64_t(h_shape[dd]);
    }
    if (elems * uint64_t(W) != nbytes) return ZC_EINVAL;
    if (!d_blob || !d_blob_bytes || (nbytes && !d_src)) return ZC_EINVAL;
    if (!aligned(d_src, W) || !aligned(d_blob, 16) || !aligned(d_blob_bytes, 8)) return ZC_EINVAL;
    const uint64_t nc = chunks_of(nbytes, chunk_bytes);
    const uint64_t planes = version == 2 ? 512ull * W : 0;  // v2: the plane tables
    if (blob_capacity < ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * nc + planes) return ZC_ECAPACITY;
    d = TensorDesc{};
    d.src = static_cast<const uint8_t *>(d_src);
    d.base = static_cast<const uint8_t *>(d_base);
    d.blob = static_cast<uint8_t *>(d_blob);
    d.d_blob_bytes = d_blob_bytes;
    d.nbytes = nbytes;
    d.cap = blob_capacity;
    d.n_chunks = uint32_t(nc);
    uint8_t head[ZC_HEADER_BYTES] = {};
    std::memcpy(head, "ZCNN", 4);
    head[4] = uint8_t(version);
    head[6] = uint8_t(dtype);
    head[7] = uint8_t(ndim);
    put32(head + 8, chunk_bytes);
    head[12] = uint8_t(kLanes);
    head[13] = uint8_t(kProbBits);
    put64(head + 16, nbytes);
    put32(head + 24, uint32_t(nc));
    for (int dd = 0; dd < ndim; dd++) put64(head + 32 + 8 * dd, uint64_t(h_shape[dd]));
    if (nc == 0) {  // the whole blob is the header (v2: and zero plane tables)
        uint32_t reg = host_crc32(head, ZC_HEADER_BYTES);
        static const uint8_t zeros[512] = {};
        for (uint64_t z = 0; z < planes; z += 512) reg = host_crc32(zeros, 512, reg);
        put32(head + 28, reg ^ 0xFFFFFFFFu);
    }
    std::memcpy(d.header, head, ZC_HEADER_BYTES);
    return ZC_OK;
}

// A batch's descriptor table reaches the device through kernel parameters
// (copied when the launch is issued): no pageable copy, no host wait.
constexpr uint32_t kParamWords = 7680;
struct TableBlock {
    uint32_t words;
    uint32_t w[kParamWords];
};
static_assert(sizeof(TableBlock) <= 32764, "kernel parameters are at most 32764 bytes");

__global__ void table_kernel(const TableBlock b, uint32_t *dst) {
    for (uint32_t i = threadIdx.x; i < b.words; i += blockDim.x) dst[i] = b.w[i];
}

int upload_table(const void *h, uint64_t bytes, void *d, cudaStream_t s) {
    static_assert(sizeof(TensorDesc) % 4 == 0 && sizeof(BlobDesc) % 4 == 0, "descriptors are whole words");
    const uint32_t *src = static_cast<const uint32_t *>(h);
    uint32_t *dst = static_cast<uint32_t *>(d);
    const uint64_t words = bytes / 4;
    static thread_local TableBlock blk;  // 30 KB: off the stack
    for (uint64_t w0 = 0; w0 < words; w0 += kParamWords) {
        blk.words = uint32_t(words - w0 < kParamWords ? words - w0 : kParamWords);
        std::memcpy(blk.w, src + w0, 4ull * blk.words);
        table_kernel<<<1, 256, 0, s>>>(blk, dst + w0);
        if (cudaGetLastError() != cudaSuccess) return ZC_ECUDA;
    }
    return ZC_OK;
}

// The address the kernels use for a data buffer: device or managed memory of
// the current device as given, page-locked host memory (cudaHostAlloc,
// cudaHostRegister) through its device mapping, so that the kernels read or
// write host memory directly over the host link. Unregistered host memory
// and other devices' memory are refused: the kernels never touch an address
// that the current device cannot reach.
int kernel_address(const void *p, const void **out) {
    *out = nullptr;
    if (!p) return ZC_OK;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not left behind for the launch checks
        return ZC_EINVAL;
    }
    if (!at.devicePointer) return ZC_EINVAL;
    if (at.type == cudaMemoryTypeDevice) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || at.device != dev) return ZC_EINVAL;
    } else if (at.type != cudaMemoryTypeHost && at.type != cudaMemoryTypeManaged) {
        return ZC_EINVAL;
    }
    *out = at.devicePointer;
    return ZC_OK;
}

template <class T>
int resolve(T *&p) {
    const void *q = nullptr;
    const int st = kernel_address(p, &q);
    p = const_cast<T *>(static_cast<const T *>(q));
    return st;
}

// Kernel addresses of a tensor's (a blob's) buffers; after all checks.
int resolve_tensor(TensorDesc &d) {
    int st = resolve(d.src);
    if (st == ZC_OK) st = resolve(d.base);
    if (st == ZC_OK) st = resolve(d.blob);
    if (st == ZC_OK) st = resolve(d.d_blob_bytes);
    return st;
}

int resolve_blob(BlobDesc &d) {
    int st = resolve(d.blob);
    if (st == ZC_OK) st = resolve(d.base);
    if (st == ZC_OK) st = resolve(d.dst);
    return st;
}

// Workspace of a compression call over n tensors and nc chunks: control
// (coder ticket; per tensor a done counter and a header-CRC accumulator),
// the tensor table (batches), the chunk status words, then a wave's
// statistics and the coding warps' slots.
uint64_t ctrl_bytes(uint64_t n) { return kCtrlBytes + pad256(16 * n); }
uint64_t table_bytes(uint64_t n) { return n > 1 ? pad256(sizeof(TensorDesc) * n) : 0; }
// v2: per tensor and plane, 256 u64 counts, then the 512-byte tables
uint64_t hist_bytes(uint64_t n, int W, uint32_t version) { return version == 2 ? pad256(2048ull * W * n) : 0; }
uint64_t ptab_bytes(uint64_t n, int W, uint32_t version) { return version == 2 ? pad256(512ull * W * n) : 0; }

// max_tc: the most chunks of one tensor (v2 waves hold whole tensors)
uint64_t ws_size(uint64_t n, uint64_t nc, int W, uint32_t chunk_bytes, uint32_t version, uint64_t max_tc) {
    const uint64_t head = ctrl_bytes(n) + table_bytes(n) + hist_bytes(n, W, version) + ptab_bytes(n, W, version);
    if (nc == 0) return head;
    uint64_t wave = wave_chunks(nc, chunk_bytes, W);
    if (version == 2 && wave < max_tc) wave = max_tc;
    // every coding warp for thresholds up to 1; at least one warp for any
    // threshold (larger thresholds then run fewer warps)
    uint64_t slots = max_workers(nc) * slot_bytes(chunk_bytes, W, 1.0, version);
    const uint64_t one_any = slot_bytes(chunk_bytes, W, 1e9, version);
    if (slots < one_any) slots = one_any;
    return head + pad256(8 * nc) + wave_layout(wave, W, chunk_bytes).slots + slots;
}

// Lay out the workspace and launch the statistics + coding waves over the
// call's chunks. `table` holds the n > 1 tensors (copied to the workspace).
int run_compress(EncodeArgs &a, const TensorDesc *table, uint32_t n, bool delta, int dtype, uint32_t chunk_bytes,
                 double threshold, uint32_t version, void *d_ws, uint64_t ws_bytes, cudaStream_t s) {
    const int W = word_bytes(dtype);
    const uint64_t nc = a.total_chunks;
    a.n_tensors = n;
    a.chunk_bytes = chunk_bytes;
    a.threshold = threshold;
    a.version = version;
    set_waits(a);
    if (!d_ws || !aligned(d_ws, 16)) return ZC_EINVAL;
    const uint64_t head = ctrl_bytes(n) + table_bytes(n);
    const uint64_t planes = hist_bytes(n, W, version) + ptab_bytes(n, W, version);
    const uint64_t fixed = head + planes + pad256(8 * nc);
    if (ws_bytes < fixed) return ZC_ECAPACITY;
    a.ws_ctrl = static_cast<uint8_t *>(d_ws);
    a.tensors = n > 1 ? reinterpret_cast<const TensorDesc *>(a.ws_ctrl + ctrl_bytes(n)) : nullptr;
    a.ws_hist = version == 2 ? reinterpret_cast<unsigned long long *>(a.ws_ctrl + head) : nullptr;
    a.ws_ptab = version == 2 ? a.ws_ctrl + head + hist_bytes(n, W, version) : nullptr;
    a.ws_status = reinterpret_cast<unsigned long long *>(a.ws_ctrl + head + planes);
    if (cudaMemsetAsync(d_ws, 0, fixed, s) != cudaSuccess) return ZC_ECUDA;
    if (n > 1) {
        const int st = upload_table(table, sizeof(TensorDesc) * n, const_cast<TensorDesc *>(a.tensors), s);
        if (st != ZC_OK) return st;
    }
    bool any_empty = false;
    uint64_t max_tc = 0;
    for (uint32_t t = 0; t < n; t++) {
        const uint32_t tc = (n == 1 ? a.one : table[t]).n_chunks;
        any_empty |= tc == 0;
        max_tc = tc > max_tc ? tc : max_tc;
    }
    if (any_empty) {
        const int st = launch_empty_blobs(a, s);
        if (st != ZC_OK) return st;
    }
    if (nc == 0) return ZC_OK;

    const uint64_t slot = slot_bytes(chunk_bytes, W, threshold, version);
    uint64_t wave = wave_chunks(nc, chunk_bytes, W);
    if (version == 2 && wave < max_tc) wave = max_tc;
    const uint64_t most_workers = max_workers(nc);
    uint64_t workers = most_workers;
    const uint64_t avail = ws_bytes - fixed;
    // room for a wave of w chunks with one coding warp per chunk (up to the
    // warps that can run at once)
    auto need = [&](uint64_t w) {
        return wave_layout(w, W, chunk_bytes).slots + std::min<uint64_t>(w, most_workers) * slot;
    };
    if (need(wave) > avail) {
        // A smaller workspace: the largest wave whose chunks all get a coding
        // warp (more waves, each as parallel as the full one), since every
        // chunk's rANS chain is a serial path that only more warps shorten.
        uint64_t lo = 0, hi = wave;  // need(lo) fits (0: nothing), need(hi) does not
        while (hi - lo > 1) {
            const uint64_t mid = lo + (hi - lo) / 2;
            if (need(mid) <= avail) lo = mid;
            else hi = mid;
        }
        if (version == 2 && lo < max_tc) {
            // v2 waves hold whole tensors: the largest tensor's statistics in
            // one wave, with the coding warps that still fit
            wave = max_tc;
            const uint64_t area = wave_layout(wave, W, chunk_bytes).slots;
            if (area + slot > avail) return ZC_ECAPACITY;
            workers = std::min<uint64_t>((avail - area) / slot, most_workers);
        } else {
            if (lo == 0) return ZC_ECAPACITY;
            wave = lo;
            workers = std::min<uint64_t>(lo, most_workers);
        }
    }
    const WaveLayout lay = wave_layout(wave, W, chunk_bytes);
    const uint64_t area0 = fixed;
    a.ws_info = a.ws_ctrl + area0 + lay.info;
    a.ws_ftab = a.ws_ctrl + area0 + lay.ftab;
    a.ws_cand = a.ws_ctrl + area0 + lay.cand;
    a.n_pad = n_pad(chunk_bytes, W);
    a.ws_slots = a.ws_ctrl + area0 + lay.slots;
    a.slot_bytes = slot;
    a.rec_stride = rec_stride(chunk_bytes, W, threshold, version);
    a.workers = uint32_t(workers < wave ? workers : wave);
    if (version != 2) {
        for (uint64_t w0 = 0; w0 < nc; w0 += wave) {
            a.wave_start = uint32_t(w0);
            a.wave_n = uint32_t(nc - w0 < wave ? nc - w0 : wave);
            const int st = launch_encode_wave(dtype, delta, a, s);
            if (st != ZC_OK) return st;
        }
        return ZC_OK;
    }
    // v2: a wave is a run of whole tensors, so that every tensor's plane
    // counts are complete before any of its chunks is coded
    uint32_t t = 0;
    while (t < n) {
        const uint32_t t0 = t;
        uint64_t chunks = 0;
        while (t < n) {
            const uint64_t tc = (n == 1 ? a.one : table[t]).n_chunks;
            if (t > t0 && chunks + tc > wave) break;
            chunks += tc;
            t++;
        }
        if (chunks == 0) continue;  // empty tensors only
        a.wave_start = (n == 1 ? a.one : table[t0]).chunk_base;
        a.wave_n = uint32_t(chunks);
        a.wave_t0 = t0;
        a.wave_t1 = t;
        a.workers = uint32_t(workers < chunks ? workers : chunks);
        const int st = launch_encode_wave(dtype, delta, a, s);
        if (st != ZC_OK) return st;
    }
    return ZC_OK;
}

// Blob format of a compression call's flags: 1 by default, 2 with shared
// plane tables, 3 with a word list per lane; 0 for flags that are invalid
// (unknown bits, or both formats at once). ZC_PACKED changes no format.
uint32_t version_of(uint32_t flags) {
    if (flags & ~(ZC_SHARED_TABLES | ZC_LANE_WORDS | ZC_PACKED)) return 0;
    if ((flags & ZC_SHARED_TABLES) && (flags & ZC_LANE_WORDS)) return 0;
    return (flags & ZC_SHARED_TABLES) ? 2u : (flags & ZC_LANE_WORDS) ? 3u : 1u;
}

int compress_impl(const void *d_src, const void *d_base, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                  uint32_t chunk_bytes, double threshold, void *d_blob, uint64_t blob_capacity,
                  uint64_t *d_blob_bytes, void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream,
                  uint32_t flags = 0) {
    const uint32_t version = version_of(flags);
    if (!d_status || version == 0) return ZC_EINVAL;
    EncodeArgs a{};
    const int st = make_tensor(d_src, d_base, nbytes, dtype, ndim, h_shape, chunk_bytes, threshold, d_blob,
                               blob_capacity, d_blob_bytes, version, a.one);
    if (st != ZC_OK) return st;
    if (resolve_tensor(a.one) != ZC_OK) return ZC_EINVAL;
    a.total_chunks = a.one.n_chunks;
    a.d_status = d_status;
    a.packed = (flags & ZC_PACKED) ? 1u : 0u;
    return run_compress(a, nullptr, 1, d_base != nullptr, dtype, chunk_bytes, threshold, version, d_ws, ws_bytes,
                        static_cast<cudaStream_t>(stream));
}

// Check one blob of a decompression call and describe it for the kernel
// (chunk_base is set by the caller).
int make_blob(const void *d_blob, const zc_info *info, const void *d_base, void *d_dst, uint64_t dst_capacity,
              BlobDesc &d) {
    if (!info || !d_blob) return ZC_EINVAL;
    const int W = word_bytes(info->dtype);
    if (!valid_params(info->nbytes, info->dtype, info->chunk_bytes, 0.95)) return ZC_EINVAL;
    if (chunks_of(info->nbytes, info->chunk_bytes) != info->n_chunks) return ZC_EINVAL;
    if (info->version < 1 || info->version > 3) return ZC_EINVAL;
    const uint64_t planes = info->version == 2 ? 512ull * W : 0;  // v2: the plane tables
    if (info->blob_bytes < ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * info->n_chunks + planes) return ZC_EINVAL;
    if (dst_capacity < info->nbytes || (info->nbytes && !d_dst)) return ZC_ECAPACITY;
    if (!aligned(d_blob, 16) || !aligned(d_dst, W)) return ZC_EINVAL;
    d = BlobDesc{};
    d.blob = static_cast<const uint8_t *>(d_blob);
    d.base = static_cast<const uint8_t *>(d_base);
    d.dst = static_cast<uint8_t *>(d_dst);
    d.blob_bytes = info->blob_bytes;
    d.nbytes = info->nbytes;
    d.n_chunks = info->n_chunks;
    return ZC_OK;
}

int decompress_impl(const void *d_blob, const zc_info *info, const void *d_base, void *d_dst, uint64_t dst_capacity,
                    uint32_t flags, int32_t *d_status, void *stream) {
    if (!d_status) return ZC_EINVAL;
    if (flags & ~(ZC_NO_VERIFY | ZC_PACKED)) return ZC_EINVAL;
    DecodeArgs a{};
    const int st = make_blob(d_blob, info, d_base, d_dst, dst_capacity, a.one);
    if (st != ZC_OK) return st;
    if (resolve_blob(a.one) != ZC_OK) return ZC_EINVAL;
    a.n_blobs = 1;
    a.total_chunks = info->n_chunks;
    a.chunk_bytes = info->chunk_bytes;
    a.flags = flags;
    a.d_status = d_status;
    a.version = info->version;
    set_waits(a);
    if (a.version == 2) {  // CTAs of a.pairs chunks
        a.pairs = decode_v2_pairs(a.total_chunks, (flags & ZC_PACKED) != 0);
        a.n_ctas = (a.total_chunks + a.pairs - 1) / a.pairs;
    }
    return launch_decode(info->dtype, d_base != nullptr, a, static_cast<cudaStream_t>(stream));
}

bool delta_dtype(int dtype) { return dtype == ZC_U8 || dtype == ZC_U16 || dtype == ZC_U32; }

} // namespace

extern "C" uint64_t zc_workspace_size_ex(uint64_t nbytes, int dtype, uint32_t chunk_bytes, uint32_t flags) {
    if (!valid_params(nbytes, dtype, chunk_bytes, 0.95) || version_of(flags) == 0) return 0;
    const uint64_t nc = chunks_of(nbytes, chunk_bytes);
    return ws_size(1, nc, word_bytes(dtype), chunk_bytes, version_of(flags), nc);
}

extern "C" uint64_t zc_workspace_size(uint64_t nbytes, int dtype, uint32_t chunk_bytes) {
    return zc_workspace_size_ex(nbytes, dtype, chunk_bytes, 0);
}

extern "C" uint64_t zc_workspace_size_batch(const uint64_t *nbytes, uint32_t n, int dtype, uint32_t chunk_bytes,
                                            uint32_t flags) {
    if (version_of(flags) == 0) return 0;
    if (n == 0) return kCtrlBytes;
    if (!nbytes) return 0;
    uint64_t nc = 0, max_tc = 0;
    for (uint32_t t = 0; t < n; t++) {
        if (!valid_params(nbytes[t], dtype, chunk_bytes, 0.95)) return 0;
        const uint64_t tc = chunks_of(nbytes[t], chunk_bytes);
        nc += tc;
        max_tc = tc > max_tc ? tc : max_tc;
    }
    if (nc > 0xFFFFFFFFull) return 0;
    return ws_size(n, nc, word_bytes(dtype), chunk_bytes, version_of(flags), max_tc);
}

extern "C" uint64_t zc_blob_size_ex(uint64_t nbytes, int dtype, uint32_t chunk_bytes, double threshold,
                                    uint32_t flags) {
    const uint32_t version = version_of(flags);
    if (version == 0 || !valid_params(nbytes, dtype, chunk_bytes, threshold)) return 0;
    const int W = word_bytes(dtype);
    const uint64_t nc = chunks_of(nbytes, chunk_bytes);
    uint64_t total = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * nc + (version == 2 ? 512ull * W : 0ull);
    if (nc == 0) return total;
    const uint64_t full = nc - 1, last = nbytes - full * chunk_bytes;
    auto worst = [&](uint64_t len) {
        uint64_t w = pad16(len);
        if (threshold > 1.0 && max_grouped(len, W, version) > w) w = max_grouped(len, W, version);
        return w;
    };
    return total + full * worst(chunk_bytes) + worst(last);
}

extern "C" int zc_compress_ex(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                              uint32_t chunk_bytes, double threshold, uint32_t flags,
                              void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                              void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream) {
    return compress_impl(d_src, nullptr, nbytes, dtype, ndim, h_shape, chunk_bytes, threshold, d_blob, blob_capacity,
                         d_blob_bytes, d_ws, ws_bytes, d_status, stream, flags);
}

extern "C" int zc_compress(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                           uint32_t chunk_bytes, double threshold,
                           void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                           void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream) {
    return compress_impl(d_src, nullptr, nbytes, dtype, ndim, h_shape, chunk_bytes, threshold, d_blob, blob_capacity,
                         d_blob_bytes, d_ws, ws_bytes, d_status, stream);
}

extern "C" int zc_compress_delta(const void *d_base, const void *d_new, uint64_t nbytes, int dtype, int ndim,
                                 const int64_t *h_shape, uint32_t chunk_bytes, double threshold,
                                 void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                                 void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream) {
    if (!delta_dtype(dtype)) return ZC_EINVAL;
    if (nbytes && (!d_base || !d_new || !aligned(d_base, 16) || !aligned(d_new, 16))) return ZC_EINVAL;
    return compress_impl(d_new, nbytes ? d_base : nullptr, nbytes, dtype, ndim, h_shape, chunk_bytes, threshold,
                         d_blob, blob_capacity, d_blob_bytes, d_ws, ws_bytes, d_status, stream);
}

extern "C" int zc_decompress(const void *d_blob, const zc_info *info, void *d_dst, uint64_t dst_capacity,
                             uint32_t flags, int32_t *d_status, void *stream) {
    return decompress_impl(d_blob, info, nullptr, d_dst, dst_capacity, flags, d_status, stream);
}

extern "C" int zc_decompress_delta(const void *d_blob, const zc_info *info, const void *d_base, void *d_dst,
                                   uint64_t dst_capacity, uint32_t flags, int32_t *d_status, void *stream) {
    if (!info || !delta_dtype(info->dtype)) return ZC_EINVAL;
    if (info->nbytes && (!d_base || !d_dst || !aligned(d_base, 16) || !aligned(d_dst, 16))) return ZC_EINVAL;
    return decompress_impl(d_blob, info, info->nbytes ? d_base : nullptr, d_dst, dst_capacity, flags, d_status,
                           stream);
}

extern "C" uint64_t zc_decompress_workspace_size_batch(uint32_t n) {
    return n > 1 ? pad256(sizeof(BlobDesc) * uint64_t(n)) : 0;
}

extern "C" int zc_compress_batch(uint32_t n, const void *const *d_srcs, const void *const *d_bases,
                                 const uint64_t *nbytes, int dtype, const int32_t *ndims, const int64_t *shapes,
                                 uint32_t chunk_bytes, double threshold, uint32_t flags, void *const *d_blobs,
                                 const uint64_t *blob_capacities, uint64_t *d_blob_bytes, void *d_ws,
                                 uint64_t ws_bytes, int32_t *d_status, void *stream) {
    const uint32_t version = version_of(flags);
    if (version == 0) return ZC_EINVAL;
    if (n == 0) return ZC_OK;
    if (!d_srcs || !nbytes || !ndims || !shapes || !d_blobs || !blob_capacities || !d_blob_bytes || !d_status)
        return ZC_EINVAL;
    if (d_bases && !delta_dtype(dtype)) return ZC_EINVAL;
    std::vector<TensorDesc> table(n);
    uint64_t nc = 0;
    for (uint32_t t = 0; t < n; t++) {
        const void *base = nullptr;
        if (d_bases && nbytes[t]) {
            base = d_bases[t];
            if (!base || !d_srcs[t] || !aligned(base, 16) || !aligned(d_srcs[t], 16)) return ZC_EINVAL;
        }
        const int st = make_tensor(d_srcs[t], base, nbytes[t], dtype, ndims[t], shapes + 8 * uint64_t(t),
                                   chunk_bytes, threshold, d_blobs[t], blob_capacities[t], d_blob_bytes + t,
                                   version, table[t]);
        if (st != ZC_OK) return st;
        table[t].chunk_base = uint32_t(nc);
        nc += table[t].n_chunks;
        if (nc > 0xFFFFFFFFull) return ZC_EINVAL;
    }
    for (auto &d : table)
        if (resolve_tensor(d) != ZC_OK) return ZC_EINVAL;
    EncodeArgs a{};
    if (n == 1) a.one = table[0];
    a.total_chunks = uint32_t(nc);
    a.d_status = d_status;
    a.packed = (flags & ZC_PACKED) ? 1u : 0u;
    return run_compress(a, table.data(), n, d_bases != nullptr, dtype, chunk_bytes, threshold, version, d_ws,
                        ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int zc_decompress_batch(uint32_t n, const void *const *d_blobs, const zc_info *infos,
                                   const void *const *d_bases, void *const *d_dsts, const uint64_t *dst_capacities,
                                   uint32_t flags, void *d_ws, uint64_t ws_bytes, int32_t *d_status, void *stream) {
    if (n == 0) return ZC_OK;
    if (!d_blobs || !infos || !d_dsts || !dst_capacities || !d_status) return ZC_EINVAL;
    if (flags & ~(ZC_NO_VERIFY | ZC_PACKED)) return ZC_EINVAL;
    const int dtype = infos[0].dtype;
    const uint32_t chunk_bytes = infos[0].chunk_bytes, version = infos[0].version;
    if (d_bases && !delta_dtype(dtype)) return ZC_EINVAL;
    if (n > 1 && (!d_ws || !aligned(d_ws, 16) || ws_bytes < zc_decompress_workspace_size_batch(n))) return ZC_EINVAL;
    std::vector<BlobDesc> table(n);
    uint64_t nc = 0;
    for (uint32_t t = 0; t < n; t++) {
        if (infos[t].dtype != dtype || infos[t].chunk_bytes != chunk_bytes || infos[t].version != version)
            return ZC_EINVAL;
        const void *base = nullptr;
        if (d_bases && infos[t].nbytes) {
            base = d_bases[t];
            if (!base || !d_dsts[t] || !aligned(base, 16) || !aligned(d_dsts[t], 16)) return ZC_EINVAL;
        }
        const int st = make_blob(d_blobs[t], &infos[t], base, d_dsts[t], dst_capacities[t], table[t]);
        if (st != ZC_OK) return st;
        table[t].chunk_base = uint32_t(nc);
        nc += table[t].n_chunks;
        if (nc > 0xFFFFFFFFull) return ZC_EINVAL;
    }
    for (auto &d : table)
        if (resolve_blob(d) != ZC_OK) return ZC_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DecodeArgs a{};
    a.version = version;
    if (version == 2) {  // CTAs of a.pairs chunks of one blob each
        a.pairs = decode_v2_pairs(nc, (flags & ZC_PACKED) != 0);
        uint64_t ctas = 0;
        for (auto &d : table) {
            d.cta_base = uint32_t(ctas);
            ctas += (d.n_chunks + a.pairs - 1) / a.pairs;
        }
        if (ctas > 0x7FFFFFFFull) return ZC_EINVAL;
        a.n_ctas = uint32_t(ctas);
    }
    if (n == 1) a.one = table[0];
    else {
        const int st = upload_table(table.data(), sizeof(BlobDesc) * n, d_ws, s);
        if (st != ZC_OK) return st;
        a.blobs = static_cast<const BlobDesc *>(d_ws);
    }
    a.n_blobs = n;
    a.total_chunks = uint32_t(nc);
    a.chunk_bytes = chunk_bytes;
    a.flags = flags;
    a.d_status = d_status;
    set_waits(a);
    return launch_decode(dtype, d_bases != nullptr, a, s);
}

extern "C" int zc_verify(const void *d_blob, const zc_info *info, int32_t *d_status, void *stream) {
    if (!d_status || !info || !d_blob) return ZC_EINVAL;
    const int W = word_bytes(info->dtype);
    if (!valid_params(info->nbytes, info->dtype, info->chunk_bytes, 0.95)) return ZC_EINVAL;
    if (chunks_of(info->nbytes, info->chunk_bytes) != info->n_chunks) return ZC_EINVAL;
    if (info->version < 1 || info->version > 3) return ZC_EINVAL;
    const uint64_t table_end = ZC_HEADER_BYTES + uint64_t(ZC_ENTRY_BYTES) * info->n_chunks +
                               (info->version == 2 ? 512ull * W : 0ull);
    if (info->blob_bytes < table_end || !aligned(d_blob, 16)) return ZC_EINVAL;
    const void *kb = nullptr;
    if (kernel_address(d_blob, &kb) != ZC_OK) return ZC_EINVAL;
    VerifyArgs a{};
    a.blob = static_cast<const uint8_t *>(kb);
    a.blob_bytes = info->blob_bytes;
    a.table_end = table_end;
    a.n_chunks = info->n_chunks;
    a.d_status = d_status;
    return launch_verify(a, static_cast<cudaStream_t>(stream));
}

extern "C" int zc_crc32(const void *d_data, uint64_t nbytes, uint64_t piece_bytes, uint32_t *d_out, void *stream) {
    if (!d_out || (nbytes && !d_data)) return ZC_EINVAL;
    const uint64_t piece = piece_bytes ? piece_bytes : (nbytes ? nbytes : 1);
    const uint64_t pieces = piece_bytes ? (nbytes + piece - 1) / piece : 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pieces == 0) return ZC_OK;
    if (cudaMemsetAsync(d_out, 0, pieces * 4, s) != cudaSuccess) return ZC_ECUDA;
    if (nbytes == 0) return ZC_OK;
    CrcArgs a{};
    a.data = static_cast<const uint8_t *>(d_data);
    a.nbytes = nbytes;
    a.piece = piece;
    a.unit = kCrcUnit;
    a.units_per_piece = (piece + kCrcUnit - 1) / kCrcUnit;
    a.n_units = pieces * a.units_per_piece;
    a.out = d_out;
    return launch_crc(a, s);
}
