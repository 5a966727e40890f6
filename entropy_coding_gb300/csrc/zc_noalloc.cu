// zc_noalloc.cu — zc_compress_noalloc: compression for callers that must
// not allocate device memory.
//
// Some callers cannot allocate: for example a service whose device memory is
// entirely owned by another allocator (a framework's caching pool reserved at
// start-up), or a runtime that forbids new device allocations after
// initialisation so that memory use and latency stay predictable. Such a
// caller cannot provide the workspace zc_compress asks for. This entry point
// uses a fixed scratch area in a file-scope device array instead, and runs
// exactly the same compression as zc_compress on it.
//
// The array is kStaticScratchBytes (64 MiB) in every device's memory once the
// library's code for this file is loaded on that device, and stays there
// until the process exits. Under CUDA's lazy module loading (the default) the
// code is loaded, and the 64 MiB committed, by the first call on a device:
// a caller whose memory pool reserves all free memory at start-up should make
// that first call before the pool does. All calls share the array: calls
// that overlap on the GPU (on different streams, or from different host
// threads without ordering) race on it and corrupt each other's results;
// callers must order them. The first call on each device looks up the
// array's device address (once per device, with that device current); that
// first call should therefore be made before any stream capture begins. The
// address is kept for the life of the process: after cudaDeviceReset the
// caller must not use this entry point on that device again.
//
// With 64 MiB the workspace planner runs waves of about 250 chunks (FP32,
// 128 KiB chunks), each with a coding warp per chunk, so a tensor larger than
// a wave is compressed in several waves on the same stream.
#include <mutex>

#include "zc_kernels.cuh"

namespace {

constexpr uint64_t kStaticScratchBytes = 64ull << 20;
constexpr uint64_t kStaticMaxChunks = 1ull << 20;  // chunk status words use 8 MiB of the array
constexpr int kMaxDevices = 64;

// Scratch shared by every zc_compress_noalloc call on a device: the chunk
// ticket and status words of the offset scan, and per-CTA staging for coded
// records. zc_compress zeroes what must start at zero on every call.
static __device__ __align__(256) uint8_t zc_static_scratch[kStaticScratchBytes];

std::mutex g_lock;
void *g_scratch[kMaxDevices] = {};

// Device address of the array on the current device (looked up once).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZC_ECUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, zc_static_scratch) != cudaSuccess || !p) return ZC_ECUDA;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return ZC_OK;
}

} // namespace

extern "C" int zc_compress_noalloc(const void *d_src, uint64_t nbytes, int dtype, int ndim, const int64_t *h_shape,
                                   uint32_t chunk_bytes, double threshold,
                                   void *d_blob, uint64_t blob_capacity, uint64_t *d_blob_bytes,
                                   int32_t *d_status, void *stream) {
    // the parameters are checked first, so that an invalid call is reported
    // as such whatever its size
    if (zc_workspace_size(nbytes, dtype, chunk_bytes) == 0) return ZC_EINVAL;
    const uint64_t n_chunks = (nbytes + chunk_bytes - 1) / chunk_bytes;
    if (n_chunks > kStaticMaxChunks) return ZC_ECAPACITY;  // tensor too large for the fixed scratch
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != ZC_OK) return st;
    return zc_compress(d_src, nbytes, dtype, ndim, h_shape, chunk_bytes, threshold, d_blob, blob_capacity,
                       d_blob_bytes, scratch, kStaticScratchBytes, d_status, stream);
}
