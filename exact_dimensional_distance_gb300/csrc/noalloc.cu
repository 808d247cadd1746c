// An exclusive prefix sum that allocates nothing: hiss_exclusive_scan_noalloc.
//
// Some callers cannot allocate device memory: a plugin running inside a host
// framework that owns all device memory through its own pool, or a
// latency-critical loop that cannot afford cudaMalloc's implicit device-wide
// synchronisation.  This entry point runs the same three scan kernels as
// hiss_exclusive_scan, but keeps their scratch (one int64 partial sum per
// 2048-element chunk, plus a total) in the file-scope device array below
// instead of a buffer owned by a context.
//
// The array costs kNoallocScratchElems * 8 bytes (256 KiB) on every device
// that loads the library, for the life of the process.  Calls share it, so two
// calls whose kernels overlap on the GPU (different streams, or different host
// threads) race on it and must be ordered by the caller.  Every scratch entry
// a call reads is written earlier in the same call, so nothing has to be
// cleared between calls.
#include <mutex>

#include "hiss_internal.cuh"

namespace {

constexpr int64_t kNoallocMaxN = int64_t(1) << 26;            // 67,108,864 elements
constexpr int64_t kNoallocScratchElems = (int64_t(1) << 15) + 64;  // >= scan_tmp_elems(kNoallocMaxN)

static __device__ __align__(256) int64_t g_scan_scratch[kNoallocScratchElems];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int64_t *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device.  In host code the
// symbol name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.  cudaDeviceReset destroys
// the module that holds the array; the cached address is then stale, so a
// process that resets a device must not call this entry point on it again.
cudaError_t scratch_address(int64_t **out)
{
    int dev = 0;
    HISS_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        HISS_TRY(cudaGetSymbolAddress(&p, g_scan_scratch));
        g_scratch_addr[dev] = static_cast<int64_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int hiss_exclusive_scan_noalloc(void *cuda_stream, const int64_t *d_in, int64_t *d_out, int64_t n)
{
    if (n < 0 || n > kNoallocMaxN || !d_out || (n > 0 && !d_in)) return HISS_E_ARG;
    if (hiss::scan_tmp_elems(n + 1) > kNoallocScratchElems) return HISS_E_ARG;
    // A pending error from the caller's own earlier work is left in place for
    // the caller to read (cudaGetLastError would clear it); this call does not
    // run on top of it, since its own launch check could not tell the two apart.
    if (cudaPeekAtLastError() != cudaSuccess) return HISS_E_CUDA;
    int64_t *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return HISS_E_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int64_t launches = 0;
    if (hiss::scan_i64(d_in, d_out, n, scratch, s, &launches) != cudaSuccess) return HISS_E_CUDA;
    return HISS_OK;
}
