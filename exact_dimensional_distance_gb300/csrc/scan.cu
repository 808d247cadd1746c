// Device-wide exclusive prefix sums (reduce, then scan of block totals, then
// scan of each chunk).  Used for the count pass and the CSR row offsets of
// the result (RT-HiSS Section IV-D builds its prefix sums on the host; here
// they stay on the device).
#include "hiss_internal.cuh"

namespace hiss {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanChunk = kScanThreads * kScanItems;

__device__ __forceinline__ int64_t warp_incl_scan(int64_t v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive scan of one value per thread across the block; returns the
// exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int64_t block_excl_scan(int64_t v, int64_t *total)
{
    __shared__ int64_t warp_sum[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t incl = warp_incl_scan(v);
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < kScanThreads / 32 ? warp_sum[lane] : 0;
        int64_t wi = warp_incl_scan(w);
        if (lane < kScanThreads / 32) warp_sum[lane] = wi - w;
        if (lane == kScanThreads / 32 - 1) *total = wi;
    }
    __syncthreads();
    int64_t r = incl - v + warp_sum[warp];
    __syncthreads();
    return r;
}

template <typename Tin>
__global__ void __launch_bounds__(kScanThreads) k_block_sums(const Tin *in, int64_t n, int64_t *sums)
{
    const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
    int64_t v = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i)
        if (base + i < n) v += (int64_t)in[base + i];
    __shared__ int64_t tot;
    block_excl_scan(v, &tot);
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_sums(int64_t *sums, int64_t nb)
{
    __shared__ int64_t tot;
    int64_t carry = 0;
    for (int64_t b0 = 0; b0 < nb; b0 += kScanThreads) {
        const int64_t i = b0 + threadIdx.x;
        int64_t v = i < nb ? sums[i] : 0;
        int64_t e = block_excl_scan(v, &tot);
        if (i < nb) sums[i] = carry + e;
        carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) sums[nb] = carry;
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kScanThreads) k_scan_chunks(const Tin *in, Tout *out, int64_t n,
                                                              const int64_t *sums, int64_t nb)
{
    const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
    int64_t v[kScanItems];
    int64_t s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        v[i] = base + i < n ? (int64_t)in[base + i] : 0;
        s += v[i];
    }
    __shared__ int64_t tot;
    int64_t e = block_excl_scan(s, &tot) + sums[blockIdx.x];
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        if (base + i < n) out[base + i] = (Tout)e;
        e += v[i];
    }
    if (blockIdx.x == nb - 1 && threadIdx.x == 0) out[n] = (Tout)sums[nb];
}

template <typename Tin, typename Tout>
cudaError_t scan_impl(const Tin *in, Tout *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches)
{
    if (n <= 0) {
        HISS_TRY(cudaMemsetAsync(out, 0, sizeof(Tout), s));
        return cudaSuccess;
    }
    const int64_t nb = (n + kScanChunk - 1) / kScanChunk;
    k_block_sums<Tin><<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, tmp);
    k_scan_sums<<<1, kScanThreads, 0, s>>>(tmp, nb);
    k_scan_chunks<Tin, Tout><<<(unsigned)nb, kScanThreads, 0, s>>>(in, out, n, tmp, nb);
    *launches += 3;
    return cudaGetLastError();
}

}  // namespace

int64_t scan_tmp_elems(int64_t n) { return (n + kScanChunk - 1) / kScanChunk + 1; }

cudaError_t scan_i64(const int64_t *in, int64_t *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches)
{
    return scan_impl<int64_t, int64_t>(in, out, n, tmp, s, launches);
}

cudaError_t scan_i32_to_i64(const int32_t *in, int64_t *out, int64_t n, int64_t *tmp, cudaStream_t s,
                            int64_t *launches)
{
    return scan_impl<int32_t, int64_t>(in, out, n, tmp, s, launches);
}

cudaError_t scan_i32(const int32_t *in, int32_t *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches)
{
    return scan_impl<int32_t, int32_t>(in, out, n, tmp, s, launches);
}

}  // namespace hiss
