// Onesweep LSD radix sort of (uint64 key, uint32 value) pairs.
//
// One kernel counts the digit histograms of every pass at once; each 8-bit
// digit pass is then a single kernel whose tiles find their output offsets
// by decoupled look-back over the tiles before them (tile ids are taken from
// an atomic ticket in launch order, so every tile a tile waits on is already
// running).  The sort is stable: inside a tile, keys are ranked warp by warp
// and item by item in index order.
//
// The look-back wait is bounded: after kSpinLimit polls a tile records
// kFlagSortTimeout and carries on, so a stalled predecessor can never hang
// the GPU; the host turns the flag into an error.
#include "hiss_internal.cuh"

namespace hiss {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;  // 4096 keys
constexpr int kBins = 256;
constexpr int kMaxPasses = 8;
constexpr uint32_t kValMask = (1u << 30) - 1;
constexpr uint32_t kAggregate = 1u, kInclusive = 2u;
constexpr uint32_t kSpinLimit = 1u << 22;

struct SortTmp {
    uint32_t *hist;     // [kMaxPasses][kBins]
    uint32_t *offsets;  // [kMaxPasses][kBins]
    uint32_t *counter;  // [kMaxPasses]
    uint32_t *status;   // [kMaxPasses][tiles][kBins]
};

int64_t num_tiles(int64_t n) { return (n + kSortTile - 1) / kSortTile; }

SortTmp carve(void *tmp, int64_t n)
{
    SortTmp t;
    uint32_t *p = static_cast<uint32_t *>(tmp);
    t.hist = p;
    t.offsets = p + kMaxPasses * kBins;
    t.counter = p + 2 * kMaxPasses * kBins;
    t.status = p + 2 * kMaxPasses * kBins + 64;
    (void)n;
    return t;
}

__device__ __forceinline__ uint32_t digit_of(uint64_t key, int shift, uint32_t dmask)
{
    return (uint32_t)(key >> shift) & dmask;
}

__global__ void __launch_bounds__(kSortThreads) k_sort_hist(const uint64_t *keys, int64_t n, int npass,
                                                            int key_bits, uint32_t *hist)
{
    __shared__ uint32_t sh[kMaxPasses][kBins];
    for (int i = threadIdx.x; i < kMaxPasses * kBins; i += kSortThreads) (&sh[0][0])[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * kSortThreads;
    for (int64_t i = (int64_t)blockIdx.x * kSortThreads + threadIdx.x; i < n; i += stride) {
        const uint64_t k = keys[i];
        for (int p = 0; p < npass; ++p) {
            const int bits = min(8, key_bits - 8 * p);
            atomicAdd(&sh[p][digit_of(k, 8 * p, (1u << bits) - 1u)], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < npass * kBins; i += kSortThreads) {
        const uint32_t c = (&sh[0][0])[i];
        if (c) atomicAdd(&hist[i], c);
    }
}

__global__ void __launch_bounds__(kBins) k_scan_hist(const uint32_t *hist, uint32_t *offsets)
{
    __shared__ uint32_t s[kBins];
    const int p = blockIdx.x, t = threadIdx.x;
    s[t] = hist[p * kBins + t];
    __syncthreads();
    for (int o = 1; o < kBins; o <<= 1) {
        uint32_t v = t >= o ? s[t - o] : 0u;
        __syncthreads();
        s[t] += v;
        __syncthreads();
    }
    offsets[p * kBins + t] = s[t] - hist[p * kBins + t];
}

__global__ void __launch_bounds__(kSortThreads) k_onesweep(const uint64_t *__restrict__ kin,
                                                           const uint32_t *__restrict__ vin,
                                                           uint64_t *__restrict__ kout, uint32_t *__restrict__ vout,
                                                           int64_t n, int shift, uint32_t dmask,
                                                           const uint32_t *offsets, uint32_t *counter,
                                                           uint32_t *status, int *flags)
{
    __shared__ uint32_t whist[kSortWarps][kBins];
    __shared__ uint32_t tile_base[kBins];
    __shared__ uint32_t s_tile;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_tile = atomicAdd(counter, 1u);
    for (int i = threadIdx.x; i < kSortWarps * kBins; i += kSortThreads) (&whist[0][0])[i] = 0;
    __syncthreads();
    const int64_t tile = s_tile;
    const int64_t base = tile * kSortTile + (int64_t)warp * (32 * kSortItems);

    uint64_t key[kSortItems];
    uint32_t val[kSortItems];
    uint32_t rank[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
        const int64_t idx = base + i * 32 + lane;
        if (idx < n) {
            key[i] = kin[idx];
            val[i] = vin[idx];
        }
    }
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
        const int64_t idx = base + i * 32 + lane;
        const bool valid = idx < n;
        const uint32_t m = __ballot_sync(0xffffffffu, valid);
        rank[i] = 0;
        if (valid) {
            const uint32_t d = digit_of(key[i], shift, dmask);
            const uint32_t peers = __match_any_sync(m, d);
            const int leader = __ffs(peers) - 1;
            uint32_t old = 0;
            if (lane == leader) {
                old = whist[warp][d];
                whist[warp][d] = old + __popc(peers);
            }
            old = __shfl_sync(m, old, leader);
            rank[i] = old + __popc(peers & lt_mask);
        }
        __syncwarp();
    }
    __syncthreads();

    // Per digit: exclusive prefix over warps, the tile's count, look-back.
    {
        const int d = threadIdx.x;
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) {
            const uint32_t c = whist[w][d];
            whist[w][d] = run;
            run += c;
        }
        uint32_t *st = status + (size_t)tile * kBins + d;
        uint32_t excl = 0;
        if (tile == 0) {
            atomicExch(st, (kInclusive << 30) | run);
        } else {
            atomicExch(st, (kAggregate << 30) | run);
            int64_t t = tile - 1;
            uint32_t spins = 0;
            while (true) {
                const uint32_t s = *(volatile uint32_t *)(status + (size_t)t * kBins + d);
                const uint32_t f = s >> 30;
                if (f == 0u) {
                    if (++spins > kSpinLimit) {
                        atomicExch(&flags[kFlagSortTimeout], 1);
                        break;
                    }
                    __nanosleep(64);
                    continue;
                }
                excl += s & kValMask;
                if (f == kInclusive || t == 0) break;
                --t;
            }
            atomicExch(st, (kInclusive << 30) | (excl + run));
        }
        tile_base[d] = offsets[d] + excl;
    }
    __syncthreads();

#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
        const int64_t idx = base + i * 32 + lane;
        if (idx < n) {
            const uint32_t d = digit_of(key[i], shift, dmask);
            const uint32_t pos = tile_base[d] + whist[warp][d] + rank[i];
            kout[pos] = key[i];
            vout[pos] = val[i];
        }
    }
}

}  // namespace

size_t sort_tmp_bytes(int64_t n)
{
    const int64_t tiles = num_tiles(n) > 0 ? num_tiles(n) : 1;
    return sizeof(uint32_t) * (size_t)(2 * kMaxPasses * kBins + 64 + (int64_t)kMaxPasses * tiles * kBins);
}

cudaError_t sort_pairs(uint64_t *keys, uint32_t *vals, uint64_t *keys_alt, uint32_t *vals_alt, int64_t n,
                       int key_bits, void *tmp, int *flags, cudaStream_t s, int64_t *launches, int *in_alt)
{
    *in_alt = 0;
    if (n <= 1 || key_bits <= 0) return cudaSuccess;
    if (key_bits > 64) key_bits = 64;
    const int npass = (key_bits + 7) / 8;
    const int64_t tiles = num_tiles(n);
    SortTmp t = carve(tmp, n);
    HISS_TRY(cudaMemsetAsync(tmp, 0, sort_tmp_bytes(n), s));
    const int hist_blocks = (int)(tiles < 4 * 152 ? tiles : 4 * 152);
    k_sort_hist<<<hist_blocks, kSortThreads, 0, s>>>(keys, n, npass, key_bits, t.hist);
    k_scan_hist<<<npass, kBins, 0, s>>>(t.hist, t.offsets);
    *launches += 2;
    uint64_t *ki = keys, *ko = keys_alt;
    uint32_t *vi = vals, *vo = vals_alt;
    for (int p = 0; p < npass; ++p) {
        const int bits = key_bits - 8 * p < 8 ? key_bits - 8 * p : 8;
        k_onesweep<<<(unsigned)tiles, kSortThreads, 0, s>>>(ki, vi, ko, vo, n, 8 * p, (1u << bits) - 1u,
                                                          t.offsets + p * kBins, t.counter + p,
                                                          t.status + (size_t)p * tiles * kBins, flags);
        ++*launches;
        uint64_t *tk = ki; ki = ko; ko = tk;
        uint32_t *tv = vi; vi = vo; vo = tv;
    }
    *in_alt = npass & 1;
    return cudaGetLastError();
}

}  // namespace hiss
