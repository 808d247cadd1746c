// Index construction: variance order of the dimensions (RT-HiSS Section
// IV-A), the three-dimensional grid with Morton-ordered points (grid indexing
// of Section II-B1, Morton order of Section IV-C), the 27-cell stencil of each
// cell, the count pass (first intersection test, Section IV-D), and the
// query tiles and batches the refinement consumes.
#include "hiss_internal.cuh"

namespace hiss {
namespace {

constexpr int kT = 256;

inline unsigned blocks_for(int64_t work, int per_block = kT)
{
    int64_t b = (work + per_block - 1) / per_block;
    return (unsigned)(b < 1 ? 1 : b);
}

// ---- per-dimension statistics -----------------------------------------------
// Each block covers a contiguous range of rows.  With g = kT / d row groups,
// thread (group, k) reads column k of every g-th row, so a warp reads whole
// consecutive rows.  Sums are shifted by the first row's value (x0) to keep
// the fp64 variance accurate when the mean is far from zero.
__global__ void __launch_bounds__(kT) k_stats_partial(const float *__restrict__ x, int64_t n, int d,
                                                      int64_t rows_per_block, double *partial, int *nonfinite)
{
    __shared__ double s_sum[kT], s_sq[kT];
    __shared__ float s_mn[kT], s_mx[kT];
    const int groups = kT / d;
    const int g = threadIdx.x / d, k = threadIdx.x % d;
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_block;
    const int64_t r1 = min(n, r0 + rows_per_block);
    double sum = 0.0, sq = 0.0;
    float mn = INFINITY, mx = -INFINITY;
    int bad = 0;
    if (g < groups) {
        const double x0 = (double)x[k];
        for (int64_t r = r0 + g; r < r1; r += groups) {
            const float v = x[r * d + k];
            if (!isfinite(v)) { ++bad; continue; }
            const double t = (double)v - x0;
            sum += t;
            sq += t * t;
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
    }
    if (bad) atomicAdd(nonfinite, bad);
    s_sum[threadIdx.x] = sum;
    s_sq[threadIdx.x] = sq;
    s_mn[threadIdx.x] = mn;
    s_mx[threadIdx.x] = mx;
    __syncthreads();
    if (threadIdx.x < d) {
        double a = 0.0, b = 0.0;
        float lo = INFINITY, hi = -INFINITY;
        for (int gg = 0; gg < groups; ++gg) {
            const int t = gg * d + threadIdx.x;
            a += s_sum[t];
            b += s_sq[t];
            lo = fminf(lo, s_mn[t]);
            hi = fmaxf(hi, s_mx[t]);
        }
        double *p = partial + ((size_t)blockIdx.x * d + threadIdx.x) * 4;
        p[0] = a;
        p[1] = b;
        p[2] = (double)lo;
        p[3] = (double)hi;
    }
}

// One block per dimension: the block partials are reduced in a fixed order
// (strided sums, then a tree), so the result does not depend on timing.
__global__ void __launch_bounds__(kT) k_stats_final(const float *x, int64_t n, int d, const double *partial,
                                                    int64_t nblocks, double *out)
{
    __shared__ double s_a[kT], s_b[kT], s_lo[kT], s_hi[kT];
    const int k = blockIdx.x;
    double a = 0.0, b = 0.0, lo = INFINITY, hi = -INFINITY;
    for (int64_t i = threadIdx.x; i < nblocks; i += kT) {
        const double *p = partial + ((size_t)i * d + k) * 4;
        a += p[0];
        b += p[1];
        lo = fmin(lo, p[2]);
        hi = fmax(hi, p[3]);
    }
    s_a[threadIdx.x] = a;
    s_b[threadIdx.x] = b;
    s_lo[threadIdx.x] = lo;
    s_hi[threadIdx.x] = hi;
    __syncthreads();
    for (int o = kT / 2; o > 0; o >>= 1) {
        if (threadIdx.x < o) {
            s_a[threadIdx.x] += s_a[threadIdx.x + o];
            s_b[threadIdx.x] += s_b[threadIdx.x + o];
            s_lo[threadIdx.x] = fmin(s_lo[threadIdx.x], s_lo[threadIdx.x + o]);
            s_hi[threadIdx.x] = fmax(s_hi[threadIdx.x], s_hi[threadIdx.x + o]);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double mean_shift = s_a[0] / (double)n;
        double var = s_b[0] / (double)n - mean_shift * mean_shift;
        if (var < 0.0) var = 0.0;
        out[0 * d + k] = s_lo[0];
        out[1 * d + k] = s_hi[0];
        out[2 * d + k] = (double)x[k] + mean_shift;
        out[3 * d + k] = var;
    }
}

__global__ void k_permute_pad(const float *__restrict__ x, int64_t n, int d, int d4, const int32_t *__restrict__ perm,
                              float *__restrict__ xv)
{
    const int64_t idx = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (idx >= n * d4) return;
    const int64_t i = idx / d4;
    const int j = (int)(idx - i * d4);
    xv[idx] = j < d ? x[i * d + perm[j]] : 0.0f;
}

// ---- grid keys ------------------------------------------------------------------
// Spread the low 21 bits of v so that bit b lands on bit 3b.
__device__ __forceinline__ uint64_t spread3(uint64_t v)
{
    v &= 0x1fffffull;
    v = (v | (v << 32)) & 0x001f00000000ffffull;
    v = (v | (v << 16)) & 0x001f0000ff0000ffull;
    v = (v | (v << 8)) & 0x100f00f00f00f00full;
    v = (v | (v << 4)) & 0x10c30c30c30c30c3ull;
    v = (v | (v << 2)) & 0x1249249249249249ull;
    return v;
}

// Inverse of spread3: gather bits 3b into bit b.
__device__ __forceinline__ uint64_t compact3(uint64_t v)
{
    v &= 0x1249249249249249ull;
    v = (v ^ (v >> 2)) & 0x10c30c30c30c30c3ull;
    v = (v ^ (v >> 4)) & 0x100f00f00f00f00full;
    v = (v ^ (v >> 8)) & 0x001f0000ff0000ffull;
    v = (v ^ (v >> 16)) & 0x001f00000000ffffull;
    v = (v ^ (v >> 32)) & 0x1fffffull;
    return v;
}

__global__ void k_cell_keys(const float *__restrict__ xv, int64_t n, int d4, GridParams gp,
                            uint64_t *__restrict__ keys, uint32_t *__restrict__ vals)
{
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= n) return;
    const double scale = (double)(1u << gp.sub_bits);
    uint64_t key = 0;
    for (int k = 0; k < gp.ndim; ++k) {
        // fp64 throughout so cell boundaries match an fp64 reading exactly
        const double u = ((double)xv[i * d4 + k] - gp.origin[k]) / gp.w;
        const uint64_t f = (uint64_t)floor(u * scale);
        key |= spread3(f) << k;
    }
    keys[i] = key;
    vals[i] = (uint32_t)i;
}

__global__ void k_gather_rows(const float4 *__restrict__ xv, const uint32_t *__restrict__ order, int64_t n, int c4,
                              float4 *__restrict__ xs, int32_t *__restrict__ ids)
{
    const int64_t idx = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (idx >= n * c4) return;
    const int64_t r = idx / c4;
    const int c = (int)(idx - r * c4);
    const uint32_t src = order[r];
    xs[idx] = xv[(int64_t)src * c4 + c];
    if (c == 0) ids[r] = (int32_t)src;
}

// Box of each aligned group of 32 index rows over the first three dimensions
// (the grid's index dimensions; zero padding where d < 3): gbox[2 g] = the
// minima, gbox[2 g + 1] = the maxima (fourth component 0).  One warp per group.
__global__ void k_group_boxes(const float *__restrict__ xs, int64_t n, int d4, float4 *__restrict__ gbox)
{
    const int64_t g = ((int64_t)blockIdx.x * kT + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (g >= (n + 31) >> 5) return;  // whole warps leave together
    const int64_t r = g * 32 + lane;
    float lo0 = INFINITY, lo1 = INFINITY, lo2 = INFINITY, hi0 = -INFINITY, hi1 = -INFINITY, hi2 = -INFINITY;
    if (r < n) {
        const float4 f = *reinterpret_cast<const float4 *>(xs + r * d4);
        lo0 = hi0 = f.x;
        lo1 = hi1 = f.y;
        lo2 = hi2 = f.z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo0 = fminf(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
        lo1 = fminf(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
        lo2 = fminf(lo2, __shfl_xor_sync(0xffffffffu, lo2, o));
        hi0 = fmaxf(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
        hi1 = fmaxf(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
        hi2 = fmaxf(hi2, __shfl_xor_sync(0xffffffffu, hi2, o));
    }
    if (lane == 0) {
        gbox[2 * g] = make_float4(lo0, lo1, lo2, 0.f);
        gbox[2 * g + 1] = make_float4(hi0, hi1, hi2, 0.f);
    }
}

__global__ void k_cell_flags(const uint64_t *__restrict__ keys, int64_t n, int shift, int32_t *__restrict__ flag)
{
    const int64_t r = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (r >= n) return;
    flag[r] = (r == 0 || (keys[r] >> shift) != (keys[r - 1] >> shift)) ? 1 : 0;
}

__global__ void k_cell_starts(const uint64_t *__restrict__ keys, const int32_t *__restrict__ e, int64_t n, int shift,
                              int32_t *__restrict__ cell_start, uint64_t *__restrict__ cell_key,
                              int32_t *__restrict__ cell_of_row)
{
    const int64_t r = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (r >= n) return;
    const int32_t c = e[r + 1] - 1;
    cell_of_row[r] = c;
    if (e[r] != e[r + 1]) {  // first row of a cell
        cell_start[c] = (int32_t)r;
        cell_key[c] = keys[r] >> shift;
    }
    if (r == 0) cell_start[e[n]] = (int32_t)n;
}

// Stencil of each cell: the existing cells among the 27 around it, in the
// order dz, dy, dx (dz outermost), found by binary search over the sorted
// cell keys.  bound = points in those cells (B_cell); work = |cell| * B_cell.
__global__ void k_stencil(const uint64_t *__restrict__ cell_key, const int32_t *__restrict__ cell_start, int64_t C,
                          int32_t *__restrict__ nbr, int32_t *__restrict__ nbr_cnt, int64_t *__restrict__ bound,
                          uint64_t *__restrict__ work_key, uint32_t *__restrict__ cell_idx,
                          int64_t *__restrict__ work)
{
    const int64_t c = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (c >= C) return;
    const uint64_t key = cell_key[c];
    const int64_t cx = (int64_t)compact3(key), cy = (int64_t)compact3(key >> 1), cz = (int64_t)compact3(key >> 2);
    const int64_t lim = 1 << 21;
    int cnt = 0;
    int64_t b = 0;
    for (int dz = -1; dz <= 1; ++dz)
        for (int dy = -1; dy <= 1; ++dy)
            for (int dx = -1; dx <= 1; ++dx) {
                const int64_t a0 = cx + dx, a1 = cy + dy, a2 = cz + dz;
                if (a0 < 0 || a1 < 0 || a2 < 0 || a0 >= lim || a1 >= lim || a2 >= lim) continue;
                const uint64_t nk = spread3((uint64_t)a0) | (spread3((uint64_t)a1) << 1) | (spread3((uint64_t)a2) << 2);
                int64_t lo = 0, hi = C;  // first index with cell_key >= nk
                while (lo < hi) {
                    const int64_t mid = (lo + hi) >> 1;
                    if (cell_key[mid] < nk) lo = mid + 1; else hi = mid;
                }
                if (lo < C && cell_key[lo] == nk) {
                    nbr[c * kStencil + cnt++] = (int32_t)lo;
                    b += cell_start[lo + 1] - cell_start[lo];
                }
            }
    nbr_cnt[c] = cnt;
    bound[c] = b;
    const int64_t w = (int64_t)(cell_start[c + 1] - cell_start[c]) * b;
    work[c] = w;
    work_key[c] = ~(uint64_t)w;  // ascending sort of ~w = descending work
    cell_idx[c] = (uint32_t)c;
}

// Semi-join: key each query into the data's grid.  Cell coordinates are
// signed; a query more than one cell outside the grid on some index dimension
// has no candidate and gets the key ~0 (it sorts last).  Otherwise the key is
// the Morton key of the coordinates shifted by +1 (so -1 maps to 0).
__global__ void k_query_keys(const float *__restrict__ xv, int64_t n, int d4, GridParams gp, int64_t cellmax,
                             uint64_t *__restrict__ keys, uint32_t *__restrict__ vals)
{
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= n) return;
    uint64_t key = 0;
    bool outside = false;
    for (int k = 0; k < 3; ++k) {
        int64_t c = 0;
        if (k < gp.ndim) {
            const double u = ((double)xv[i * d4 + k] - gp.origin[k]) / gp.w;
            const double f = floor(u);
            if (f < -1.0 || f > (double)(cellmax + 1)) outside = true;
            else c = (int64_t)f;
        }
        key |= spread3((uint64_t)(c + 1)) << k;
    }
    keys[i] = outside ? ~0ull : key;
    vals[i] = (uint32_t)i;
}

// Stencil of each query cell in the data's grid (cells of D around it, order
// dz, dy, dx), its candidate count and work, as k_stencil does for D's cells.
__global__ void k_query_stencil(const uint64_t *__restrict__ qcell_key, const int32_t *__restrict__ qcell_start,
                                int64_t Cq, const uint64_t *__restrict__ cell_key,
                                const int32_t *__restrict__ cell_start, int64_t C, int32_t *__restrict__ nbr,
                                int32_t *__restrict__ nbr_cnt, int64_t *__restrict__ bound,
                                uint64_t *__restrict__ work_key, uint32_t *__restrict__ cell_idx,
                                int64_t *__restrict__ work)
{
    const int64_t c = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (c >= Cq) return;
    const uint64_t key = qcell_key[c];
    int cnt = 0;
    int64_t b = 0;
    if (key != ~0ull) {
        const int64_t cx = (int64_t)compact3(key) - 1, cy = (int64_t)compact3(key >> 1) - 1,
                      cz = (int64_t)compact3(key >> 2) - 1;
        const int64_t lim = 1 << 21;
        for (int dz = -1; dz <= 1; ++dz)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dx = -1; dx <= 1; ++dx) {
                    const int64_t a0 = cx + dx, a1 = cy + dy, a2 = cz + dz;
                    if (a0 < 0 || a1 < 0 || a2 < 0 || a0 >= lim || a1 >= lim || a2 >= lim) continue;
                    const uint64_t nk =
                        spread3((uint64_t)a0) | (spread3((uint64_t)a1) << 1) | (spread3((uint64_t)a2) << 2);
                    int64_t lo = 0, hi = C;
                    while (lo < hi) {
                        const int64_t mid = (lo + hi) >> 1;
                        if (cell_key[mid] < nk) lo = mid + 1; else hi = mid;
                    }
                    if (lo < C && cell_key[lo] == nk) {
                        nbr[c * kStencil + cnt++] = (int32_t)lo;
                        b += cell_start[lo + 1] - cell_start[lo];
                    }
                }
    }
    nbr_cnt[c] = cnt;
    bound[c] = b;
    const int64_t w = (int64_t)(qcell_start[c + 1] - qcell_start[c]) * b;
    work[c] = w;
    work_key[c] = ~(uint64_t)w;
    cell_idx[c] = (uint32_t)c;
}

__global__ void k_scatter_counts(const int32_t *__restrict__ ids, const int32_t *__restrict__ cell_of_row,
                                 const int64_t *__restrict__ bound, int64_t n, int64_t *__restrict__ counts)
{
    const int64_t r = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (r >= n) return;
    counts[ids[r]] = bound[cell_of_row[r]];
}

__global__ void k_tile_counts(const uint32_t *__restrict__ order, const int32_t *__restrict__ cell_start, int64_t C,
                              int tq, int32_t *__restrict__ ntiles)
{
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= C) return;
    const uint32_t c = order[i];
    const int32_t sz = cell_start[c + 1] - cell_start[c];
    ntiles[i] = (sz + tq - 1) / tq;
}

__global__ void k_tile_fill(const uint32_t *__restrict__ order, const int32_t *__restrict__ cell_start,
                            const int64_t *__restrict__ bound, const int64_t *__restrict__ tile_off, int64_t C,
                            int tq, int chunk, int32_t *__restrict__ tile_cell, int32_t *__restrict__ tile_q0,
                            int32_t *__restrict__ tile_nq, int64_t *__restrict__ tile_words,
                            int64_t *__restrict__ tile_units)
{
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= C) return;
    const uint32_t c = order[i];
    const int32_t s0 = cell_start[c], sz = cell_start[c + 1] - s0;
    const int64_t B = bound[c];
    const int64_t words = (((B + 31) / 32) + 3) & ~int64_t(3);  // mask row stride: 16-byte rows
    const int64_t units = (B + chunk - 1) / chunk;
    int64_t t = tile_off[i];
    for (int32_t q = 0; q < sz; q += tq, ++t) {
        const int32_t nq = min(tq, sz - q);
        tile_cell[t] = (int32_t)c;
        tile_q0[t] = s0 + q;
        tile_nq[t] = nq;
        tile_words[t] = (int64_t)nq * words;
        tile_units[t] = units;
    }
}

// Greedy batches: each batch takes the longest run of tiles whose device
// memory fits in cap_words 32-bit words: the mask words, their occupancy
// bitmap (one bit per word, plus two words of slack) and per_query words for
// each query (counts, row offsets, ids).  One thread; the number of batches
// is small.
__device__ __forceinline__ int64_t batch_cost(const int64_t *word_off, const int64_t *qoff, int64_t b0, int64_t b1,
                                              int64_t per_query)
{
    const int64_t dw = word_off[b1] - word_off[b0];
    return dw + (dw >> 5) + 2 + per_query * (qoff[b1] - qoff[b0]);
}

__global__ void k_plan_batches(const int64_t *__restrict__ word_off, const int64_t *__restrict__ unit_off,
                               const int64_t *__restrict__ qoff, int64_t T, int64_t cap_words, int64_t per_query,
                               int64_t *__restrict__ boundaries, int64_t *__restrict__ info,
                               int64_t *__restrict__ nb_out, int *flags)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int64_t nb = 0, start = 0;
    while (start < T) {
        boundaries[nb++] = start;
        // largest end in (start, T] whose cost fits in cap_words
        int64_t lo = start + 1, hi = T;
        if (batch_cost(word_off, qoff, start, lo, per_query) > cap_words) {
            flags[kFlagPlanTooSmall] = 1;
            break;
        }
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (batch_cost(word_off, qoff, start, mid, per_query) <= cap_words) lo = mid; else hi = mid - 1;
        }
        start = lo;
    }
    boundaries[nb] = T;
    for (int64_t k = 0; k <= nb; ++k) {
        const int64_t b = boundaries[k];
        info[4 * k + 0] = word_off[b];
        info[4 * k + 1] = unit_off[b];
        info[4 * k + 2] = qoff[b];
        info[4 * k + 3] = b;
    }
    *nb_out = nb;
}

}  // namespace

int64_t stats_blocks(int64_t n, int d)
{
    int64_t b = (n * d + 8191) / 8192;
    if (b > 4 * 152) b = 4 * 152;
    return b < 1 ? 1 : b;
}

cudaError_t dim_stats(const float *x, int64_t n, int d, double *partial, double *out, int *nonfinite,
                      cudaStream_t s, int64_t *launches)
{
    const int64_t nb = stats_blocks(n, d);
    const int64_t rows = (n + nb - 1) / nb;
    HISS_TRY(cudaMemsetAsync(nonfinite, 0, sizeof(int), s));
    k_stats_partial<<<(unsigned)nb, kT, 0, s>>>(x, n, d, rows, partial, nonfinite);
    k_stats_final<<<d, kT, 0, s>>>(x, n, d, partial, nb, out);
    *launches += 2;
    return cudaGetLastError();
}

cudaError_t permute_pad(const float *x, int64_t n, int d, int d4, const int32_t *perm, float *xv, cudaStream_t s,
                        int64_t *launches)
{
    k_permute_pad<<<blocks_for(n * d4), kT, 0, s>>>(x, n, d, d4, perm, xv);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t cell_keys(const float *xv, int64_t n, int d4, GridParams gp, uint64_t *keys, uint32_t *vals,
                      cudaStream_t s, int64_t *launches)
{
    k_cell_keys<<<blocks_for(n), kT, 0, s>>>(xv, n, d4, gp, keys, vals);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t gather_rows(const float *xv, const uint32_t *order, int64_t n, int d4, float *xs, int32_t *ids,
                        cudaStream_t s, int64_t *launches)
{
    const int c4 = d4 / 4;
    k_gather_rows<<<blocks_for(n * c4), kT, 0, s>>>(reinterpret_cast<const float4 *>(xv), order, n, c4,
                                                   reinterpret_cast<float4 *>(xs), ids);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t group_boxes(const float *xs, int64_t n, int d4, float4 *gbox, cudaStream_t s, int64_t *launches)
{
    if (n <= 0) return cudaSuccess;
    k_group_boxes<<<blocks_for(((n + 31) >> 5) * 32), kT, 0, s>>>(xs, n, d4, gbox);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t cell_flags(const uint64_t *keys, int64_t n, int shift, int32_t *flag, cudaStream_t s, int64_t *launches)
{
    k_cell_flags<<<blocks_for(n), kT, 0, s>>>(keys, n, shift, flag);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t cell_starts(const uint64_t *keys, const int32_t *flag_scan, int64_t n, int shift, int32_t *cell_start,
                        uint64_t *cell_key, int32_t *cell_of_row, cudaStream_t s, int64_t *launches)
{
    k_cell_starts<<<blocks_for(n), kT, 0, s>>>(keys, flag_scan, n, shift, cell_start, cell_key, cell_of_row);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t stencil(const uint64_t *cell_key, const int32_t *cell_start, int64_t C, int32_t *nbr, int32_t *nbr_cnt,
                    int64_t *bound, uint64_t *work_key, uint32_t *cell_idx, int64_t *work, cudaStream_t s,
                    int64_t *launches)
{
    k_stencil<<<blocks_for(C), kT, 0, s>>>(cell_key, cell_start, C, nbr, nbr_cnt, bound, work_key, cell_idx, work);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t query_keys(const float *xv, int64_t n, int d4, GridParams gp, int64_t cellmax, uint64_t *keys,
                       uint32_t *vals, cudaStream_t s, int64_t *launches)
{
    k_query_keys<<<blocks_for(n), kT, 0, s>>>(xv, n, d4, gp, cellmax, keys, vals);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t query_stencil(const uint64_t *qcell_key, const int32_t *qcell_start, int64_t Cq, const uint64_t *cell_key,
                          const int32_t *cell_start, int64_t C, int32_t *nbr, int32_t *nbr_cnt, int64_t *bound,
                          uint64_t *work_key, uint32_t *cell_idx, int64_t *work, cudaStream_t s, int64_t *launches)
{
    k_query_stencil<<<blocks_for(Cq), kT, 0, s>>>(qcell_key, qcell_start, Cq, cell_key, cell_start, C, nbr, nbr_cnt,
                                                  bound, work_key, cell_idx, work);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t scatter_counts(const int32_t *ids, const int32_t *cell_of_row, const int64_t *bound, int64_t n,
                           int64_t *counts, cudaStream_t s, int64_t *launches)
{
    k_scatter_counts<<<blocks_for(n), kT, 0, s>>>(ids, cell_of_row, bound, n, counts);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t tile_counts(const uint32_t *order, const int32_t *cell_start, int64_t C, int tq, int32_t *ntiles,
                        cudaStream_t s, int64_t *launches)
{
    k_tile_counts<<<blocks_for(C), kT, 0, s>>>(order, cell_start, C, tq, ntiles);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t tile_fill(const uint32_t *order, const int32_t *cell_start, const int64_t *bound,
                      const int64_t *tile_off, int64_t C, int tq, int chunk, int32_t *tile_cell, int32_t *tile_q0,
                      int32_t *tile_nq, int64_t *tile_words, int64_t *tile_units, cudaStream_t s,
                      int64_t *launches)
{
    k_tile_fill<<<blocks_for(C), kT, 0, s>>>(order, cell_start, bound, tile_off, C, tq, chunk, tile_cell, tile_q0,
                                             tile_nq, tile_words, tile_units);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t plan_batches(const int64_t *tile_word_off, const int64_t *tile_unit, const int64_t *tile_qoff,
                         int64_t T, int64_t cap_words, int64_t per_query_words, int64_t *boundaries, int64_t *info,
                         int64_t *nb_out, int *flags, cudaStream_t s, int64_t *launches)
{
    k_plan_batches<<<1, 32, 0, s>>>(tile_word_off, tile_unit, tile_qoff, T, cap_words, per_query_words, boundaries,
                                    info, nb_out, flags);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace hiss
