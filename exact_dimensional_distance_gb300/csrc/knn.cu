// Exact k nearest neighbours by epsilon expansion (the use of the epsilon join
// that RT-HiSS names for exact kNN): kernels that turn one CSR batch of an
// epsilon join into the k nearest neighbours of every query of the batch that
// has at least k neighbours within eps.
//
// Per batch: the squared distance of every (query, neighbour) pair is
// recomputed in float32 with the refinement's arithmetic (refine_dist2); pairs are ordered by neighbour id, then stably by (query,
// squared distance) with the library's radix sort, so each query's pairs end
// up by increasing distance, equal distances by increasing id; the first k of
// each query with at least k pairs are its result.
#include "hiss_internal.cuh"

namespace hiss {
namespace {

constexpr int kKnnWarps = 8;

// One warp per query row of the batch: distances of its pairs, the sort key
// (neighbour id) and the pair's row.
__global__ void __launch_bounds__(kKnnWarps * 32) k_knn_pairs(KnnBatchArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kKnnWarps + (threadIdx.x >> 5);
    if (r >= a.nq) return;
    const int64_t p0 = a.row_ptr[r] - a.pair0, p1 = a.row_ptr[r + 1] - a.pair0;
    const float *q = a.xq + (int64_t)a.query_rows[r] * a.d4;
    for (int64_t p = p0 + lane; p < p1; p += 32) {
        const int32_t c = a.cols[a.pair0 + p];
        const float *x = a.xv + (int64_t)c * a.d4;
        a.d2[p] = refine_dist2(q, x, a.d4);
        a.prow[p] = (int32_t)r;
        a.keys[p] = (uint64_t)(uint32_t)c;
        a.vals[p] = (uint32_t)p;
    }
}

// After the sort by neighbour id: key = (row << 32) | bits of the squared
// distance (non-negative floats order like their bit patterns).
__global__ void k_knn_rekey(KnnBatchArgs a)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.nnz) return;
    const uint32_t p = a.vals[i];
    a.keys[i] = ((uint64_t)(uint32_t)a.prow[p] << 32) | (uint64_t)__float_as_uint(a.d2[p]);
}

// First k pairs of every row with at least k pairs; marks the query done.
__global__ void k_knn_take(KnnBatchArgs a)
{
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= a.nq) return;
    const int64_t p0 = a.row_ptr[r] - a.pair0, cnt = a.row_ptr[r + 1] - a.row_ptr[r];
    if (cnt < a.k) return;
    const int64_t id = a.query_map ? (int64_t)a.query_map[a.query_ids[r]] : a.query_ids[r];
    for (int t = lane; t < a.k; t += 32) {
        const uint32_t p = a.vals[p0 + t];
        a.out_ids[id * a.k + t] = a.cols[a.pair0 + p];
        if (a.out_d2) a.out_d2[id * a.k + t] = a.d2[p];
    }
    if (lane == 0) a.done[id] = 1;
}

}  // namespace

cudaError_t knn_batch_pairs(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches)
{
    if (a.nq <= 0) return cudaSuccess;
    k_knn_pairs<<<(unsigned)((a.nq + kKnnWarps - 1) / kKnnWarps), kKnnWarps * 32, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t knn_batch_rekey(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches)
{
    if (a.nnz <= 0) return cudaSuccess;
    k_knn_rekey<<<(unsigned)((a.nnz + 255) / 256), 256, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t knn_batch_take(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches)
{
    if (a.nq <= 0) return cudaSuccess;
    k_knn_take<<<(unsigned)((a.nq + 7) / 8), 256, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace hiss
