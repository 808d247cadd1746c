// Internal declarations shared by the translation units of libhiss.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "hiss.h"

namespace hiss {

// ---- tiling of the refinement kernel ---------------------------------------
// A refinement unit is one query tile (up to refine_tq() queries of one cell)
// against one chunk of up to refine_chunk() of the cell's stencil candidates.
constexpr int kStencil = 27;

// Device-side error flags (one int each in ctx->d_flags).
enum { kFlagSortTimeout = 0, kFlagPlanTooSmall = 1, kFlagOverflow = 2, kFlagRefineTimeout = 3, kNumFlags = 4 };

// Sticky-error launch check used by every host wrapper.
#define HISS_TRY(expr)                                      \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return e_;                   \
    } while (0)

// ---- scan (scan.cu) --------------------------------------------------------
// Exclusive prefix sums; out has n + 1 entries (out[n] = total).  tmp must
// hold scan_tmp_elems(n) int64 values.  in and out may alias for the
// int64 -> int64 form.
int64_t scan_tmp_elems(int64_t n);
cudaError_t scan_i64(const int64_t *in, int64_t *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches);
cudaError_t scan_i32_to_i64(const int32_t *in, int64_t *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches);
cudaError_t scan_i32(const int32_t *in, int32_t *out, int64_t n, int64_t *tmp, cudaStream_t s, int64_t *launches);

// ---- onesweep radix sort (sort.cu) -----------------------------------------
size_t sort_tmp_bytes(int64_t n);
// Sorts (keys, vals) by the low key_bits bits.  keys_alt/vals_alt are
// ping-pong buffers of n entries.  On return *in_alt tells whether the
// sorted data are in the alt buffers.  flags: device int[kNumFlags].
cudaError_t sort_pairs(uint64_t *keys, uint32_t *vals, uint64_t *keys_alt, uint32_t *vals_alt, int64_t n,
                       int key_bits, void *tmp, int *flags, cudaStream_t s, int64_t *launches, int *in_alt);

// ---- index kernels (index.cu) ----------------------------------------------
int64_t stats_blocks(int64_t n, int d);
// partial: [blocks][d][4] doubles; out: [4][d] doubles (min, max, mean, var)
// and nonfinite: device int (count of non-finite inputs).
cudaError_t dim_stats(const float *x, int64_t n, int d, double *partial, double *out, int *nonfinite,
                      cudaStream_t s, int64_t *launches);
cudaError_t permute_pad(const float *x, int64_t n, int d, int d4, const int32_t *perm, float *xv,
                        cudaStream_t s, int64_t *launches);

struct GridParams {
    double origin[3];
    double w;
    int sub_bits;
    int key_bits;
    int ndim;  // index dimensions used (min(d, 3))
};
cudaError_t cell_keys(const float *xv, int64_t n, int d4, GridParams gp, uint64_t *keys, uint32_t *vals,
                      cudaStream_t s, int64_t *launches);
cudaError_t gather_rows(const float *xv, const uint32_t *order, int64_t n, int d4, float *xs, int32_t *ids,
                        cudaStream_t s, int64_t *launches);
// Per aligned 32-row group of xs: box over the first three dimensions,
// gbox[2 g] = minima, gbox[2 g + 1] = maxima ((n + 31) / 32 groups).
cudaError_t group_boxes(const float *xs, int64_t n, int d4, float4 *gbox, cudaStream_t s, int64_t *launches);
cudaError_t cell_flags(const uint64_t *keys, int64_t n, int shift, int32_t *flag, cudaStream_t s, int64_t *launches);
cudaError_t cell_starts(const uint64_t *keys, const int32_t *flag_scan, int64_t n, int shift, int32_t *cell_start,
                        uint64_t *cell_key, int32_t *cell_of_row, cudaStream_t s, int64_t *launches);
cudaError_t stencil(const uint64_t *cell_key, const int32_t *cell_start, int64_t C, int32_t *nbr, int32_t *nbr_cnt,
                    int64_t *bound, uint64_t *work_key, uint32_t *cell_idx, int64_t *work, cudaStream_t s,
                    int64_t *launches);
// Semi-join: queries keyed into the data's grid (see k_query_keys) and the
// stencil of each query cell among the data's cells.
cudaError_t query_keys(const float *xv, int64_t n, int d4, GridParams gp, int64_t cellmax, uint64_t *keys,
                       uint32_t *vals, cudaStream_t s, int64_t *launches);
cudaError_t query_stencil(const uint64_t *qcell_key, const int32_t *qcell_start, int64_t Cq, const uint64_t *cell_key,
                          const int32_t *cell_start, int64_t C, int32_t *nbr, int32_t *nbr_cnt, int64_t *bound,
                          uint64_t *work_key, uint32_t *cell_idx, int64_t *work, cudaStream_t s, int64_t *launches);
cudaError_t scatter_counts(const int32_t *ids, const int32_t *cell_of_row, const int64_t *bound, int64_t n,
                           int64_t *counts, cudaStream_t s, int64_t *launches);
// Per cell in processing order: tiles and their sizes.
cudaError_t tile_counts(const uint32_t *order, const int32_t *cell_start, int64_t C, int tq, int32_t *ntiles,
                        cudaStream_t s, int64_t *launches);
cudaError_t tile_fill(const uint32_t *order, const int32_t *cell_start, const int64_t *bound,
                      const int64_t *tile_off, int64_t C, int tq, int chunk, int32_t *tile_cell, int32_t *tile_q0,
                      int32_t *tile_nq, int64_t *tile_words, int64_t *tile_units, cudaStream_t s,
                      int64_t *launches);
// Greedy batches over query tiles: boundaries[k] = first tile of batch k,
// boundaries[nb] = T; *nb written to nb_out (device).  info[4 k + 0..2] =
// (word offset, unit offset, query offset) at boundary k, for k = 0..nb.
// A batch's cost in 32-bit words is its mask words + occupancy words
// (words / 32 + 2) + per_query_words per query; it is at most cap_words.
// flags[kFlagPlanTooSmall] is set when one tile alone exceeds cap_words.
cudaError_t plan_batches(const int64_t *tile_word_off, const int64_t *tile_unit, const int64_t *tile_qoff,
                         int64_t T, int64_t cap_words, int64_t per_query_words, int64_t *boundaries, int64_t *info,
                         int64_t *nb_out, int *flags, cudaStream_t s, int64_t *launches);

// ---- refinement and compaction (refine.cu) ---------------------------------
struct RefineArgs {
    const float *xs;            // index-ordered points, n x d4 (row stride d4)
    const float *xq;            // query rows (== xs for the self-join)
    const int32_t *cell_start;  // [C+1]
    const int32_t *nbr;         // [C*27]
    const int32_t *nbr_cnt;     // [C]
    const int64_t *bound;       // [C]
    const int32_t *tile_cell;   // [T]
    const int32_t *tile_q0;     // [T] first index row of the tile
    const int32_t *tile_nq;     // [T]
    const int64_t *tile_word;   // [T+1] mask word offset (absolute)
    const int64_t *tile_unit;   // [T+1] first unit of each tile (absolute)
    const int64_t *tile_qoff;   // [T+1] first query (absolute, processing order)
    int64_t t0, t1;             // batch: tiles [t0, t1)
    int64_t unit0, nunits;      // units of the batch
    const int32_t *unit_tile;   // [nunits] tile of block u (NULL: found by search, units in tile order)
    const int32_t *unit_chunk;  // [nunits] candidate chunk of block u
    int64_t word0, q0;          // batch origin in words and queries
    uint32_t *mask;             // batch mask: only nonzero words are written
    uint32_t *occ;              // occupancy: bit (w & 31) of occ[w >> 5] set when mask word w is nonzero (zeroed per batch)
    int32_t *qcount;            // [nq of batch] neighbour count per query (accumulated)
    int d4;
    int d;                      // true dimension (profile mode caps the last step at d)
    float eps2;
    int64_t *prof;              // profile mode: [2] counters (sum of per-pair exit dims, executed dims)
    const float4 *gbox;         // boxes of xs's 32-row groups (see group_boxes); NULL: every staged tile is streamed
    unsigned long long *kept;   // if set: candidate pairs of the staged tiles kept for refinement are added here
    int *flags;                 // device int[kNumFlags]; kFlagRefineTimeout set if a stage wait gave up
};
int refine_tq(int d4);
int refine_chunk(int d4);
// The float32 squared distance of two rows of d4 values (variance order,
// padded) with the refinement's own arithmetic (the first product, then a
// fused multiply-add per dimension, in dimension order), so that values
// recomputed elsewhere (tensor-core recheck, kNN ranking) agree with its bits.
__device__ __forceinline__ float refine_dist2(const float *q, const float *p, int d4)
{
    float s = 0.0f;
    for (int k = 0; k < d4; k += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(q + k);
        const float4 b = *reinterpret_cast<const float4 *>(p + k);
        float e = __fsub_rn(a.x, b.x);
        s = k == 0 ? __fmul_rn(e, e) : __fmaf_rn(e, e, s);
        e = __fsub_rn(a.y, b.y);
        s = __fmaf_rn(e, e, s);
        e = __fsub_rn(a.z, b.z);
        s = __fmaf_rn(e, e, s);
        e = __fsub_rn(a.w, b.w);
        s = __fmaf_rn(e, e, s);
    }
    return s;
}
cudaError_t refine(const RefineArgs &a, cudaStream_t s, int64_t *launches);
// The order in which a batch's blocks take its units: within each cell's run
// of tiles in the batch, chunk by chunk (every query tile of the cell on
// candidate chunk 0, then chunk 1, ...), so that blocks running at the same
// time read the same candidate rows.  Fills unit_tile / unit_chunk (device
// arrays of a.nunits entries) from the batch's tiles; qcell_start: the query
// side's cell ranges (the data's own for the self-join).
cudaError_t unit_order(const RefineArgs &a, const int32_t *qcell_start, int tq, int32_t *unit_tile,
                       int32_t *unit_chunk, cudaStream_t s, int64_t *launches);
cudaError_t refine_profile(const RefineArgs &a, cudaStream_t s, int64_t *launches);

struct CompactArgs {
    const int32_t *ids;         // [n] original id per index row
    const int32_t *qids;        // original id per query row (== ids for the self-join)
    const int32_t *cell_start;
    const int32_t *nbr;
    const int32_t *nbr_cnt;
    const int64_t *bound;
    const int32_t *tile_cell;
    const int32_t *tile_q0;
    const int64_t *tile_word;
    const int64_t *tile_qoff;
    int64_t t0, t1, word0, q0, nq;
    const uint32_t *mask;
    const uint32_t *occ;        // occupancy bitmap of the mask (nonzero words)
    const int64_t *row_ptr;     // [nq+1] batch-relative
    int64_t col0;               // row_ptr value of this call's first query: row gq goes to cols + row_ptr[gq] - col0
    int64_t *row_ptr_out;       // [nq+1] row_ptr - col0 (may be NULL)
    int32_t *cols;              // CSR output (NULL: only query ids/rows/cand)
    int64_t *query_ids;         // [nq]
    int32_t *query_rows;        // [nq]
    int64_t *cand;              // [nq] B_q (may be NULL)
    int64_t *mask_row_ptr;      // [nq+1] word offsets (may be NULL)
};
cudaError_t compact(const CompactArgs &a, cudaStream_t s, int64_t *launches);
cudaError_t mask_positions(const uint32_t *words, int64_t nbits, int64_t *pos, int64_t *count,
                           int64_t *tmp, cudaStream_t s, int64_t *launches);

// ---- exact kNN by epsilon expansion (knn.cu) --------------------------------------
// A group of rows of one CSR batch of an epsilon join (row_ptr, query_rows and
// query_ids point at the group's first row; scratch arrays are indexed from the
// group's first pair): per pair p of row r, the float32
// squared distance d2[p] between query row query_rows[r] of xq and data point
// cols[p] of xv (original order, variance-ordered dimensions).
struct KnnBatchArgs {
    const float *xq;             // query rows (index order of the query side), row stride d4
    const float *xv;             // data points in original order, row stride d4
    const int64_t *row_ptr;      // [nq + 1]
    const int32_t *cols;         // [nnz] neighbour ids
    const int32_t *query_rows;   // [nq] row of each query in xq
    const int64_t *query_ids;    // [nq] id of each query in the join's query set
    const int32_t *query_map;    // query set -> point id (NULL: identity)
    int64_t nq, nnz;
    int64_t pair0;               // pairs of this group start at cols[pair0] (= row_ptr[0])
    int d4, k;
    float *d2;                   // [nnz] scratch: squared distances
    int32_t *prow;               // [nnz] scratch: row of each pair
    uint64_t *keys;              // [nnz] sort keys
    uint32_t *vals;              // [nnz] sort values (pair index)
    int64_t *out_ids;            // [n * k]
    float *out_d2;               // [n * k] or NULL
    int8_t *done;                // [n] set to 1 for queries completed in this batch
};
cudaError_t knn_batch_pairs(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches);   // d2, prow, keys = col, vals = p
cudaError_t knn_batch_rekey(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches);   // keys = (prow << 32) | d2 bits
cudaError_t knn_batch_take(const KnnBatchArgs &a, cudaStream_t s, int64_t *launches);    // first k per row with >= k pairs

// ---- tensor cores (refine_tc.cu) ----------------------------------------------
// Refinement of a batch with the squared distances from TF32 Gram matrices on
// the tensor cores and an exact float32 recheck of every undecided pair;
// same units, tiles (refine_tc_tq() queries, refine_tc_chunk() candidates
// per unit) and mask as refine().  d4 <= refine_tc_max_d4().
int refine_tc_max_d4();
int refine_tc_tq();
int refine_tc_chunk();
cudaError_t refine_tc(const RefineArgs &a, float eps, cudaStream_t s, int64_t *launches);
// G = tf32(a) tf32(b)^T for two 128 x k float32 blocks (k % 8 == 0, k <= 128).
cudaError_t gram_tf32(const float *a, const float *b, int k, float *out, int *flags, cudaStream_t s,
                      int64_t *launches);

}  // namespace hiss
