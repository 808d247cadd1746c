/*
 * hiss.h -- C ABI of the GB300 exact epsilon self-join library (libhiss.so).
 *
 * The operation (RT-HiSS, Munugala & Gowanlock, "RT-HiSS: Ray Tracing
 * Accelerated High Dimensional Vector Similarity Searches", Section II-A,
 * "Problem Statement"): for a dataset D of n points in R^d, return every pair
 * (i, j) with Euclidean distance dist(p_i, p_j) <= eps, inclusive; each point
 * is its own neighbour.  The library computes it in the three steps of the
 * paper's Section IV, rebuilt for one GPU without ray-tracing cores:
 *
 *   hiss_build  -- per-dimension variance and the variance order of the
 *                  dimensions (Section IV-A); the data are kept on the device
 *                  in that order.
 *   hiss_count  -- a three-dimensional grid over the three highest-variance
 *                  dimensions (grid indexing, Section II-B1) with Morton-ordered
 *                  points (Section IV-C), and the count pass that bounds every
 *                  query's candidate count (first intersection test and pass 1,
 *                  Section IV-D).
 *   hiss_join   -- batches sized from the count pass (Section IV-D), exact
 *                  refinement on CUDA cores with shared-memory tiling and early
 *                  termination in variance order (Sections IV-A and IV-E), a
 *                  one-bit-per-candidate result mask and its stream compaction
 *                  (Section IV-F1, Fig. 5), and optional delivery to host memory
 *                  (Section IV-F2).
 *
 * Conventions shared by every call
 *   - Every call returns HISS_OK (0) or a negative hiss_status; none aborts.
 *     A CUDA error inside the library is sticky: the call that meets it
 *     returns HISS_E_CUDA and every later call on the context returns
 *     HISS_E_STATE (destroy the context and create a new one).
 *   - "device pointer" means memory of the current CUDA device (cudaMalloc,
 *     a torch CUDA tensor, ...); "host pointer" means ordinary or pinned host
 *     memory.  The library never frees memory it did not allocate.
 *   - A context is bound to the CUDA stream given at creation and to the
 *     device current at that time.  All device work of a call is ordered on
 *     that stream; calls return after the work they describe is complete
 *     unless stated otherwise.  A context is not thread-safe.
 *   - Point ids are the row indices of the array given to hiss_build
 *     (0-based).  n must be below 2^30 and d at most HISS_MAX_DIM.
 */
#ifndef HISS_H
#define HISS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HISS_MAX_DIM 256

typedef enum {
    HISS_OK = 0,
    HISS_E_ARG = -1,             /* invalid argument (NULL, n < 1, d out of range, eps < 0 or NaN, non-finite input) */
    HISS_E_NOMEM = -2,           /* a device or pinned allocation failed (or exceeded the allocation limit) */
    HISS_E_STATE = -3,           /* call out of order (join before build), or the context holds a sticky CUDA error */
    HISS_E_BATCH_TOO_SMALL = -4, /* batch_bytes is smaller than the result mask of one query tile */
    HISS_E_OVERFLOW = -5,        /* a count exceeded the library's integer ranges */
    HISS_E_CUDA = -6,            /* a CUDA runtime call or kernel failed; see hiss_last_cuda_error */
    HISS_E_CALLBACK = -7         /* the batch callback returned non-zero; the join stopped */
} hiss_status;

typedef struct hiss_ctx hiss_ctx;

/* Create a context on the current CUDA device.  cuda_stream is a
 * cudaStream_t (NULL = the legacy default stream).  The context owns every
 * internal device buffer; none is allocated before the first build. */
int hiss_create(hiss_ctx **out, void *cuda_stream);

/* Free every resource of the context.  NULL is ignored. */
void hiss_destroy(hiss_ctx *ctx);

/* Load the dataset.  d_points: device pointer to n x d float32, row-major
 * (row i = point i), read only during the call; the library keeps its own
 * copy, so the caller may free or overwrite the array afterwards.  Computes
 * the per-dimension min, max and variance (fp64 accumulation) and the
 * variance order of the dimensions, descending, equal variances by lower
 * index (RT-HiSS Section IV-A), and stores the points with their dimensions in
 * that order, padded with zeros to a multiple of 4.  Rejects non-finite
 * coordinates with HISS_E_ARG.  Discards any index built for an earlier
 * dataset. */
int hiss_build(hiss_ctx *ctx, const float *d_points, int64_t n, int32_t d);

/* As hiss_build, with h_points a host pointer; the copy to the device is part
 * of the call. */
int hiss_build_host(hiss_ctx *ctx, const float *h_points, int64_t n, int32_t d);

/* Build the grid index for eps (reused while eps is unchanged) and write the
 * count bound of every point: d_counts (device pointer, int64[n], original
 * point order; may be NULL to build the index only) receives B_q, the number
 * of points in the 27 grid cells around q's cell, q's own cell included.
 * B_q >= |{j : dist(q, p_j) <= eps}| for every q (the grid cell side exceeds
 * eps).  This is the per-query intersection count of the first intersection
 * test (RT-HiSS Section IV-D) for the grid index.  eps must be finite and
 * >= 0. */
int hiss_count(hiss_ctx *ctx, float eps, int64_t *d_counts);

/* One batch of results handed to the caller. */
typedef struct {
    int64_t index;              /* batch number, 0-based */
    int64_t nq;                 /* queries in this batch */
    const int64_t *query_ids;   /* [nq] original id of each query, in processing order */
    const int64_t *row_ptr;     /* [nq+1] CSR: offsets into cols; MASK: offsets into mask (32-bit words;
                                   rows are padded to a multiple of 4 words, bits at or beyond cand[i] are 0
                                   or unspecified) */
    const int32_t *cols;        /* CSR: [nnz] original ids of the neighbours (unordered within a row); else NULL */
    const uint32_t *mask;       /* MASK: [n_words] result mask; else NULL */
    const int64_t *cand;        /* MASK: [nq] candidate count B_q (bits used in the row); else NULL */
    const int32_t *query_rows;  /* [nq] row of each query in the index order (see hiss_index) */
    int64_t nnz;                /* CSR: pairs in this batch (self pairs included) */
    int64_t n_words;            /* MASK: mask words in this batch */
    int32_t on_host;            /* 1: every pointer above is host memory; 0: device memory */
    int32_t mode;               /* HISS_OUT_CSR or HISS_OUT_MASK */
} hiss_batch;

/* Called once per batch, in batch order, after the batch is complete on the
 * device (and copied to the host when copy_to_host = 1).  The pointers are
 * valid only until the callback returns.  A non-zero return stops the join
 * with HISS_E_CALLBACK. */
typedef int (*hiss_batch_fn)(void *user, const hiss_batch *batch);

enum { HISS_OUT_CSR = 0, HISS_OUT_MASK = 1 };

typedef struct {
    int32_t mode;            /* HISS_OUT_CSR (default) or HISS_OUT_MASK */
    int32_t copy_to_host;    /* 1: copy each batch to pinned host memory before the callback */
    hiss_batch_fn on_batch;  /* may be NULL: results are produced on the device and dropped */
    void *user;              /* passed to on_batch */
} hiss_out;

/* The self-join for eps.  Builds (or reuses) the grid index of hiss_count,
 * orders the grid cells by decreasing work |cell| * B_cell so that the
 * largest work goes first (RT-HiSS Section IV-D), and cuts them, one query
 * tile at a time, into batches whose result mask (one bit per candidate
 * pair, ceil(B_q / 32) words per query rounded up to a multiple of 4) fits
 * in three quarters of batch_bytes together with its occupancy bitmap (one
 * bit per mask word) and its per-query arrays (counts, row offsets, ids; 24
 * bytes per query, 40 with HISS_OUT_MASK, 44 for CSR copied to the host,
 * whose batches alternate between two sets).  The CSR columns of a batch get
 * the rest of batch_bytes (half of it per set when copied to the host); a
 * batch whose result is larger is compacted and handed over in parts of
 * consecutive queries, each a batch of its own for the callback, so the
 * library's batch memory stays within batch_bytes.  HISS_E_BATCH_TOO_SMALL:
 * one query tile, or one query's row of results, does not fit.  Each batch is
 * refined exactly on CUDA cores (float32 squared distances summed in
 * variance order, pair rejected once the partial sum exceeds eps^2; bit =
 * sum <= eps^2; candidate tiles whose boxes over the index dimensions are
 * provably farther than eps from the query tile's box are skipped with
 * their bits 0, see hiss_stats.candidates_refined), compacted from the mask
 * to CSR (Section IV-F1) unless out->mode is HISS_OUT_MASK, and handed to
 * out->on_batch.  Every query
 * appears in exactly one batch; every row contains the query itself.
 * batch_bytes = 0 selects 1/4 of the free device memory.  out may be NULL
 * (CSR, device, no callback).
 *
 * Mask layout (HISS_OUT_MASK): bit v of a query's row (word v / 32, bit
 * v % 32) is the v-th candidate of the query's cell: the cells of the
 * stencil in the order given by hiss_index (dz, dy, dx, dz outermost), each
 * cell's points in index order. */
int hiss_join(hiss_ctx *ctx, float eps, size_t batch_bytes, const hiss_out *out);

/* One shard of the self-join, for spreading one join over nranks GPUs (one
 * context per GPU, each built from the same points: the index is
 * deterministic, so every rank derives the same query tiles).  The query
 * tiles in processing order are cut into nranks contiguous ranges with about
 * equal refinement units (split at the unit prefix sums); this call runs
 * range rank (0 <= rank < nranks) exactly as hiss_join runs all of them.
 * Every query belongs to exactly one shard, so the union of the shards'
 * batches is the join; no data moves between ranks.  RT-HiSS suggests
 * offloading batches to other GPUs (Section VI); this is that split. */
int hiss_join_shard(hiss_ctx *ctx, float eps, size_t batch_bytes, const hiss_out *out, int32_t rank,
                    int32_t nranks);

/* Semi-join (RT-HiSS Section II-A: "D and Q are distinct"; the method
 * applies unchanged): for each of nq query points (d_queries: device pointer,
 * nq x d float32 row-major, same d as the dataset, read only during the call)
 * every point of the dataset within eps, inclusive.  The queries are keyed
 * into the dataset's grid for eps (built or reused as by hiss_count); a query
 * more than one cell outside the grid on an index dimension has no candidate
 * and an empty row.  Batches, output modes and the callback are those of
 * hiss_join, with query_ids = row indices of d_queries (0 .. nq-1) and
 * query_rows = rows of the queries in their own cell order; cols are dataset
 * ids.  No query is its own neighbour unless it coincides with a data point
 * within eps.  nq = 0 is valid (no batch).  Invalidates the self-join's
 * cached tiles (the next hiss_join rebuilds them). */
int hiss_join_queries(hiss_ctx *ctx, const float *d_queries, int64_t nq, float eps, size_t batch_bytes,
                      const hiss_out *out);

/* Count bound of the semi-join: d_counts (device int64[nq], query order)
 * receives, per query, the number of dataset points in the 27 grid cells
 * around the query's cell, >= its true neighbour count. */
int hiss_count_queries(hiss_ctx *ctx, const float *d_queries, int64_t nq, float eps, int64_t *d_counts);

/* Exact k nearest neighbours by epsilon expansion (RT-HiSS names exact kNN
 * as a use of the epsilon join: repeat the join with a growing eps for the
 * queries that have fewer than k neighbours, then keep the k nearest).  For
 * every point of the dataset (the point itself included, at distance 0):
 * d_ids (device int64[n * k], row i = point i) receives the ids of its k
 * nearest points by float32 squared distance summed in variance order,
 * increasing, equal distances by increasing id; d_dist2 (device
 * float32[n * k], may be NULL) receives those squared distances.  Round 1 is
 * the self-join for eps0 (eps0 <= 0: a start from the point spacing over the
 * three index dimensions); each later round multiplies eps by sqrt(2), capped
 * at the dataset's diameter, and semi-joins only the points still short of k
 * neighbours.  A point is finished in the first round where it has at least
 * k neighbours within eps, which holds its k nearest.  1 <= k <= n.  Join
 * batches hold up to 1 GiB of result mask; their pairs are ranked in groups
 * of rows of at most 2^27 pairs (one longer row forms its own group). */
int hiss_knn(hiss_ctx *ctx, int32_t k, float eps0, int64_t *d_ids, float *d_dist2);

/* Read-only view of the index built for the last eps (device pointers owned
 * by the context, valid until the next build or a call with another eps). */
typedef struct {
    int64_t n;                  /* points */
    int64_t cells;              /* non-empty grid cells C */
    const int32_t *ids;         /* [n] original id of the point at each index row (Morton order) */
    const int32_t *cell_start;  /* [C+1] first index row of each cell; cell_start[C] = n */
    const int32_t *cell_of_row; /* [n] cell of each index row */
    const int32_t *nbr;         /* [C*27] existing stencil cells of each cell, first nbr_count[c] used */
    const int32_t *nbr_count;   /* [C] */
    const int64_t *cell_bound;  /* [C] B_cell: points in the cell's stencil */
    const uint64_t *cell_key;   /* [C] Morton key of each cell's grid coordinates */
    int32_t perm[3];            /* index dimensions (original dimension numbers), highest variance first */
    int32_t sub_bits;           /* sub-cell bits per dimension used to order points inside a cell */
    double cell_width;          /* grid cell side w > eps */
    double origin[3];           /* grid origin on the three index dimensions */
} hiss_index_view;

int hiss_index(hiss_ctx *ctx, hiss_index_view *out);

/* Counters and timings of the last hiss_count / hiss_join. */
typedef struct {
    int64_t n, cells, cell_pairs;   /* points, non-empty cells, stencil cell pairs */
    int64_t candidates;             /* sum of B_q over all queries (candidate distance evaluations) */
    int64_t pairs;                  /* result pairs |R| of the last join, self pairs included */
    int64_t batches, query_tiles, refine_units;
    int64_t mask_words_max;         /* largest batch mask, 32-bit words */
    int64_t kernel_launches;        /* kernels launched by the last call */
    int32_t d, d_pad, sub_bits, key_bits;
    float eps;
    double cell_width;
    double ms_build, ms_index, ms_count, ms_refine, ms_compact, ms_deliver, ms_total;
    int64_t deliveries;             /* batches handed to the callback: more than batches when a batch's
                                       CSR result outgrew its share of batch_bytes and came in parts */
    int64_t candidates_refined;     /* candidate pairs of the last join in the staged tiles the CUDA-core
                                       refinement kept after its group-box test (at most candidates; the
                                       rest were proved farther than eps without being streamed); -1 with
                                       the tensor-core refinement */
} hiss_stats;

int hiss_last_stats(const hiss_ctx *ctx, hiss_stats *out);

/* Kernels launched by this context since creation (all calls). */
int64_t hiss_launch_count(const hiss_ctx *ctx);

/* Human-readable name of a status code (static string). */
const char *hiss_strerror(int status);

/* The CUDA error string behind the last HISS_E_CUDA of this context. */
const char *hiss_last_cuda_error(const hiss_ctx *ctx);

/* Options.  HISS_OPT_ALLOC_LIMIT: cap, in bytes, on the device memory the
 * context may hold (0 = no cap); an allocation beyond it fails with
 * HISS_E_NOMEM without calling the CUDA allocator.  Used to test the
 * out-of-memory path without exhausting the device.
 *
 * HISS_OPT_REFINE selects the refinement of hiss_join and hiss_join_queries:
 *   HISS_REFINE_CUDA_CORES (default): float32 squared distances on the CUDA
 *     cores, summed in variance order with early termination (RT-HiSS
 *     Sections IV-A and IV-E);
 *   HISS_REFINE_TENSOR_CORES: the same result mask from a prefilter on the
 *     tensor cores (d <= 128; larger d uses the CUDA cores).  Per 128 x 128
 *     tile of (query, candidate) pairs, the points are centred on the query
 *     tile's mean and rounded to TF32, and the squared distance minus eps^2 is
 *     obtained as a Gram matrix (tcgen05.mma) with the norms carried in extra
 *     K columns.  A rigorous bound on the rounding and accumulation errors
 *     decides most pairs from the sign; every pair inside the bound is
 *     rechecked exactly (float32 sum in variance order).  Decided pairs agree
 *     with the exact predicate dist <= eps; rechecked pairs are those of the
 *     CUDA-core refinement.  No pages' counterpart: RT-HiSS refines on CUDA
 *     cores only.
 * Other options or values return HISS_E_ARG. */
enum { HISS_OPT_ALLOC_LIMIT = 1, HISS_OPT_REFINE = 2 };
enum { HISS_REFINE_CUDA_CORES = 0, HISS_REFINE_TENSOR_CORES = 1 };
int hiss_set_option(hiss_ctx *ctx, int option, int64_t value);

/* Work accounting for the refinement roofline (diagnostic; no result
 * output).  For eps, over every candidate pair of the join: out[0] = the
 * sum, over pairs, of the dimensions the pair needs when it is abandoned at
 * the first multiple of 4 dimensions whose variance-ordered float32 partial
 * sum exceeds eps^2 (capped at d) -- the method's minimal refinement work
 * with early termination (RT-HiSS Section IV-A); out[1] = the dimensions
 * hiss_join's refinement kernel actually evaluates, whose warps skip a
 * block of pairs when the boxes of its queries and candidates over the three
 * index dimensions are farther apart than eps, and otherwise abandon it only
 * when all of its pairs exceed eps^2 (checked after every 2 dimensions up to
 * d4 = 64, from the 10th at d4 = 16 and the 6th at d4 = 32 on, and after
 * every 4 above d4 = 64); from d4 = 64 on, a warp left with at most 64 pairs
 * within eps^2 after 16 dimensions, or with any when the dimensions staged in
 * shared memory run out (16 at d4 = 64, 32 above), finishes those pairs
 * alone, each stopping when it exceeds eps^2.  out is a host int64[2].
 * Costs about one join's refinement with no early termination. */
int hiss_work_profile(hiss_ctx *ctx, float eps, int64_t *out);

/* ---- building blocks exposed for testing ---------------------------------
 * These run the library's own kernels on caller data (device pointers) on
 * the context's stream and return when done. */

/* Stable LSD radix sort (onesweep: one digit histogram pass, then one
 * decoupled-look-back scatter pass per 8-bit digit) of n (key, value) pairs
 * by the low key_bits bits of the key (1..64); keys and vals are sorted in
 * place.  n < 2^30. */
int hiss_sort_pairs(hiss_ctx *ctx, uint64_t *d_keys, uint32_t *d_vals, int64_t n, int32_t key_bits);

/* Exclusive prefix sum of n int64 values: out[i] = sum(in[0..i)), out[n] =
 * total (out has n + 1 entries).  in and out may alias. */
int hiss_exclusive_scan(hiss_ctx *ctx, const int64_t *d_in, int64_t *d_out, int64_t n);

/* Stream compaction of one result mask (RT-HiSS Section IV-F1, Fig. 5):
 * writes the positions of the ones among the first nbits bits of d_words
 * (bit v = word v / 32, bit v % 32) to d_pos in increasing order and their
 * number to *h_count (host).  d_pos must hold nbits entries. */
int hiss_mask_positions(hiss_ctx *ctx, const uint32_t *d_words, int64_t nbits, int64_t *d_pos, int64_t *h_count);

/* Gram matrix on the tensor cores: out[i][j] = sum_k tf32(a[i][k]) *
 * tf32(b[j][k]) for two 128 x k float32 row-major device blocks (k a
 * multiple of 8, 8 <= k <= 128), out a device float32[128][128].  tf32(x)
 * rounds to 10 explicit mantissa bits, to nearest with ties away from zero;
 * the products are exact in float32 and the sums are accumulated in float32
 * by tcgen05.mma (kind::tf32).  This is the inner product that the
 * tensor-core refinement evaluates (see HISS_OPT_REFINE); exposed to test the
 * tensor-core operand layout. */
int hiss_gram_tf32(hiss_ctx *ctx, const float *d_a, const float *d_b, int32_t k, float *d_out);

/* ---- allocation-free variant ---------------------------------------------
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory (a plugin inside a host framework that
 * owns all device memory through its own pool, or a latency-critical loop that
 * cannot afford cudaMalloc's implicit device-wide synchronisation).
 *
 * Same result as hiss_exclusive_scan (out[i] = sum(in[0..i)), out[n] =
 * total; in and out may alias), computed by the same kernels on cuda_stream
 * (a cudaStream_t; NULL = legacy default stream), but with no context and no
 * allocation: the scratch lives in a static device array of 256 KiB that
 * every device loading the library holds until the process exits.  The call
 * is asynchronous with respect to the host.
 *   - n must be at most 2^26 (67,108,864); larger n returns HISS_E_ARG.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - cudaDeviceReset makes the cached address stale: after resetting a
 *     device, do not call this entry point on it again in the same process.
 *   - All calls share the array: calls whose kernels may overlap on the GPU
 *     (other streams, other host threads) race and must be ordered by the
 *     caller.  Nothing in the array needs clearing between calls.
 *   - A CUDA error already pending on the calling thread (left by the
 *     caller's earlier work) is not cleared: the call returns HISS_E_CUDA
 *     without launching, and the caller can still read the error with
 *     cudaGetLastError.
 * Returns HISS_OK, HISS_E_ARG, or HISS_E_CUDA if a launch failed or an error
 * was already pending. */
int hiss_exclusive_scan_noalloc(void *cuda_stream, const int64_t *d_in, int64_t *d_out, int64_t n);

#ifdef __cplusplus
}
#endif
#endif /* HISS_H */
