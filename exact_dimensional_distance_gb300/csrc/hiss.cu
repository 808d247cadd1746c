// C ABI of libhiss.so: context, buffers, and the orchestration of build,
// count and join (RT-HiSS Sections IV-A to IV-F rebuilt for one GPU without
// ray-tracing cores).  All device work runs on the context's stream; the
// host only sizes launches from a few counts it reads back.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "hiss_internal.cuh"

using namespace hiss;

namespace {

struct DBuf {
    void *p = nullptr;
    size_t cap = 0;
};

template <typename T>
T *as(DBuf &b) { return static_cast<T *>(b.p); }

}  // namespace

struct hiss_ctx {
    int device = 0;
    cudaStream_t stream = nullptr;
    int sticky = 0;
    char cuda_err[256] = {0};
    int64_t alloc_limit = 0;
    int64_t alloc_held = 0;
    int64_t launches = 0;

    // dataset (variance-ordered, padded to d4)
    bool built = false;
    int64_t n = 0;
    int d = 0, d4 = 0;
    std::vector<int32_t> perm;
    std::vector<double> stats;  // [4][d]: min, max, mean, var (original dimension order)
    DBuf x_stage, xv, perm_d, stats_partial, stats_out, flags;

    // grid index for one eps
    bool grid_valid = false;
    float grid_eps = 0.0f;
    GridParams gp{};
    int64_t C = 0, cell_pairs = 0, candidates = 0;
    DBuf keys, vals, keys_alt, vals_alt, sort_tmp, xs, ids, flag, flag_scan, cell_start, cell_key, cell_of_row;
    DBuf gbox;  // boxes of xs's 32-row groups over the index dimensions
    DBuf nbr, nbr_cnt, bound, work_key, cell_idx, work, scan_tmp, sums2;
    uint64_t *sorted_keys = nullptr;
    uint32_t *sorted_vals = nullptr;

    // query tiles in processing order
    bool tiles_valid = false;
    int tiles_tc = 0;           // the cached tiles were cut for the tensor-core refinement
    int refine_mode = HISS_REFINE_CUDA_CORES;
    int64_t T = 0, total_units = 0, total_words = 0;
    DBuf lpt_keys, lpt_order, ntiles, tile_off, tile_cell, tile_q0, tile_nq, tile_word, tile_unit, tile_qoff;
    uint32_t *order = nullptr;

    // batches
    DBuf boundaries, binfo, nb_d, mask, occ, qcount, row_ptr, cols, query_ids, query_rows, cand, mask_row_ptr;

    // host staging for copy_to_host
    void *h_pinned = nullptr;
    size_t h_cap = 0;

    // overlapped host delivery (CSR to host): second set of batch outputs and
    // pinned staging, a copy stream and its events (created on first use)
    DBuf row_ptr2, cols2, query_ids2, query_rows2;
    DBuf row_ptr_sub;  // row offsets of a batch delivered in parts
    DBuf unit_tile, unit_chunk;  // order in which a batch's refinement blocks take its units
    void *h_pinned2 = nullptr;
    size_t h_cap2 = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_compacted[2] = {}, ev_copy0[2] = {}, ev_copied[2] = {};

    // test helpers
    DBuf t_keys_alt, t_vals_alt, t_sort_tmp, t_scan_tmp;

    // semi-join query side
    DBuf q_xv, q_xs, q_ids, q_cell_of_row, q_cell_start, q_cell_key, q_nbr, q_nbr_cnt, q_bound, q_work_key, q_cell_idx,
        q_work;

    // exact kNN: per-batch pair scratch, done flags, active query ids
    DBuf k_keys, k_vals, k_keys_alt, k_vals_alt, k_sort_tmp, k_d2, k_prow, k_done, k_active;

    hiss_stats st{};
    cudaEvent_t ev[8] = {};
};

namespace {

constexpr double kCellMargin = 1.0 / 1024.0;  // cell side = eps (1 + 2^-10)
constexpr int kMortonBits = 21;
constexpr int kSubBitsMax = 5;
constexpr int kExtentBits = 20;

int fail_cuda(hiss_ctx *c, cudaError_t e)
{
    snprintf(c->cuda_err, sizeof(c->cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    c->sticky = HISS_E_CUDA;
    return HISS_E_CUDA;
}

#define CK(expr)                                          \
    do {                                                  \
        cudaError_t e__ = (expr);                         \
        if (e__ != cudaSuccess) return fail_cuda(ctx, e__); \
    } while (0)

#define ST(expr)                       \
    do {                               \
        int r__ = (expr);              \
        if (r__ != HISS_OK) return r__; \
    } while (0)

int enter(hiss_ctx *ctx)
{
    if (!ctx) return HISS_E_ARG;
    if (ctx->sticky) return HISS_E_STATE;
    cudaGetLastError();  // drop a stale non-sticky error left by an earlier runtime call
    cudaError_t e = cudaSetDevice(ctx->device);
    if (e != cudaSuccess) return fail_cuda(ctx, e);
    return HISS_OK;
}

// Grow-only device buffer on the context's stream.
int ensure(hiss_ctx *ctx, DBuf &b, size_t bytes)
{
    if (bytes == 0) bytes = 16;
    bytes = (bytes + 255) & ~(size_t)255;
    if (b.cap >= bytes) return HISS_OK;
    if (ctx->alloc_limit > 0 && ctx->alloc_held - (int64_t)b.cap + (int64_t)bytes > ctx->alloc_limit)
        return HISS_E_NOMEM;
    if (b.p) {
        CK(cudaFreeAsync(b.p, ctx->stream));
        ctx->alloc_held -= (int64_t)b.cap;
        b.p = nullptr;
        b.cap = 0;
    }
    cudaError_t e = cudaMallocAsync(&b.p, bytes, ctx->stream);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        b.p = nullptr;
        return HISS_E_NOMEM;
    }
    CK(e);
    b.cap = bytes;
    ctx->alloc_held += (int64_t)bytes;
    return HISS_OK;
}

void release(hiss_ctx *ctx, DBuf &b)
{
    if (b.p) cudaFreeAsync(b.p, ctx->stream);
    b.p = nullptr;
    b.cap = 0;
}

int sync(hiss_ctx *ctx)
{
    CK(cudaStreamSynchronize(ctx->stream));
    return HISS_OK;
}

float elapsed(hiss_ctx *ctx, int a, int b)
{
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, ctx->ev[a], ctx->ev[b]) != cudaSuccess) {
        cudaGetLastError();
        return 0.0f;
    }
    return ms;
}

int check_flags(hiss_ctx *ctx)
{
    int h[kNumFlags];
    CK(cudaMemcpyAsync(h, ctx->flags.p, sizeof(h), cudaMemcpyDeviceToHost, ctx->stream));
    ST(sync(ctx));
    if (h[kFlagSortTimeout]) {
        snprintf(ctx->cuda_err, sizeof(ctx->cuda_err), "radix sort look-back exceeded its wait limit");
        ctx->sticky = HISS_E_CUDA;
        return HISS_E_CUDA;
    }
    if (h[kFlagRefineTimeout]) {
        snprintf(ctx->cuda_err, sizeof(ctx->cuda_err), "refinement stage wait exceeded its limit");
        ctx->sticky = HISS_E_CUDA;
        return HISS_E_CUDA;
    }
    return HISS_OK;
}

int bit_length(int64_t v)
{
    int b = 0;
    while (v > 0) {
        ++b;
        v >>= 1;
    }
    return b;
}

// ---- build -------------------------------------------------------------------
int do_build(hiss_ctx *ctx, const float *d_points, int64_t n, int32_t d)
{
    ctx->built = false;
    ctx->grid_valid = false;
    ctx->tiles_valid = false;
    ctx->st = hiss_stats{};
    const int64_t launches0 = ctx->launches;
    CK(cudaEventRecord(ctx->ev[0], ctx->stream));
    const int d4 = (d + 3) & ~3;
    const int64_t nb = stats_blocks(n, d);
    ST(ensure(ctx, ctx->stats_partial, sizeof(double) * (size_t)nb * d * 4));
    ST(ensure(ctx, ctx->stats_out, sizeof(double) * 4 * (size_t)d + 16));
    ST(ensure(ctx, ctx->flags, sizeof(int) * kNumFlags * 2));
    CK(cudaMemsetAsync(ctx->flags.p, 0, sizeof(int) * kNumFlags * 2, ctx->stream));
    int *nonfinite_d = as<int>(ctx->flags) + kNumFlags;
    CK(dim_stats(d_points, n, d, as<double>(ctx->stats_partial), as<double>(ctx->stats_out), nonfinite_d,
                 ctx->stream, &ctx->launches));
    ctx->stats.assign(4 * (size_t)d, 0.0);
    int nonfinite = 0;
    CK(cudaMemcpyAsync(ctx->stats.data(), ctx->stats_out.p, sizeof(double) * 4 * d, cudaMemcpyDeviceToHost,
                       ctx->stream));
    CK(cudaMemcpyAsync(&nonfinite, nonfinite_d, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
    ST(sync(ctx));
    if (nonfinite) return HISS_E_ARG;

    // variance order, descending; equal variances keep the lower index first
    ctx->perm.resize(d);
    for (int k = 0; k < d; ++k) ctx->perm[k] = k;
    const double *var = ctx->stats.data() + 3 * (size_t)d;
    std::stable_sort(ctx->perm.begin(), ctx->perm.end(), [var](int a, int b) { return var[a] > var[b]; });

    ST(ensure(ctx, ctx->perm_d, sizeof(int32_t) * d));
    ST(ensure(ctx, ctx->xv, sizeof(float) * (size_t)n * d4));
    CK(cudaMemcpyAsync(ctx->perm_d.p, ctx->perm.data(), sizeof(int32_t) * d, cudaMemcpyHostToDevice, ctx->stream));
    CK(permute_pad(d_points, n, d, d4, as<int32_t>(ctx->perm_d), as<float>(ctx->xv), ctx->stream, &ctx->launches));
    CK(cudaEventRecord(ctx->ev[1], ctx->stream));
    ST(sync(ctx));
    ctx->n = n;
    ctx->d = d;
    ctx->d4 = d4;
    ctx->built = true;
    ctx->st.n = n;
    ctx->st.d = d;
    ctx->st.d_pad = d4;
    ctx->st.ms_build = elapsed(ctx, 0, 1);
    ctx->st.kernel_launches = ctx->launches - launches0;
    return HISS_OK;
}

// ---- grid index for eps --------------------------------------------------------
int ensure_grid(hiss_ctx *ctx, float eps)
{
    if (!ctx->built) return HISS_E_STATE;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    if (ctx->grid_valid && ctx->grid_eps == eps) return HISS_OK;
    ctx->grid_valid = false;
    ctx->tiles_valid = false;
    const int64_t n = ctx->n;
    const int d = ctx->d, d4 = ctx->d4;
    cudaStream_t s = ctx->stream;

    // grid parameters (fp64 on the host, identical to an fp64 reading)
    GridParams gp{};
    gp.ndim = d < 3 ? d : 3;
    double extent = 0.0, ext[3] = {0.0, 0.0, 0.0};
    for (int k = 0; k < gp.ndim; ++k) {
        const int dim = ctx->perm[k];
        const double mn = ctx->stats[0 * (size_t)d + dim], mx = ctx->stats[1 * (size_t)d + dim];
        gp.origin[k] = mn;
        ext[k] = mx - mn;
        extent = std::max(extent, ext[k]);
    }
    double w = std::max((double)eps * (1.0 + kCellMargin), std::ldexp(extent, -kExtentBits));
    if (w == 0.0) w = 1.0;
    gp.w = w;
    int64_t cellmax = 0;
    for (int k = 0; k < gp.ndim; ++k) cellmax = std::max(cellmax, (int64_t)std::floor(ext[k] / w));
    const int cellbits = bit_length(cellmax);
    gp.sub_bits = std::min(kSubBitsMax, kMortonBits - cellbits);
    gp.key_bits = 3 * (cellbits + gp.sub_bits);

    CK(cudaEventRecord(ctx->ev[0], s));
    ST(ensure(ctx, ctx->keys, 8 * (size_t)n));
    ST(ensure(ctx, ctx->vals, 4 * (size_t)n));
    ST(ensure(ctx, ctx->keys_alt, 8 * (size_t)n));
    ST(ensure(ctx, ctx->vals_alt, 4 * (size_t)n));
    ST(ensure(ctx, ctx->sort_tmp, sort_tmp_bytes(n)));
    ST(ensure(ctx, ctx->xs, sizeof(float) * (size_t)n * d4));
    ST(ensure(ctx, ctx->ids, 4 * (size_t)n));
    ST(ensure(ctx, ctx->flag, 4 * (size_t)n));
    ST(ensure(ctx, ctx->flag_scan, 4 * (size_t)(n + 1)));
    ST(ensure(ctx, ctx->cell_of_row, 4 * (size_t)n));
    ST(ensure(ctx, ctx->scan_tmp, 8 * (size_t)scan_tmp_elems(n + 1) + 64));

    CK(cell_keys(as<float>(ctx->xv), n, d4, gp, as<uint64_t>(ctx->keys), as<uint32_t>(ctx->vals), s,
                 &ctx->launches));
    int in_alt = 0;
    CK(sort_pairs(as<uint64_t>(ctx->keys), as<uint32_t>(ctx->vals), as<uint64_t>(ctx->keys_alt),
                  as<uint32_t>(ctx->vals_alt), n, gp.key_bits, ctx->sort_tmp.p, as<int>(ctx->flags), s,
                  &ctx->launches, &in_alt));
    ctx->sorted_keys = in_alt ? as<uint64_t>(ctx->keys_alt) : as<uint64_t>(ctx->keys);
    ctx->sorted_vals = in_alt ? as<uint32_t>(ctx->vals_alt) : as<uint32_t>(ctx->vals);
    CK(gather_rows(as<float>(ctx->xv), ctx->sorted_vals, n, d4, as<float>(ctx->xs), as<int32_t>(ctx->ids), s,
                   &ctx->launches));
    ST(ensure(ctx, ctx->gbox, 32 * (size_t)((n + 31) / 32) + 32));
    CK(group_boxes(as<float>(ctx->xs), n, d4, as<float4>(ctx->gbox), s, &ctx->launches));
    const int shift = 3 * gp.sub_bits;
    CK(cell_flags(ctx->sorted_keys, n, shift, as<int32_t>(ctx->flag), s, &ctx->launches));
    CK(scan_i32(as<int32_t>(ctx->flag), as<int32_t>(ctx->flag_scan), n, as<int64_t>(ctx->scan_tmp), s,
                &ctx->launches));
    int32_t C32 = 0;
    CK(cudaMemcpyAsync(&C32, as<int32_t>(ctx->flag_scan) + n, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ST(check_flags(ctx));
    const int64_t C = C32;

    ST(ensure(ctx, ctx->cell_start, 4 * (size_t)(C + 1)));
    ST(ensure(ctx, ctx->cell_key, 8 * (size_t)C));
    ST(ensure(ctx, ctx->nbr, 4 * (size_t)C * kStencil));
    ST(ensure(ctx, ctx->nbr_cnt, 4 * (size_t)(C + 1)));
    ST(ensure(ctx, ctx->bound, 8 * (size_t)(C + 1)));
    ST(ensure(ctx, ctx->work_key, 8 * (size_t)C));
    ST(ensure(ctx, ctx->cell_idx, 4 * (size_t)C));
    ST(ensure(ctx, ctx->work, 8 * (size_t)(C + 1)));
    ST(ensure(ctx, ctx->sums2, 8 * (size_t)(C + 1)));
    CK(cell_starts(ctx->sorted_keys, as<int32_t>(ctx->flag_scan), n, shift, as<int32_t>(ctx->cell_start),
                   as<uint64_t>(ctx->cell_key), as<int32_t>(ctx->cell_of_row), s, &ctx->launches));
    CK(stencil(as<uint64_t>(ctx->cell_key), as<int32_t>(ctx->cell_start), C, as<int32_t>(ctx->nbr),
               as<int32_t>(ctx->nbr_cnt), as<int64_t>(ctx->bound), as<uint64_t>(ctx->work_key),
               as<uint32_t>(ctx->cell_idx), as<int64_t>(ctx->work), s, &ctx->launches));
    // totals: candidates = sum |cell| B_cell, cell pairs = sum of stencil sizes
    CK(scan_i64(as<int64_t>(ctx->work), as<int64_t>(ctx->sums2), C, as<int64_t>(ctx->scan_tmp), s, &ctx->launches));
    int64_t tot[2] = {0, 0};
    CK(cudaMemcpyAsync(&tot[0], as<int64_t>(ctx->sums2) + C, 8, cudaMemcpyDeviceToHost, s));
    CK(scan_i32_to_i64(as<int32_t>(ctx->nbr_cnt), as<int64_t>(ctx->sums2), C, as<int64_t>(ctx->scan_tmp), s,
                       &ctx->launches));
    CK(cudaMemcpyAsync(&tot[1], as<int64_t>(ctx->sums2) + C, 8, cudaMemcpyDeviceToHost, s));
    CK(cudaEventRecord(ctx->ev[1], s));
    ST(sync(ctx));

    ctx->gp = gp;
    ctx->C = C;
    ctx->candidates = tot[0];
    ctx->cell_pairs = tot[1];
    ctx->grid_eps = eps;
    ctx->grid_valid = true;
    ctx->st.ms_index = elapsed(ctx, 0, 1);
    return HISS_OK;
}

void fill_grid_stats(hiss_ctx *ctx)
{
    ctx->st.n = ctx->n;
    ctx->st.d = ctx->d;
    ctx->st.d_pad = ctx->d4;
    ctx->st.cells = ctx->C;
    ctx->st.cell_pairs = ctx->cell_pairs;
    ctx->st.candidates = ctx->candidates;
    ctx->st.sub_bits = ctx->gp.sub_bits;
    ctx->st.key_bits = ctx->gp.key_bits;
    ctx->st.cell_width = ctx->gp.w;
    ctx->st.eps = ctx->grid_eps;
}

}  // namespace

namespace {

// The query side of a join: query rows and ids (index order) and the query
// cells with their stencils among the data's cells.  For the self-join it is
// the data's own index; for the semi-join it is built from the queries.
struct QuerySide {
    const float *xq;
    const int32_t *qids;
    int64_t C;                  // query cells
    const int32_t *qcell_start; // [C+1] first query row of each query cell
    const int32_t *nbr;         // [C*27] data cells of each query cell's stencil
    const int32_t *nbr_cnt;     // [C]
    const int64_t *bound;       // [C] candidates of each query cell
    const uint64_t *work_key;   // [C] ~(|cell| * bound)
    const uint32_t *cell_idx;   // [C] 0 .. C-1
};

QuerySide self_side(hiss_ctx *ctx)
{
    QuerySide q;
    q.xq = as<float>(ctx->xs);
    q.qids = as<int32_t>(ctx->ids);
    q.C = ctx->C;
    q.qcell_start = as<int32_t>(ctx->cell_start);
    q.nbr = as<int32_t>(ctx->nbr);
    q.nbr_cnt = as<int32_t>(ctx->nbr_cnt);
    q.bound = as<int64_t>(ctx->bound);
    q.work_key = as<uint64_t>(ctx->work_key);
    q.cell_idx = as<uint32_t>(ctx->cell_idx);
    return q;
}

// The refinement a join runs: the tensor-core one when selected and the
// dimension fits it, else the CUDA-core one.
bool use_tc(const hiss_ctx *ctx)
{
    return ctx->refine_mode == HISS_REFINE_TENSOR_CORES && ctx->d4 <= refine_tc_max_d4();
}

// ---- query tiles in processing order (largest work first) ------------------------
int build_tiles(hiss_ctx *ctx, const QuerySide &qs, bool tc)
{
    cudaStream_t s = ctx->stream;
    const int64_t C = qs.C;
    const int tq = tc ? refine_tc_tq() : refine_tq(ctx->d4);
    const int chunk = tc ? refine_tc_chunk() : refine_chunk(ctx->d4);
    ST(ensure(ctx, ctx->lpt_keys, 8 * (size_t)C));
    ST(ensure(ctx, ctx->lpt_order, 4 * (size_t)C));
    ST(ensure(ctx, ctx->ntiles, 4 * (size_t)C));
    ST(ensure(ctx, ctx->tile_off, 8 * (size_t)(C + 1)));
    ST(ensure(ctx, ctx->sort_tmp, sort_tmp_bytes(C)));
    ST(ensure(ctx, ctx->scan_tmp, 8 * (size_t)scan_tmp_elems(C + 1) + 64));
    // the work keys are consumed by the sort; copy them so the index stays intact
    CK(cudaMemcpyAsync(ctx->lpt_keys.p, qs.work_key, 8 * (size_t)C, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(ctx->lpt_order.p, qs.cell_idx, 4 * (size_t)C, cudaMemcpyDeviceToDevice, s));
    int in_alt = 0;
    ST(ensure(ctx, ctx->keys_alt, 8 * (size_t)C));
    ST(ensure(ctx, ctx->vals_alt, 4 * (size_t)C));
    CK(sort_pairs(as<uint64_t>(ctx->lpt_keys), as<uint32_t>(ctx->lpt_order), as<uint64_t>(ctx->keys_alt),
                  as<uint32_t>(ctx->vals_alt), C, 64, ctx->sort_tmp.p, as<int>(ctx->flags), s, &ctx->launches,
                  &in_alt));
    if (in_alt)
        CK(cudaMemcpyAsync(ctx->lpt_order.p, ctx->vals_alt.p, 4 * (size_t)C, cudaMemcpyDeviceToDevice, s));
    ctx->order = as<uint32_t>(ctx->lpt_order);
    // keys_alt / vals_alt held the sorted grid keys: the index keeps only the
    // gathered points, ids and cell arrays, so they are free to reuse here.
    ctx->sorted_keys = nullptr;
    ctx->sorted_vals = nullptr;

    CK(tile_counts(ctx->order, qs.qcell_start, C, tq, as<int32_t>(ctx->ntiles), s, &ctx->launches));
    CK(scan_i32_to_i64(as<int32_t>(ctx->ntiles), as<int64_t>(ctx->tile_off), C, as<int64_t>(ctx->scan_tmp), s,
                       &ctx->launches));
    int64_t T = 0;
    CK(cudaMemcpyAsync(&T, as<int64_t>(ctx->tile_off) + C, 8, cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ST(check_flags(ctx));
    ST(ensure(ctx, ctx->tile_cell, 4 * (size_t)T));
    ST(ensure(ctx, ctx->tile_q0, 4 * (size_t)T));
    ST(ensure(ctx, ctx->tile_nq, 4 * (size_t)(T + 1)));
    ST(ensure(ctx, ctx->tile_word, 8 * (size_t)(T + 1)));
    ST(ensure(ctx, ctx->tile_unit, 8 * (size_t)(T + 1)));
    ST(ensure(ctx, ctx->tile_qoff, 8 * (size_t)(T + 1)));
    ST(ensure(ctx, ctx->scan_tmp, 8 * (size_t)scan_tmp_elems(T + 1) + 64));
    CK(tile_fill(ctx->order, qs.qcell_start, qs.bound, as<int64_t>(ctx->tile_off), C, tq, chunk,
                 as<int32_t>(ctx->tile_cell), as<int32_t>(ctx->tile_q0), as<int32_t>(ctx->tile_nq),
                 as<int64_t>(ctx->tile_word), as<int64_t>(ctx->tile_unit), s, &ctx->launches));
    CK(scan_i64(as<int64_t>(ctx->tile_word), as<int64_t>(ctx->tile_word), T, as<int64_t>(ctx->scan_tmp), s,
                &ctx->launches));
    CK(scan_i64(as<int64_t>(ctx->tile_unit), as<int64_t>(ctx->tile_unit), T, as<int64_t>(ctx->scan_tmp), s,
                &ctx->launches));
    CK(scan_i32_to_i64(as<int32_t>(ctx->tile_nq), as<int64_t>(ctx->tile_qoff), T, as<int64_t>(ctx->scan_tmp), s,
                       &ctx->launches));
    int64_t tot[2] = {0, 0};
    CK(cudaMemcpyAsync(&tot[0], as<int64_t>(ctx->tile_word) + T, 8, cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(&tot[1], as<int64_t>(ctx->tile_unit) + T, 8, cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ctx->T = T;
    ctx->total_words = tot[0];
    ctx->total_units = tot[1];
    return HISS_OK;
}

// Tiles of the self-join, cached with the index.
int ensure_tiles(hiss_ctx *ctx, bool tc)
{
    if (ctx->tiles_valid && ctx->tiles_tc == (int)tc) return HISS_OK;
    ctx->tiles_valid = false;
    ST(build_tiles(ctx, self_side(ctx), tc));
    ctx->tiles_valid = true;
    ctx->tiles_tc = (int)tc;
    return HISS_OK;
}

int ensure_pinned_slot(void *&ptr, size_t &cap, size_t bytes)
{
    if (cap >= bytes) return HISS_OK;
    if (ptr) cudaFreeHost(ptr);
    ptr = nullptr;
    cap = 0;
    cudaError_t e = cudaMallocHost(&ptr, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ptr = nullptr;
        return HISS_E_NOMEM;
    }
    cap = bytes;
    return HISS_OK;
}

int ensure_pinned(hiss_ctx *ctx, size_t bytes) { return ensure_pinned_slot(ctx->h_pinned, ctx->h_cap, bytes); }

// The copy stream and events of the overlapped host delivery.
int ensure_copy_stream(hiss_ctx *ctx)
{
    if (ctx->copy_stream) return HISS_OK;
    CK(cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
        CK(cudaEventCreateWithFlags(&ctx->ev_compacted[i], cudaEventDisableTiming));
        CK(cudaEventCreate(&ctx->ev_copy0[i]));
        CK(cudaEventCreate(&ctx->ev_copied[i]));
    }
    return HISS_OK;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Above 32 dimensions the refinement blocks take a batch's units chunk by
// chunk within each cell (unit_order) rather than tile by tile, so that
// blocks running together read the same candidate rows (which the
// survivors re-read from global memory).  Measured on GB300: subspace (d4 =
// 64) 2.44 -> 2.35 s, spectrum (d4 = 128) 385 -> 366 ms; gmm (d4 = 32) no
// change; exp (d4 = 16) 12.91 -> 13.14 s, so builds up to 32 dimensions keep
// the tile order.
#ifndef HISS_UNIT_ORDER_MIN_D4
#define HISS_UNIT_ORDER_MIN_D4 33
#endif
bool chunk_major(int d4) { return d4 >= HISS_UNIT_ORDER_MIN_D4; }

// Plan the batches over the current tiles and run them: refinement,
// compaction, delivery and the callback, batch by batch.
// tlo, thi: the query tiles (processing order) to run; thi < 0 means all.
int run_batches(hiss_ctx *ctx, const QuerySide &qs, float eps, size_t batch_bytes, const hiss_out *out,
                double ms_index, int64_t launches0, int64_t tlo = 0, int64_t thi = -1)
{
    const int mode = out ? out->mode : HISS_OUT_CSR;
    const int to_host = out ? out->copy_to_host : 0;
    const bool tc = use_tc(ctx);  // the tiles were cut for this refinement
    // CSR to host: batch b's copies run on the copy stream while batch b + 1
    // is refined; outputs and pinned staging alternate between two slots
    const bool ov = to_host && mode == HISS_OUT_CSR;
    hiss_batch_fn fn = out ? out->on_batch : nullptr;
    void *user = out ? out->user : nullptr;
    cudaStream_t s = ctx->stream;
    if (batch_bytes == 0) {
        size_t fr = 0, tot = 0;
        CK(cudaMemGetInfo(&fr, &tot));
        batch_bytes = fr / 4;
    }
    // batch_bytes bounds a batch's device memory.  The planner fits the mask,
    // its occupancy bitmap and the per-query arrays (counts, row offsets, ids;
    // doubled for the overlapped host delivery) in three quarters of it; the
    // CSR columns get the rest.  A batch whose result outgrows that is
    // compacted and delivered in several parts (RT-HiSS Section IV-D sizes
    // batches so that their results fit in device memory).
    const int64_t per_query_words = (24 + (mode == HISS_OUT_MASK ? 16 : 0) + (ov ? 20 : 0)) / 4;
    const int64_t budget_words = (int64_t)(batch_bytes / 4);
    const int64_t cap_words = budget_words - budget_words / 4;
    if (thi < 0) thi = ctx->T;
    const int64_t T = thi - tlo;  // tiles of this call; batch tile indices are relative to tlo
    ST(ensure(ctx, ctx->boundaries, 8 * (size_t)(T + 2)));
    ST(ensure(ctx, ctx->binfo, 32 * (size_t)(T + 2)));
    ST(ensure(ctx, ctx->nb_d, 64));
    CK(cudaMemsetAsync(ctx->flags.p, 0, sizeof(int) * kNumFlags, s));
    CK(plan_batches(as<int64_t>(ctx->tile_word) + tlo, as<int64_t>(ctx->tile_unit) + tlo,
                    as<int64_t>(ctx->tile_qoff) + tlo, T, cap_words, per_query_words, as<int64_t>(ctx->boundaries),
                    as<int64_t>(ctx->binfo), as<int64_t>(ctx->nb_d), as<int>(ctx->flags), s, &ctx->launches));
    int64_t nb = 0;
    int hflags[kNumFlags];
    CK(cudaMemcpyAsync(&nb, ctx->nb_d.p, 8, cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(hflags, ctx->flags.p, sizeof(hflags), cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    if (hflags[kFlagPlanTooSmall]) return HISS_E_BATCH_TOO_SMALL;
    std::vector<int64_t> info(4 * (size_t)(nb + 1));
    CK(cudaMemcpyAsync(info.data(), ctx->binfo.p, 32 * (size_t)(nb + 1), cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));

    int64_t max_words = 0, max_nq = 0, max_cost = 0, max_units = 0;
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t dw = info[4 * (b + 1)] - info[4 * b], dq = info[4 * (b + 1) + 2] - info[4 * b + 2];
        max_words = std::max(max_words, dw);
        max_nq = std::max(max_nq, dq);
        max_cost = std::max(max_cost, dw + (dw >> 5) + 2 + per_query_words * dq);
        max_units = std::max(max_units, info[4 * (b + 1) + 1] - info[4 * b + 1]);
    }
    if (!tc && chunk_major(ctx->d4)) {
        ST(ensure(ctx, ctx->unit_tile, 4 * (size_t)max_units));
        ST(ensure(ctx, ctx->unit_chunk, 4 * (size_t)max_units));
    }
    // CSR columns per delivery (per slot with the overlapped delivery)
    const int64_t cols_cap = std::max<int64_t>(1, (budget_words - max_cost) / (ov ? 2 : 1));
    ST(ensure(ctx, ctx->mask, 4 * (size_t)max_words));
    ST(ensure(ctx, ctx->occ, 4 * (size_t)(max_words / 32 + 2)));
    ST(ensure(ctx, ctx->qcount, 4 * (size_t)(max_nq + 1)));
    ST(ensure(ctx, ctx->row_ptr, 8 * (size_t)(max_nq + 1)));
    ST(ensure(ctx, ctx->query_ids, 8 * (size_t)max_nq));
    ST(ensure(ctx, ctx->query_rows, 4 * (size_t)max_nq));
    ST(ensure(ctx, ctx->scan_tmp, 8 * (size_t)scan_tmp_elems(max_nq + 1) + 64));
    if (mode == HISS_OUT_MASK) {
        ST(ensure(ctx, ctx->cand, 8 * (size_t)max_nq));
        ST(ensure(ctx, ctx->mask_row_ptr, 8 * (size_t)(max_nq + 1)));
    }
    if (ov) {
        ST(ensure_copy_stream(ctx));
        ST(ensure(ctx, ctx->row_ptr2, 8 * (size_t)(max_nq + 1)));
        ST(ensure(ctx, ctx->query_ids2, 8 * (size_t)max_nq));
        ST(ensure(ctx, ctx->query_rows2, 4 * (size_t)max_nq));
    }
    int64_t pending = -1;  // overlapped delivery: batch whose copies are in flight
    int pslot = 0;
    hiss_batch pending_hb{};

    double ms_refine = 0.0, ms_compact = 0.0, ms_deliver = 0.0;
    int64_t pairs = 0, delivered = 0;
    // candidate pairs of the staged tiles the CUDA-core refinement keeps,
    // summed over the batches on the device (nb_d[4])
    unsigned long long *kept_d = reinterpret_cast<unsigned long long *>(as<int64_t>(ctx->nb_d) + 4);
    CK(cudaMemsetAsync(kept_d, 0, 8, s));
    // Hands over the overlapped delivery still in flight, if any.
    auto flush_pending = [&]() -> int {
        if (pending < 0) return HISS_OK;
        CK(cudaEventSynchronize(ctx->ev_copied[pslot]));
        float cms = 0.0f;
        if (cudaEventElapsedTime(&cms, ctx->ev_copy0[pslot], ctx->ev_copied[pslot]) == cudaSuccess) ms_deliver += cms;
        cudaGetLastError();
        pending = -1;
        if (fn && fn(user, &pending_hb) != 0) return HISS_E_CALLBACK;
        return HISS_OK;
    };
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t *lo = &info[4 * b], *hi = &info[4 * (b + 1)];
        const int64_t nq = hi[2] - lo[2];
        const int64_t nwords = hi[0] - lo[0];
        const int slot = ov ? (int)(b & 1) : 0;
        DBuf &rp_buf = slot ? ctx->row_ptr2 : ctx->row_ptr;
        DBuf &cols_buf = slot ? ctx->cols2 : ctx->cols;
        DBuf &qid_buf = slot ? ctx->query_ids2 : ctx->query_ids;
        DBuf &qrow_buf = slot ? ctx->query_rows2 : ctx->query_rows;
        CK(cudaMemsetAsync(ctx->qcount.p, 0, 4 * (size_t)nq, s));
        // the refinement stores only nonzero mask words and marks them in occ;
        // the raw-mask output needs the zero words too
        CK(cudaMemsetAsync(ctx->occ.p, 0, 4 * (size_t)(nwords / 32 + 2), s));
        if (mode == HISS_OUT_MASK) CK(cudaMemsetAsync(ctx->mask.p, 0, 4 * (size_t)nwords, s));
        RefineArgs ra{};
        ra.xs = as<float>(ctx->xs);
        ra.xq = qs.xq;
        ra.cell_start = as<int32_t>(ctx->cell_start);
        ra.nbr = qs.nbr;
        ra.nbr_cnt = qs.nbr_cnt;
        ra.bound = qs.bound;
        ra.tile_cell = as<int32_t>(ctx->tile_cell);
        ra.tile_q0 = as<int32_t>(ctx->tile_q0);
        ra.tile_nq = as<int32_t>(ctx->tile_nq);
        ra.tile_word = as<int64_t>(ctx->tile_word);
        ra.tile_unit = as<int64_t>(ctx->tile_unit);
        ra.tile_qoff = as<int64_t>(ctx->tile_qoff);
        ra.t0 = tlo + lo[3];
        ra.t1 = tlo + hi[3];
        ra.unit0 = lo[1];
        ra.nunits = hi[1] - lo[1];
        ra.word0 = lo[0];
        ra.q0 = lo[2];
        ra.mask = as<uint32_t>(ctx->mask);
        ra.occ = as<uint32_t>(ctx->occ);
        ra.qcount = as<int32_t>(ctx->qcount);
        ra.d4 = ctx->d4;
        ra.d = ctx->d;
        ra.eps2 = eps * eps;
        ra.prof = nullptr;
        ra.gbox = as<float4>(ctx->gbox);
        ra.kept = kept_d;
        ra.flags = as<int>(ctx->flags);
        if (!tc && chunk_major(ctx->d4)) {
            CK(unit_order(ra, qs.qcell_start, refine_tq(ctx->d4), as<int32_t>(ctx->unit_tile),
                          as<int32_t>(ctx->unit_chunk), s, &ctx->launches));
            ra.unit_tile = as<int32_t>(ctx->unit_tile);
            ra.unit_chunk = as<int32_t>(ctx->unit_chunk);
        }
        CK(cudaEventRecord(ctx->ev[4], s));
        if (tc) CK(refine_tc(ra, eps, s, &ctx->launches));
        else CK(refine(ra, s, &ctx->launches));
        CK(cudaEventRecord(ctx->ev[5], s));

        CompactArgs ca{};
        ca.ids = as<int32_t>(ctx->ids);
        ca.qids = qs.qids;
        ca.cell_start = ra.cell_start;
        ca.nbr = ra.nbr;
        ca.nbr_cnt = ra.nbr_cnt;
        ca.bound = ra.bound;
        ca.tile_cell = ra.tile_cell;
        ca.tile_q0 = ra.tile_q0;
        ca.tile_word = ra.tile_word;
        ca.tile_qoff = ra.tile_qoff;
        ca.t0 = ra.t0;
        ca.t1 = ra.t1;
        ca.word0 = ra.word0;
        ca.q0 = ra.q0;
        ca.nq = nq;
        ca.mask = ra.mask;
        ca.occ = ra.occ;
        ca.query_ids = as<int64_t>(qid_buf);
        ca.query_rows = as<int32_t>(qrow_buf);
        int64_t nnz = 0;
        CK(scan_i32_to_i64(as<int32_t>(ctx->qcount), as<int64_t>(rp_buf), nq, as<int64_t>(ctx->scan_tmp), s,
                           &ctx->launches));
        CK(cudaMemcpyAsync(&nnz, as<int64_t>(rp_buf) + nq, 8, cudaMemcpyDeviceToHost, s));
        ST(sync(ctx));
        if (mode == HISS_OUT_CSR && nnz > cols_cap) {
            // The batch's result does not fit its CSR budget: compact and
            // deliver it in parts of consecutive queries, each within the
            // budget, one after another on the context's stream.
            ST(flush_pending());
            std::vector<int64_t> rph((size_t)nq + 1);
            CK(cudaMemcpyAsync(rph.data(), rp_buf.p, 8 * (size_t)(nq + 1), cudaMemcpyDeviceToHost, s));
            ST(sync(ctx));
            ms_refine += elapsed(ctx, 4, 5);
            ST(ensure(ctx, ctx->cols, 4 * (size_t)cols_cap));
            ST(ensure(ctx, ctx->row_ptr_sub, 8 * (size_t)(max_nq + 1)));
            for (int64_t q = 0; q < nq;) {
                int64_t e = q + 1;
                if (rph[e] - rph[q] > cols_cap) return HISS_E_BATCH_TOO_SMALL;  // one row alone is larger
                e = std::upper_bound(rph.begin() + e, rph.end(), rph[q] + cols_cap) - rph.begin() - 1;
                const int64_t nsub = e - q, nnz_sub = rph[e] - rph[q];
                CompactArgs cs = ca;
                cs.q0 = ca.q0 + q;
                cs.nq = nsub;
                cs.row_ptr = as<int64_t>(rp_buf) + q;
                cs.col0 = rph[q];
                cs.row_ptr_out = as<int64_t>(ctx->row_ptr_sub);
                cs.cols = as<int32_t>(ctx->cols);
                cs.query_ids = as<int64_t>(ctx->query_ids);
                cs.query_rows = as<int32_t>(ctx->query_rows);
                CK(cudaEventRecord(ctx->ev[5], s));
                CK(compact(cs, s, &ctx->launches));
                CK(cudaEventRecord(ctx->ev[6], s));
                hiss_batch hb{};
                hb.index = delivered++;
                hb.nq = nsub;
                hb.nnz = nnz_sub;
                hb.mode = mode;
                if (to_host) {
                    const size_t o_ids = 0, o_rp = align256(8 * nsub), o_rows = o_rp + align256(8 * (nsub + 1));
                    const size_t o_data = o_rows + align256(4 * nsub);
                    ST(ensure_pinned(ctx, o_data + 4 * (size_t)nnz_sub + 256));
                    char *h = static_cast<char *>(ctx->h_pinned);
                    CK(cudaMemcpyAsync(h + o_ids, ctx->query_ids.p, 8 * nsub, cudaMemcpyDeviceToHost, s));
                    CK(cudaMemcpyAsync(h + o_rows, ctx->query_rows.p, 4 * nsub, cudaMemcpyDeviceToHost, s));
                    CK(cudaMemcpyAsync(h + o_rp, ctx->row_ptr_sub.p, 8 * (nsub + 1), cudaMemcpyDeviceToHost, s));
                    CK(cudaMemcpyAsync(h + o_data, ctx->cols.p, 4 * (size_t)nnz_sub, cudaMemcpyDeviceToHost, s));
                    hb.query_ids = reinterpret_cast<const int64_t *>(h + o_ids);
                    hb.row_ptr = reinterpret_cast<const int64_t *>(h + o_rp);
                    hb.query_rows = reinterpret_cast<const int32_t *>(h + o_rows);
                    hb.cols = reinterpret_cast<const int32_t *>(h + o_data);
                    hb.on_host = 1;
                } else {
                    hb.query_ids = as<int64_t>(ctx->query_ids);
                    hb.row_ptr = as<int64_t>(ctx->row_ptr_sub);
                    hb.query_rows = as<int32_t>(ctx->query_rows);
                    hb.cols = as<int32_t>(ctx->cols);
                }
                CK(cudaEventRecord(ctx->ev[7], s));
                ST(sync(ctx));
                ms_compact += elapsed(ctx, 5, 6);
                ms_deliver += elapsed(ctx, 6, 7);
                if (fn && fn(user, &hb) != 0) return HISS_E_CALLBACK;
                q = e;
            }
            pairs += nnz;
            continue;
        }
        if (mode == HISS_OUT_CSR) {
            ST(ensure(ctx, cols_buf, 4 * (size_t)nnz));
            ca.row_ptr = as<int64_t>(rp_buf);
            ca.cols = as<int32_t>(cols_buf);
        } else {
            ca.cand = as<int64_t>(ctx->cand);
            ca.mask_row_ptr = as<int64_t>(ctx->mask_row_ptr);
        }
        CK(compact(ca, s, &ctx->launches));
        CK(cudaEventRecord(ctx->ev[6], s));

        hiss_batch hb{};
        hb.index = delivered++;
        hb.nq = nq;
        hb.nnz = nnz;
        hb.mode = mode;
        hb.n_words = mode == HISS_OUT_MASK ? nwords : 0;
        if (ov) {
            const size_t o_ids = 0, o_rp = align256(8 * nq), o_rows = o_rp + align256(8 * (nq + 1));
            const size_t o_data = o_rows + align256(4 * nq);
            const size_t bytes = o_data + 4 * (size_t)nnz + 256;
            void *&hp = slot ? ctx->h_pinned2 : ctx->h_pinned;
            size_t &hc = slot ? ctx->h_cap2 : ctx->h_cap;
            ST(ensure_pinned_slot(hp, hc, bytes));
            char *h = static_cast<char *>(hp);
            cudaStream_t cs = ctx->copy_stream;
            CK(cudaEventRecord(ctx->ev_compacted[slot], s));
            CK(cudaStreamWaitEvent(cs, ctx->ev_compacted[slot], 0));
            CK(cudaEventRecord(ctx->ev_copy0[slot], cs));
            CK(cudaMemcpyAsync(h + o_ids, qid_buf.p, 8 * nq, cudaMemcpyDeviceToHost, cs));
            CK(cudaMemcpyAsync(h + o_rows, qrow_buf.p, 4 * nq, cudaMemcpyDeviceToHost, cs));
            CK(cudaMemcpyAsync(h + o_rp, rp_buf.p, 8 * (nq + 1), cudaMemcpyDeviceToHost, cs));
            CK(cudaMemcpyAsync(h + o_data, cols_buf.p, 4 * (size_t)nnz, cudaMemcpyDeviceToHost, cs));
            CK(cudaEventRecord(ctx->ev_copied[slot], cs));
            hb.query_ids = reinterpret_cast<const int64_t *>(h + o_ids);
            hb.row_ptr = reinterpret_cast<const int64_t *>(h + o_rp);
            hb.query_rows = reinterpret_cast<const int32_t *>(h + o_rows);
            hb.cols = reinterpret_cast<const int32_t *>(h + o_data);
            hb.on_host = 1;
            // hand over the previous batch, whose copies ran during this batch's refinement
            if (pending >= 0) {
                const int r = flush_pending();
                if (r != HISS_OK) {
                    cudaStreamSynchronize(cs);
                    return r;
                }
            }
            ST(sync(ctx));
            ms_refine += elapsed(ctx, 4, 5);
            ms_compact += elapsed(ctx, 5, 6);
            pairs += nnz;
            pending = b;
            pslot = slot;
            pending_hb = hb;
            continue;
        }
        if (to_host) {
            const size_t o_ids = 0, o_rp = align256(8 * nq), o_rows = o_rp + align256(8 * (nq + 1));
            const size_t o_cand = o_rows + align256(4 * nq), o_data = o_cand + align256(8 * nq);
            const size_t bytes = o_data + (mode == HISS_OUT_CSR ? 4 * (size_t)nnz : 4 * (size_t)nwords) + 256;
            ST(ensure_pinned(ctx, bytes));
            char *h = static_cast<char *>(ctx->h_pinned);
            CK(cudaMemcpyAsync(h + o_ids, ctx->query_ids.p, 8 * nq, cudaMemcpyDeviceToHost, s));
            CK(cudaMemcpyAsync(h + o_rows, ctx->query_rows.p, 4 * nq, cudaMemcpyDeviceToHost, s));
            if (mode == HISS_OUT_CSR) {
                CK(cudaMemcpyAsync(h + o_rp, ctx->row_ptr.p, 8 * (nq + 1), cudaMemcpyDeviceToHost, s));
                CK(cudaMemcpyAsync(h + o_data, ctx->cols.p, 4 * (size_t)nnz, cudaMemcpyDeviceToHost, s));
                hb.cols = reinterpret_cast<const int32_t *>(h + o_data);
            } else {
                CK(cudaMemcpyAsync(h + o_rp, ctx->mask_row_ptr.p, 8 * (nq + 1), cudaMemcpyDeviceToHost, s));
                CK(cudaMemcpyAsync(h + o_cand, ctx->cand.p, 8 * nq, cudaMemcpyDeviceToHost, s));
                CK(cudaMemcpyAsync(h + o_data, ctx->mask.p, 4 * (size_t)nwords, cudaMemcpyDeviceToHost, s));
                hb.mask = reinterpret_cast<const uint32_t *>(h + o_data);
                hb.cand = reinterpret_cast<const int64_t *>(h + o_cand);
            }
            hb.query_ids = reinterpret_cast<const int64_t *>(h + o_ids);
            hb.row_ptr = reinterpret_cast<const int64_t *>(h + o_rp);
            hb.query_rows = reinterpret_cast<const int32_t *>(h + o_rows);
            hb.on_host = 1;
        } else {
            hb.query_ids = as<int64_t>(ctx->query_ids);
            hb.query_rows = as<int32_t>(ctx->query_rows);
            if (mode == HISS_OUT_CSR) {
                hb.row_ptr = as<int64_t>(ctx->row_ptr);
                hb.cols = as<int32_t>(ctx->cols);
            } else {
                hb.row_ptr = as<int64_t>(ctx->mask_row_ptr);
                hb.mask = as<uint32_t>(ctx->mask);
                hb.cand = as<int64_t>(ctx->cand);
            }
        }
        CK(cudaEventRecord(ctx->ev[7], s));
        ST(sync(ctx));
        ms_refine += elapsed(ctx, 4, 5);
        ms_compact += elapsed(ctx, 5, 6);
        ms_deliver += elapsed(ctx, 6, 7);
        pairs += nnz;
        if (fn && fn(user, &hb) != 0) return HISS_E_CALLBACK;
    }
    ST(flush_pending());
    ST(check_flags(ctx));
    int64_t kept = 0;
    CK(cudaMemcpyAsync(&kept, kept_d, 8, cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ctx->st.candidates_refined = tc ? -1 : kept;
    ctx->st.pairs = mode == HISS_OUT_CSR ? pairs : -1;
    ctx->st.batches = nb;
    ctx->st.deliveries = delivered;
    ctx->st.query_tiles = T;
    ctx->st.refine_units = info[4 * (size_t)nb + 1] - info[1];
    ctx->st.mask_words_max = max_words;
    ctx->st.ms_index = ms_index;
    ctx->st.ms_count = elapsed(ctx, 2, 3);
    ctx->st.ms_refine = ms_refine;
    ctx->st.ms_compact = ms_compact;
    ctx->st.ms_deliver = ms_deliver;
    ctx->st.ms_total = ms_index + ctx->st.ms_count + ms_refine + ms_compact + ms_deliver;
    ctx->st.kernel_launches = ctx->launches - launches0;
    return HISS_OK;
}


// rank / nranks: run only the rank-th of nranks contiguous ranges of the
// query tiles in processing order, balanced by refinement units.
int do_join(hiss_ctx *ctx, float eps, size_t batch_bytes, const hiss_out *out, int32_t rank = 0, int32_t nranks = 1)
{
    const int mode = out ? out->mode : HISS_OUT_CSR;
    if (mode != HISS_OUT_CSR && mode != HISS_OUT_MASK) return HISS_E_ARG;
    cudaStream_t s = ctx->stream;
    const int64_t launches0 = ctx->launches;
    double ms_index = 0.0;
    if (!(ctx->grid_valid && ctx->grid_eps == eps)) {
        ST(ensure_grid(ctx, eps));
        ms_index = ctx->st.ms_index;
    }
    CK(cudaEventRecord(ctx->ev[2], s));
    ST(ensure_tiles(ctx, use_tc(ctx)));
    CK(cudaEventRecord(ctx->ev[3], s));
    fill_grid_stats(ctx);
    int64_t tlo = 0, thi = ctx->T;
    if (nranks > 1) {
        // split points of the unit prefix sums: tile t belongs to the shard of its first unit
        std::vector<int64_t> tu((size_t)ctx->T + 1);
        CK(cudaMemcpyAsync(tu.data(), ctx->tile_unit.p, 8 * tu.size(), cudaMemcpyDeviceToHost, s));
        ST(sync(ctx));
        const int64_t U = tu[(size_t)ctx->T];
        auto split = [&](int32_t r) -> int64_t {
            if (r >= nranks) return ctx->T;
            const int64_t target = (int64_t)((__int128)U * r / nranks);
            return std::lower_bound(tu.begin(), tu.end() - 1, target) - tu.begin();
        };
        tlo = split(rank);
        thi = split(rank + 1);
    }
    return run_batches(ctx, self_side(ctx), eps, batch_bytes, out, ms_index, launches0, tlo, thi);
}

// ---- semi-join: the query side built from separate query points -------------------
// d_queries: nq x d rows in the dataset's original dimension order, or NULL
// when ctx->q_xv already holds the nq rows permuted and padded (kNN rounds).
int build_query_side(hiss_ctx *ctx, const float *d_queries, int64_t nq, QuerySide *out)
{
    cudaStream_t s = ctx->stream;
    const int d = ctx->d, d4 = ctx->d4;
    if (d_queries) ST(ensure(ctx, ctx->q_xv, sizeof(float) * (size_t)nq * d4));
    ST(ensure(ctx, ctx->q_xs, sizeof(float) * (size_t)nq * d4));
    ST(ensure(ctx, ctx->q_ids, 4 * (size_t)nq));
    ST(ensure(ctx, ctx->q_cell_of_row, 4 * (size_t)nq));
    ST(ensure(ctx, ctx->keys, 8 * (size_t)nq));
    ST(ensure(ctx, ctx->vals, 4 * (size_t)nq));
    ST(ensure(ctx, ctx->keys_alt, 8 * (size_t)nq));
    ST(ensure(ctx, ctx->vals_alt, 4 * (size_t)nq));
    ST(ensure(ctx, ctx->sort_tmp, sort_tmp_bytes(nq)));
    ST(ensure(ctx, ctx->flag, 4 * (size_t)nq));
    ST(ensure(ctx, ctx->flag_scan, 4 * (size_t)(nq + 1)));
    ST(ensure(ctx, ctx->scan_tmp, 8 * (size_t)scan_tmp_elems(nq + 1) + 64));
    if (d_queries)
        CK(permute_pad(d_queries, nq, d, d4, as<int32_t>(ctx->perm_d), as<float>(ctx->q_xv), s, &ctx->launches));
    int64_t cellmax = 0;
    for (int k = 0; k < ctx->gp.ndim; ++k) {
        const int dim = ctx->perm[k];
        const double ext = ctx->stats[1 * (size_t)d + dim] - ctx->stats[0 * (size_t)d + dim];
        cellmax = std::max(cellmax, (int64_t)std::floor(ext / ctx->gp.w));
    }
    CK(query_keys(as<float>(ctx->q_xv), nq, d4, ctx->gp, cellmax, as<uint64_t>(ctx->keys), as<uint32_t>(ctx->vals), s,
                  &ctx->launches));
    int in_alt = 0;
    CK(sort_pairs(as<uint64_t>(ctx->keys), as<uint32_t>(ctx->vals), as<uint64_t>(ctx->keys_alt),
                  as<uint32_t>(ctx->vals_alt), nq, 64, ctx->sort_tmp.p, as<int>(ctx->flags), s, &ctx->launches,
                  &in_alt));
    const uint64_t *skeys = in_alt ? as<uint64_t>(ctx->keys_alt) : as<uint64_t>(ctx->keys);
    const uint32_t *svals = in_alt ? as<uint32_t>(ctx->vals_alt) : as<uint32_t>(ctx->vals);
    CK(gather_rows(as<float>(ctx->q_xv), svals, nq, d4, as<float>(ctx->q_xs), as<int32_t>(ctx->q_ids), s,
                   &ctx->launches));
    CK(cell_flags(skeys, nq, 0, as<int32_t>(ctx->flag), s, &ctx->launches));
    CK(scan_i32(as<int32_t>(ctx->flag), as<int32_t>(ctx->flag_scan), nq, as<int64_t>(ctx->scan_tmp), s,
                &ctx->launches));
    int32_t Cq32 = 0;
    CK(cudaMemcpyAsync(&Cq32, as<int32_t>(ctx->flag_scan) + nq, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ST(check_flags(ctx));
    const int64_t Cq = Cq32;
    ST(ensure(ctx, ctx->q_cell_start, 4 * (size_t)(Cq + 1)));
    ST(ensure(ctx, ctx->q_cell_key, 8 * (size_t)Cq));
    ST(ensure(ctx, ctx->q_nbr, 4 * (size_t)Cq * kStencil));
    ST(ensure(ctx, ctx->q_nbr_cnt, 4 * (size_t)(Cq + 1)));
    ST(ensure(ctx, ctx->q_bound, 8 * (size_t)(Cq + 1)));
    ST(ensure(ctx, ctx->q_work_key, 8 * (size_t)Cq));
    ST(ensure(ctx, ctx->q_cell_idx, 4 * (size_t)Cq));
    ST(ensure(ctx, ctx->q_work, 8 * (size_t)(Cq + 1)));
    CK(cell_starts(skeys, as<int32_t>(ctx->flag_scan), nq, 0, as<int32_t>(ctx->q_cell_start),
                   as<uint64_t>(ctx->q_cell_key), as<int32_t>(ctx->q_cell_of_row), s, &ctx->launches));
    CK(query_stencil(as<uint64_t>(ctx->q_cell_key), as<int32_t>(ctx->q_cell_start), Cq, as<uint64_t>(ctx->cell_key),
                     as<int32_t>(ctx->cell_start), ctx->C, as<int32_t>(ctx->q_nbr), as<int32_t>(ctx->q_nbr_cnt),
                     as<int64_t>(ctx->q_bound), as<uint64_t>(ctx->q_work_key), as<uint32_t>(ctx->q_cell_idx),
                     as<int64_t>(ctx->q_work), s, &ctx->launches));
    // candidates = sum over query cells of |cell| * bound
    ST(ensure(ctx, ctx->sums2, 8 * (size_t)(Cq + 1)));
    CK(scan_i64(as<int64_t>(ctx->q_work), as<int64_t>(ctx->sums2), Cq, as<int64_t>(ctx->scan_tmp), s, &ctx->launches));
    int64_t cand = 0;
    CK(cudaMemcpyAsync(&cand, as<int64_t>(ctx->sums2) + Cq, 8, cudaMemcpyDeviceToHost, s));
    ST(sync(ctx));
    ctx->st.candidates = cand;
    QuerySide q;
    q.xq = as<float>(ctx->q_xs);
    q.qids = as<int32_t>(ctx->q_ids);
    q.C = Cq;
    q.qcell_start = as<int32_t>(ctx->q_cell_start);
    q.nbr = as<int32_t>(ctx->q_nbr);
    q.nbr_cnt = as<int32_t>(ctx->q_nbr_cnt);
    q.bound = as<int64_t>(ctx->q_bound);
    q.work_key = as<uint64_t>(ctx->q_work_key);
    q.cell_idx = as<uint32_t>(ctx->q_cell_idx);
    *out = q;
    return HISS_OK;
}

int do_semi(hiss_ctx *ctx, const float *d_queries, int64_t nq, float eps, size_t batch_bytes, const hiss_out *out,
            int64_t *d_counts)
{
    const int mode = out ? out->mode : HISS_OUT_CSR;
    if (mode != HISS_OUT_CSR && mode != HISS_OUT_MASK) return HISS_E_ARG;
    cudaStream_t s = ctx->stream;
    const int64_t launches0 = ctx->launches;
    double ms_index = 0.0;
    if (!(ctx->grid_valid && ctx->grid_eps == eps)) {
        ST(ensure_grid(ctx, eps));
        ms_index = ctx->st.ms_index;
    }
    fill_grid_stats(ctx);
    ctx->st.pairs = 0;
    ctx->st.batches = 0;
    ctx->st.candidates_refined = 0;
    if (nq == 0) return HISS_OK;
    CK(cudaEventRecord(ctx->ev[2], s));
    QuerySide qs;
    ST(build_query_side(ctx, d_queries, nq, &qs));
    if (d_counts) {
        CK(scatter_counts(qs.qids, as<int32_t>(ctx->q_cell_of_row), qs.bound, nq, d_counts, s, &ctx->launches));
        CK(cudaEventRecord(ctx->ev[3], s));
        ST(sync(ctx));
        ctx->st.ms_count = elapsed(ctx, 2, 3);
        ctx->st.kernel_launches = ctx->launches - launches0;
        return HISS_OK;
    }
    ctx->tiles_valid = false;  // the tile arrays now describe the queries
    ST(build_tiles(ctx, qs, use_tc(ctx)));
    CK(cudaEventRecord(ctx->ev[3], s));
    return run_batches(ctx, qs, eps, batch_bytes, out, ms_index, launches0);
}


// ---- exact kNN by epsilon expansion -------------------------------------------------
constexpr size_t kKnnBatchBytes = size_t(1) << 30;   // mask per join batch
constexpr int kKnnMaxRounds = 256;

struct KnnState {
    hiss_ctx *ctx;
    int semi;                   // 0: first round (self-join, query rows = xs); 1: semi-join (query rows = q_xs)
    const int32_t *query_map;   // round's query index -> point id (NULL in the first round)
    int k;
    int64_t *out_ids;
    float *out_d2;
    int status;
};

// A group of rows of one batch whose pairs fit the group limit (a single row
// may exceed it; every count stays below the radix sort's 2^30).
int knn_group(KnnState *st, const hiss_batch *b, int64_t r0, int64_t r1, int64_t pair0, int64_t nnz)
{
    hiss_ctx *ctx = st->ctx;
    cudaStream_t s = ctx->stream;
    ST(ensure(ctx, ctx->k_keys, 8 * (size_t)nnz));
    ST(ensure(ctx, ctx->k_vals, 4 * (size_t)nnz));
    ST(ensure(ctx, ctx->k_keys_alt, 8 * (size_t)nnz));
    ST(ensure(ctx, ctx->k_vals_alt, 4 * (size_t)nnz));
    ST(ensure(ctx, ctx->k_sort_tmp, sort_tmp_bytes(nnz)));
    ST(ensure(ctx, ctx->k_d2, 4 * (size_t)nnz));
    ST(ensure(ctx, ctx->k_prow, 4 * (size_t)nnz));
    KnnBatchArgs a{};
    // the query side's buffers are (re)allocated inside the round: read them now
    a.xq = st->semi ? as<float>(ctx->q_xs) : as<float>(ctx->xs);
    a.xv = as<float>(ctx->xv);
    a.row_ptr = b->row_ptr + r0;
    a.cols = b->cols;
    a.query_rows = b->query_rows + r0;
    a.query_ids = b->query_ids + r0;
    a.query_map = st->query_map;
    a.nq = r1 - r0;
    a.nnz = nnz;
    a.pair0 = pair0;
    a.d4 = ctx->d4;
    a.k = st->k;
    a.d2 = as<float>(ctx->k_d2);
    a.prow = as<int32_t>(ctx->k_prow);
    a.keys = as<uint64_t>(ctx->k_keys);
    a.vals = as<uint32_t>(ctx->k_vals);
    a.out_ids = st->out_ids;
    a.out_d2 = st->out_d2;
    a.done = as<int8_t>(ctx->k_done);
    CK(knn_batch_pairs(a, s, &ctx->launches));
    // by neighbour id, then stably by (row, squared distance)
    int in_alt = 0;
    CK(sort_pairs(a.keys, a.vals, as<uint64_t>(ctx->k_keys_alt), as<uint32_t>(ctx->k_vals_alt), nnz, 31,
                  ctx->k_sort_tmp.p, as<int>(ctx->flags), s, &ctx->launches, &in_alt));
    if (in_alt) {
        a.keys = as<uint64_t>(ctx->k_keys_alt);
        a.vals = as<uint32_t>(ctx->k_vals_alt);
    }
    CK(knn_batch_rekey(a, s, &ctx->launches));
    uint64_t *ka = in_alt ? as<uint64_t>(ctx->k_keys) : as<uint64_t>(ctx->k_keys_alt);
    uint32_t *va = in_alt ? as<uint32_t>(ctx->k_vals) : as<uint32_t>(ctx->k_vals_alt);
    CK(sort_pairs(a.keys, a.vals, ka, va, nnz, 32 + bit_length(a.nq), ctx->k_sort_tmp.p, as<int>(ctx->flags), s,
                  &ctx->launches, &in_alt));
    if (in_alt) a.vals = va;
    CK(knn_batch_take(a, s, &ctx->launches));
    return HISS_OK;
}

// Called by run_batches for every CSR batch of a kNN round (device pointers).
int knn_on_batch(void *user, const hiss_batch *b)
{
    KnnState *st = static_cast<KnnState *>(user);
    hiss_ctx *ctx = st->ctx;
    std::vector<int64_t> rp((size_t)b->nq + 1);
    int rc = HISS_OK;
    if (cudaMemcpyAsync(rp.data(), b->row_ptr, 8 * rp.size(), cudaMemcpyDeviceToHost, ctx->stream) != cudaSuccess)
        rc = fail_cuda(ctx, cudaGetLastError());
    if (rc == HISS_OK) rc = sync(ctx);
    constexpr int64_t kMaxPairs = int64_t(1) << 27;  // about 3.8 GB of sort scratch per group
    for (int64_t r0 = 0; rc == HISS_OK && r0 < b->nq;) {
        int64_t r1 = r0 + 1;  // one row never exceeds n < 2^30 pairs
        while (r1 < b->nq && rp[r1 + 1] - rp[r0] <= kMaxPairs) ++r1;
        rc = knn_group(st, b, r0, r1, rp[r0], rp[r1] - rp[r0]);
        r0 = r1;
    }
    if (rc != HISS_OK) {
        st->status = rc;
        return 1;
    }
    return 0;
}

int do_knn(hiss_ctx *ctx, int32_t k, float eps0, int64_t *out_ids, float *out_d2)
{
    const int64_t n = ctx->n;
    const int d = ctx->d;
    cudaStream_t s = ctx->stream;
    // a radius that holds every point: the dataset's diameter (fp64, padded)
    double diam2 = 0.0;
    for (int j = 0; j < d; ++j) {
        const double e = ctx->stats[1 * (size_t)d + j] - ctx->stats[0 * (size_t)d + j];
        diam2 += e * e;
    }
    const float diam = (float)(std::sqrt(diam2) * (1.0 + 1e-3) + 1e-30);
    float eps = eps0;
    if (!(eps > 0.0f)) {
        // start from the spacing of n points over the three index dimensions
        double ext = 0.0;
        for (int j = 0; j < std::min(d, 3); ++j) {
            const int dim = ctx->perm[j];
            ext = std::max(ext, ctx->stats[1 * (size_t)d + dim] - ctx->stats[0 * (size_t)d + dim]);
        }
        eps = (float)(0.5 * ext * std::pow((double)k / (double)n, 1.0 / std::min(d, 3)));
        if (!(eps > 0.0f)) eps = diam;
    }
    ST(ensure(ctx, ctx->k_done, (size_t)n));
    ST(ensure(ctx, ctx->k_active, 4 * (size_t)n));
    CK(cudaMemsetAsync(ctx->k_done.p, 0, (size_t)n, s));
    std::vector<int8_t> done(n);
    std::vector<uint32_t> active;
    hiss_out out{};
    out.mode = HISS_OUT_CSR;
    out.copy_to_host = 0;
    out.on_batch = knn_on_batch;
    KnnState st{ctx, 0, nullptr, k, out_ids, out_d2, HISS_OK};
    out.user = &st;
    for (int round = 0; round < kKnnMaxRounds; ++round) {
        int rc;
        if (round == 0) {
            st.semi = 0;
            st.query_map = nullptr;
            rc = do_join(ctx, eps, kKnnBatchBytes, &out);
        } else {
            // the queries still short of k neighbours, as a semi-join against the data
            const int64_t nq = (int64_t)active.size();
            ST(ensure(ctx, ctx->q_xv, sizeof(float) * (size_t)nq * ctx->d4));
            ST(ensure(ctx, ctx->q_ids, 4 * (size_t)nq));
            CK(cudaMemcpyAsync(ctx->k_active.p, active.data(), 4 * (size_t)nq, cudaMemcpyHostToDevice, s));
            CK(gather_rows(as<float>(ctx->xv), as<uint32_t>(ctx->k_active), nq, ctx->d4, as<float>(ctx->q_xv),
                           as<int32_t>(ctx->q_ids), s, &ctx->launches));
            st.semi = 1;
            st.query_map = as<int32_t>(ctx->k_active);
            rc = do_semi(ctx, nullptr, nq, eps, kKnnBatchBytes, &out, nullptr);
        }
        if (rc == HISS_E_CALLBACK) return st.status != HISS_OK ? st.status : HISS_E_CUDA;
        if (rc != HISS_OK) return rc;
        CK(cudaMemcpyAsync(done.data(), ctx->k_done.p, (size_t)n, cudaMemcpyDeviceToHost, s));
        ST(sync(ctx));
        active.clear();
        for (int64_t i = 0; i < n; ++i)
            if (!done[i]) active.push_back((uint32_t)i);
        if (active.empty()) return HISS_OK;
        if (eps >= diam) return HISS_E_STATE;  // cannot happen: eps = diameter holds every point
        eps = std::min(diam, std::max(eps * 1.41421356f, std::nextafter(eps, INFINITY)));
    }
    return HISS_E_OVERFLOW;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

int hiss_create(hiss_ctx **out, void *cuda_stream)
{
    if (!out) return HISS_E_ARG;
    *out = nullptr;
    hiss_ctx *ctx = new (std::nothrow) hiss_ctx();
    if (!ctx) return HISS_E_NOMEM;
    if (cudaGetDevice(&ctx->device) != cudaSuccess) {
        cudaGetLastError();
        delete ctx;
        return HISS_E_CUDA;
    }
    ctx->stream = static_cast<cudaStream_t>(cuda_stream);
    for (auto &e : ctx->ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            cudaGetLastError();
            for (auto &f : ctx->ev)
                if (f) cudaEventDestroy(f);
            delete ctx;
            return HISS_E_CUDA;
        }
    }
    *out = ctx;
    return HISS_OK;
}

void hiss_destroy(hiss_ctx *ctx)
{
    if (!ctx) return;
    cudaSetDevice(ctx->device);
    cudaStreamSynchronize(ctx->stream);
    DBuf *all[] = {&ctx->x_stage, &ctx->xv, &ctx->perm_d, &ctx->stats_partial, &ctx->stats_out, &ctx->flags,
                   &ctx->keys, &ctx->vals, &ctx->keys_alt, &ctx->vals_alt, &ctx->sort_tmp, &ctx->xs, &ctx->gbox, &ctx->ids,
                   &ctx->flag, &ctx->flag_scan, &ctx->cell_start, &ctx->cell_key, &ctx->cell_of_row, &ctx->nbr,
                   &ctx->nbr_cnt, &ctx->bound, &ctx->work_key, &ctx->cell_idx, &ctx->work, &ctx->scan_tmp,
                   &ctx->sums2, &ctx->lpt_keys, &ctx->lpt_order, &ctx->ntiles, &ctx->tile_off, &ctx->tile_cell,
                   &ctx->tile_q0, &ctx->tile_nq, &ctx->tile_word, &ctx->tile_unit, &ctx->tile_qoff,
                   &ctx->boundaries, &ctx->binfo, &ctx->nb_d, &ctx->mask, &ctx->occ, &ctx->qcount, &ctx->row_ptr, &ctx->cols,
                   &ctx->query_ids, &ctx->query_rows, &ctx->cand, &ctx->mask_row_ptr, &ctx->t_keys_alt,
                   &ctx->t_vals_alt, &ctx->t_sort_tmp, &ctx->t_scan_tmp, &ctx->q_xv, &ctx->q_xs, &ctx->q_ids,
                   &ctx->q_cell_of_row, &ctx->q_cell_start, &ctx->q_cell_key, &ctx->q_nbr, &ctx->q_nbr_cnt,
                   &ctx->q_bound, &ctx->q_work_key, &ctx->q_cell_idx, &ctx->q_work, &ctx->k_keys,
                   &ctx->k_vals, &ctx->k_keys_alt, &ctx->k_vals_alt, &ctx->k_sort_tmp, &ctx->k_d2, &ctx->k_prow,
                   &ctx->k_done, &ctx->k_active, &ctx->row_ptr2, &ctx->cols2, &ctx->row_ptr_sub, &ctx->unit_tile, &ctx->unit_chunk,
                   &ctx->query_ids2, &ctx->query_rows2};
    if (ctx->copy_stream) cudaStreamSynchronize(ctx->copy_stream);
    for (DBuf *b : all) release(ctx, *b);
    cudaStreamSynchronize(ctx->stream);
    if (ctx->h_pinned) cudaFreeHost(ctx->h_pinned);
    if (ctx->h_pinned2) cudaFreeHost(ctx->h_pinned2);
    for (int i = 0; i < 2; ++i) {
        if (ctx->ev_compacted[i]) cudaEventDestroy(ctx->ev_compacted[i]);
        if (ctx->ev_copy0[i]) cudaEventDestroy(ctx->ev_copy0[i]);
        if (ctx->ev_copied[i]) cudaEventDestroy(ctx->ev_copied[i]);
    }
    if (ctx->copy_stream) cudaStreamDestroy(ctx->copy_stream);
    for (auto &e : ctx->ev)
        if (e) cudaEventDestroy(e);
    cudaGetLastError();
    delete ctx;
}

int hiss_build(hiss_ctx *ctx, const float *d_points, int64_t n, int32_t d)
{
    ST(enter(ctx));
    if (!d_points || n < 1 || n >= (int64_t(1) << 30) || d < 1 || d > HISS_MAX_DIM) return HISS_E_ARG;
    return do_build(ctx, d_points, n, d);
}

int hiss_build_host(hiss_ctx *ctx, const float *h_points, int64_t n, int32_t d)
{
    ST(enter(ctx));
    if (!h_points || n < 1 || n >= (int64_t(1) << 30) || d < 1 || d > HISS_MAX_DIM) return HISS_E_ARG;
    ST(ensure(ctx, ctx->x_stage, sizeof(float) * (size_t)n * d));
    CK(cudaMemcpyAsync(ctx->x_stage.p, h_points, sizeof(float) * (size_t)n * d, cudaMemcpyHostToDevice,
                       ctx->stream));
    return do_build(ctx, as<float>(ctx->x_stage), n, d);
}

int hiss_count(hiss_ctx *ctx, float eps, int64_t *d_counts)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    const int64_t launches0 = ctx->launches;
    ctx->st.ms_index = 0.0;
    ST(ensure_grid(ctx, eps));
    CK(cudaEventRecord(ctx->ev[2], ctx->stream));
    if (d_counts)
        CK(scatter_counts(as<int32_t>(ctx->ids), as<int32_t>(ctx->cell_of_row), as<int64_t>(ctx->bound), ctx->n,
                          d_counts, ctx->stream, &ctx->launches));
    CK(cudaEventRecord(ctx->ev[3], ctx->stream));
    ST(sync(ctx));
    fill_grid_stats(ctx);
    ctx->st.ms_count = elapsed(ctx, 2, 3);
    ctx->st.kernel_launches = ctx->launches - launches0;
    return HISS_OK;
}

int hiss_join(hiss_ctx *ctx, float eps, size_t batch_bytes, const hiss_out *out)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    return do_join(ctx, eps, batch_bytes, out);
}

int hiss_join_queries(hiss_ctx *ctx, const float *d_queries, int64_t nq, float eps, size_t batch_bytes,
                      const hiss_out *out)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    if (nq < 0 || nq >= (int64_t(1) << 30) || (nq > 0 && !d_queries)) return HISS_E_ARG;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    return do_semi(ctx, d_queries, nq, eps, batch_bytes, out, nullptr);
}

int hiss_count_queries(hiss_ctx *ctx, const float *d_queries, int64_t nq, float eps, int64_t *d_counts)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    if (nq < 0 || nq >= (int64_t(1) << 30) || (nq > 0 && (!d_queries || !d_counts))) return HISS_E_ARG;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    return do_semi(ctx, d_queries, nq, eps, 0, nullptr, d_counts);
}

int hiss_work_profile(hiss_ctx *ctx, float eps, int64_t *out)
{
    ST(enter(ctx));
    if (!out) return HISS_E_ARG;
    if (!ctx->built) return HISS_E_STATE;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    ST(ensure_grid(ctx, eps));
    ST(ensure_tiles(ctx, false));  // the work counter is the CUDA-core kernel's
    ST(ensure(ctx, ctx->nb_d, 64));
    CK(cudaMemsetAsync(ctx->nb_d.p, 0, 16, ctx->stream));
    RefineArgs ra{};
    ra.xs = as<float>(ctx->xs);
    ra.xq = as<float>(ctx->xs);
    ra.cell_start = as<int32_t>(ctx->cell_start);
    ra.nbr = as<int32_t>(ctx->nbr);
    ra.nbr_cnt = as<int32_t>(ctx->nbr_cnt);
    ra.bound = as<int64_t>(ctx->bound);
    ra.tile_cell = as<int32_t>(ctx->tile_cell);
    ra.tile_q0 = as<int32_t>(ctx->tile_q0);
    ra.tile_nq = as<int32_t>(ctx->tile_nq);
    ra.tile_word = as<int64_t>(ctx->tile_word);
    ra.tile_unit = as<int64_t>(ctx->tile_unit);
    ra.tile_qoff = as<int64_t>(ctx->tile_qoff);
    ra.t0 = 0;
    ra.t1 = ctx->T;
    ra.unit0 = 0;
    ra.nunits = ctx->total_units;
    ra.d4 = ctx->d4;
    ra.d = ctx->d;
    ra.eps2 = eps * eps;
    ra.prof = as<int64_t>(ctx->nb_d);
    ra.flags = as<int>(ctx->flags);
    CK(refine_profile(ra, ctx->stream, &ctx->launches));
    CK(cudaMemcpyAsync(out, ctx->nb_d.p, 16, cudaMemcpyDeviceToHost, ctx->stream));
    ST(sync(ctx));
    return check_flags(ctx);
}

int hiss_index(hiss_ctx *ctx, hiss_index_view *v)
{
    ST(enter(ctx));
    if (!v) return HISS_E_ARG;
    if (!ctx->grid_valid) return HISS_E_STATE;
    memset(v, 0, sizeof(*v));
    v->n = ctx->n;
    v->cells = ctx->C;
    v->ids = as<int32_t>(ctx->ids);
    v->cell_start = as<int32_t>(ctx->cell_start);
    v->cell_of_row = as<int32_t>(ctx->cell_of_row);
    v->nbr = as<int32_t>(ctx->nbr);
    v->nbr_count = as<int32_t>(ctx->nbr_cnt);
    v->cell_bound = as<int64_t>(ctx->bound);
    v->cell_key = as<uint64_t>(ctx->cell_key);
    for (int k = 0; k < 3; ++k) {
        v->perm[k] = k < ctx->gp.ndim ? ctx->perm[k] : -1;
        v->origin[k] = ctx->gp.origin[k];
    }
    v->sub_bits = ctx->gp.sub_bits;
    v->cell_width = ctx->gp.w;
    return HISS_OK;
}

int hiss_last_stats(const hiss_ctx *ctx, hiss_stats *out)
{
    if (!ctx || !out) return HISS_E_ARG;
    *out = ctx->st;
    return HISS_OK;
}

int64_t hiss_launch_count(const hiss_ctx *ctx) { return ctx ? ctx->launches : 0; }

const char *hiss_strerror(int status)
{
    switch (status) {
    case HISS_OK: return "ok";
    case HISS_E_ARG: return "invalid argument";
    case HISS_E_NOMEM: return "out of memory";
    case HISS_E_STATE: return "call out of order or context in error state";
    case HISS_E_BATCH_TOO_SMALL: return "batch_bytes smaller than one query tile's result mask";
    case HISS_E_OVERFLOW: return "integer overflow";
    case HISS_E_CUDA: return "CUDA error";
    case HISS_E_CALLBACK: return "batch callback requested stop";
    default: return "unknown status";
    }
}

const char *hiss_last_cuda_error(const hiss_ctx *ctx) { return ctx ? ctx->cuda_err : ""; }

int hiss_set_option(hiss_ctx *ctx, int option, int64_t value)
{
    if (!ctx) return HISS_E_ARG;
    if (option == HISS_OPT_ALLOC_LIMIT) {
        if (value < 0) return HISS_E_ARG;
        ctx->alloc_limit = value;
        return HISS_OK;
    }
    if (option == HISS_OPT_REFINE) {
        if (value != HISS_REFINE_CUDA_CORES && value != HISS_REFINE_TENSOR_CORES) return HISS_E_ARG;
        ctx->refine_mode = (int)value;
        return HISS_OK;
    }
    return HISS_E_ARG;
}

int hiss_sort_pairs(hiss_ctx *ctx, uint64_t *d_keys, uint32_t *d_vals, int64_t n, int32_t key_bits)
{
    ST(enter(ctx));
    if (!d_keys || !d_vals || n < 0 || n >= (int64_t(1) << 30) || key_bits < 1 || key_bits > 64) return HISS_E_ARG;
    if (n <= 1) return HISS_OK;
    ST(ensure(ctx, ctx->t_keys_alt, 8 * (size_t)n));
    ST(ensure(ctx, ctx->t_vals_alt, 4 * (size_t)n));
    ST(ensure(ctx, ctx->t_sort_tmp, sort_tmp_bytes(n)));
    ST(ensure(ctx, ctx->flags, sizeof(int) * kNumFlags * 2));
    CK(cudaMemsetAsync(ctx->flags.p, 0, sizeof(int) * kNumFlags, ctx->stream));
    int in_alt = 0;
    CK(sort_pairs(d_keys, d_vals, as<uint64_t>(ctx->t_keys_alt), as<uint32_t>(ctx->t_vals_alt), n, key_bits,
                  ctx->t_sort_tmp.p, as<int>(ctx->flags), ctx->stream, &ctx->launches, &in_alt));
    if (in_alt) {
        CK(cudaMemcpyAsync(d_keys, ctx->t_keys_alt.p, 8 * (size_t)n, cudaMemcpyDeviceToDevice, ctx->stream));
        CK(cudaMemcpyAsync(d_vals, ctx->t_vals_alt.p, 4 * (size_t)n, cudaMemcpyDeviceToDevice, ctx->stream));
    }
    return check_flags(ctx);
}

int hiss_exclusive_scan(hiss_ctx *ctx, const int64_t *d_in, int64_t *d_out, int64_t n)
{
    ST(enter(ctx));
    if ((n > 0 && !d_in) || !d_out || n < 0) return HISS_E_ARG;
    ST(ensure(ctx, ctx->t_scan_tmp, 8 * (size_t)scan_tmp_elems(n + 1) + 64));
    CK(scan_i64(d_in, d_out, n, as<int64_t>(ctx->t_scan_tmp), ctx->stream, &ctx->launches));
    return sync(ctx);
}

int hiss_mask_positions(hiss_ctx *ctx, const uint32_t *d_words, int64_t nbits, int64_t *d_pos, int64_t *h_count)
{
    ST(enter(ctx));
    if (!d_words || !d_pos || !h_count || nbits < 0) return HISS_E_ARG;
    const int64_t nw = (nbits + 31) >> 5;
    ST(ensure(ctx, ctx->t_scan_tmp, 8 * (size_t)((nw + 1) / 2 + 1 + nw + 1 + scan_tmp_elems(nw + 1)) + 64));
    ST(ensure(ctx, ctx->nb_d, 64));
    CK(mask_positions(d_words, nbits, d_pos, as<int64_t>(ctx->nb_d), as<int64_t>(ctx->t_scan_tmp), ctx->stream,
                      &ctx->launches));
    CK(cudaMemcpyAsync(h_count, ctx->nb_d.p, 8, cudaMemcpyDeviceToHost, ctx->stream));
    return sync(ctx);
}

int hiss_gram_tf32(hiss_ctx *ctx, const float *d_a, const float *d_b, int32_t k, float *d_out)
{
    ST(enter(ctx));
    if (!d_a || !d_b || !d_out || k < 8 || k > 128 || k % 8 != 0) return HISS_E_ARG;
    ST(ensure(ctx, ctx->flags, sizeof(int) * kNumFlags * 2));
    CK(cudaMemsetAsync(ctx->flags.p, 0, sizeof(int) * kNumFlags, ctx->stream));
    CK(gram_tf32(d_a, d_b, k, d_out, as<int>(ctx->flags), ctx->stream, &ctx->launches));
    ST(sync(ctx));
    return check_flags(ctx);
}

int hiss_join_shard(hiss_ctx *ctx, float eps, size_t batch_bytes, const hiss_out *out, int32_t rank,
                    int32_t nranks)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    if (!(eps >= 0.0f) || std::isinf(eps)) return HISS_E_ARG;
    if (nranks < 1 || rank < 0 || rank >= nranks) return HISS_E_ARG;
    return do_join(ctx, eps, batch_bytes, out, rank, nranks);
}

int hiss_knn(hiss_ctx *ctx, int32_t k, float eps0, int64_t *d_ids, float *d_dist2)
{
    ST(enter(ctx));
    if (!ctx->built) return HISS_E_STATE;
    if (!d_ids || k < 1 || (int64_t)k > ctx->n || std::isnan(eps0) || std::isinf(eps0)) return HISS_E_ARG;
    const int64_t launches0 = ctx->launches;
    const int rc = do_knn(ctx, k, eps0, d_ids, d_dist2);
    ctx->st.kernel_launches = ctx->launches - launches0;
    return rc;
}

}  // extern "C"
