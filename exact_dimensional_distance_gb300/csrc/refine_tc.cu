// Tensor-core (tcgen05) refinement and its Gram building block.
//
// gram_tf32: the Gram matrix G = A B^T of two 128-row float32 blocks after
// rounding both to TF32, computed by one CTA with tcgen05.mma (kind::tf32,
// M = N = 128, accumulator in tensor memory) from operands staged in shared
// memory in the no-swizzle K-major core-matrix layout.
//
// refine_tc: the refinement of a batch (the same units, tiles and result
// mask as the CUDA-core refinement) with the squared distances of each
// 128 x 128 tile of (query, candidate) pairs obtained as a Gram matrix on the
// tensor cores, and every pair whose TF32 estimate is not decisive rechecked
// exactly in float32 (see k_refine_tc).
#include "hiss_internal.cuh"
#include "ptx.cuh"

namespace hiss {
namespace {

constexpr int kGramRows = 128;

// Byte offset of element (row, k) of a K-major operand with kpad columns in
// the no-swizzle core-matrix layout: core matrices of 8 rows x 4 TF32
// elements (128 bytes) are contiguous along K (lbo = 128 bytes); groups of 8
// rows follow each other (sbo = kpad / 4 * 128 bytes).
__host__ __device__ __forceinline__ uint32_t core_offset(int row, int k, int kpad)
{
    return (uint32_t)((row >> 3) * (kpad / 4) * 128 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

__global__ void __launch_bounds__(128, 1) k_gram_tf32(const float *a, const float *b, int k, float *out, int *flags)
{
    extern __shared__ __align__(128) unsigned char gsm[];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned char *As = gsm;
    unsigned char *Bs = gsm + (size_t)kGramRows * k * 4;
    // row tid of both operands, TF32-rounded, into the core-matrix layout
    for (int kc = 0; kc < k / 4; ++kc) {
        const float4 va = *reinterpret_cast<const float4 *>(a + (int64_t)tid * k + 4 * kc);
        const float4 vb = *reinterpret_cast<const float4 *>(b + (int64_t)tid * k + 4 * kc);
        *reinterpret_cast<float4 *>(As + core_offset(tid, 4 * kc, k)) =
            make_float4(to_tf32(va.x), to_tf32(va.y), to_tf32(va.z), to_tf32(va.w));
        *reinterpret_cast<float4 *>(Bs + core_offset(tid, 4 * kc, k)) =
            make_float4(to_tf32(vb.x), to_tf32(vb.y), to_tf32(vb.z), to_tf32(vb.w));
    }
    fence_proxy_async_smem();
    if (warp == 0) tmem_alloc(&s_tmem, 128);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        const uint32_t sbo = (uint32_t)(k / 4) * 128u;
        const uint32_t idesc = idesc_tf32(kGramRows, kGramRows);
        for (int s = 0; s < k / 8; ++s) {
            const uint64_t ad = smem_desc(smem_u32(As) + 256u * s, 128u, sbo);
            const uint64_t bd = smem_desc(smem_u32(Bs) + 256u * s, 128u, sbo);
            mma_tf32(tmem, ad, bd, idesc, s > 0 ? 1u : 0u);
        }
        mma_commit(&s_bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&s_bar, 0);
    if (!ok && lane == 0) atomicExch(&flags[kFlagRefineTimeout], 1);
    tc_fence_after_sync();
    if (ok) {
        for (int cb = 0; cb < kGramRows / 32; ++cb) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32u * cb, v);
            tmem_ld_wait();
            float *row = out + (int64_t)(32 * warp + lane) * kGramRows + 32 * cb;
#pragma unroll
            for (int j = 0; j < 32; ++j) row[j] = __uint_as_float(v[j]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---- tensor-core refinement -------------------------------------------------------
//
// One CTA refines one unit (a tile of up to 128 queries of one cell against a
// chunk of up to kTcChunk stencil candidates), in 128-candidate tiles.  Warp
// roles: warps 0-3 read the accumulator (warp w owns tensor-memory lanes
// 32 w .. 32 w + 31, i.e. query rows) and write the mask; warps 4-7 stage the
// operands; one thread of warp 8 issues the MMAs.
//
// Arithmetic.  c = the query tile's mean (any float32 vector works; the mean
// keeps the values small).  Every query row q and candidate row p is centred
// and rounded, q~ = tf32(q - c), p~ = tf32(p - c), and gets a = |q~|, b = |p~|
// (rounded up).  One MMA chain over K = d4 + 8 computes, per pair,
//     u = (|q~|^2 - eps^2 + alpha) + (|p~|^2 + beta) - 2 q~ . p~
// with the two bracketed terms carried exactly as hi + lo TF32 pairs in 8
// extra K columns (A: [q~, X_hi, X_lo, 1, 1, 0..], B: [-2 p~, 1, 1, Y_hi,
// Y_lo, 0..]).  Rounding moves each point by at most 2^-10 of its norm, so
// |dist(q, p) - |q~ - p~|| <= 2^-10 (a + b); with the float32 and tensor-core
// accumulation errors bounded by g (a + b)^2 + g eps^2, the margins
//     alpha = c1 a + c2 a^2 + c0,  beta = c1 b + c2 b^2,
//     c1 = 2^-9 eps (1 + 2^-10), c2 = 2^-19 + 2 g (1 + 2^-10), c0 = g eps^2 (1 + 2^-10),
// g = (K + 24) 2^-22, make the signs decisive:
//     u < 0                   => dist(q, p) <  eps  (bit 1),
//     u > 2 (alpha + beta)    => dist(q, p) >  eps  (bit 0),
// and only pairs with 0 <= u <= 2 (alpha + beta) are rechecked exactly with
// the CUDA-core refinement's float32 arithmetic (refine_dist2), bit =
// sum <= eps^2.
constexpr int kTcRows = 128;                 // queries per tile (M) = candidates per tile (N)
constexpr int kTcThreads = 9 * 32;
constexpr int kTcXf0 = 4 * 32;               // first transform thread
constexpr int kTcChunk = 8192;               // candidates per unit
constexpr int kTcSide = 8;                   // slots of the per-tile side ring
constexpr int kTcMaxStages = 4;
constexpr int kTcTmemCols = 256;             // two 128-column accumulators
constexpr float kTcBig = 1e30f;              // augmented value of padding rows: u >= 1e30

struct TcLayout {
    int kpad, stages;
    uint32_t op_bytes, off_b, off_c, off_alpha, off_beta, off_src, off_bmax, total;
};

// Operand width: d4 rounded up to a power of two (zero columns change no
// distance) so that the lanes sharing a row form a fixed shuffle group.
__host__ __device__ __forceinline__ int tc_d4p(int d4)
{
    int p = 4;
    while (p < d4) p *= 2;
    return p;
}

__host__ __device__ __forceinline__ TcLayout tc_layout(int d4)
{
    TcLayout L;
    L.kpad = tc_d4p(d4) + 8;
    L.op_bytes = (uint32_t)kTcRows * L.kpad * 4;
    const uint32_t misc = (uint32_t)d4 * 4 + kTcRows * 4 + 2 * kTcSide * kTcRows * 4 + kTcSide * 4 * 4 + 256;
    int ns = (int)((113u * 1024u - misc) / L.op_bytes) - 1;  // two CTAs per SM when it fits
    if (ns < 2) ns = (int)((220u * 1024u - misc) / L.op_bytes) - 1;
    L.stages = ns > kTcMaxStages ? kTcMaxStages : ns;
    L.off_b = L.op_bytes;
    L.off_c = L.off_b + (uint32_t)L.stages * L.op_bytes;
    L.off_alpha = L.off_c + (uint32_t)((d4 * 4 + 15) & ~15);
    L.off_beta = L.off_alpha + kTcRows * 4;
    L.off_src = L.off_beta + kTcSide * kTcRows * 4;
    L.off_bmax = L.off_src + kTcSide * kTcRows * 4;
    L.total = L.off_bmax + kTcSide * 4 * 4;
    return L;
}

struct TcConst {
    float c0, c1, c2;   // margins: alpha = c1 a + c2 a^2 + c0, beta = c1 b + c2 b^2
};

__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo)
{
    hi = to_tf32(x);
    lo = to_tf32(x - hi);  // x - hi is exact in float32
}

// Exact recheck of one pair: the CUDA-core refinement's float32 squared
// distance (refine_dist2).
__device__ __noinline__ bool tc_recheck(const float *q, const float *p, int d4, float eps2)
{
    return refine_dist2(q, p, d4) <= eps2;
}

// Stage 128 rows into a K-major core-matrix operand with the 4 transform
// warps.  Lane l of transform warp wx handles row 8 (wx + 4 gi) + l % 8 and
// the 16-byte column chunks kc = l / 8 + 4 h: a warp's store of one (gi, h)
// fills four whole core matrices (conflict-free), its loads read 8 rows x 64
// contiguous bytes.  Element k of a row becomes scale * tf32(x[k] - c[k]) for
// k < d4 and rows with data (rowptr(row) != nullptr), else 0.  nrm[gi]
// receives the row's squared norm of the tf32 values (summed over the row's
// four lanes with a fixed shuffle tree; the same value in all four).
template <int C4P, typename RowPtr>
__device__ __forceinline__ void stage_rows(unsigned char *op, int kpad, int d4, const float *s_c,
                                           const RowPtr &rowptr, float scale, float (&nrm)[4], int wx, int lane)
{
    constexpr int H = (C4P + 3) / 4;               // chunks per lane per row
    constexpr int GB = H >= 8 ? 1 : (H >= 4 ? 2 : 4);  // rows per batch: at most 8 loads in flight
    const int rl = lane & 7, cs = lane >> 3;
#pragma unroll
    for (int g0 = 0; g0 < 4; g0 += GB) {
        float4 x[GB][H];
        bool has[GB];
#pragma unroll
        for (int gb = 0; gb < GB; ++gb) {
            const float *rp = rowptr(8 * (wx + 4 * (g0 + gb)) + rl);
            has[gb] = rp != nullptr;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const int kc = cs + 4 * h;
                x[gb][h] = (kc < C4P && 4 * kc < d4 && rp) ? *reinterpret_cast<const float4 *>(rp + 4 * kc)
                                                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int gb = 0; gb < GB; ++gb) {
            const int row = 8 * (wx + 4 * (g0 + gb)) + rl;
            float sq = 0.0f;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const int kc = cs + 4 * h;
                if (kc < C4P) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (4 * kc < d4 && has[gb]) {
                        const float4 cc = *reinterpret_cast<const float4 *>(s_c + 4 * kc);
                        const float4 xv = x[gb][h];
                        v = make_float4(to_tf32(xv.x - cc.x), to_tf32(xv.y - cc.y), to_tf32(xv.z - cc.z),
                                        to_tf32(xv.w - cc.w));
                        sq = fmaf(v.x, v.x, sq);
                        sq = fmaf(v.y, v.y, sq);
                        sq = fmaf(v.z, v.z, sq);
                        sq = fmaf(v.w, v.w, sq);
                    }
                    *reinterpret_cast<float4 *>(op + core_offset(row, 4 * kc, kpad)) =
                        make_float4(scale * v.x, scale * v.y, scale * v.z, scale * v.w);
                }
            }
            sq += __shfl_xor_sync(0xffffffffu, sq, 8);
            sq += __shfl_xor_sync(0xffffffffu, sq, 16);
            nrm[g0 + gb] = sq;
        }
    }
}

template <int C4P>
__global__ void __maxnreg__(96) k_refine_tc(const RefineArgs a, const TcConst cst)
{
    extern __shared__ __align__(128) unsigned char tsm[];
    __shared__ __align__(8) uint64_t s_full_b[kTcMaxStages], s_empty_b[kTcMaxStages];
    __shared__ __align__(8) uint64_t s_full_d[2], s_empty_d[2], s_a_full, s_side[kTcSide];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int32_t s_nstart[kStencil];
    __shared__ int32_t s_vpre[kStencil + 1];
    __shared__ int64_t s_info[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d4 = a.d4;
    const TcLayout L = tc_layout(d4);
    const int nst = L.stages, kpad = L.kpad;
    unsigned char *As = tsm;
    unsigned char *Bs0 = tsm + L.off_b;
    float *s_c = reinterpret_cast<float *>(tsm + L.off_c);
    float *s_alpha = reinterpret_cast<float *>(tsm + L.off_alpha);
    float *s_beta = reinterpret_cast<float *>(tsm + L.off_beta);
    int32_t *s_src = reinterpret_cast<int32_t *>(tsm + L.off_src);
    float *s_bmax = reinterpret_cast<float *>(tsm + L.off_bmax);

    if (tid == 0) {
        const int64_t u = a.unit0 + blockIdx.x;
        int64_t lo = a.t0, hi = a.t1 - 1;  // last tile with tile_unit[t] <= u
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (a.tile_unit[mid] <= u) lo = mid; else hi = mid - 1;
        }
        s_info[0] = lo;
        s_info[1] = u - a.tile_unit[lo];
        for (int i = 0; i < nst; ++i) {
            mbar_init(&s_full_b[i], 4);
            mbar_init(&s_empty_b[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full_d[i], 1);
            mbar_init(&s_empty_d[i], 4);
        }
        for (int i = 0; i < kTcSide; ++i) mbar_init(&s_side[i], 4);
        mbar_init(&s_a_full, 4);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, kTcTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    const int64_t t = s_info[0];
    const int64_t chunk = s_info[1];
    const int32_t cell = a.tile_cell[t];
    const int32_t q0 = a.tile_q0[t];
    const int nq = a.tile_nq[t];
    const int64_t B = a.bound[cell];
    const int64_t W = (B + 31) >> 5;
    const int64_t W4 = (W + 3) & ~int64_t(3);
    const int ncell = a.nbr_cnt[cell];
    if (tid < ncell) {
        const int32_t nb = a.nbr[(int64_t)cell * kStencil + tid];
        s_nstart[tid] = a.cell_start[nb];
        s_vpre[tid + 1] = a.cell_start[nb + 1] - a.cell_start[nb];
    }
    __syncthreads();
    if (tid == 0) {
        s_vpre[0] = 0;
        for (int i = 1; i <= ncell; ++i) s_vpre[i] += s_vpre[i - 1];
    }
    __syncthreads();
    const int64_t vbeg = chunk * kTcChunk;
    const int64_t vend = min(B, vbeg + (int64_t)kTcChunk);
    const int ntiles = (int)((vend - vbeg + kTcRows - 1) / kTcRows);
    const float eps2 = a.eps2;
    volatile int *abort_flag = &s_abort;
    auto give_up = [&]() {
        s_abort = 1;
        atomicExch(&a.flags[kFlagRefineTimeout], 1);
    };

    if (warp >= 4 && warp < 8) {
        // ---- operand staging (128 threads) ----
        const int t4 = tid - kTcXf0;
        const int wx = warp - 4;
        const int d4p = 4 * C4P;
        // centre: mean of the first (up to) 8 query rows
        for (int k = t4; k < d4; k += 128) {
            const int m = nq < 8 ? nq : 8;
            float sum = 0.0f;
            for (int i = 0; i < m; ++i) sum += a.xq[(int64_t)(q0 + i) * d4 + k];
            s_c[k] = sum / (float)m;
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");
        {
            auto qrow = [&](int row) -> const float * {
                return row < nq ? a.xq + (int64_t)(q0 + row) * d4 : nullptr;
            };
            float nrm[4];
            stage_rows<C4P>(As, kpad, d4, s_c, qrow, 1.0f, nrm, wx, lane);
            if (lane < 8) {
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) {
                    const int row = 8 * (wx + 4 * gi) + lane;
                    float xh = kTcBig, xl = 0.0f, alpha = 0.0f;
                    if (row < nq) {
                        const float an = sqrtf(nrm[gi]) * (1.0f + 0x1p-12f);
                        alpha = fmaf(fmaf(cst.c2, an, cst.c1), an, cst.c0);
                        split_tf32((nrm[gi] - eps2) + alpha, xh, xl);
                    }
                    *reinterpret_cast<float4 *>(As + core_offset(row, d4p, kpad)) = make_float4(xh, xl, 1.0f, 1.0f);
                    *reinterpret_cast<float4 *>(As + core_offset(row, d4p + 4, kpad)) =
                        make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    s_alpha[row] = alpha;
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_a_full);
        for (int it = 0; it < ntiles; ++it) {
            const int st = it % nst;
            if (it >= nst && !mbar_wait(&s_empty_b[st], (uint32_t)(it / nst - 1) & 1u, abort_flag)) give_up();
            unsigned char *Bs = Bs0 + (size_t)st * L.op_bytes;
            const int slot = it % kTcSide;
            {
                // source row of candidate row t4 of this tile
                const int64_t v = vbeg + (int64_t)it * kTcRows + t4;
                int32_t src = -1;
                if (v < vend) {
                    int lo = 0, hi = ncell - 1;  // last slot with s_vpre[slot] <= v
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (s_vpre[mid] <= v) lo = mid; else hi = mid - 1;
                    }
                    src = s_nstart[lo] + (int32_t)(v - s_vpre[lo]);
                }
                s_src[slot * kTcRows + t4] = src;
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");  // every transform warp reaches it
            if (s_abort) break;                               // uniform: read after the barrier
            auto prow = [&](int row) -> const float * {
                const int32_t src = s_src[slot * kTcRows + row];
                return src >= 0 ? a.xs + (int64_t)src * d4 : nullptr;
            };
            float nrm[4];
            stage_rows<C4P>(Bs, kpad, d4, s_c, prow, -2.0f, nrm, wx, lane);
            float bm = 0.0f;
            if (lane < 8) {
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) {
                    const int row = 8 * (wx + 4 * gi) + lane;
                    float yh = kTcBig, yl = 0.0f, beta = 0.0f;
                    if (s_src[slot * kTcRows + row] >= 0) {
                        const float bn = sqrtf(nrm[gi]) * (1.0f + 0x1p-12f);
                        beta = fmaf(cst.c2, bn, cst.c1) * bn;
                        split_tf32(nrm[gi] + beta, yh, yl);
                    }
                    *reinterpret_cast<float4 *>(Bs + core_offset(row, d4p, kpad)) = make_float4(1.0f, 1.0f, yh, yl);
                    *reinterpret_cast<float4 *>(Bs + core_offset(row, d4p + 4, kpad)) =
                        make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    s_beta[slot * kTcRows + row] = beta;
                    bm = fmaxf(bm, beta);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            if (lane == 0) s_bmax[slot * 4 + wx] = bm;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s_side[slot]);
                mbar_arrive(&s_full_b[st]);
            }
        }
    } else if (warp == 8) {
        // ---- MMA issue (one thread) ----
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(kTcRows, kTcRows);
            const uint32_t sbo = (uint32_t)(kpad / 4) * 128u;
            const uint32_t a_base = smem_u32(As), b_base = smem_u32(Bs0);
            int issued = 0;
            bool ok = mbar_wait(&s_a_full, 0, abort_flag);
            if (!ok) give_up();
            tc_fence_after_sync();
            for (int it = 0; ok && it < ntiles; ++it) {
                const int st = it % nst, buf = it & 1;
                if (!mbar_wait(&s_full_b[st], (uint32_t)(it / nst) & 1u, abort_flag) ||
                    (it >= 2 && !mbar_wait(&s_empty_d[buf], (uint32_t)((it >> 1) - 1) & 1u, abort_flag))) {
                    give_up();
                    break;
                }
                tc_fence_after_sync();
                const uint32_t bb = b_base + (uint32_t)st * L.op_bytes;
                for (int s = 0; s < kpad / 8; ++s)
                    mma_tf32(tmem + (uint32_t)buf * kTcRows, smem_desc(a_base + 256u * s, 128u, sbo),
                             smem_desc(bb + 256u * s, 128u, sbo), idesc, s > 0 ? 1u : 0u);
                mma_commit(&s_empty_b[st]);
                mma_commit(&s_full_d[buf]);
                issued = it + 1;
            }
            // every issued MMA has completed before tensor memory is released
            if (issued > 0 && !mbar_wait(&s_full_d[(issued - 1) & 1], (uint32_t)((issued - 1) >> 1) & 1u))
                give_up();
        }
    } else {
        // ---- accumulator readout and mask (warps 0-3; row i = tensor-memory lane i) ----
        const int i = 32 * warp + lane;
        uint32_t my_count = 0;
        bool ok = mbar_wait(&s_a_full, 0, abort_flag);
        if (!ok) give_up();
        const float alpha = ok ? s_alpha[i] : 0.0f;
        const float *qrow = a.xq + (int64_t)(q0 + (i < nq ? i : 0)) * d4;
        const int64_t row_word0 = a.tile_word[t] - a.word0;
        for (int it = 0; ok && it < ntiles; ++it) {
            const int buf = it & 1, slot = it % kTcSide;
            if (!mbar_wait(&s_side[slot], (uint32_t)(it / kTcSide) & 1u, abort_flag) ||
                !mbar_wait(&s_full_d[buf], (uint32_t)(it >> 1) & 1u, abort_flag)) {
                give_up();
                break;
            }
            tc_fence_after_sync();
            const float bmax = fmaxf(fmaxf(s_bmax[slot * 4], s_bmax[slot * 4 + 1]),
                                     fmaxf(s_bmax[slot * 4 + 2], s_bmax[slot * 4 + 3]));
            const float theta = 2.0f * (alpha + bmax) * (1.0f + 0x1p-20f);
            uint32_t words[4];
#pragma unroll
            for (int wc = 0; wc < 4; ++wc) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)buf * kTcRows + 32u * wc, v);
                tmem_ld_wait();
                uint32_t w = 0;
                float m = INFINITY;
#pragma unroll
                for (int j = 31; j >= 0; --j) {
                    w = __funnelshift_l(v[j], w, 1);  // (w << 1) | sign bit of u_j
                    m = fminf(m, fabsf(__uint_as_float(v[j])));
                }
                if (m <= theta) {
                    // a pair of this word may lie in the uncertain band: recheck exactly
                    // every pair with 0 <= u <= 2 (alpha + beta_j)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float uj = __uint_as_float(v[j]);
                        const int col = 32 * wc + j;
                        if (uj >= 0.0f && uj <= 2.0f * (alpha + s_beta[slot * kTcRows + col]) * (1.0f + 0x1p-20f)) {
                            const int32_t src = s_src[slot * kTcRows + col];
                            if (src >= 0 && tc_recheck(qrow, a.xs + (int64_t)src * d4, d4, eps2)) w |= 1u << j;
                        }
                    }
                }
                words[wc] = w;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty_d[buf]);
            const uint32_t nz = (words[0] ? 1u : 0u) | (words[1] ? 2u : 0u) | (words[2] ? 4u : 0u) | (words[3] ? 8u : 0u);
            if (i < nq && nz) {
                // only rows with a nonzero word store; the occupancy bitmap marks the
                // nonzero words (4 consecutive words share one 32-bit occupancy word)
                const int64_t v0 = vbeg + (int64_t)it * kTcRows;
                const int64_t wi = row_word0 + (int64_t)i * W4 + (v0 >> 5);
                *reinterpret_cast<uint4 *>(a.mask + wi) = make_uint4(words[0], words[1], words[2], words[3]);
                atomicOr(&a.occ[wi >> 5], nz << (wi & 31));
                my_count += __popc(words[0]) + __popc(words[1]) + __popc(words[2]) + __popc(words[3]);
            }
        }
        if (i < nq && my_count) atomicAdd(&a.qcount[a.tile_qoff[t] - a.q0 + i], (int32_t)my_count);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

template <int C4P>
cudaError_t launch_tc(const RefineArgs &a, const TcConst &c, const TcLayout &L, cudaStream_t s)
{
    static uint32_t configured = 0;  // largest dynamic shared memory requested so far
    if (L.total > configured) {
        HISS_TRY(cudaFuncSetAttribute(k_refine_tc<C4P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total));
        HISS_TRY(cudaFuncSetAttribute(k_refine_tc<C4P>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      (int)cudaSharedmemCarveoutMaxShared));
        configured = L.total;
    }
    k_refine_tc<C4P><<<(unsigned)a.nunits, kTcThreads, L.total, s>>>(a, c);
    return cudaGetLastError();
}

}  // namespace

int refine_tc_max_d4() { return 128; }

cudaError_t refine_tc(const RefineArgs &a, float eps, cudaStream_t s, int64_t *launches)
{
    if (a.d4 > refine_tc_max_d4()) return cudaErrorInvalidValue;
    const TcLayout L = tc_layout(a.d4);
    // margins (see k_refine_tc); computed in double, rounded up to float
    const double g = (double)(L.kpad + 24) * 0x1p-22;
    const double e = (double)eps, e2 = e * e;
    TcConst c;
    c.c1 = (float)(0x1p-9 * e * (1.0 + 0x1p-10) * (1.0 + 0x1p-20));
    c.c2 = (float)((0x1p-19 + 2.0 * g * (1.0 + 0x1p-10)) * (1.0 + 0x1p-20));
    c.c0 = (float)(g * e2 * (1.0 + 0x1p-10) * (1.0 + 0x1p-20) + 0x1p-100);
    ++*launches;
    if (a.nunits <= 0) return cudaSuccess;
    switch (tc_d4p(a.d4) / 4) {
    case 1: return launch_tc<1>(a, c, L, s);
    case 2: return launch_tc<2>(a, c, L, s);
    case 4: return launch_tc<4>(a, c, L, s);
    case 8: return launch_tc<8>(a, c, L, s);
    case 16: return launch_tc<16>(a, c, L, s);
    default: return launch_tc<32>(a, c, L, s);
    }
}

int refine_tc_tq() { return kTcRows; }
int refine_tc_chunk() { return kTcChunk; }

cudaError_t gram_tf32(const float *a, const float *b, int k, float *out, int *flags, cudaStream_t s,
                      int64_t *launches)
{
    const size_t smem = (size_t)2 * kGramRows * k * 4;
    HISS_TRY(cudaFuncSetAttribute(k_gram_tf32, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    k_gram_tf32<<<1, 128, smem, s>>>(a, b, k, out, flags);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace hiss
