// Candidate refinement on CUDA cores (RT-HiSS Section IV-E) and stream
// compaction of the result mask (Section IV-F1, Fig. 5).
//
// One thread block refines one unit: a tile of up to TQ queries of one grid
// cell against one chunk of the cell's stencil candidates (the cells around
// it, concatenated in stencil order).  The query tile stays in shared memory
// (two query rows interleaved per pair row); candidate tiles of TP points are
// staged through shared memory with cp.async, double-buffered, gathered row by
// row from the stencil cells.  Each thread owns an MQ x MP block of (query,
// candidate) squared distances, held as packed float32 pairs, and adds two
// dimensions per step with f32x2 subtract / multiply-add instructions (one
// instruction per pair and dimension instead of two).  Dimensions are in
// variance order, so after 4, 8 and 12 dimensions and then every 8 a warp checks
// whether all of its partial sums already exceed eps^2 and, if so, leaves the
// tile (early termination, Section IV-A).  The result is one bit per pair,
// sum <= eps^2, written to the query's mask row; the popcount of each word is
// accumulated into the query's neighbour count.
#include "hiss_internal.cuh"

namespace hiss {
namespace {

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Row stride of a staged tile, in floats: d4 plus padding chosen so that
// stride / 4 is odd, which makes the 16-byte loads of 8 consecutive rows hit
// 8 distinct bank quads.
__host__ __device__ __forceinline__ int tile_stride(int d4) { return ((d4 / 4) % 2 == 0) ? d4 + 4 : d4 + 8; }

template <int MQ, int MP>
struct Tile {
    static constexpr int TQ = 16 * MQ;   // 4 warps x 4 lanes x MQ queries
    static constexpr int TP = 16 * MP;   // 2 warps x 8 lanes x MP candidates
    static constexpr int CH = kChunkTiles * TP;
    static constexpr int WPW = MP / 4;   // mask words per query row per warp column
};

// Row stride of the pair-interleaved query tile, in floats: 2 d4 plus padding
// so that stride / 4 is odd (4 consecutive pair rows hit distinct bank quads).
__host__ __device__ __forceinline__ int pair_stride(int d4) { return (d4 % 8 == 0) ? 2 * d4 + 4 : 2 * d4 + 8; }

// Packed float32 pairs (two lanes of one 64-bit register), computed with the
// sm_100-family f32x2 instructions: each is two independent round-to-nearest
// float32 operations, so the results equal the scalar ones bit for bit.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo_of(f32x2 v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    (void)hi;
    return lo;
}
__device__ __forceinline__ float hi_of(f32x2 v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    (void)lo;
    return hi;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// The thread's MQ x MP block of squared distances is held as MQ/2 x MP
// packed pairs: acc[i2][j] = (query i = 2 i2, query i = 2 i2 + 1) x
// candidate j, i.e. query rows qbase + 8 i2 and qbase + 8 i2 + 4, candidate
// row pbase + 8 j.  The query tile Q2 stores those two rows interleaved
// (pair row pid = 16 wq + lq + 4 i2), so one 16-byte load gives both queries'
// dimensions k and k+1.
template <int MQ, int MP>
__device__ __forceinline__ float acc_at(const f32x2 (&acc)[MQ / 2][MP], int i, int j)
{
    return (i & 1) ? hi_of(acc[i >> 1][j]) : lo_of(acc[i >> 1][j]);
}

// Squared-distance increments of dimensions k and k+1 for the whole block.
// FIRST starts the sums (the first product is not added to a zeroed register).
template <int MQ, int MP, bool FIRST>
__device__ __forceinline__ void block_step2(f32x2 (&acc)[MQ / 2][MP], const float *Q2, const float *P, int S2, int S,
                                            int pidbase, int pbase, int k)
{
    f32x2 qa[MQ / 2], qb[MQ / 2];
#pragma unroll
    for (int i2 = 0; i2 < MQ / 2; ++i2) {
        const float4 v = *reinterpret_cast<const float4 *>(Q2 + (pidbase + 4 * i2) * S2 + 2 * k);
        qa[i2] = pk(v.x, v.y);  // dimension k of both queries
        qb[i2] = pk(v.z, v.w);  // dimension k + 1
    }
#pragma unroll
    for (int j = 0; j < MP; ++j) {
        const float2 pv = *reinterpret_cast<const float2 *>(P + (pbase + 8 * j) * S + k);
        const f32x2 p0 = pk(pv.x, pv.x), p1 = pk(pv.y, pv.y);
#pragma unroll
        for (int i2 = 0; i2 < MQ / 2; ++i2) {
            const f32x2 e0 = sub2(qa[i2], p0), e1 = sub2(qb[i2], p1);
            if constexpr (FIRST) acc[i2][j] = mul2(e0, e0);
            else acc[i2][j] = fma2(e0, e0, acc[i2][j]);
            acc[i2][j] = fma2(e1, e1, acc[i2][j]);
        }
    }
}

__device__ __forceinline__ float min3(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Smallest of the thread's MQ x MP partial sums (three-input minima).
template <int MQ, int MP>
__device__ __forceinline__ float block_min(const f32x2 (&acc)[MQ / 2][MP])
{
    float m = lo_of(acc[0][0]);
#pragma unroll
    for (int i2 = 0; i2 < MQ / 2; ++i2)
#pragma unroll
        for (int j = 0; j < MP; ++j) m = min3(m, lo_of(acc[i2][j]), hi_of(acc[i2][j]));
    return m;
}

// Resident blocks per SM the register budget is sized for.
#ifndef HISS_REFINE_MINB
#define HISS_REFINE_MINB 2
#endif

// PROF = true: no mask output; instead count, over all candidate pairs, the
// dimensions a pair needs when it stops at the first multiple of 4 whose
// partial sum exceeds eps^2 (prof[0]), and the dimensions the warp-level
// schedule of the PROF = false kernel executes (prof[1]).
template <int MQ, int MP, bool PROF>
__global__ void __launch_bounds__(kThreads, HISS_REFINE_MINB) k_refine(const RefineArgs a)
{
    using T = Tile<MQ, MP>;
    extern __shared__ __align__(16) float smem[];
    __shared__ int32_t s_nstart[kStencil];
    __shared__ int32_t s_vpre[kStencil + 1];
    __shared__ int64_t s_info[2];
    __shared__ int32_t s_src[2][T::TP];  // source row of each candidate row of a staged tile (-1: none)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d4 = a.d4, S = tile_stride(d4), S2 = pair_stride(d4), C4 = d4 / 4;
    float *Q2 = smem;
    float *Ps0 = smem + (T::TQ / 2) * S2;

    if (tid == 0) {
        const int64_t u = a.unit0 + blockIdx.x;
        int64_t lo = a.t0, hi = a.t1 - 1;  // last tile with tile_unit[t] <= u
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (a.tile_unit[mid] <= u) lo = mid; else hi = mid - 1;
        }
        s_info[0] = lo;
        s_info[1] = u - a.tile_unit[lo];
    }
    __syncthreads();
    const int64_t t = s_info[0];
    const int64_t chunk = s_info[1];
    const int32_t c = a.tile_cell[t];
    const int32_t q0 = a.tile_q0[t];
    const int nq = a.tile_nq[t];
    const int64_t B = a.bound[c];
    const int64_t W = (B + 31) >> 5;           // meaningful words of a mask row
    const int64_t W4 = (W + 3) & ~int64_t(3);  // row stride (16-byte rows)
    const int ns = a.nbr_cnt[c];
    if (tid < ns) {
        const int32_t nb = a.nbr[(int64_t)c * kStencil + tid];
        s_nstart[tid] = a.cell_start[nb];
        s_vpre[tid + 1] = a.cell_start[nb + 1] - a.cell_start[nb];
    }
    __syncthreads();
    if (tid == 0) {
        s_vpre[0] = 0;
        for (int i = 1; i <= ns; ++i) s_vpre[i] += s_vpre[i - 1];
    }

    // query tile, pair-interleaved: pair row pid holds rows a = 8 (pid / 4) +
    // pid % 4 and a + 4, dimension by dimension; rows >= nq are +inf
    for (int idx = tid; idx < (T::TQ / 2) * C4; idx += kThreads) {
        const int pid = idx / C4, cc = idx - pid * C4;
        const int ra = 8 * (pid >> 2) + (pid & 3), rb = ra + 4;
        const float4 inf4 = make_float4(INFINITY, INFINITY, INFINITY, INFINITY);
        const float4 x = ra < nq ? *reinterpret_cast<const float4 *>(a.xq + (int64_t)(q0 + ra) * d4 + 4 * cc) : inf4;
        const float4 y = rb < nq ? *reinterpret_cast<const float4 *>(a.xq + (int64_t)(q0 + rb) * d4 + 4 * cc) : inf4;
        float4 *dst = reinterpret_cast<float4 *>(Q2 + pid * S2 + 8 * cc);
        dst[0] = make_float4(x.x, y.x, x.y, y.y);
        dst[1] = make_float4(x.z, y.z, x.w, y.w);
    }
    __syncthreads();  // s_vpre complete

    const int64_t vbeg = chunk * T::CH;
    const int64_t vend = min(B, vbeg + (int64_t)T::CH);
    const int ntiles = (int)((vend - vbeg + T::TP - 1) / T::TP);

    // source rows of candidate tile v0 .. v0 + TP, looked up once per row
    auto fill_src = [&](int buf, int64_t v0) {
        for (int r = tid; r < T::TP; r += kThreads) {
            const int64_t v = v0 + r;
            int32_t src = -1;
            if (v < vend) {
                int lo = 0, hi = ns - 1;  // last slot with s_vpre[slot] <= v
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_vpre[mid] <= v) lo = mid; else hi = mid - 1;
                }
                src = s_nstart[lo] + (int32_t)(v - s_vpre[lo]);
            }
            s_src[buf][r] = src;
        }
    };
    // this thread's first (row, 16-byte chunk) of a staged tile and the step
    const int r_first = tid / C4, c_first = tid - (tid / C4) * C4;
    const int r_step = kThreads / C4, c_step = kThreads - (kThreads / C4) * C4;
    auto load_p = [&](int buf) {
        float *P = Ps0 + buf * T::TP * S;
        int r = r_first, cc = c_first;
        for (int idx = tid; idx < T::TP * C4; idx += kThreads) {
            float *dst = P + r * S + 4 * cc;
            const int32_t src = s_src[buf][r];
            if (src >= 0) cp_async16(dst, a.xs + (int64_t)src * d4 + 4 * cc);
            else *reinterpret_cast<float4 *>(dst) = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            r += r_step;
            cc += c_step;
            if (cc >= C4) {
                cc -= C4;
                ++r;
            }
        }
    };

    fill_src(0, vbeg);
    if (ntiles > 1) fill_src(1, vbeg + T::TP);
    __syncthreads();
    load_p(0);
    cp_async_commit();

    const int wq = warp >> 1, wp = warp & 1;
    const int lq = lane >> 3, lp = lane & 7;
    const int qbase = wq * (4 * MQ) + lq;  // query row i: qbase + 4 i
    const int pidbase = wq * (2 * MQ) + lq; // pair row of queries 2 i2, 2 i2 + 1: pidbase + 4 i2
    const int pbase = wp * (8 * MP) + lp;  // candidate row j: pbase + 8 j
    const float eps2 = a.eps2;
    uint32_t my_count = 0;                 // neighbours of query row qbase + 4 lp (lp < MQ)
    const int64_t row_word0 = a.tile_word[t] - a.word0;
    uint64_t prof_alg = 0, prof_exec = 0;

    for (int it = 0; it < ntiles; ++it) {
        const int64_t v0 = vbeg + (int64_t)it * T::TP;
        if (it + 1 < ntiles) {
            load_p((it + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const float *P = Ps0 + (it & 1) * T::TP * S;
        f32x2 acc[MQ / 2][MP];
        if constexpr (PROF) {
            // all dimensions, counting live pairs step by step
            bool warp_live = true;
            block_step2<MQ, MP, true>(acc, Q2, P, S2, S, pidbase, pbase, 0);
            block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, 2);
            int live = 0;
#pragma unroll
            for (int i = 0; i < MQ; ++i)
#pragma unroll
                for (int j = 0; j < MP; ++j) live += (qbase + 4 * i < nq && v0 + pbase + 8 * j < vend) ? 1 : 0;
            const int valid = live;
            prof_alg += (uint64_t)valid * (uint64_t)min(4, a.d);
            prof_exec += (uint64_t)valid * (uint64_t)min(4, a.d);
            for (int k = 4; k < d4; k += 4) {
                live = 0;
#pragma unroll
                for (int i = 0; i < MQ; ++i)
#pragma unroll
                    for (int j = 0; j < MP; ++j) live += (acc_at<MQ, MP>(acc, i, j) <= eps2) ? 1 : 0;
                if (k < 16 || (k & 7) == 0)
                    if (__all_sync(0xffffffffu, block_min<MQ, MP>(acc) > eps2)) warp_live = false;
                if (!__any_sync(0xffffffffu, live > 0) && !warp_live) break;
                const uint64_t step = (uint64_t)min(4, a.d - k);
                prof_alg += (uint64_t)live * step;
                if (warp_live) prof_exec += (uint64_t)valid * step;
                block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k);
                block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k + 2);
            }
            if (it + 2 < ntiles) fill_src(it & 1, v0 + 2 * T::TP);
            __syncthreads();
            continue;
        }
        block_step2<MQ, MP, true>(acc, Q2, P, S2, S, pidbase, pbase, 0);
        block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, 2);
        // warp-level early termination: checked after 4, 8 and 12 dimensions,
        // then every 8 (the pairs are in variance order, most leave early)
        bool any_close = true;
        for (int k = 4;; k += 4) {
            if (k == d4) {
                any_close = __any_sync(0xffffffffu, block_min<MQ, MP>(acc) <= eps2);
                break;
            }
            if (k < 16 || (k & 7) == 0) {
                if (__all_sync(0xffffffffu, block_min<MQ, MP>(acc) > eps2)) {
                    any_close = false;
                    break;
                }
            }
            block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k);
            block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k + 2);
        }

        // one bit per pair; OR across the 8 lanes of a query row; lane lp
        // writes the words of query j = lp
        const int64_t word_tile = v0 >> 5;
        if (any_close) {
#pragma unroll
            for (int i = 0; i < MQ; ++i) {
#pragma unroll
                for (int wi = 0; wi < T::WPW; ++wi) {
                    uint32_t w = 0;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        w |= (acc_at<MQ, MP>(acc, i, 4 * wi + jj) <= eps2 ? 1u : 0u) << (lp + 8 * jj);
                    w |= __shfl_xor_sync(0xffffffffu, w, 1);
                    w |= __shfl_xor_sync(0xffffffffu, w, 2);
                    w |= __shfl_xor_sync(0xffffffffu, w, 4);
                    const int qr = qbase + 4 * i;
                    const int64_t wcol = word_tile + wp * T::WPW + wi;
                    if (lp == i && qr < nq && wcol < W) {
                        a.mask[row_word0 + (int64_t)qr * W4 + wcol] = w;
                        my_count += __popc(w);
                    }
                }
            }
        } else if (lp < MQ && qbase + 4 * lp < nq) {
            // no pair of the warp is within eps: zero words for this lane's row
            uint32_t *row = a.mask + row_word0 + (int64_t)(qbase + 4 * lp) * W4;
#pragma unroll
            for (int wi = 0; wi < T::WPW; ++wi) {
                const int64_t wcol = word_tile + wp * T::WPW + wi;
                if (wcol < W) row[wcol] = 0u;
            }
        }
        if (it + 2 < ntiles) fill_src(it & 1, v0 + 2 * T::TP);
        __syncthreads();
    }
    if constexpr (PROF) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            prof_alg += __shfl_xor_sync(0xffffffffu, prof_alg, o);
            prof_exec += __shfl_xor_sync(0xffffffffu, prof_exec, o);
        }
        if (lane == 0) {
            atomicAdd(reinterpret_cast<unsigned long long *>(a.prof), (unsigned long long)prof_alg);
            atomicAdd(reinterpret_cast<unsigned long long *>(a.prof) + 1, (unsigned long long)prof_exec);
        }
        return;
    }
    if (lp < MQ) {
        const int qr = qbase + 4 * lp;
        if (qr < nq && my_count) atomicAdd(&a.qcount[a.tile_qoff[t] - a.q0 + qr], (int32_t)my_count);
    }
}

template <int MQ, int MP, bool PROF>
cudaError_t launch_refine(const RefineArgs &a, cudaStream_t s)
{
    using T = Tile<MQ, MP>;
    const size_t smem = sizeof(float) * ((size_t)(T::TQ / 2) * pair_stride(a.d4) + (size_t)2 * T::TP * tile_stride(a.d4));
    static size_t configured = 0;  // largest dynamic shared memory requested so far
    if (smem > configured) {
        HISS_TRY(cudaFuncSetAttribute(k_refine<MQ, MP, PROF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
        configured = smem;
    }
    if (a.nunits <= 0) return cudaSuccess;
    k_refine<MQ, MP, PROF><<<(unsigned)a.nunits, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// ---- compaction: one warp per query row --------------------------------------
constexpr int kCompactWarps = 8;

__global__ void __launch_bounds__(kCompactWarps * 32) k_compact(const CompactArgs a)
{
    __shared__ int32_t s_start[kCompactWarps][kStencil];
    __shared__ int32_t s_vpre[kCompactWarps][kStencil + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gq = (int64_t)blockIdx.x * kCompactWarps + warp;
    if (gq >= a.nq) return;
    const int64_t qa = a.q0 + gq;
    int64_t lo = a.t0, hi = a.t1 - 1;  // last tile with tile_qoff[t] <= qa
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (a.tile_qoff[mid] <= qa) lo = mid; else hi = mid - 1;
    }
    const int64_t t = lo;
    const int64_t i = qa - a.tile_qoff[t];
    const int32_t c = a.tile_cell[t];
    const int32_t row = a.tile_q0[t] + (int32_t)i;
    const int64_t B = a.bound[c];
    const int64_t W = (B + 31) >> 5;
    const int64_t W4 = (W + 3) & ~int64_t(3);
    const int64_t woff = a.tile_word[t] - a.word0 + i * W4;
    if (lane == 0) {
        a.query_ids[gq] = a.qids[row];
        a.query_rows[gq] = row;
        if (a.cand) a.cand[gq] = B;
        if (a.mask_row_ptr) {
            a.mask_row_ptr[gq] = woff;
            if (gq == a.nq - 1) a.mask_row_ptr[a.nq] = woff + W4;
        }
    }
    if (!a.cols) return;
    const int ns = a.nbr_cnt[c];
    int32_t sz = 0;
    if (lane < ns) {
        const int32_t nb = a.nbr[(int64_t)c * kStencil + lane];
        s_start[warp][lane] = a.cell_start[nb];
        sz = a.cell_start[nb + 1] - a.cell_start[nb];
    }
    int32_t incl = sz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane < ns) s_vpre[warp][lane] = incl - sz;
    __syncwarp();

    // rows are 16-byte aligned: each lane takes four words per step
    const uint4 *mrow = reinterpret_cast<const uint4 *>(a.mask + woff);
    int32_t *out = a.cols + a.row_ptr[gq];
    int64_t run = 0;
    for (int64_t w0 = 0; w0 < W; w0 += 128) {
        const int64_t w = w0 + 4 * lane;
        uint32_t wd[4] = {0u, 0u, 0u, 0u};
        if (w < W) {
            const uint4 v = mrow[w >> 2];
            wd[0] = v.x;
            wd[1] = w + 1 < W ? v.y : 0u;
            wd[2] = w + 2 < W ? v.z : 0u;
            wd[3] = w + 3 < W ? v.w : 0u;
        }
        const int cnt = __popc(wd[0]) + __popc(wd[1]) + __popc(wd[2]) + __popc(wd[3]);
        int ex = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, ex, o);
            if (lane >= o) ex += v;
        }
        const int total = __shfl_sync(0xffffffffu, ex, 31);
        int64_t pos = run + ex - cnt;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint32_t word = wd[h];
            while (word) {
                const int b = __ffs(word) - 1;
                word &= word - 1;
                const int64_t v = (w + h) * 32 + b;
                int l = 0, hh = ns - 1;
                while (l < hh) {
                    const int m = (l + hh + 1) >> 1;
                    if (s_vpre[warp][m] <= v) l = m; else hh = m - 1;
                }
                out[pos++] = a.ids[s_start[warp][l] + (v - s_vpre[warp][l])];
            }
        }
        run += total;
    }
}

__global__ void k_word_popc(const uint32_t *words, int64_t nbits, int32_t *cnt)
{
    const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nw = (nbits + 31) >> 5;
    if (w >= nw) return;
    uint32_t x = words[w];
    const int64_t rem = nbits - w * 32;
    if (rem < 32) x &= (1u << rem) - 1u;
    cnt[w] = __popc(x);
}

__global__ void k_word_positions(const uint32_t *words, int64_t nbits, const int64_t *off, int64_t *pos)
{
    const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nw = (nbits + 31) >> 5;
    if (w >= nw) return;
    uint32_t x = words[w];
    const int64_t rem = nbits - w * 32;
    if (rem < 32) x &= (1u << rem) - 1u;
    int64_t o = off[w];
    while (x) {
        const int b = __ffs(x) - 1;
        x &= x - 1;
        pos[o++] = w * 32 + b;
    }
}

}  // namespace

int refine_tq(int d4) { return d4 <= 128 ? Tile<8, 8>::TQ : Tile<4, 4>::TQ; }

cudaError_t refine(const RefineArgs &a, cudaStream_t s, int64_t *launches)
{
    ++*launches;
    if (a.d4 <= 128) return launch_refine<8, 8, false>(a, s);
    return launch_refine<4, 4, false>(a, s);
}

cudaError_t refine_profile(const RefineArgs &a, cudaStream_t s, int64_t *launches)
{
    ++*launches;
    if (a.d4 <= 128) return launch_refine<8, 8, true>(a, s);
    return launch_refine<4, 4, true>(a, s);
}

int refine_chunk(int d4) { return d4 <= 128 ? Tile<8, 8>::CH : Tile<4, 4>::CH; }

cudaError_t compact(const CompactArgs &a, cudaStream_t s, int64_t *launches)
{
    if (a.nq <= 0) return cudaSuccess;
    const int64_t blocks = (a.nq + kCompactWarps - 1) / kCompactWarps;
    k_compact<<<(unsigned)blocks, kCompactWarps * 32, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t mask_positions(const uint32_t *words, int64_t nbits, int64_t *pos, int64_t *count, int64_t *tmp,
                           cudaStream_t s, int64_t *launches)
{
    // tmp: [nw] int32 counts, then [nw+1] int64 offsets, then scan scratch
    const int64_t nw = (nbits + 31) >> 5;
    int32_t *cnt = reinterpret_cast<int32_t *>(tmp);
    int64_t *off = tmp + (nw + 1) / 2 + 1;
    int64_t *scratch = off + nw + 1;
    const unsigned blocks = (unsigned)((nw + 255) / 256);
    if (nw == 0) return cudaMemsetAsync(count, 0, sizeof(int64_t), s);
    k_word_popc<<<blocks, 256, 0, s>>>(words, nbits, cnt);
    HISS_TRY(scan_i32_to_i64(cnt, off, nw, scratch, s, launches));
    k_word_positions<<<blocks, 256, 0, s>>>(words, nbits, off, pos);
    *launches += 2;
    HISS_TRY(cudaMemcpyAsync(count, off + nw, sizeof(int64_t), cudaMemcpyDeviceToDevice, s));
    return cudaGetLastError();
}

}  // namespace hiss
