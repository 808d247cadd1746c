// Candidate refinement on CUDA cores (RT-HiSS Section IV-E) and stream
// compaction of the result mask (Section IV-F1, Fig. 5).
//
// One thread block refines one unit: a tile of up to TQ queries of one grid
// cell against one chunk of the cell's stencil candidates (the cells around
// it, concatenated in stencil order).  The query tile stays in shared memory
// (two query rows interleaved per pair row).  A producer warp streams the
// candidates through a ring of shared-memory stages, gathering each candidate
// row (its first 16 or 32 dimensions above 32) from its stencil cell with
// cp.async, completion tracked by mbarriers.  Each compute thread owns an
// 8 x 4 block of (query, candidate) squared distances (4 x 4 above 64
// dimensions), held as packed float32 pairs, and adds two dimensions per
// step with f32x2 subtract / multiply-add instructions (one instruction per
// pair and dimension instead of two).  A block first drops the candidate
// tiles whose rows' 32-row group boxes (over the three index dimensions,
// built with the index) are all farther than eps from its query tile's box:
// they are neither streamed nor refined.  Before any arithmetic a warp also
// skips a staged tile whose exact box is farther than eps from its queries'
// box.  Dimensions are in variance order, so after every
// 2 dimensions (8 x 4 blocks) or 4 (4 x 4 blocks) a warp checks whether all
// of its partial sums already exceed eps^2 and, if so, leaves the tile
// (early termination, Section IV-A); at 64 dimensions and more, a warp left
// with few pairs within eps^2, or with any when the staged dimensions run
// out, finishes them one pair per lane.  The result is one bit per pair,
// sum <= eps^2, written to the query's mask row; the popcount of each word
// is accumulated into the query's neighbour count.
#include "hiss_internal.cuh"
#include "ptx.cuh"

namespace hiss {
namespace {

// ---- staging geometry ---------------------------------------------------------
// Row stride of a staged candidate tile, in floats: d4 plus padding chosen so
// that stride / 4 is odd, which makes the 8-byte loads of 8 consecutive rows
// hit 8 distinct bank quads.

__host__ __device__ __forceinline__ int tile_stride(int d4) { return ((d4 / 4) % 2 == 0) ? d4 + 4 : d4 + 8; }

// Row stride of the pair-interleaved query tile, in floats: 2 d4 + 4, so that
// stride / 4 is odd (4 consecutive pair rows hit distinct bank quads).
__host__ __device__ __forceinline__ int pair_stride(int d4) { return 2 * d4 + 4; }

// Thread-block shape of the refinement.  Eight compute warps (4 query warps x
// 2 candidate warps) and one producer warp.  A compute warp owns a 4 MQ x 32
// block of (query, candidate) pairs of the staged tile; each of its threads
// owns MQ x MP of them.
constexpr int kQueryWarps = 4, kCandWarps = 2;
constexpr int kComputeWarps = kQueryWarps * kCandWarps;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kRefineThreads = kComputeThreads + 32;
#ifndef HISS_REFINE_CHUNK
#define HISS_REFINE_CHUNK 8192
#endif
constexpr int kCH = HISS_REFINE_CHUNK;  // candidates per unit (a multiple of 64)
__host__ __device__ __forceinline__ int refine_chunk_of(int) { return kCH; }

// Per-thread block MQ x MP: 8 x 4 up to d4 = 64 (tiles of 128 queries x 64
// candidates), 4 x 4 above (64 x 64), so that two blocks fit per SM.
template <int MQ, int MP>
struct Geo {
    static constexpr int TQ = kQueryWarps * 4 * MQ;  // queries per tile
    static constexpr int TP = kCandWarps * 8 * MP;   // candidates per staged tile
};
#ifndef HISS_REFINE_STAGES
#define HISS_REFINE_STAGES 6
#endif
constexpr int kMaxStages = HISS_REFINE_STAGES;

// Dimensions of each candidate row that the ring stages: all of them up to
// HISS_STAGE_DIMS, else the first HISS_STAGE_DIMS.  Most pairs leave within
// the first few dimensions (variance order), so staging whole rows of 64 or
// 128 dimensions would fill the ring with data that is never read and leave
// room for only two stages; the few pairs still within eps^2 after the staged
// dimensions read the rest of their candidate's row from global memory (see
// finish_pairs).  The work-profile build stages every dimension.
// Measured on GB300: 64-dimensional subspace data 2.73 s with 32 dimensions
// staged, 2.62 s with 16 (six stages instead of four); 128-dimensional
// spectrum data 0.38 s with 32, 0.49 s with 16.
#ifndef HISS_STAGE_DIMS
#define HISS_STAGE_DIMS 32
#endif
#ifndef HISS_STAGE_DIMS64
#define HISS_STAGE_DIMS64 16
#endif
template <bool PROF>
__host__ __device__ __forceinline__ constexpr int staged_dims(int d4)
{
    return (PROF || d4 <= 32) ? d4 : (d4 <= 64 ? HISS_STAGE_DIMS64 : HISS_STAGE_DIMS);
}

// Survivor mode.  A warp still in a tile after surv_dim dimensions counts its
// pairs whose partial sum is still <= eps^2; if there are at most kSurvMax
// of them and at least 8 dimensions are left, it stops the blocked
// arithmetic and finishes those pairs one per lane, continuing each pair's
// own float32 sum in dimension order (the same subtract and multiply-add, so
// the same sums and bits), with a per-pair exit.  A warp still in a tile when
// the staged dimensions run out finishes all of its live pairs that way,
// kSurvMax at a time.  The early switch is used with 4 x 4 blocks (d4 > 64)
// and with 8 x 4 blocks at d4 = 64.  With fewer dimensions the
// one-pair-per-lane path (2 scalar instructions and about 0.75 shared loads
// per pair-dimension, against 1 packed instruction in a register block) costs
// more than the blocked dimensions it saves.  The lists sit in dynamic shared
// memory after the ring, only in builds that use them.
#ifndef HISS_SURV8_DIM
#define HISS_SURV8_DIM 16
#endif
#ifndef HISS_SURV4_DIM
#define HISS_SURV4_DIM 16
#endif
constexpr int kSurvMax = 64;  // survivors a warp takes at a time (a multiple of 32)
// 16-byte chunks of a candidate row a survivor loads from global memory at
// once (its latency is paid once per chunk group).  Measured on GB300:
// spectrum (d4 = 128) 397 / 374 / 490 ms and subspace (d4 = 64) 2.39 / 2.57 /
// 5.03 s with 2 / 4 / 8 chunks (8 spills registers of the blocked loop).
#ifndef HISS_SURV_AHEAD
#define HISS_SURV_AHEAD 4
#endif
#ifndef HISS_SURV_AHEAD64
#define HISS_SURV_AHEAD64 2
#endif
__host__ __device__ __forceinline__ constexpr int surv_ahead(int d4) { return d4 <= 64 ? HISS_SURV_AHEAD64 : HISS_SURV_AHEAD; }
// Dimension after which a warp may switch to survivor mode (a multiple of 4),
// 0 for none.
__host__ __device__ __forceinline__ constexpr int surv_dim(int mq, int d4)
{
    return mq == 4 ? HISS_SURV4_DIM : (d4 == 64 ? HISS_SURV8_DIM : 0);
}
template <bool PROF>
__host__ __device__ __forceinline__ constexpr bool uses_survivors(int mq, int d4)
{
    return surv_dim(mq, d4) > 0 || staged_dims<PROF>(d4) < d4;
}
template <bool PROF>
__host__ __device__ __forceinline__ constexpr size_t surv_bytes(int mq, int d4)
{
    // per compute warp: kSurvMax partial sums (float) and pair codes (uint16),
    // and 32 mask words
    return uses_survivors<PROF>(mq, d4) ? (size_t)kComputeWarps * (kSurvMax * 6 + 32 * 4) : 0;
}

// Bytes of one ring stage: the staged rows, then (when rows are staged
// partly) the global row index of each staged candidate.
template <int MQ, int MP, bool PROF>
__host__ __device__ __forceinline__ int stage_bytes(int d4)
{
    const int ds = staged_dims<PROF>(d4);
    return Geo<MQ, MP>::TP * (tile_stride(ds) * 4 + (ds < d4 ? 4 : 0));
}

// Stages of the candidate ring: as many as fit (up to 6, at least 2) in
// about a third of the SM's shared memory, so that two or three blocks stay
// resident per SM.
template <int MQ, int MP, bool PROF>
__host__ __device__ __forceinline__ int refine_stages(int d4)
{
    const int q2 = (Geo<MQ, MP>::TQ / 2) * pair_stride(d4) * 4 + (int)surv_bytes<PROF>(MQ, d4);
    int ns = (75 * 1024 - q2) / stage_bytes<MQ, MP, PROF>(d4);
    return ns < 2 ? 2 : (ns > kMaxStages ? kMaxStages : ns);
}

template <int MQ, int MP, bool PROF>
__host__ __forceinline__ size_t refine_smem(int d4)
{
    using G = Geo<MQ, MP>;
    return sizeof(float) * (size_t)(G::TQ / 2) * pair_stride(d4) +
           (size_t)refine_stages<MQ, MP, PROF>(d4) * stage_bytes<MQ, MP, PROF>(d4) + surv_bytes<PROF>(MQ, d4);
}

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

__device__ __forceinline__ void compute_warps_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}

// The thread's MQ x MP block of squared distances is held as MQ/2 x MP
// packed pairs: acc[i2][j] = (query i = 2 i2, query i = 2 i2 + 1) x
// candidate j, i.e. query rows qbase + 8 i2 and qbase + 8 i2 + 4, candidate
// row pbase + 8 j.  The query tile Q2 stores those two rows interleaved
// (pair row pid = pidbase + 4 i2), so one 16-byte load gives both queries'
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

// Minimum / maximum over the warp in one instruction (sm_100-family
// redux.sync on float32; NaN-free inputs here).
__device__ __forceinline__ float warp_min(float v)
{
    float r;
    asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float min3(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// One level of a min tree over v[0..N): v[t] = min(v[3t], v[3t+1], v[3t+2]),
// repeated until one value is left (indices are compile-time constants, so v
// stays in registers).
template <int N>
__device__ __forceinline__ void min_levels(float (&v)[32])
{
    constexpr int M = (N + 2) / 3;
#pragma unroll
    for (int t = 0; t < M; ++t) {
        const int b = 3 * t;
        if (b + 2 < N) v[t] = min3(v[b], v[b + 1], v[b + 2]);
        else if (b + 1 < N) v[t] = fminf(v[b], v[b + 1]);
        else v[t] = v[b];
    }
    if constexpr (M > 1) min_levels<M>(v);
}

// Smallest of the thread's MQ x MP partial sums: a tree of three-input
// minima (depth 4 for 32 values instead of a chain of 16 dependent ones).
template <int MQ, int MP>
__device__ __forceinline__ float block_min(const f32x2 (&acc)[MQ / 2][MP])
{
    constexpr int N = MQ * MP;
    static_assert(N <= 32, "min tree size");
    float v[32];
#pragma unroll
    for (int i2 = 0; i2 < MQ / 2; ++i2)
#pragma unroll
        for (int j = 0; j < MP; ++j) {
            v[2 * (i2 * MP + j)] = lo_of(acc[i2][j]);
            v[2 * (i2 * MP + j) + 1] = hi_of(acc[i2][j]);
        }
    min_levels<N>(v);
    return v[0];
}

// Rank of this thread's first live pair among the warp's (exclusive prefix
// of the per-thread counts of partial sums <= eps^2) and the warp's total.
template <int MQ, int MP>
__device__ __forceinline__ void live_scan(const f32x2 (&acc)[MQ / 2][MP], float eps2, int lane, int *first,
                                          int *total)
{
    int live = 0;
#pragma unroll
    for (int i = 0; i < MQ; ++i)
#pragma unroll
        for (int j = 0; j < MP; ++j) live += (acc_at<MQ, MP>(acc, i, j) <= eps2) ? 1 : 0;
    int incl = live;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    *first = incl - live;
    *total = __shfl_sync(0xffffffffu, incl, 31);
}

// Survivor mode of one warp at dimension k: the pairs of its MQ x MP blocks
// whose partial sum is still <= eps^2 (total of them over the warp; this
// thread's rank from first) are listed in shared memory, kSurvMax at a time
// (query row << 5 | candidate column within the warp tile, and the partial
// sum), then finished one per lane: dimensions k, k+1, ... are added to the
// pair's own partial sum with the blocked path's round-to-nearest subtract
// and fused multiply-add, in the same order, so the final sum and bit are
// those of the blocked path.  Dimensions below ds come from the staged tile
// P; the rest from the candidate's row in global memory (xs, row srow[column],
// 16 dimensions loaded ahead).  A pair stops once its sum exceeds eps^2.  The
// bits of the pairs within eps^2 are gathered in sword[query row of the warp
// tile] (bit = candidate column), ready for the caller after the closing
// __syncwarp.
template <int MQ, int MP, int AHEAD>
__device__ __forceinline__ void survivors(const f32x2 (&acc)[MQ / 2][MP], const float *Q2, const float *P,
                                          const float *xs, const int32_t *srow, int S2, int S, int k, int ds, int d4,
                                          float eps2, int first, int total, int lane, int wq, int wp, float *spart,
                                          uint16_t *sidx, uint32_t *sword)
{
    const int lq = lane >> 3, lp = lane & 7;
    sword[lane] = 0u;
    for (int b0 = 0; b0 < total; b0 += kSurvMax) {
        __syncwarp();
        int pos = first;
#pragma unroll
        for (int i = 0; i < MQ; ++i)
#pragma unroll
            for (int j = 0; j < MP; ++j) {
                const float v = acc_at<MQ, MP>(acc, i, j);
                if (v <= eps2) {
                    if (pos >= b0 && pos < b0 + kSurvMax) {
                        sidx[pos - b0] = (uint16_t)(((lq + 4 * i) << 5) | (lp + 8 * j));
                        spart[pos - b0] = v;
                    }
                    ++pos;
                }
            }
        __syncwarp();
        const int cnt = min(kSurvMax, total - b0);
        for (int e = lane; e < cnt; e += 32) {
            const int code = sidx[e];
            const int r = code >> 5, pc = code & 31;
            const int qt = wq * (4 * MQ) + r;  // query row of the tile
            // the query's values: every other float of its pair row, from the
            // first or the second slot
            const float *qv = Q2 + (4 * (qt >> 3) + (qt & 3)) * S2 + ((qt >> 2) & 1);
            const int prow_i = wp * (8 * MP) + pc;
            const float *prow = P + prow_i * S;
            float sum = spart[e];
            int kk = k;
            for (; kk < ds; kk += 4) {
                const float4 pv = *reinterpret_cast<const float4 *>(prow + kk);
                float df;
                df = __fsub_rn(qv[2 * kk], pv.x);
                sum = __fmaf_rn(df, df, sum);
                df = __fsub_rn(qv[2 * kk + 2], pv.y);
                sum = __fmaf_rn(df, df, sum);
                df = __fsub_rn(qv[2 * kk + 4], pv.z);
                sum = __fmaf_rn(df, df, sum);
                df = __fsub_rn(qv[2 * kk + 6], pv.w);
                sum = __fmaf_rn(df, df, sum);
                if (sum > eps2) break;
            }
            if (sum <= eps2 && kk < d4) {
                // dimensions past the staged ones, from the candidate's row
                // (a live pair's candidate is a real row: padding rows are at
                // +inf distance)
                const float4 *pg = reinterpret_cast<const float4 *>(xs + (int64_t)srow[prow_i] * d4);
                for (; kk < d4; kk += 4 * AHEAD) {
                    float4 pv[AHEAD];
#pragma unroll
                    for (int u = 0; u < AHEAD; ++u)
                        if (kk + 4 * u < d4) pv[u] = __ldg(pg + (kk >> 2) + u);
#pragma unroll
                    for (int u = 0; u < AHEAD; ++u) {
                        const int k4 = kk + 4 * u;
                        if (k4 < d4) {
                            float df;
                            df = __fsub_rn(qv[2 * k4], pv[u].x);
                            sum = __fmaf_rn(df, df, sum);
                            df = __fsub_rn(qv[2 * k4 + 2], pv[u].y);
                            sum = __fmaf_rn(df, df, sum);
                            df = __fsub_rn(qv[2 * k4 + 4], pv[u].z);
                            sum = __fmaf_rn(df, df, sum);
                            df = __fsub_rn(qv[2 * k4 + 6], pv[u].w);
                            sum = __fmaf_rn(df, df, sum);
                        }
                    }
                    if (sum > eps2) break;
                }
            }
            if (sum <= eps2) atomicOr(&sword[r], 1u << pc);
        }
    }
    __syncwarp();
}

// Where a warp checks for early termination (k = dimensions summed so far):
// with 8 x 4 blocks (d4 <= 64) after every 2 dimensions from the first check
// on, with 4 x 4 blocks after every 4 (there the pairs leave later, and the
// shorter steps need two per loop iteration to overlap their loads).  The box
// test has already removed most of the tiles that an early check would end,
// so the first check comes later: after 10 dimensions at d4 = 16, 6 at
// d4 = 32, 8 at d4 = 64 (and at most half the dimensions elsewhere), 4 with
// 4 x 4 blocks.  Measured on GB300 (refinement): exp (d = 16) 15.3 s with the
// first check after 2, 14.7 s after 10; gmm (d = 32) 35.2 ms after 2, 34.4
// after 6; subspace (d = 64) 2.35 / 2.32 / 2.30 / 2.29 / 2.32 / 2.39 s after
// 2 / 4 / 6 / 8 / 10 / 12; spectrum (d = 128, 4 x 4 blocks) 366 / 366 /
// 367 / 370 ms after 4 / 8 / 12 / 16.
#ifndef HISS_FIRST_CHECK16
#define HISS_FIRST_CHECK16 10
#endif
#ifndef HISS_FIRST_CHECK32
#define HISS_FIRST_CHECK32 6
#endif
#ifndef HISS_FIRST_CHECK64
#define HISS_FIRST_CHECK64 8
#endif
#ifndef HISS_FIRST_CHECK4
#define HISS_FIRST_CHECK4 4
#endif
__host__ __device__ __forceinline__ constexpr int first_check(int d4)
{
    return d4 == 16 ? HISS_FIRST_CHECK16
                    : (d4 == 32 ? HISS_FIRST_CHECK32 : (d4 / 2 < HISS_FIRST_CHECK64 ? d4 / 2 : HISS_FIRST_CHECK64));
}
template <int MQ>
__device__ __forceinline__ bool exit_check_at(int k, int d4)
{
    return MQ == 8 ? k >= first_check(d4) : ((k & 3) == 0 && k >= HISS_FIRST_CHECK4);
}


// Stage waits sleep in the barrier (mbarrier.try_wait with a suspend-time
// hint) rather than polling it, so that waiting warps (mostly the producer,
// which runs ahead of the compute warps) leave the issue slots to the
// arithmetic.  0: poll.
#ifndef HISS_WAIT_SUSPEND
#define HISS_WAIT_SUSPEND 1
#endif
__device__ __forceinline__ bool refine_wait(uint64_t *bar, uint32_t parity)
{
#if HISS_WAIT_SUSPEND
    return mbar_wait_suspend(bar, parity);
#else
    return mbar_wait(bar, parity);
#endif
}

// Resident blocks per SM the register budget is sized for.
#ifndef HISS_REFINE_MINB
#define HISS_REFINE_MINB 3
#endif


// Per-unit state of a refinement block.
struct Unit {
    int64_t t;           // query tile
    int64_t B, W, W4;    // candidates of the tile's cell, meaningful mask words per row, row stride
    int64_t vbeg, vend;  // this unit's chunk of the cell's concatenated stencil
    int32_t c, q0;       // cell, first query row
    int nq, ncell, ntiles;
};

// Finds the block's unit (the last query tile whose first unit is at most
// the block's), initialises the stage barriers and the stencil's cell
// offsets.  All threads of the block call it.
template <int TP>
__device__ __forceinline__ Unit unit_begin(const RefineArgs &a, int nst, uint64_t *s_full, uint64_t *s_empty,
                                           int32_t *s_nstart, int32_t *s_vpre, int64_t *s_info)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        if (a.unit_tile) {
            s_info[0] = a.unit_tile[blockIdx.x];
            s_info[1] = a.unit_chunk[blockIdx.x];
        } else {
            const int64_t u = a.unit0 + blockIdx.x;
            int64_t lo = a.t0, hi = a.t1 - 1;  // last tile with tile_unit[t] <= u
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (a.tile_unit[mid] <= u) lo = mid; else hi = mid - 1;
            }
            s_info[0] = lo;
            s_info[1] = u - a.tile_unit[lo];
        }
        for (int st = 0; st < nst; ++st) {
            mbar_init(&s_full[st], 32);
            mbar_init(&s_empty[st], kComputeWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    Unit un;
    un.t = s_info[0];
    const int64_t chunk = s_info[1];
    un.c = a.tile_cell[un.t];
    un.q0 = a.tile_q0[un.t];
    un.nq = a.tile_nq[un.t];
    un.B = a.bound[un.c];
    un.W = (un.B + 31) >> 5;
    un.W4 = (un.W + 3) & ~int64_t(3);
    un.ncell = a.nbr_cnt[un.c];
    if (tid < un.ncell) {
        const int32_t nb = a.nbr[(int64_t)un.c * kStencil + tid];
        s_nstart[tid] = a.cell_start[nb];
        s_vpre[tid + 1] = a.cell_start[nb + 1] - a.cell_start[nb];
    }
    __syncthreads();
    if (tid == 0) {
        s_vpre[0] = 0;
        for (int i = 1; i <= un.ncell; ++i) s_vpre[i] += s_vpre[i - 1];
    }
    __syncthreads();
    const int64_t ch = refine_chunk_of(a.d4);
    un.vbeg = chunk * ch;
    un.vend = min(un.B, un.vbeg + ch);
    un.ntiles = (int)((un.vend - un.vbeg + TP - 1) / TP);
    return un;
}

// Boxes of the query tile over the three index dimensions, and the staged
// tiles of the unit worth streaming.
//
// s_qbox[8 g ...] = (lo0, lo1, lo2, hi0, hi1, hi2) of query rows g QG ...
// g QG + QG - 1 (QG = 4 MQ, the rows of the compute warps with wq = g; no
// row: +inf / -inf), for the compute warps' box test.
//
// Return value nkeep and s_list[0 .. nkeep): the staged tiles, in increasing
// order, that are not provably farther than eps from every query of the tile
// (tile it = candidate positions vbeg + it TP ...).  The test is the compute
// warps' box test (below) on larger boxes: the query tile's box against the
// union of the boxes of the 32-row groups of xs that hold the tile's
// candidates.  Both contain the exact boxes, so the rounded gap bound is at
// most that of any warp tile of the stage, and a skipped tile is one every
// warp would have skipped.  Threads tid < ntiles each test one tile (a unit
// has at most 128).  Without group boxes (and in the work-profile build)
// every tile is kept.  All threads of the block call it.
#ifndef HISS_STAGE_SKIP
#define HISS_STAGE_SKIP 1
#endif
template <int TP, int TQ, int QG, bool PROF>
__device__ __forceinline__ int stage_keep(const RefineArgs &a, const Unit &un, const int32_t *s_nstart,
                                          const int32_t *s_vpre, float *s_qbox, uint32_t *s_keep, uint8_t *s_list,
                                          int *s_kept)
{
    static_assert(kCH / TP <= 128 && TQ / 32 <= kComputeWarps && (QG == 16 || QG == 32), "keep mask geometry");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp < TQ / 32) {
        const int r = warp * 32 + lane;
        float lo0 = INFINITY, lo1 = INFINITY, lo2 = INFINITY, hi0 = -INFINITY, hi1 = -INFINITY, hi2 = -INFINITY;
        if (r < un.nq) {
            const float4 f = *reinterpret_cast<const float4 *>(a.xq + (int64_t)(un.q0 + r) * a.d4);
            lo0 = hi0 = f.x;
            lo1 = hi1 = f.y;
            lo2 = hi2 = f.z;
        }
#pragma unroll
        for (int o = QG / 2; o > 0; o >>= 1) {
            lo0 = fminf(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
            lo1 = fminf(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
            lo2 = fminf(lo2, __shfl_xor_sync(0xffffffffu, lo2, o));
            hi0 = fmaxf(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
            hi1 = fmaxf(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
            hi2 = fmaxf(hi2, __shfl_xor_sync(0xffffffffu, hi2, o));
        }
        if ((lane & (QG - 1)) == 0) {
            float *b = s_qbox + 8 * (r / QG);
            b[0] = lo0, b[1] = lo1, b[2] = lo2, b[3] = hi0, b[4] = hi1, b[5] = hi2, b[6] = 0.f, b[7] = 0.f;
        }
    }
    if (PROF || !HISS_STAGE_SKIP || a.gbox == nullptr) {
        if (tid < un.ntiles) s_list[tid] = (uint8_t)tid;
        if (tid == 0 && a.kept) atomicAdd(a.kept, (unsigned long long)(un.vend - un.vbeg) * (unsigned long long)un.nq);
        __syncthreads();
        return un.ntiles;
    }
    if (tid == 0) *s_kept = 0;
    __syncthreads();
    bool keep = false;
    if (tid < un.ntiles) {
        float qlo0 = s_qbox[0], qlo1 = s_qbox[1], qlo2 = s_qbox[2], qhi0 = s_qbox[3], qhi1 = s_qbox[4],
              qhi2 = s_qbox[5];
#pragma unroll
        for (int w = 1; w < TQ / QG; ++w) {
            const float *b = s_qbox + 8 * w;
            qlo0 = fminf(qlo0, b[0]), qlo1 = fminf(qlo1, b[1]), qlo2 = fminf(qlo2, b[2]);
            qhi0 = fmaxf(qhi0, b[3]), qhi1 = fmaxf(qhi1, b[4]), qhi2 = fmaxf(qhi2, b[5]);
        }
        const int64_t v0 = un.vbeg + (int64_t)tid * TP;
        const int64_t v1 = min(v0 + TP, un.vend) - 1;  // last candidate position of the tile
        int seg = 0, hi = un.ncell - 1;                 // last slot with s_vpre[slot] <= v0
        while (seg < hi) {
            const int mid = (seg + hi + 1) >> 1;
            if (s_vpre[mid] <= v0) seg = mid; else hi = mid - 1;
        }
        float plo0 = INFINITY, plo1 = INFINITY, plo2 = INFINITY, phi0 = -INFINITY, phi1 = -INFINITY,
              phi2 = -INFINITY;
        for (; seg < un.ncell && s_vpre[seg] <= v1; ++seg) {
            const int64_t pa = max(v0, (int64_t)s_vpre[seg]), pb = min(v1, (int64_t)s_vpre[seg + 1] - 1);
            const int64_t ga = (s_nstart[seg] + (pa - s_vpre[seg])) >> 5;
            const int64_t gb = (s_nstart[seg] + (pb - s_vpre[seg])) >> 5;
            for (int64_t g = ga; g <= gb; ++g) {
                const float4 l = __ldg(a.gbox + 2 * g), h = __ldg(a.gbox + 2 * g + 1);
                plo0 = fminf(plo0, l.x), plo1 = fminf(plo1, l.y), plo2 = fminf(plo2, l.z);
                phi0 = fmaxf(phi0, h.x), phi1 = fmaxf(phi1, h.y), phi2 = fmaxf(phi2, h.z);
            }
        }
        const float g0 = fmaxf(0.f, fmaxf(__fsub_rn(plo0, qhi0), __fsub_rn(qlo0, phi0)));
        const float g1 = fmaxf(0.f, fmaxf(__fsub_rn(plo1, qhi1), __fsub_rn(qlo1, phi1)));
        const float g2 = fmaxf(0.f, fmaxf(__fsub_rn(plo2, qhi2), __fsub_rn(qlo2, phi2)));
        keep = !(__fmaf_rn(g2, g2, __fmaf_rn(g1, g1, __fmul_rn(g0, g0))) > a.eps2);
        if (keep && a.kept) atomicAdd(s_kept, (int)(v1 - v0 + 1));
    }
    // the kept tiles in increasing order: s_list[0 .. nkeep)
    const uint32_t b = __ballot_sync(0xffffffffu, keep);
    if (warp < 4 && lane == 0) s_keep[warp] = b;
    __syncthreads();
    int base = 0, nkeep = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int c = __popc(s_keep[w]);
        base += w < warp ? c : 0;
        nkeep += c;
    }
    if (keep) s_list[base + __popc(b & ((1u << lane) - 1u))] = (uint8_t)tid;
    __syncthreads();
    if (tid == 0 && a.kept) atomicAdd(a.kept, (unsigned long long)*s_kept * (unsigned long long)un.nq);
    return nkeep;
}

// The producer warp: streams the unit's chunk through the stage ring.  Each
// lane copies the 16-byte chunks of the staged dimensions (C4 chunks) of rows
// lane and lane + 32 of a tile (cp.async), then arrives on the stage's full
// barrier twice: once asynchronously when its copies land, once now.  With
// partly staged rows it also records each row's index (-1 past the chunk
// end).
template <int TP>
__device__ __forceinline__ void produce(const RefineArgs &a, const Unit &un, float *P0, int32_t *s_row, int S, int C4,
                                        int d4, bool partial_rows, int nst, uint64_t *s_full, uint64_t *s_empty,
                                        const int32_t *s_nstart, const int32_t *s_vpre, const uint8_t *s_list,
                                        int nkeep, int lane)
{
    // stencil slot of each of the lane's rows: positions only grow from one
    // staged tile to the next, so the slot is found by walking forward from
    // the previous one (usually no step in a large cell)
    int seg[TP / 32];
#pragma unroll
    for (int h = 0; h < TP / 32; ++h) seg[h] = 0;
    for (int slot = 0; slot < nkeep; ++slot) {
        const int it = s_list[slot];
        const int st = slot % nst;
        const uint32_t round = (uint32_t)(slot / nst);
        if (slot >= nst && !refine_wait(&s_empty[st], (round - 1u) & 1u)) {
            atomicExch(&a.flags[kFlagRefineTimeout], 1);
            return;
        }
        float *P = P0 + st * TP * S;
        const int64_t v0 = un.vbeg + (int64_t)it * TP;
#pragma unroll
        for (int h = 0; h < TP / 32; ++h) {
            const int r = lane + 32 * h;
            const int64_t v = v0 + r;
            float4 *row = reinterpret_cast<float4 *>(P + r * S);
            if (v < un.vend) {
                int lo = seg[h];  // last slot with s_vpre[slot] <= v
                while (lo + 1 < un.ncell && s_vpre[lo + 1] <= v) ++lo;
                seg[h] = lo;
                const int32_t grow = s_nstart[lo] + (int32_t)(v - s_vpre[lo]);
                const float *src = a.xs + (int64_t)grow * d4;
                for (int cc = 0; cc < C4; ++cc) cp_async16(row + cc, src + 4 * cc);
                if (partial_rows) s_row[st * TP + r] = grow;
            } else {
                // no candidate: -inf makes every distance to this row +inf
                for (int cc = 0; cc < C4; ++cc) row[cc] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                if (partial_rows) s_row[st * TP + r] = -1;
            }
        }
        cp_async_arrive_on(&s_full[st]);
        mbar_arrive(&s_full[st]);
    }
}

// One thread block refines one unit: a tile of up to TQ queries of one grid
// cell against one chunk of up to kCH candidates of the cell's concatenated
// stencil.  The producer warp streams the chunk through a ring of staged
// candidate tiles (cp.async per 16-byte chunk, completion tracked by the
// stage's "full" mbarrier); each compute warp waits for a stage, refines its
// 4 MQ x 32 block of pairs with early termination, writes its mask words and
// releases the stage on its "empty" mbarrier.  Warps never wait for one
// another within a tile, so a warp whose pairs all leave after 4 dimensions
// moves on to the next tile while others finish.
//
// PROF = true: no mask output; instead count, over all candidate pairs, the
// dimensions a pair needs when it stops at the first multiple of 4 whose
// partial sum exceeds eps^2 (prof[0]), and the dimensions the warp-level
// schedule of the PROF = false kernel executes (prof[1]).
//
// D4 > 0: the kernel is compiled for that padded dimension (equal to a.d4),
// so every shared-memory row offset is an immediate and the dimension loop
// has a constant trip count; D4 = 0 takes a.d4 at run time.
template <int MQ, int MP, bool PROF, int D4>
__global__ void __launch_bounds__(kRefineThreads, HISS_REFINE_MINB) k_refine(const RefineArgs a)
{
    constexpr int kTQ = Geo<MQ, MP>::TQ, kTP = Geo<MQ, MP>::TP;
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t s_full[kMaxStages];
    __shared__ __align__(8) uint64_t s_empty[kMaxStages];
    __shared__ int32_t s_nstart[kStencil];
    __shared__ int32_t s_vpre[kStencil + 1];
    __shared__ int64_t s_info[2];
    __shared__ __align__(16) float s_qbox[8 * kQueryWarps];
    __shared__ uint32_t s_keep[4];
    __shared__ uint8_t s_list[kCH / kTP];
    __shared__ int s_kept;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d4 = D4 > 0 ? D4 : a.d4, S2 = pair_stride(d4);
    // staged dimensions per candidate row, their row stride and 16-byte chunks
    const int ds = staged_dims<PROF>(d4), S = tile_stride(ds), C4 = ds / 4;
    const bool partial_rows = ds < d4;
    const int nst = refine_stages<MQ, MP, PROF>(d4);
    float *Q2 = smem;
    float *P0 = smem + (kTQ / 2) * S2;
    // with partly staged rows: the global row of each staged candidate, per stage
    int32_t *s_row = reinterpret_cast<int32_t *>(P0 + nst * kTP * S);
    // survivor lists after the stage ring
    float *s_spart = reinterpret_cast<float *>(s_row + (partial_rows ? nst * kTP : 0));
    uint16_t *s_sidx = reinterpret_cast<uint16_t *>(s_spart + kComputeWarps * kSurvMax);
    uint32_t *s_sword = reinterpret_cast<uint32_t *>(s_sidx + kComputeWarps * kSurvMax);

    const Unit un = unit_begin<kTP>(a, nst, s_full, s_empty, s_nstart, s_vpre, s_info);
    // staged tiles to stream and refine (slot i of the ring takes tile s_list[i])
    const int nkeep = stage_keep<kTP, kTQ, 4 * MQ, PROF>(a, un, s_nstart, s_vpre, s_qbox, s_keep, s_list, &s_kept);
    const int64_t t = un.t;
    const int32_t q0 = un.q0;
    const int nq = un.nq;
    const int64_t W = un.W, W4 = un.W4;
    const int64_t vbeg = un.vbeg, vend = un.vend;

    if (warp == kComputeWarps) {
        produce<kTP>(a, un, P0, s_row, S, C4, d4, partial_rows, nst, s_full, s_empty, s_nstart, s_vpre, s_list,
                     nkeep, lane);
        return;
    }

    // ---- compute warps ----
    // query tile, pair-interleaved: pair row pid holds rows a = 8 (pid / 4) +
    // pid % 4 and a + 4, dimension by dimension; rows >= nq are +inf
    const int Q4 = d4 / 4;  // the query tile holds every dimension
    for (int idx = tid; idx < (kTQ / 2) * Q4; idx += kComputeThreads) {
        const int pid = idx / Q4, cc = idx - pid * Q4;
        const int ra = 8 * (pid >> 2) + (pid & 3), rb = ra + 4;
        const float4 inf4 = make_float4(INFINITY, INFINITY, INFINITY, INFINITY);
        const float4 x = ra < nq ? *reinterpret_cast<const float4 *>(a.xq + (int64_t)(q0 + ra) * d4 + 4 * cc) : inf4;
        const float4 y = rb < nq ? *reinterpret_cast<const float4 *>(a.xq + (int64_t)(q0 + rb) * d4 + 4 * cc) : inf4;
        float4 *dst = reinterpret_cast<float4 *>(Q2 + pid * S2 + 8 * cc);
        dst[0] = make_float4(x.x, y.x, x.y, y.y);
        dst[1] = make_float4(x.z, y.z, x.w, y.w);
    }
    compute_warps_sync();

    const int wq = warp >> 1, wp = warp & 1;
    const int lq = lane >> 3, lp = lane & 7;
    const int qbase = wq * (4 * MQ) + lq;    // query row i: qbase + 4 i
    const int pidbase = wq * (2 * MQ) + lq;  // pair row of queries 2 i2, 2 i2 + 1: pidbase + 4 i2
    const int pbase = wp * (8 * MP) + lp;    // candidate row j: pbase + 8 j
    const float eps2 = a.eps2;
    uint32_t my_count = 0;                   // neighbours of query row qbase + 4 lp (lp < MQ)
    const int64_t row_word0 = a.tile_word[t] - a.word0;
    uint64_t prof_alg = 0, prof_exec = 0;
    // Box of the warp's query rows (wq * 4 MQ ... + 4 MQ - 1) over the three
    // index dimensions (no query row: lo = +inf, hi = -inf).  With 8 x 4
    // blocks the warp reduces it into registers here; with 4 x 4 blocks it is
    // read per tile from stage_keep's copy in shared memory, which leaves the
    // registers to the larger survivor state.  Measured on GB300 (refinement):
    // spectrum (d = 128) 342 ms with the shared-memory copy against 364;
    // exp (d = 16) 12.1 s with registers against 12.3 s.
    constexpr bool kQBoxRegs = MQ == 8;
    float qlo0 = 0.f, qlo1 = 0.f, qlo2 = 0.f, qhi0 = 0.f, qhi1 = 0.f, qhi2 = 0.f;
    if constexpr (kQBoxRegs) {
        const int r = wq * (4 * MQ) + (lane & (4 * MQ - 1));
        qlo0 = qlo1 = qlo2 = INFINITY;
        qhi0 = qhi1 = qhi2 = -INFINITY;
        if (r < nq) {
            const float4 f = *reinterpret_cast<const float4 *>(a.xq + (int64_t)(q0 + r) * d4);
            qlo0 = qhi0 = f.x;
            qlo1 = qhi1 = f.y;
            qlo2 = qhi2 = f.z;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            qlo0 = fminf(qlo0, __shfl_xor_sync(0xffffffffu, qlo0, o));
            qlo1 = fminf(qlo1, __shfl_xor_sync(0xffffffffu, qlo1, o));
            qlo2 = fminf(qlo2, __shfl_xor_sync(0xffffffffu, qlo2, o));
            qhi0 = fmaxf(qhi0, __shfl_xor_sync(0xffffffffu, qhi0, o));
            qhi1 = fmaxf(qhi1, __shfl_xor_sync(0xffffffffu, qhi1, o));
            qhi2 = fmaxf(qhi2, __shfl_xor_sync(0xffffffffu, qhi2, o));
        }
    }

    for (int slot = 0; slot < nkeep; ++slot) {
        const int it = s_list[slot];
        const int st = slot % nst;
        const uint32_t round = (uint32_t)(slot / nst);
        if (!refine_wait(&s_full[st], round & 1u)) {
            atomicExch(&a.flags[kFlagRefineTimeout], 1);
            return;
        }
        const int64_t v0 = vbeg + (int64_t)it * kTP;
        const float *P = P0 + st * kTP * S;
        // Box test over the three index dimensions: for every pair of the
        // warp tile, |q_k - p_k| rounded is at least the rounded box gap g_k,
        // and the kernel's first three operations are e0 * e0, then fused
        // e1 * e1 + s, e2 * e2 + s, so with rounding monotone G below is at
        // most each pair's float32 partial sum after 3 dimensions, which the
        // later terms only increase.  G > eps^2: every pair's bit is 0.
        // The box of the warp's 32 staged candidates (rows 32 wp ...) is
        // reduced from shared memory with single-instruction warp minima and
        // maxima; rows past the chunk end hold -inf, which only widens it.
        bool far = false;
        {
            float blo0 = qlo0, blo1 = qlo1, blo2 = qlo2, bhi0 = qhi0, bhi1 = qhi1, bhi2 = qhi2;
            if constexpr (!kQBoxRegs) {
                const float4 qa = *reinterpret_cast<const float4 *>(s_qbox + 8 * wq);
                const float4 qb = *reinterpret_cast<const float4 *>(s_qbox + 8 * wq + 4);
                blo0 = qa.x, blo1 = qa.y, blo2 = qa.z, bhi0 = qa.w, bhi1 = qb.x, bhi2 = qb.y;
            }
            const float4 c = *reinterpret_cast<const float4 *>(P + (wp * 32 + lane) * S);
            const float plo0 = warp_min(c.x), plo1 = warp_min(c.y), plo2 = warp_min(c.z);
            const float phi0 = warp_max(c.x), phi1 = warp_max(c.y), phi2 = warp_max(c.z);
            const float g0 = fmaxf(0.f, fmaxf(__fsub_rn(plo0, bhi0), __fsub_rn(blo0, phi0)));
            const float g1 = fmaxf(0.f, fmaxf(__fsub_rn(plo1, bhi1), __fsub_rn(blo1, phi1)));
            const float g2 = fmaxf(0.f, fmaxf(__fsub_rn(plo2, bhi2), __fsub_rn(blo2, phi2)));
            far = __fmaf_rn(g2, g2, __fmaf_rn(g1, g1, __fmul_rn(g0, g0))) > eps2;
        }
        f32x2 acc[MQ / 2][MP];
        if constexpr (PROF) {
            // all dimensions, counting live pairs step by step: the
            // method's per-pair exit every 4 dimensions (prof_alg) and the
            // warp schedule of the kernel below (prof_exec)
            bool warp_live = !far, surv = false;
            block_step2<MQ, MP, true>(acc, Q2, P, S2, S, pidbase, pbase, 0);
            int valid = 0;
#pragma unroll
            for (int i = 0; i < MQ; ++i)
#pragma unroll
                for (int j = 0; j < MP; ++j) valid += (qbase + 4 * i < nq && v0 + pbase + 8 * j < vend) ? 1 : 0;
            prof_alg += (uint64_t)valid * (uint64_t)min(4, a.d);
            if (warp_live) prof_exec += (uint64_t)valid * (uint64_t)min(2, a.d);
            // dimensions the timed kernel stages: a warp still live there
            // finishes its pairs one per lane
            const int dsk = staged_dims<false>(d4);
            int live = 0;
            for (int k = 2; k < d4; k += 2) {
                if (warp_live && !surv && exit_check_at<MQ>(k, d4) &&
                    __all_sync(0xffffffffu, block_min<MQ, MP>(acc) > eps2))
                    warp_live = false;
                if ((k & 3) == 0) {
                    live = 0;
#pragma unroll
                    for (int i = 0; i < MQ; ++i)
#pragma unroll
                        for (int j = 0; j < MP; ++j) live += (acc_at<MQ, MP>(acc, i, j) <= eps2) ? 1 : 0;
                    if (warp_live && !surv &&
                        ((k == surv_dim(MQ, d4) && k < dsk && d4 - k >= 8 &&
                          __reduce_add_sync(0xffffffffu, live) <= kSurvMax) ||
                         k == dsk))
                        surv = true;  // survivor mode: each live pair runs on alone
                    if (!__any_sync(0xffffffffu, live > 0) && (!warp_live || surv)) break;
                    prof_alg += (uint64_t)live * (uint64_t)min(4, a.d - k);
                }
                if (surv) prof_exec += (uint64_t)live * (uint64_t)max(0, min(2, a.d - k));
                else if (warp_live) prof_exec += (uint64_t)valid * (uint64_t)max(0, min(2, a.d - k));
                block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k);
            }
        } else if (!far) {
            block_step2<MQ, MP, true>(acc, Q2, P, S2, S, pidbase, pbase, 0);
            // warp-level early termination (the pairs are in variance order,
            // most leave early)
            bool any_close = true, surv = false;
            // A warp still live when the staged dimensions run out finishes
            // its pairs one per lane (the rest of each candidate row comes
            // from global memory); with whole rows staged that point is d4,
            // where the bits are read from the sums.
            int sk = 0, sfirst = 0, stotal = 0;  // survivor mode from dimension sk
            if constexpr (MQ == 8) {
                // a check after every 2 dimensions
                for (int k = 2;; k += 2) {
                    if (k == ds) {
                        if (ds == d4) {
                            any_close = __any_sync(0xffffffffu, block_min<MQ, MP>(acc) <= eps2);
                        } else {
                            live_scan<MQ, MP>(acc, eps2, lane, &sfirst, &stotal);
                            any_close = surv = stotal > 0;
                            sk = k;
                        }
                        break;
                    }
                    if (exit_check_at<MQ>(k, d4) && __all_sync(0xffffffffu, block_min<MQ, MP>(acc) > eps2)) {
                        any_close = false;
                        break;
                    }
                    if (k == surv_dim(MQ, d4) && d4 - k >= 8) {
                        live_scan<MQ, MP>(acc, eps2, lane, &sfirst, &stotal);
                        if (stotal <= kSurvMax) {
                            surv = true;
                            sk = k;
                            break;
                        }
                    }
                    block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k);
                }
            } else {
                // a check after every 4 dimensions; two steps per iteration
                // let the compiler overlap one step's loads with the other
                block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, 2);
                for (int k = 4;; k += 4) {
                    if (k == ds) {
                        if (ds == d4) {
                            any_close = __any_sync(0xffffffffu, block_min<MQ, MP>(acc) <= eps2);
                        } else {
                            live_scan<MQ, MP>(acc, eps2, lane, &sfirst, &stotal);
                            any_close = surv = stotal > 0;
                            sk = k;
                        }
                        break;
                    }
                    if (exit_check_at<MQ>(k, d4) && __all_sync(0xffffffffu, block_min<MQ, MP>(acc) > eps2)) {
                        any_close = false;
                        break;
                    }
                    if (k == surv_dim(MQ, d4) && d4 - k >= 8) {
                        live_scan<MQ, MP>(acc, eps2, lane, &sfirst, &stotal);
                        if (stotal <= kSurvMax) {
                            surv = true;
                            sk = k;
                            break;
                        }
                    }
                    block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k);
                    block_step2<MQ, MP, false>(acc, Q2, P, S2, S, pidbase, pbase, k + 2);
                }
            }
            if (uses_survivors<false>(MQ, d4) && surv)
                survivors<MQ, MP, surv_ahead(D4 > 0 ? D4 : 64)>(acc, Q2, P, a.xs, s_row + st * kTP, S2, S, sk, ds, d4, eps2, sfirst, stotal, lane,
                                  wq, wp, s_spart + warp * kSurvMax, s_sidx + warp * kSurvMax, s_sword + warp * 32);
            // one bit per pair.  The warp's 32 candidate columns (pbase + 8 j)
            // form one mask word per query row: bit lp + 8 j.  A ballot per
            // (i, j) gives, for each lq, byte lq = the 8 lanes' bits; three
            // byte permutes assemble the word of query row qbase + 4 i.  Lane
            // lp keeps the word of i = lp and writes it.
            static_assert(MP == 4, "one mask word per query row per warp");
            const int64_t wcol = (v0 >> 5) + wp;
            const int qr = qbase + 4 * lp;
            if (any_close) {
                const uint32_t sel = (uint32_t)lq | ((uint32_t)(lq + 4) << 4);
                uint32_t mine = 0;
                if (surv) {
                    if (lp < MQ) mine = s_sword[warp * 32 + lq + 4 * lp];
                } else {
#pragma unroll
                for (int i = 0; i < MQ; ++i) {
                    uint32_t bj[MP];
#pragma unroll
                    for (int j = 0; j < MP; ++j) bj[j] = __ballot_sync(0xffffffffu, acc_at<MQ, MP>(acc, i, j) <= eps2);
                    const uint32_t w01 = __byte_perm(bj[0], bj[1], sel), w23 = __byte_perm(bj[2], bj[3], sel);
                    const uint32_t w = __byte_perm(w01, w23, 0x5410);
                    if (lp == i) mine = w;
                }
                }
                if (lp < MQ && qr < nq && wcol < W && mine) {
                    // only nonzero words are stored; the occupancy bitmap marks them
                    const int64_t wi = row_word0 + (int64_t)qr * W4 + wcol;
                    a.mask[wi] = mine;
                    atomicOr(&a.occ[wi >> 5], 1u << (wi & 31));
                    my_count += __popc(mine);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[st]);
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

template <int MQ, int MP, bool PROF, int D4 = 0>
cudaError_t launch_refine(const RefineArgs &a, cudaStream_t s)
{
    const size_t smem = refine_smem<MQ, MP, PROF>(a.d4);
    static size_t configured = 0;  // largest dynamic shared memory requested so far
    if (smem > configured) {
        HISS_TRY(cudaFuncSetAttribute(k_refine<MQ, MP, PROF, D4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
        configured = smem;
    }
    if (a.nunits <= 0) return cudaSuccess;
    k_refine<MQ, MP, PROF, D4><<<(unsigned)a.nunits, kRefineThreads, smem, s>>>(a);
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
        if (a.row_ptr_out) {
            a.row_ptr_out[gq] = a.row_ptr[gq] - a.col0;
            if (gq == a.nq - 1) a.row_ptr_out[a.nq] = a.row_ptr[a.nq] - a.col0;
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

    // only the nonzero words of the row are visited: lane l takes occupancy
    // word o = o0 + 32 s + l (bits = mask words 32 o .. 32 o + 31), clipped to
    // the row's words [woff, woff + W)
    int32_t *out = a.cols + (a.row_ptr[gq] - a.col0);
    int64_t run = 0;
    const int64_t o0 = woff >> 5, o1 = (woff + W - 1) >> 5;
    // occupancy words are loaded two sweeps ahead, so that their latency
    // overlaps the mask-word work of the current sweep
    uint32_t ahead0 = o0 + lane <= o1 ? a.occ[o0 + lane] : 0u;
    uint32_t ahead1 = o0 + 32 + lane <= o1 ? a.occ[o0 + 32 + lane] : 0u;
    for (int64_t ob = o0; ob <= o1; ob += 32) {
        const int64_t o = ob + lane;
        uint32_t bits = ahead0;
        ahead0 = ahead1;
        ahead1 = o + 64 <= o1 ? a.occ[o + 64] : 0u;
        if (o <= o1) {
            const int64_t wlo = 32 * o;
            if (wlo < woff) bits &= ~0u << (int)(woff - wlo);
            const int64_t n_in = woff + W - wlo;
            if (n_in < 32) bits &= (1u << (int)n_in) - 1u;
        }
        int cnt = 0;
        for (uint32_t bb = bits; bb; bb &= bb - 1) cnt += __popc(a.mask[32 * o + __ffs(bb) - 1]);
        int ex = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, ex, off);
            if (lane >= off) ex += v;
        }
        const int total = __shfl_sync(0xffffffffu, ex, 31);
        int64_t pos = run + ex - cnt;
        for (uint32_t bb = bits; bb; bb &= bb - 1) {
            const int64_t w = 32 * o + __ffs(bb) - 1;
            uint32_t word = a.mask[w];
            // stencil slot of the word's first candidate (binary search),
            // then forward: the bits are visited in increasing order
            const int64_t v0 = (w - woff) * 32;
            int l = 0, hh = ns - 1;
            while (l < hh) {
                const int m = (l + hh + 1) >> 1;
                if (s_vpre[warp][m] <= v0) l = m; else hh = m - 1;
            }
            while (word) {
                const int b = __ffs(word) - 1;
                word &= word - 1;
                const int64_t v = v0 + b;
                while (l + 1 < ns && s_vpre[warp][l + 1] <= v) ++l;
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

// One thread per tile of the batch: its units go to positions chunk x (tiles
// of its cell in the batch) + (its rank among them), counted from the unit
// of the first of those tiles.  A cell's tiles are consecutive in
// processing order and share one chunk count.
__global__ void k_unit_order(const RefineArgs a, const int32_t *qcell_start, int tq, int32_t *unit_tile,
                             int32_t *unit_chunk)
{
    const int64_t t = a.t0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= a.t1) return;
    const int32_t c = a.tile_cell[t];
    const int32_t s0 = qcell_start[c], sz = qcell_start[c + 1] - s0;
    const int64_t first = t - (a.tile_q0[t] - s0) / tq;     // the cell's first tile
    const int64_t ta = max(first, a.t0);
    const int64_t tb = min(first + (sz + tq - 1) / tq, a.t1);
    const int64_t nt = tb - ta;
    const int64_t base = a.tile_unit[ta] - a.unit0;
    const int64_t k_units = a.tile_unit[t + 1] - a.tile_unit[t];
    for (int64_t k = 0; k < k_units; ++k) {
        const int64_t u = base + k * nt + (t - ta);
        unit_tile[u] = (int32_t)t;
        unit_chunk[u] = (int32_t)k;
    }
}

}  // namespace

cudaError_t unit_order(const RefineArgs &a, const int32_t *qcell_start, int tq, int32_t *unit_tile,
                       int32_t *unit_chunk, cudaStream_t s, int64_t *launches)
{
    const int64_t nt = a.t1 - a.t0;
    if (nt <= 0) return cudaSuccess;
    k_unit_order<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(a, qcell_start, tq, unit_tile, unit_chunk);
    ++*launches;
    return cudaGetLastError();
}

int refine_tq(int d4) { return d4 <= 64 ? Geo<8, 4>::TQ : Geo<4, 4>::TQ; }

#ifndef HISS_REFINE_SPECIALIZE
#define HISS_REFINE_SPECIALIZE 1
#endif

cudaError_t refine(const RefineArgs &a, cudaStream_t s, int64_t *launches)
{
    ++*launches;
#if HISS_REFINE_SPECIALIZE
    // the padded dimensions of the common workloads get their own builds
    switch (a.d4) {
        case 16: return launch_refine<8, 4, false, 16>(a, s);
        case 32: return launch_refine<8, 4, false, 32>(a, s);
        case 64: return launch_refine<8, 4, false, 64>(a, s);
        case 128: return launch_refine<4, 4, false, 128>(a, s);
        default: break;
    }
#endif
    return a.d4 <= 64 ? launch_refine<8, 4, false>(a, s) : launch_refine<4, 4, false>(a, s);
}

cudaError_t refine_profile(const RefineArgs &a, cudaStream_t s, int64_t *launches)
{
    ++*launches;
    return a.d4 <= 64 ? launch_refine<8, 4, true>(a, s) : launch_refine<4, 4, true>(a, s);
}

int refine_chunk(int d4) { return refine_chunk_of(d4); }

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
