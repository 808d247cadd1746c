/*
 * Oracle for the exact epsilon self-join -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 brute force on the CPU.  Nothing in the
 * product path links, loads or calls this file; only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark do.  It shares no code,
 * header or constant with the CUDA library.
 *
 * Definition followed (RT-HiSS, Munugala & Gowanlock, Section II-A "Problem
 * Statement"): two points are neighbours iff their Euclidean distance is at
 * most epsilon, inclusive.  We compare squared distances,
 *     s(i,j) = sum_{k=0}^{d-1} (x[i][k] - x[j][k])^2   <=   eps^2,
 * in double precision from the float32 inputs (exact in double), with
 * eps^2 = (double)eps * (double)eps for the float32 eps the GPU receives.
 * The self pair (i,i) has s = 0 and therefore belongs to every row, which is
 * what the selectivity definition of Section V-B ("z = (|R| - |D|)/|D|")
 * presumes.
 *
 * Summation runs over k in increasing index order, one term at a time; the
 * build passes -ffp-contract=off so the arithmetic is the same on every host.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

static double sqdist(const float *a, const float *b, int d)
{
    double s = 0.0;
    for (int k = 0; k < d; ++k) {
        double t = (double)a[k] - (double)b[k];
        s += t * t;
    }
    return s;
}

/*
 * For each listed query row i = rows[r], count the points j (all of [0,n),
 * the query itself included) with s(i,j) <= hi, where hi = eps2 * (1 + band).
 * band = 0 gives the exact neighbour count of the definition.
 */
void orc_rows_count(const float *x, int64_t n, int32_t d, double eps2, double band,
                    const int64_t *rows, int64_t nrows, int64_t *out_count)
{
    const double hi = eps2 * (1.0 + band);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const float *q = x + rows[r] * (int64_t)d;
        int64_t c = 0;
        for (int64_t j = 0; j < n; ++j)
            if (sqdist(q, x + j * (int64_t)d, d) <= hi)
                ++c;
        out_count[r] = c;
    }
}

/*
 * List, for each listed query row, every j with s(i,j) <= eps2 * (1 + band),
 * in increasing j.  row_ptr (nrows+1) must come from orc_rows_count with the
 * same band.  flag[k] = 1 marks a pair inside the boundary band
 * |s - eps2| <= band * eps2 (such pairs may legitimately differ between two
 * correct float32 implementations); flag[k] = 0 marks a pair that is a
 * neighbour beyond doubt (s < eps2 * (1 - band)).  dist2 receives s.
 */
void orc_rows_fill(const float *x, int64_t n, int32_t d, double eps2, double band,
                   const int64_t *rows, int64_t nrows, const int64_t *row_ptr,
                   int32_t *cols, uint8_t *flag, double *dist2)
{
    const double hi = eps2 * (1.0 + band);
    const double lo = eps2 * (1.0 - band);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const float *q = x + rows[r] * (int64_t)d;
        int64_t o = row_ptr[r];
        for (int64_t j = 0; j < n; ++j) {
            double s = sqdist(q, x + j * (int64_t)d, d);
            if (s <= hi) {
                cols[o] = (int32_t)j;
                flag[o] = (uint8_t)(s >= lo);
                dist2[o] = s;
                ++o;
            }
        }
    }
}

/*
 * splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna): the
 * first output of a generator seeded with v.  Used only to fingerprint
 * neighbour sets, so that large rows can be compared without listing them.
 */
static uint64_t splitmix64(uint64_t v)
{
    uint64_t z = v + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/*
 * A digest of each listed query row i = rows[r] of the definition's result
 * (no band): out_count[r] = |{j : s(i,j) <= eps2}|, out_hash[r] = the sum,
 * modulo 2^64, of splitmix64(j) over those j, and out_band[r] = the number of
 * j with |s(i,j) - eps2| <= band * eps2 (pairs a correct float32
 * implementation may decide either way).  One pass, nothing listed.
 */
void orc_rows_digest(const float *x, int64_t n, int32_t d, double eps2, double band,
                     const int64_t *rows, int64_t nrows, int64_t *out_count, uint64_t *out_hash,
                     int64_t *out_band)
{
    const double hi = eps2 * (1.0 + band);
    const double lo = eps2 * (1.0 - band);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const float *q = x + rows[r] * (int64_t)d;
        int64_t c = 0, b = 0;
        uint64_t h = 0;
        for (int64_t j = 0; j < n; ++j) {
            const double s = sqdist(q, x + j * (int64_t)d, d);
            if (s <= eps2) {
                ++c;
                h += splitmix64((uint64_t)j);
            }
            if (s >= lo && s <= hi) ++b;
        }
        out_count[r] = c;
        out_hash[r] = h;
        out_band[r] = b;
    }
}

/*
 * Semi-join (RT-HiSS Section II-A: "D and Q are distinct"): for each query
 * row r of xq (nq x d), count the points j of xd (nd x d) with
 * s(q_r, p_j) <= eps2 * (1 + band); then list them (increasing j) with the
 * same band flags as orc_rows_fill.  No point is implicitly its own
 * neighbour: only distances count.
 */
void orc_semi_count(const float *xq, int64_t nq, const float *xd, int64_t nd, int32_t d, double eps2,
                    double band, int64_t *out_count)
{
    const double hi = eps2 * (1.0 + band);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nq; ++r) {
        const float *q = xq + r * (int64_t)d;
        int64_t c = 0;
        for (int64_t j = 0; j < nd; ++j)
            if (sqdist(q, xd + j * (int64_t)d, d) <= hi)
                ++c;
        out_count[r] = c;
    }
}

void orc_semi_fill(const float *xq, int64_t nq, const float *xd, int64_t nd, int32_t d, double eps2,
                   double band, const int64_t *row_ptr, int32_t *cols, uint8_t *flag, double *dist2)
{
    const double hi = eps2 * (1.0 + band);
    const double lo = eps2 * (1.0 - band);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nq; ++r) {
        const float *q = xq + r * (int64_t)d;
        int64_t o = row_ptr[r];
        for (int64_t j = 0; j < nd; ++j) {
            double s = sqdist(q, xd + j * (int64_t)d, d);
            if (s <= hi) {
                cols[o] = (int32_t)j;
                flag[o] = (uint8_t)(s >= lo);
                dist2[o] = s;
                ++o;
            }
        }
    }
}

/* Exact neighbour count of every point (band = 0), rows 0..n-1. */
void orc_counts(const float *x, int64_t n, int32_t d, double eps2, int64_t *out_count)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
        const float *q = x + i * (int64_t)d;
        int64_t c = 0;
        for (int64_t j = 0; j < n; ++j)
            if (sqdist(q, x + j * (int64_t)d, d) <= eps2)
                ++c;
        out_count[i] = c;
    }
}

/* ---- epsilon picker (workload definition, not the join itself) ----------
 *
 * The workloads fix epsilon by a target mean neighbour count K (self
 * excluded), measured on a seeded sample of queries.  For each sampled query
 * the squared distances to all other points are pooled; a = the (nq*K)-th
 * and b = the (nq*K+1)-th smallest pooled value.  Only the M smallest values
 * of each query are kept; the result is exact when b is below every query's
 * M-th smallest value, which the function reports (return 0) or not (return 1,
 * the caller retries with a larger M).
 */

static void swap_d(double *a, double *b) { double t = *a; *a = *b; *b = t; }

/* Rearrange v[0..n) so that v[0..m) hold the m smallest values (any order). */
static void select_smallest(double *v, int64_t n, int64_t m)
{
    int64_t lo = 0, hi = n - 1;
    if (m <= 0 || m >= n) return;
    while (lo < hi) {
        double pivot = v[lo + (hi - lo) / 2];
        int64_t i = lo, j = hi;
        while (i <= j) {
            while (v[i] < pivot) ++i;
            while (v[j] > pivot) --j;
            if (i <= j) { swap_d(&v[i], &v[j]); ++i; --j; }
        }
        if (m - 1 <= j) hi = j;
        else if (m - 1 >= i) lo = i;
        else break;
    }
}

static int cmp_d(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

int orc_pick_eps2(const float *x, int64_t n, int32_t d, const int64_t *qidx, int64_t nq,
                  int64_t K, int64_t M, double *out_a, double *out_b)
{
    const int all_kept = (M >= n - 1);
    if (all_kept) M = n - 1;
    if (nq * K + 1 > nq * M) return 2;
    double *pool = (double *)malloc(sizeof(double) * (size_t)(nq * M));
    double *kth = (double *)malloc(sizeof(double) * (size_t)nq);
    if (!pool || !kth) { free(pool); free(kth); return 3; }
#pragma omp parallel
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nq; ++r) {
            const int64_t i = qidx[r];
            const float *q = x + i * (int64_t)d;
            int64_t m = 0;
            for (int64_t j = 0; j < n; ++j)
                if (j != i) buf[m++] = sqdist(q, x + j * (int64_t)d, d);
            select_smallest(buf, m, M);
            double mx = -1.0;
            for (int64_t t = 0; t < M; ++t) {
                pool[r * M + t] = buf[t];
                if (buf[t] > mx) mx = buf[t];
            }
            kth[r] = mx; /* the M-th smallest of this query */
        }
        free(buf);
    }
    qsort(pool, (size_t)(nq * M), sizeof(double), cmp_d);
    const double a = pool[nq * K - 1], b = pool[nq * K];
    int status = 0; /* 0: exact, 1: retry with a larger M */
    for (int64_t r = 0; r < nq && !all_kept; ++r)
        if (!(b < kth[r])) { status = 1; break; }
    *out_a = a;
    *out_b = b;
    free(pool);
    free(kth);
    return status;
}
