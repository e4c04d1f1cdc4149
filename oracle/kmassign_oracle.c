/*
 * kmassign_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the k-means assignment step, used to
 * check the CUDA library.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * constant with the CUDA path (means_nearest_centroid_gb300/csrc).
 *
 * What it computes (flashlib PR #22 "Optimize Blackwell k-means assignment
 * reduction", Summary: score tiles, then centroid norms applied, then the
 * winning centroid chosen, with lowest-index tie breaking):
 *
 *   x_id, c_jd  = bf16 inputs decoded exactly and promoted to double
 *   cnorm_j     = sum_d c_jd^2                  (sequential in d, fp64)
 *   dot_ij      = sum_d x_id * c_jd             (sequential in d, fp64)
 *   s_ij        = cnorm_j - 2 * dot_ij          (fp64)
 *   idx_i       = the lowest j whose s_ij is minimal, where -0 equals +0 and
 *                 NaN is greater than every number
 *   minscore_i  = s_i,idx_i
 *
 * A row whose scores are all NaN gets idx 0 and minscore NaN: with NaN ordered
 * above every number and ties going to the lowest index, index 0 is the first
 * of the equal (all-NaN) candidates.  The pages test NaN rows but fix no
 * convention; this is the reading the library documents too.
 *
 * Parallelism: rows are independent, so an OpenMP loop runs over rows; the
 * scan over centroids inside one row is strictly sequential in j, which is
 * what makes "first minimum wins" the lowest index.
 *
 * Build (no fast-math: every sum must keep its written order):
 *   gcc -O2 -fopenmp -fPIC -shared kmassign_oracle.c -o liboracle.so
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32; widening it is exact. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The order the method minimises over: NaN above every number; otherwise the
 * usual order of the reals (so -0 and +0 are equal, neither is less). */
static int score_less(double a, double b)
{
    if (isnan(a))
        return 0;
    if (isnan(b))
        return 1;
    return a < b;
}

static double sq_norm(const uint16_t *row, int64_t D)
{
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) {
        double v = bf16_to_double(row[d]);
        acc += v * v;
    }
    return acc;
}

static double dot(const uint16_t *a, const uint16_t *b, int64_t D)
{
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d)
        acc += bf16_to_double(a[d]) * bf16_to_double(b[d]);
    return acc;
}

static double score(const uint16_t *x, const uint16_t *c, double cnorm, int64_t D)
{
    return cnorm - 2.0 * dot(x, c, D);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the OpenMP runtime will use for the next parallel loop. */
int oracle_max_threads(int nthreads)
{
    set_threads(nthreads);
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* cnorm[j] = ||c_j||^2 in fp64, for j in [0, K). */
void oracle_norms(const uint16_t *C, int64_t K, int64_t D, double *cnorm, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < K; ++j)
        cnorm[j] = sq_norm(C + j * D, D);
}

/*
 * Assign rows.  rows == NULL means every row 0..N-1 (nrows must equal N);
 * otherwise rows[r] names the X row whose answer goes to idx[r], minscore[r].
 * cnorm: fp64 norms from oracle_norms (the oracle always uses its own).
 */
void oracle_assign(const uint16_t *X, const uint16_t *C, const double *cnorm,
                   int64_t N, int64_t K, int64_t D,
                   const int64_t *rows, int64_t nrows,
                   int32_t *idx, double *minscore, int nthreads)
{
    (void)N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        const uint16_t *x = X + i * D;
        int64_t best_j = 0;
        double best_s = score(x, C, cnorm[0], D);
        for (int64_t j = 1; j < K; ++j) {
            double s = score(x, C + j * D, cnorm[j], D);
            if (score_less(s, best_s)) {
                best_s = s;
                best_j = j;
            }
        }
        idx[r] = (int32_t)best_j;
        minscore[r] = best_s;
    }
}

/* out[p] = s_{ii[p], jj[p]} in fp64, for p in [0, npairs). */
void oracle_scores(const uint16_t *X, const uint16_t *C, const double *cnorm, int64_t D,
                   const int64_t *ii, const int64_t *jj, int64_t npairs, double *out,
                   int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; ++p)
        out[p] = score(X + ii[p] * D, C + jj[p] * D, cnorm[jj[p]], D);
}

/*
 * The k-means update step, which follows the assignment in a Lloyd iteration
 * (flashlib PR #22 covers the assignment only; this is the textbook update):
 * for every centroid j,
 *   counts[j] = number of points with idx[i] == j
 *   sums[j][d] = sum over those points, in increasing i, of x_id (fp64)
 * idx values outside [0, K) are skipped.
 */
void oracle_update(const uint16_t *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                   double *sums, int64_t *counts)
{
    for (int64_t j = 0; j < K; ++j) {
        counts[j] = 0;
        for (int64_t d = 0; d < D; ++d)
            sums[j * D + d] = 0.0;
    }
    for (int64_t i = 0; i < N; ++i) {
        int32_t j = idx[i];
        if (j < 0 || j >= K)
            continue;
        counts[j] += 1;
        for (int64_t d = 0; d < D; ++d)
            sums[(int64_t)j * D + d] += bf16_to_double(X[i * D + d]);
    }
}

/*
 * The k nearest centroids of each point: the k smallest pairs (s_ij, j) in
 * the order the assignment uses (NaN above every number, -0 equal to +0, the
 * lower index first among equal scores), ascending.  With k = 1 this is the
 * assignment itself.  Requires 1 <= k <= K.  rows as in oracle_assign;
 * results go to idx[r * k + e] and score[r * k + e].
 */
static int pair_less(double a, int64_t ja, double b, int64_t jb)
{
    if (score_less(a, b))
        return 1;
    if (score_less(b, a))
        return 0;
    return ja < jb;   /* equal scores, or both NaN */
}

void oracle_topk(const uint16_t *X, const uint16_t *C, const double *cnorm, int64_t N, int64_t K,
                 int64_t D, const int64_t *rows, int64_t nrows, int64_t k, int32_t *idx,
                 double *score_out, int nthreads)
{
    (void)N;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        const uint16_t *xi = X + i * D;
        int32_t *bi = idx + r * k;
        double *bs = score_out + r * k;
        int64_t filled = 0;
        for (int64_t j = 0; j < K; ++j) {
            double s = score(xi, C + j * D, cnorm[j], D);
            /* insert (s, j) into the sorted list bs/bi of length filled (<= k) */
            int64_t pos = filled;
            while (pos > 0 && pair_less(s, j, bs[pos - 1], bi[pos - 1]))
                --pos;
            if (pos >= k)
                continue;
            int64_t last = filled < k ? filled : k - 1;
            for (int64_t e = last; e > pos; --e) {
                bs[e] = bs[e - 1];
                bi[e] = bi[e - 1];
            }
            bs[pos] = s;
            bi[pos] = (int32_t)j;
            if (filled < k)
                ++filled;
        }
    }
}

/*
 * The true squared Euclidean distance ||x_i - c_j||^2 = sum_d (x_id - c_jd)^2
 * (fp64, sequential in d) for each pair (ii[p], jj[p]): the textbook
 * definition, written without the norm expansion the assignment uses.
 */
void oracle_sqdist(const uint16_t *X, const uint16_t *C, int64_t D, const int64_t *ii,
                   const int64_t *jj, int64_t npairs, double *out, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; ++p) {
        const uint16_t *x = X + ii[p] * D;
        const uint16_t *c = C + jj[p] * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double diff = bf16_to_double(x[d]) - bf16_to_double(c[d]);
            acc += diff * diff;
        }
        out[p] = acc;
    }
}
