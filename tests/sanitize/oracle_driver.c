/*
 * oracle_driver.c -- runs every function of the C oracle (oracle/kmassign_oracle.c)
 * on small inputs with special values and edge shapes, for a build with
 * AddressSanitizer and UndefinedBehaviorSanitizer (compiled and run by
 * tests/test_sanitize_host.py; any report aborts with a non-zero status).
 * It also checks properties every answer must have, so the run does real
 * work: indices in range, minscore equal to the pair score at the chosen
 * index, top-k lists ascending and distinct with the assignment first, and
 * exact squared distances on integer data.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int oracle_max_threads(int nthreads);
void oracle_norms(const uint16_t *C, int64_t K, int64_t D, double *cnorm, int nthreads);
void oracle_assign(const uint16_t *X, const uint16_t *C, const double *cnorm, int64_t N, int64_t K,
                   int64_t D, const int64_t *rows, int64_t nrows, int32_t *idx, double *minscore,
                   int nthreads);
void oracle_scores(const uint16_t *X, const uint16_t *C, const double *cnorm, int64_t D,
                   const int64_t *ii, const int64_t *jj, int64_t npairs, double *out, int nthreads);
void oracle_update(const uint16_t *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                   double *sums, int64_t *counts);
void oracle_topk(const uint16_t *X, const uint16_t *C, const double *cnorm, int64_t N, int64_t K,
                 int64_t D, const int64_t *rows, int64_t nrows, int64_t k, int32_t *idx,
                 double *score_out, int nthreads);
void oracle_sqdist(const uint16_t *X, const uint16_t *C, int64_t D, const int64_t *ii,
                   const int64_t *jj, int64_t npairs, double *out, int nthreads);

static uint64_t rng = 88172645463325252ull;
static uint32_t next_u32(void)
{
    rng ^= rng << 13;
    rng ^= rng >> 7;
    rng ^= rng << 17;
    return (uint32_t)(rng >> 32);
}

/* bf16 bits of a small integer in [-4, 4] (exact in bf16) */
static uint16_t small_int_bf16(void)
{
    float f = (float)((int)(next_u32() % 9) - 4);
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CHECK(c, msg)                                                                             \
    do {                                                                                          \
        if (!(c)) {                                                                               \
            fprintf(stderr, "FAIL %s (line %d)\n", msg, __LINE__);                               \
            return 1;                                                                             \
        }                                                                                         \
    } while (0)

static int score_lt(double a, double b)
{
    if (isnan(a))
        return 0;
    if (isnan(b))
        return 1;
    return a < b;
}

static int run(int64_t N, int64_t K, int64_t D, int specials)
{
    /* exact-size heap buffers, so any overrun is a sanitizer report */
    uint16_t *X = malloc(sizeof(uint16_t) * (size_t)(N * D));
    uint16_t *C = malloc(sizeof(uint16_t) * (size_t)(K * D));
    double *cn = malloc(sizeof(double) * (size_t)K);
    int32_t *idx = malloc(sizeof(int32_t) * (size_t)N);
    double *ms = malloc(sizeof(double) * (size_t)N);
    int64_t *ii = malloc(sizeof(int64_t) * (size_t)N);
    double *sc = malloc(sizeof(double) * (size_t)N);
    for (int64_t t = 0; t < N * D; ++t)
        X[t] = small_int_bf16();
    for (int64_t t = 0; t < K * D; ++t)
        C[t] = small_int_bf16();
    if (specials && N > 3) {
        const uint16_t sp[4] = {0x7fc0, 0x7f80, 0xff80, 0x8000}; /* NaN, +inf, -inf, -0 */
        for (int s = 0; s < 4; ++s)
            X[(int64_t)s * D + (int64_t)(next_u32() % (uint32_t)D)] = sp[s];
    }
    oracle_norms(C, K, D, cn, 1);
    oracle_assign(X, C, cn, N, K, D, NULL, N, idx, ms, 1);
    for (int64_t i = 0; i < N; ++i) {
        CHECK(idx[i] >= 0 && idx[i] < K, "idx in range");
        ii[i] = i;
    }
    int64_t *jj = malloc(sizeof(int64_t) * (size_t)N);
    for (int64_t i = 0; i < N; ++i)
        jj[i] = idx[i];
    oracle_scores(X, C, cn, D, ii, jj, N, sc, 1);
    for (int64_t i = 0; i < N; ++i)
        CHECK((isnan(sc[i]) && isnan(ms[i])) || sc[i] == ms[i], "minscore is the pair score");
    /* a subset of rows, in reverse order */
    int64_t nr = N < 5 ? N : 5;
    int64_t *rows = malloc(sizeof(int64_t) * (size_t)nr);
    int32_t *idx2 = malloc(sizeof(int32_t) * (size_t)nr);
    double *ms2 = malloc(sizeof(double) * (size_t)nr);
    for (int64_t r = 0; r < nr; ++r)
        rows[r] = N - 1 - r;
    oracle_assign(X, C, cn, N, K, D, rows, nr, idx2, ms2, 1);
    for (int64_t r = 0; r < nr; ++r)
        CHECK(idx2[r] == idx[rows[r]], "row subset agrees");
    /* top-k with k = min(K, 7) and k = K */
    for (int pass = 0; pass < 2; ++pass) {
        int64_t k = pass == 0 ? (K < 7 ? K : 7) : K;
        int32_t *ti = malloc(sizeof(int32_t) * (size_t)(N * k));
        double *ts = malloc(sizeof(double) * (size_t)(N * k));
        oracle_topk(X, C, cn, N, K, D, NULL, N, k, ti, ts, 1);
        for (int64_t i = 0; i < N; ++i) {
            CHECK(ti[i * k] == idx[i], "top-1 is the assignment");
            for (int64_t e = 0; e < k; ++e) {
                CHECK(ti[i * k + e] >= 0 && ti[i * k + e] < K, "top-k index in range");
                for (int64_t f = 0; f < e; ++f)
                    CHECK(ti[i * k + f] != ti[i * k + e], "top-k indices distinct");
                if (e > 0)
                    CHECK(!score_lt(ts[i * k + e], ts[i * k + e - 1]), "top-k ascending");
            }
        }
        free(ti);
        free(ts);
    }
    /* distances: exact on integer rows without specials */
    double *dist = malloc(sizeof(double) * (size_t)N);
    oracle_sqdist(X, C, D, ii, jj, N, dist, 1);
    for (int64_t i = specials ? 4 : 0; i < N; ++i) {
        double xn = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            uint32_t u = (uint32_t)X[i * D + d] << 16;
            float f;
            memcpy(&f, &u, 4);
            xn += (double)f * f;
        }
        CHECK(dist[i] >= 0.0 && dist[i] == xn + ms[i], "distance identity");
    }
    /* update with ids out of range, which are skipped */
    int32_t *uid = malloc(sizeof(int32_t) * (size_t)N);
    for (int64_t i = 0; i < N; ++i)
        uid[i] = (i % 5 == 4) ? (int32_t)(K + (int64_t)i) : ((i % 7 == 6) ? -1 : idx[i]);
    double *sums = malloc(sizeof(double) * (size_t)(K * D));
    int64_t *counts = malloc(sizeof(int64_t) * (size_t)K);
    oracle_update(X, uid, N, K, D, sums, counts);
    int64_t total = 0, valid = 0;
    for (int64_t j = 0; j < K; ++j)
        total += counts[j];
    for (int64_t i = 0; i < N; ++i)
        valid += (uid[i] >= 0 && uid[i] < K);
    CHECK(total == valid, "update counts every valid id once");
    free(X); free(C); free(cn); free(idx); free(ms); free(ii); free(jj); free(sc);
    free(rows); free(idx2); free(ms2); free(dist); free(uid); free(sums); free(counts);
    return 0;
}

int main(void)
{
    CHECK(oracle_max_threads(1) >= 1, "threads");
    const int64_t shapes[][3] = {{1, 1, 16}, {1, 3, 16}, {5, 1, 32}, {17, 9, 48}, {33, 65, 64},
                                 {7, 130, 96}, {64, 40, 128}, {3, 5, 256}, {40, 12, 192}};
    for (size_t s = 0; s < sizeof shapes / sizeof shapes[0]; ++s)
        for (int sp = 0; sp < 2; ++sp)
            if (run(shapes[s][0], shapes[s][1], shapes[s][2], sp) != 0)
                return 1;
    printf("oracle under sanitizers: ok\n");
    return 0;
}
