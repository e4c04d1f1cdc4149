/*
 * host_driver.c -- exercises the host code of libkmassign built with
 * AddressSanitizer and UndefinedBehaviorSanitizer, on a machine with or
 * without a GPU (compiled and run by tests/test_sanitize_host.py; any report
 * aborts with a non-zero status).  Without a GPU nothing is launched: it
 * covers every entry point's argument checks, the error texts, and the
 * planner (kmassign_plan_for) over extreme shapes and every forcing, checking
 * that each plan is one the kernels can run.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "kmassign.h"

#define CHECK(c, msg)                                                                             \
    do {                                                                                          \
        if (!(c)) {                                                                               \
            fprintf(stderr, "FAIL %s (line %d)\n", msg, __LINE__);                               \
            return 1;                                                                             \
        }                                                                                         \
    } while (0)

static int plan_ok(const int32_t *p, int64_t N, int64_t K, int64_t D, int sms, int pairs)
{
    const int rows = p[1], nt = p[2], cw = p[8];
    const int pair = rows == 256 && nt == 256;
    if (!((rows == 128 && nt == 128 && cw == 4) || (rows == 256 && nt == 128 && (cw == 8 || cw == 16)) ||
          (rows == 128 && nt == 256 && (cw == 8 || cw == 16)) || (pair && (cw == 8 || cw == 16))))
        return 0;
    if (p[3] < 1 || p[3] > sms || (pair && (p[3] % 2 != 0 || p[3] / 2 > pairs)))
        return 0;
    if (p[4] < 2 || p[4] > 16 || (p[5] != 1 && p[5] != 2))
        return 0;
    /* a folding pair's ring holds whole tiles: a multiple of the k-blocks,
       at least two tiles */
    const int kb = (int)((D + 63) / 64);
    if (pair && D <= 128 && (p[4] % kb != 0 || p[4] < 2 * kb))
        return 0;
    const int64_t rowtiles = ((N < 1 ? 1 : N) + rows - 1) / rows;
    if ((int64_t)p[6] + p[7] != rowtiles || p[0] < 1 || (p[0] > 1) != (p[7] > 0))
        return 0;
    return p[0] <= (K + nt - 1) / nt;
}

int main(void)
{
    /* every status has a text */
    for (int c = -12; c <= 1; ++c)
        CHECK(kmassign_strerror(c) != NULL && strlen(kmassign_strerror(c)) > 0, "strerror");

    /* argument errors, returned before any CUDA call */
    void *A = (void *)0x10000, *B = (void *)0x20000;
    int32_t *I = (int32_t *)0x30000;
    float *F = (float *)0x40000;
    CHECK(kmassign(A, B, NULL, -1, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_SHAPE, "N < 0");
    CHECK(kmassign(A, B, NULL, 10, 0, 64, I, NULL, NULL) == KMASSIGN_ERR_SHAPE, "K < 1");
    CHECK(kmassign(A, B, NULL, 10, 5, 40, I, NULL, NULL) == KMASSIGN_ERR_UNSUPPORTED_D, "D");
    CHECK(kmassign(NULL, NULL, NULL, 0, 5, 64, NULL, NULL, NULL) == KMASSIGN_OK, "N == 0");
    CHECK(kmassign(NULL, B, NULL, 10, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_NULL, "X NULL");
    CHECK(kmassign((char *)A + 8, B, NULL, 10, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_ALIGN,
          "X misaligned");
    CHECK(kmassign_ex(A, B, NULL, 10, 5, 64, I, NULL, -1, 0, 0, 0, NULL) == KMASSIGN_ERR_ARG,
          "ksplit -1");
    CHECK(kmassign_ex(A, B, NULL, 10, 5, 64, I, NULL, 0, 64, 0, 0, NULL) == KMASSIGN_ERR_ARG,
          "rows 64");
    CHECK(kmassign_norms(NULL, 5, 64, F, NULL) == KMASSIGN_ERR_NULL, "norms NULL");
    CHECK(kmassign_norms(A, 5, 24, F, NULL) == KMASSIGN_ERR_UNSUPPORTED_D, "norms D");
    CHECK(kmassign_noalloc(A, B, NULL, -3, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_SHAPE,
          "noalloc shape");
    CHECK(kmassign_topk(A, B, NULL, 10, 5, 64, 0, I, F, 0, NULL) == KMASSIGN_ERR_ARG, "k 0");
    CHECK(kmassign_topk(A, B, NULL, 10, 5, 64, 6, I, F, 0, NULL) == KMASSIGN_ERR_ARG, "k > K");
    CHECK(kmassign_topk(A, B, NULL, 10, 50, 64, 33, I, F, 0, NULL) == KMASSIGN_ERR_ARG, "k > 32");
    CHECK(kmassign_topk(A, B, NULL, 10, 50, 64, 4, I, NULL, 1, NULL) == KMASSIGN_ERR_NULL,
          "distances without score");
    CHECK(kmassign_topk_ex(A, B, NULL, 10, 50, 64, 4, I, F, 0, -1, NULL) == KMASSIGN_ERR_ARG,
          "topk ksplit -1");
    CHECK(kmassign_update(A, I, 10, 0, 64, F, I, NULL) == KMASSIGN_ERR_SHAPE, "update K");
    CHECK(kmassign_update_ex(A, I, 10, 5, 64, F, I, 3, NULL) == KMASSIGN_ERR_ARG, "method 3");
    CHECK(kmassign_centroids(F, I, A, 5, 40, B, NULL, NULL) == KMASSIGN_ERR_UNSUPPORTED_D,
          "centroids D");
    CHECK(kmassign_lloyd(A, B, 10, 5, 64, -1, I, NULL) == KMASSIGN_ERR_ARG, "iters < 0");
    CHECK(kmassign_host(A, B, NULL, -1, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_SHAPE, "host N");
    CHECK(kmassign_host_ex(A, B, NULL, 10, 5, 64, I, NULL, -5, NULL) == KMASSIGN_ERR_ARG,
          "host rows");
    CHECK(kmassign_host(NULL, B, NULL, 10, 5, 64, I, NULL, NULL) == KMASSIGN_ERR_NULL, "host NULL");
    CHECK(kmassign_plan_for(10, 10, 64, 0, 232448, 76, 0, 0, 0, 0, (int32_t *)F) ==
              KMASSIGN_ERR_ARG,
          "plan_for sms");
    CHECK(kmassign_plan_for(10, 10, 64, 152, 232448, 76, 0, 0, 0, 0, NULL) == KMASSIGN_ERR_NULL,
          "plan_for out");

    /* the planner over extreme shapes, every forcing, three devices */
    const int64_t Ns[] = {1, 2, 127, 129, 4096, 65536, 65537, 262144, 1048576, 330000,
                          (int64_t)1 << 30, ((int64_t)1 << 31) - 1};
    const int64_t Ks[] = {1, 3, 128, 129, 512, 4096, 16384, 65536, 524288, ((int64_t)1 << 31) - 1};
    const int64_t Ds[] = {16, 48, 64, 96, 128, 192, 256};
    const int devs[][3] = {{152, 232448, 76}, {8, 232448, 4}, {152, 232448, 0}, {1, 232448, 0}};
    const int ks_force[] = {0, 1, 2, 5, 64, -2, -3};
    const int rows_force[] = {0, 128, 256};
    const int nt_force[] = {0, 128, 256};
    const int cw_force[] = {0, 4, 8, 16};
    long plans = 0;
    for (size_t dv = 0; dv < sizeof devs / sizeof devs[0]; ++dv)
        for (size_t a = 0; a < sizeof Ns / sizeof Ns[0]; ++a)
            for (size_t b = 0; b < sizeof Ks / sizeof Ks[0]; ++b)
                for (size_t c = 0; c < sizeof Ds / sizeof Ds[0]; ++c)
                    for (size_t f = 0; f < sizeof ks_force / sizeof ks_force[0]; ++f)
                        for (size_t r = 0; r < 3; ++r)
                            for (size_t t = 0; t < 3; ++t)
                                for (size_t w = 0; w < 4; ++w) {
                                    if ((f | r | t | w) != 0 && (a % 3 != 0 || b % 2 != 0))
                                        continue;   /* forcings on a subset of shapes */
                                    int32_t p[9];
                                    const int rc = kmassign_plan_for(
                                        Ns[a], Ks[b], Ds[c], devs[dv][0], devs[dv][1],
                                        devs[dv][2], ks_force[f], rows_force[r], nt_force[t],
                                        cw_force[w], p);
                                    if (rc == KMASSIGN_ERR_ARG)
                                        continue;
                                    CHECK(rc == KMASSIGN_OK, "plan_for status");
                                    CHECK(plan_ok(p, Ns[a], Ks[b], Ds[c], devs[dv][0], devs[dv][2]),
                                          "plan is runnable");
                                    ++plans;
                                }
    CHECK(plans > 1000, "planner exercised");
    printf("host code under sanitizers: ok (%ld plans)\n", plans);
    return 0;
}
