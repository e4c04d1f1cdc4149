/*
 * Calling libkmassign from plain C (no Python, no PyTorch): a tiny problem
 * with a known answer.  Centroid j is the one-hot vector e_j scaled by 2, and
 * point i equals centroid (i * 7) % K, so the nearest centroid of point i is
 * (i * 7) % K and its score ||c||^2 - 2 x.c = 4 - 8 = -4.  The problem is
 * solved from device buffers, then from host buffers (kmassign_host).
 * Exit status 0 when every check passes.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kmassign.h"

#define N 1000
#define K 64
#define D 64

static uint16_t bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);   /* exact for the small integers used here */
}

#define CHECK(cond, msg)                                                                          \
    do {                                                                                         \
        if (!(cond)) {                                                                           \
            fprintf(stderr, "FAIL: %s\n", msg);                                                  \
            return 1;                                                                            \
        }                                                                                        \
    } while (0)

int main(void)
{
    static uint16_t hx[N * D], hc[K * D];
    static int32_t hidx[N], htop[N * 2], hidx2[N];
    static float hms[N], hsc[N * 2], hms2[N];
    memset(hx, 0, sizeof hx);
    memset(hc, 0, sizeof hc);
    for (int j = 0; j < K; ++j)
        hc[j * D + j] = bf16(2.0f);
    for (int i = 0; i < N; ++i)
        hx[i * D + (i * 7) % K] = bf16(2.0f);

    void *dx, *dc;
    float *dn, *dms, *dsc;
    int32_t *didx, *dtop;
    CHECK(cudaMalloc(&dx, sizeof hx) == cudaSuccess, "cudaMalloc X");
    CHECK(cudaMalloc(&dc, sizeof hc) == cudaSuccess, "cudaMalloc C");
    CHECK(cudaMalloc((void **)&dn, K * sizeof(float)) == cudaSuccess, "cudaMalloc cnorm");
    CHECK(cudaMalloc((void **)&dms, N * sizeof(float)) == cudaSuccess, "cudaMalloc minscore");
    CHECK(cudaMalloc((void **)&didx, N * sizeof(int32_t)) == cudaSuccess, "cudaMalloc idx");
    CHECK(cudaMalloc((void **)&dtop, sizeof htop) == cudaSuccess, "cudaMalloc top idx");
    CHECK(cudaMalloc((void **)&dsc, sizeof hsc) == cudaSuccess, "cudaMalloc top score");
    cudaMemcpy(dx, hx, sizeof hx, cudaMemcpyHostToDevice);
    cudaMemcpy(dc, hc, sizeof hc, cudaMemcpyHostToDevice);

    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess, "stream");
    CHECK(kmassign_norms(dc, K, D, dn, s) == KMASSIGN_OK, "kmassign_norms");
    CHECK(kmassign(dx, dc, dn, N, K, D, didx, dms, s) == KMASSIGN_OK, "kmassign");
    CHECK(kmassign_topk(dx, dc, NULL, N, K, D, 2, dtop, dsc, 1, s) == KMASSIGN_OK, "kmassign_topk");
    CHECK(kmassign_check(s) == KMASSIGN_OK, "kmassign_check");
    /* argument errors come back as codes, with text */
    CHECK(kmassign(dx, dc, dn, N, K, 40, didx, dms, s) == KMASSIGN_ERR_UNSUPPORTED_D, "bad D");
    CHECK(strlen(kmassign_strerror(KMASSIGN_ERR_UNSUPPORTED_D)) > 0, "strerror");

    cudaMemcpy(hidx, didx, sizeof hidx, cudaMemcpyDeviceToHost);
    cudaMemcpy(hms, dms, sizeof hms, cudaMemcpyDeviceToHost);
    cudaMemcpy(htop, dtop, sizeof htop, cudaMemcpyDeviceToHost);
    cudaMemcpy(hsc, dsc, sizeof hsc, cudaMemcpyDeviceToHost);
    for (int i = 0; i < N; ++i) {
        const int want = (i * 7) % K;
        CHECK(hidx[i] == want, "idx");
        CHECK(hms[i] == -4.0f, "minscore");
        /* nearest: distance 0; every other centroid: 2^2 + 2^2 = 8; the
           second nearest is the lowest other index */
        CHECK(htop[2 * i] == want && hsc[2 * i] == 0.0f, "top-1 distance");
        CHECK(htop[2 * i + 1] == (want == 0 ? 1 : 0) && hsc[2 * i + 1] == 8.0f, "top-2 distance");
    }
    /* the same problem end to end from host buffers: copies inside the call */
    CHECK(kmassign_host(hx, hc, NULL, N, K, D, hidx2, hms2, s) == KMASSIGN_OK, "kmassign_host");
    for (int i = 0; i < N; ++i) {
        CHECK(hidx2[i] == (i * 7) % K, "host idx");
        CHECK(hms2[i] == -4.0f, "host minscore");
    }
    CHECK(kmassign_host(dx, dc, NULL, N, K, D, hidx2, NULL, s) == KMASSIGN_ERR_NOT_HOST,
          "device pointers refused by kmassign_host");
    cudaStreamDestroy(s);
    cudaFree(dx);
    cudaFree(dc);
    cudaFree(dn);
    cudaFree(dms);
    cudaFree(didx);
    cudaFree(dtop);
    cudaFree(dsc);
    printf("c abi example: ok\n");
    return 0;
}
