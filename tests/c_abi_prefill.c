/* A plain C caller of libcca.so on the GPU: device buffers from the CUDA runtime, a
 * seeded bf16 input, cca_pool then cca_attn_fwd on a created stream, and the inputs and
 * outputs written to one binary file (Q, K, V as bf16 bits; O as bf16 bits; LSE as fp32) for
 * the test to check against the oracle.  Usage: c_abi_prefill <out-file>. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "cca.h"

enum { B = 1, HQ = 4, HKV = 2, N = 768, D = 128, G = 16, W = 200 };

static uint32_t lcg(uint32_t *s) { return *s = *s * 1664525u + 1013904223u; }

/* uniform in [-0.5, 0.5), rounded to bf16 by truncation (any bf16 input will do) */
static uint16_t rand_bf16(uint32_t *s) {
    float f = (float)(lcg(s) >> 8) / 16777216.0f - 0.5f;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CK(x)                                                                  \
    do {                                                                       \
        int rc_ = (int)(x);                                                    \
        if (rc_ != 0) {                                                        \
            fprintf(stderr, "%s failed (%d) at line %d\n", #x, rc_, __LINE__); \
            return 1;                                                          \
        }                                                                      \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 2) return 2;
    const size_t nq = (size_t)B * HQ * N * D, nk = (size_t)B * HKV * N * D, nc = (size_t)B * HKV * (N / G) * D;
    uint16_t *hQ = malloc(nq * 2), *hK = malloc(nk * 2), *hV = malloc(nk * 2), *hO = malloc(nq * 2);
    float *hL = malloc((size_t)B * HQ * N * 4);
    if (!hQ || !hK || !hV || !hO || !hL) return 3;
    uint32_t seed = 12345u;
    for (size_t i = 0; i < nq; ++i) hQ[i] = rand_bf16(&seed);
    for (size_t i = 0; i < nk; ++i) hK[i] = rand_bf16(&seed);
    for (size_t i = 0; i < nk; ++i) hV[i] = rand_bf16(&seed);
    void *dQ, *dK, *dV, *dKc, *dVc, *dO;
    float *dL;
    CK(cudaMalloc(&dQ, nq * 2));
    CK(cudaMalloc(&dK, nk * 2));
    CK(cudaMalloc(&dV, nk * 2));
    CK(cudaMalloc(&dKc, nc * 2));
    CK(cudaMalloc(&dVc, nc * 2));
    CK(cudaMalloc(&dO, nq * 2));
    CK(cudaMalloc((void **)&dL, (size_t)B * HQ * N * 4));
    CK(cudaMemcpy(dQ, hQ, nq * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dK, hK, nk * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dV, hV, nk * 2, cudaMemcpyHostToDevice));
    cudaStream_t st;
    CK(cudaStreamCreate(&st));
    cca_params_t p = {0};
    p.B = B;
    p.Hq = HQ;
    p.Hkv = HKV;
    p.N = N;
    p.d = D;
    p.g = G;
    p.w = W;
    p.dtype = CCA_BF16;
    CK(cca_pool(dQ, dK, dV, dKc, dVc, &p, st));
    CK(cca_attn_fwd(dQ, dK, dV, dKc, dVc, dO, dL, &p, st));
    CK(cudaStreamSynchronize(st));
    CK(cudaMemcpy(hO, dO, nq * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(hL, dL, (size_t)B * HQ * N * 4, cudaMemcpyDeviceToHost));
    FILE *f = fopen(argv[1], "wb");
    if (!f) return 4;
    fwrite(hQ, 2, nq, f);
    fwrite(hK, 2, nk, f);
    fwrite(hV, 2, nk, f);
    fwrite(hO, 2, nq, f);
    fwrite(hL, 4, (size_t)B * HQ * N, f);
    fclose(f);
    cudaFree(dQ);
    cudaFree(dK);
    cudaFree(dV);
    cudaFree(dKc);
    cudaFree(dVc);
    cudaFree(dO);
    cudaFree(dL);
    cudaStreamDestroy(st);
    printf("c prefill ok\n");
    return 0;
}
