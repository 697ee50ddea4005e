/*
 * A plain C caller of libsb: device memory from cudaMalloc, the projection through the C ABI
 * of sb.h, results compared with the fp64 oracle (liboracle) linked into this test program;
 * then the host-buffer call with pinned and with pageable host memory against those results.
 * Built and run by tests/test_c_abi.py on a GPU machine; exits 0 on agreement.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sb.h"

int oracle_project(const uint16_t *H, const uint16_t *W, const int64_t *row_ids, int64_t M,
                   int64_t d, int64_t V, int32_t k, int32_t gumbel, double temperature,
                   uint64_t seed, const int32_t *targets, int32_t *token, double *lse,
                   double *logprob, double *target_logprob, double *key_top1, double *key_top2,
                   double *shard_max, int32_t *shard_token, double *shard_lse, double *Z);

/* bf16 bits of a float (round to nearest even; inputs are finite) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* a small deterministic generator for the test inputs (not the method's) */
static uint64_t lcg = 88172645463325252ull;
static float unif(void) {
    lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((lcg >> 40) + 0.5) / 16777216.0f - 0.5f;
}

#define CHECK(x)                                                                          \
    do {                                                                                  \
        if (!(x)) {                                                                       \
            fprintf(stderr, "check failed: %s (line %d)\n", #x, __LINE__);                \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

int main(void) {
    const int64_t M = 8, d = 192, V = 3000, k = 3;
    uint16_t *H = malloc(M * d * 2), *W = malloc(V * d * 2);
    for (int64_t i = 0; i < M * d; ++i) H[i] = to_bf16(4.0f * unif());
    for (int64_t i = 0; i < V * d; ++i) W[i] = to_bf16(0.3f * unif());

    void *dH, *dW, *dTok, *dLp, *dLse, *dWs;
    const size_t ws = sb_workspace_bytes(M, V, (int32_t)k, SB_TOKEN_LOGPROB);
    CHECK(ws > 0);
    CHECK(cudaMalloc(&dH, M * d * 2) == cudaSuccess);
    CHECK(cudaMalloc(&dW, V * d * 2) == cudaSuccess);
    CHECK(cudaMalloc(&dTok, M * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dLp, M * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dLse, M * 4) == cudaSuccess);
    CHECK(cudaMalloc(&dWs, ws) == cudaSuccess);
    CHECK(cudaMemcpy(dH, H, M * d * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dW, W, V * d * 2, cudaMemcpyHostToDevice) == cudaSuccess);

    sb_outputs out;
    memset(&out, 0, sizeof out);
    out.token = dTok;
    out.token_logprob = dLp;
    out.lse = dLse;
    out.workspace = dWs;
    out.workspace_bytes = ws;
    int32_t st = sb_lmhead_project(dH, dW, M, d, V, (int32_t)k, SB_TOKEN_LOGPROB, 1.0f, 0, &out,
                                   NULL);
    if (st != SB_OK) {
        fprintf(stderr, "sb_lmhead_project: %s\n", sb_status_string(st));
        return 1;
    }
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(sb_last_device_status(&out) == SB_OK);
    int32_t tok[8];
    float lp[8], lse[8];
    CHECK(cudaMemcpy(tok, dTok, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(lp, dLp, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(lse, dLse, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);

    int32_t rtok[8];
    double rlse[8], rlp[8], t1[8], t2[8];
    double *Z = malloc(sizeof(double) * M * V);
    CHECK(oracle_project(H, W, NULL, M, d, V, (int32_t)k, 0, 1.0, 0, NULL, rtok, rlse, rlp, NULL,
                         t1, t2, NULL, NULL, NULL, Z) == 0);
    for (int r = 0; r < M; ++r) {
        if (t1[r] - t2[r] > 1e-2)
            CHECK(tok[r] == rtok[r]);
        else
            CHECK(Z[r * V + tok[r]] >= t1[r] - 1e-2);
        CHECK(fabs(lse[r] - rlse[r]) <= 5e-3);
        CHECK(fabs(lp[r] - (Z[r * V + tok[r]] - rlse[r])) <= 5e-3);
    }
    /* the host-buffer call: pinned buffers (moved by the kernels) and pageable ones (copied)
       give the device call's bits */
    for (int pinned = 0; pinned < 2; ++pinned) {
        uint16_t *hH = NULL;
        int32_t *hTok = NULL;
        float *hLp = NULL;
        if (pinned) {
            CHECK(cudaMallocHost((void **)&hH, M * d * 2) == cudaSuccess);
            CHECK(cudaMallocHost((void **)&hTok, M * 4) == cudaSuccess);
            CHECK(cudaMallocHost((void **)&hLp, M * 4) == cudaSuccess);
        } else {
            hH = malloc(M * d * 2);
            hTok = malloc(M * 4);
            hLp = malloc(M * 4);
        }
        memcpy(hH, H, M * d * 2);
        memset(hTok, 0xFF, M * 4);
        memset(hLp, 0xFF, M * 4);
        void *dStage;
        CHECK(cudaMalloc(&dStage, M * d * 2) == cudaSuccess);
        st = sb_lmhead_project_from_host(hH, dStage, dW, M, d, V, (int32_t)k, SB_TOKEN_LOGPROB,
                                         1.0f, 0, &out, hTok, hLp, NULL);
        CHECK(st == SB_OK);
        CHECK(cudaDeviceSynchronize() == cudaSuccess);
        CHECK(memcmp(hTok, tok, M * 4) == 0);
        CHECK(memcmp(hLp, lp, M * 4) == 0);
        cudaFree(dStage);
        if (pinned) {
            cudaFreeHost(hH);
            cudaFreeHost(hTok);
            cudaFreeHost(hLp);
        } else {
            free(hH);
            free(hTok);
            free(hLp);
        }
    }
    /* the same call on a packed copy of W gives the same bits */
    {
        const size_t pb = sb_packed_weight_bytes(V, d, (int32_t)k);
        void *dWp = NULL;
        CHECK(pb > 0 && cudaMalloc(&dWp, pb) == cudaSuccess);
        CHECK(sb_pack_weights(dW, V, d, (int32_t)k, dWp, pb, NULL) == SB_OK);
        CHECK(sb_lmhead_project(dH, dWp, M, d, V, (int32_t)k, SB_TOKEN_LOGPROB | SB_W_PACKED,
                                1.0f, 0, &out, NULL) == SB_OK);
        CHECK(cudaDeviceSynchronize() == cudaSuccess);
        int32_t ptok[8];
        float plp[8], plse[8];
        CHECK(cudaMemcpy(ptok, dTok, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
        CHECK(cudaMemcpy(plp, dLp, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
        CHECK(cudaMemcpy(plse, dLse, M * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
        CHECK(memcmp(ptok, tok, M * 4) == 0 && memcmp(plp, lp, M * 4) == 0 &&
              memcmp(plse, lse, M * 4) == 0);
        cudaFree(dWp);
    }
    /* invalid arguments are refused before anything runs */
    CHECK(sb_lmhead_project(dH, dW, M, d, V + 1, (int32_t)k, SB_TOKEN, 1.0f, 0, &out, NULL) ==
          SB_ERR_INVALID_ARG);
    out.workspace_bytes = 16;
    CHECK(sb_lmhead_project(dH, dW, M, d, V, (int32_t)k, SB_TOKEN, 1.0f, 0, &out, NULL) ==
          SB_ERR_WORKSPACE_TOO_SMALL);
    cudaFree(dH);
    cudaFree(dW);
    cudaFree(dTok);
    cudaFree(dLp);
    cudaFree(dLse);
    cudaFree(dWs);
    free(H);
    free(W);
    free(Z);
    printf("C ABI ok: tokens %d %d %d %d\n", tok[0], tok[1], tok[2], tok[3]);
    return 0;
}
