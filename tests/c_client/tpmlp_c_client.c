/*
 * A plain C11 client of libtpmlp (test infrastructure): it includes only include/tpmlp.h and
 * the CUDA runtime API, and drives the tensor-parallel MLP block through the C ABI with device
 * buffers of its own, as a user of the library without PyTorch would:
 *   tpmlp_create -> tpmlp_pack_shards -> tpmlp_forward -> tpmlp_get_status -> tpmlp_destroy.
 * The result is checked against the fp64 CPU oracle (linked in from oracle/tpmlp_oracle.c) on
 * the seeded inputs of synth/synth.c, with the block's bars: relative Frobenius error <= 1e-2
 * and max |dZ| <= 3e-2 max |Z_ref|. It also checks a shape error and the error strings.
 * Usage: tpmlp_c_client [H F k M seed]   (default: the tiny workload, 256 1024 2 128 0)
 * Exit status 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tpmlp.h"

/* synth/synth.c */
void synth_normal_bf16(uint64_t seed, uint64_t stream, double mean, double std, int64_t first,
                       int64_t n, uint16_t *out);
/* oracle/tpmlp_oracle.c */
int oracle_tpmlp_f64(const uint16_t *X, int64_t x_rows, const int64_t *rows, int64_t R,
                     const uint16_t *W1, const uint16_t *b1, const uint16_t *W2,
                     const uint16_t *b2, int64_t H, int64_t F, int32_t k, int32_t act,
                     double *Z, double *Y, double *P);

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

#define CHECK_CUDA(call)                                                                  \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));           \
            return 2;                                                                     \
        }                                                                                 \
    } while (0)

#define CHECK_TPMLP(call)                                                                 \
    do {                                                                                  \
        int s_ = (call);                                                                  \
        if (s_ != TPMLP_OK) {                                                             \
            fprintf(stderr, "%s failed: %s (%d)\n", #call, tpmlp_strerror(s_), s_);       \
            return 3;                                                                     \
        }                                                                                 \
    } while (0)

int main(int argc, char **argv) {
    int64_t H = 256, F = 1024, M = 128;
    int32_t k = 2;
    uint64_t seed = 0;
    if (argc == 6) {
        H = atoll(argv[1]);
        F = atoll(argv[2]);
        k = (int32_t)atoi(argv[3]);
        M = atoll(argv[4]);
        seed = (uint64_t)atoll(argv[5]);
    }
    /* the seeded draws of synth: streams X 0, W1 1, b1 2, W2 3, b2 4 */
    uint16_t *X = malloc((size_t)(M * H) * 2), *W1 = malloc((size_t)(H * F) * 2);
    uint16_t *b1 = malloc((size_t)F * 2), *W2 = malloc((size_t)(F * H) * 2);
    uint16_t *b2 = malloc((size_t)H * 2), *Z = malloc((size_t)(M * H) * 2);
    double *Zref = malloc((size_t)(M * H) * sizeof(double));
    if (!X || !W1 || !b1 || !W2 || !b2 || !Z || !Zref) return 4;
    synth_normal_bf16(seed, 0, 0.0, 1.0, 0, M * H, X);
    synth_normal_bf16(seed, 1, 0.0, 1.0 / sqrt((double)H), 0, H * F, W1);
    synth_normal_bf16(seed, 2, 0.0, 0.02, 0, F, b1);
    synth_normal_bf16(seed, 3, 0.0, 1.0 / sqrt((double)F), 0, F * H, W2);
    synth_normal_bf16(seed, 4, 0.0, 0.02, 0, H, b2);

    /* the shape rules of tpmlp_create: F % k != 0 is rejected, and no context is returned */
    tpmlp_ctx *bad = (tpmlp_ctx *)&bad;
    if (tpmlp_create(&bad, H, F, (int32_t)(F + 1), 0) != TPMLP_ERR_UNSUPPORTED_SHAPE || bad != NULL) {
        fprintf(stderr, "tpmlp_create accepted F %% k != 0\n");
        return 5;
    }
    if (strlen(tpmlp_strerror(TPMLP_ERR_UNSUPPORTED_SHAPE)) == 0) return 5;

    void *dX, *dW1, *db1, *dW2, *db2, *dZ;
    CHECK_CUDA(cudaMalloc(&dX, (size_t)(M * H) * 2));
    CHECK_CUDA(cudaMalloc(&dW1, (size_t)(H * F) * 2));
    CHECK_CUDA(cudaMalloc(&db1, (size_t)F * 2));
    CHECK_CUDA(cudaMalloc(&dW2, (size_t)(F * H) * 2));
    CHECK_CUDA(cudaMalloc(&db2, (size_t)H * 2));
    CHECK_CUDA(cudaMalloc(&dZ, (size_t)(M * H) * 2));
    CHECK_CUDA(cudaMemcpy(dX, X, (size_t)(M * H) * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dW1, W1, (size_t)(H * F) * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db1, b1, (size_t)F * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dW2, W2, (size_t)(F * H) * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db2, b2, (size_t)H * 2, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));

    tpmlp_ctx *ctx = NULL;
    CHECK_TPMLP(tpmlp_create(&ctx, H, F, k, 0));
    CHECK_TPMLP(tpmlp_pack_shards(ctx, dW1, db1, dW2, db2, (void *)stream));
    /* the raw weights may be released once the stream has passed the pack */
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaFree(dW1));
    CHECK_CUDA(cudaFree(dW2));
    CHECK_TPMLP(tpmlp_forward(ctx, dX, 1, M, dZ, (void *)stream));
    int32_t detail = 0;
    CHECK_TPMLP(tpmlp_get_status(ctx, (void *)stream, &detail));
    CHECK_CUDA(cudaMemcpy(Z, dZ, (size_t)(M * H) * 2, cudaMemcpyDeviceToHost));
    const int64_t launches = tpmlp_launch_count(ctx);
    tpmlp_destroy(ctx);
    tpmlp_destroy(NULL); /* NULL-safe */

    if (oracle_tpmlp_f64(X, M, NULL, M, W1, b1, W2, b2, H, F, k, 0, Zref, NULL, NULL) != 0) {
        fprintf(stderr, "oracle rejected its arguments\n");
        return 6;
    }
    double num = 0.0, den = 0.0, maxd = 0.0, maxr = 0.0;
    for (int64_t i = 0; i < M * H; ++i) {
        const double d = bf16_to_double(Z[i]) - Zref[i];
        num += d * d;
        den += Zref[i] * Zref[i];
        if (fabs(d) > maxd) maxd = fabs(d);
        if (fabs(Zref[i]) > maxr) maxr = fabs(Zref[i]);
    }
    const double rel = sqrt(num / den), mx = maxd / maxr;
    printf("c client: H=%lld F=%lld k=%d M=%lld launches=%lld rel_fro=%.3e max_abs/max|Z|=%.3e\n",
           (long long)H, (long long)F, k, (long long)M, (long long)launches, rel, mx);
    cudaFree(dX);
    cudaFree(db1);
    cudaFree(db2);
    cudaFree(dZ);
    cudaStreamDestroy(stream);
    return (rel <= 1e-2 && mx <= 3e-2 && launches >= 2) ? 0 : 1;
}
