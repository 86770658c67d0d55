/*
 * CPU oracle for the tensor-parallel MLP block -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load this code. It shares nothing with the CUDA library: plain fp64 loops on
 * bf16 inputs widened exactly to double, no blocking, no fusion, no reordering of
 * any sum beyond what the definition below states.
 *
 * What it computes (the block as the pages define it):
 *
 *   Column-parallel first layer: W1 [H, F] is split by columns into k equal,
 *   contiguous shards W1_i = W1[:, i*f:(i+1)*f], f = F/k; every shard sees the
 *   same X and produces Y_i = X W1_i, and concatenating the Y_i gives X W1.
 *   (千亿参数模型如何拆分到多张GPU上训练, "方案一：按列切分权重矩阵";
 *    大模型分布式并行策略详解 §4.1; AI大模型分布式训练 §2.1 ColumnParallelLinear,
 *    whose bias is sliced with the output columns.)
 *
 *   GeLU is applied to each shard's output on its own, with no exchange before
 *   it, because it acts element by element (same section of the first page).
 *   Reading: the exact form GeLU(a) = a * Phi(a) = a/2 * (1 + erf(a / sqrt 2)).
 *
 *   Row-parallel second layer: W2 [F, H] is split by rows into the matching
 *   shards W2_i = W2[i*f:(i+1)*f, :]; shard i forms the partial Z_i = Y_i W2_i and
 *   the block output is the sum Z = sum_i Z_i, which the pages obtain with one
 *   All-Reduce (千亿参数模型…, "方案二：按行切分权重矩阵", Z = Y1 V1 + Y2 V2;
 *   大模型分布式并行策略详解 §4.1; AI大模型分布式训练 §2.2 RowParallelLinear).
 *
 *   Reading for the output bias: b2 is added once, after the sum over shards.
 *
 *   Z[m, n] = b2[n] + sum_{i=0}^{k-1} sum_{j=i f}^{(i+1) f - 1}
 *                 GeLU(b1[j] + sum_h X[m, h] W1[h, j]) * W2[j, n]
 *
 * Sums run in index order: over h for each pre-activation, over j inside a shard
 * for each partial, then over shards i = 0..k-1 (the "all-reduce"), then + b2.
 * Rows of X are independent, so any subset of rows is evaluated exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double, exact: a bf16 is the upper 16 bits of an IEEE fp32. */
static double widen_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* GeLU(a) = a * Phi(a), Phi the standard normal CDF = (1 + erf(a / sqrt(2))) / 2. */
double oracle_gelu(double a) { return 0.5 * a * (1.0 + erf(a / sqrt(2.0))); }

#define ORACLE_ACT_GELU 0
#define ORACLE_ACT_IDENTITY 1 /* test-only: drops the nonlinearity so the block is two plain products */

/*
 * Evaluate the block for R token rows.
 *   X        bf16 [x_rows][H]; rows[r] (or r if rows == NULL) selects the row of X
 *   W1       bf16 [H][F] (math orientation: Y = X W1), b1 bf16 [F]
 *   W2       bf16 [F][H], b2 bf16 [H]
 *   k        shard count, F % k == 0
 *   act      ORACLE_ACT_GELU or ORACLE_ACT_IDENTITY
 *   Z        out, double [R][H]
 *   Y        out or NULL, double [R][F]: the concatenated shard activations
 *   P        out or NULL, double [R][k][H]: each shard's partial Z_i (before the sum)
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_tpmlp_f64(const uint16_t *X, int64_t x_rows, const int64_t *rows, int64_t R,
                     const uint16_t *W1, const uint16_t *b1, const uint16_t *W2,
                     const uint16_t *b2, int64_t H, int64_t F, int32_t k, int32_t act,
                     double *Z, double *Y, double *P) {
    if (!X || !W1 || !b1 || !W2 || !b2 || !Z || H <= 0 || F <= 0 || k <= 0 || R < 0) return -1;
    if (F % k != 0) return -1;
    if (act != ORACLE_ACT_GELU && act != ORACLE_ACT_IDENTITY) return -1;
    const int64_t f = F / k;
    int failed = 0;

#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)f);
        double *part = (double *)malloc(sizeof(double) * (size_t)H);
        double *zsum = (double *)malloc(sizeof(double) * (size_t)H);
        if (!acc || !part || !zsum) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < R; ++r) {
                const int64_t m = rows ? rows[r] : r;
                if (m < 0 || m >= x_rows) {
#pragma omp atomic write
                    failed = 1;
                    continue;
                }
                const uint16_t *x = X + m * H;
                for (int64_t n = 0; n < H; ++n) zsum[n] = 0.0;

                for (int32_t i = 0; i < k; ++i) {
                    const int64_t j0 = (int64_t)i * f; /* first column of shard i */

                    /* Column shard i: acc[jj] = sum_h X[m,h] * W1[h, j0+jj] */
                    for (int64_t jj = 0; jj < f; ++jj) acc[jj] = 0.0;
                    for (int64_t h = 0; h < H; ++h) {
                        const double xh = widen_bf16(x[h]);
                        const uint16_t *w = W1 + h * F + j0;
                        for (int64_t jj = 0; jj < f; ++jj) acc[jj] += xh * widen_bf16(w[jj]);
                    }
                    /* + b1 slice, then the activation, element by element */
                    for (int64_t jj = 0; jj < f; ++jj) {
                        const double a = acc[jj] + widen_bf16(b1[j0 + jj]);
                        acc[jj] = (act == ORACLE_ACT_GELU) ? oracle_gelu(a) : a;
                        if (Y) Y[r * F + j0 + jj] = acc[jj];
                    }

                    /* Row shard i: part[n] = sum_{jj} Y_i[jj] * W2[j0+jj, n] */
                    for (int64_t n = 0; n < H; ++n) part[n] = 0.0;
                    for (int64_t jj = 0; jj < f; ++jj) {
                        const double y = acc[jj];
                        const uint16_t *w = W2 + (j0 + jj) * H;
                        for (int64_t n = 0; n < H; ++n) part[n] += y * widen_bf16(w[n]);
                    }
                    if (P)
                        for (int64_t n = 0; n < H; ++n) P[(r * k + i) * H + n] = part[n];

                    /* The all-reduce: sum of the shards' partials, in shard order */
                    for (int64_t n = 0; n < H; ++n) zsum[n] += part[n];
                }
                /* Output bias, once, after the sum */
                for (int64_t n = 0; n < H; ++n) Z[r * H + n] = zsum[n] + widen_bf16(b2[n]);
            }
        }
        free(acc);
        free(part);
        free(zsum);
    }
    return failed ? -1 : 0;
}

/*
 * Gated variant (the NEXT step the pages point to): the FFN's gate_up_proj is
 * column-parallel and its down_proj row-parallel (大模型分布式优化技术（一） §5.1;
 * AI大模型分布式训练 §6.1 gate_proj / up_proj ColwiseParallel, down_proj RowwiseParallel),
 * with the SwiGLU activation named in §3.3 of the first of those pages.
 * Reading: Y = SiLU(X Wg + bg) * (X Wu + bu), SiLU(a) = a / (1 + exp(-a)), element by
 * element; shard i owns columns [i f, (i+1) f) of BOTH Wg and Wu and rows [i f, (i+1) f) of W2.
 *   Z[m, n] = b2[n] + sum_i sum_{j in shard i} SiLU(ag_j) * au_j * W2[j, n]
 *   ag_j = bg[j] + sum_h X[m, h] Wg[h, j],   au_j = bu[j] + sum_h X[m, h] Wu[h, j]
 */
double oracle_silu(double a) { return a / (1.0 + exp(-a)); }

int oracle_tpmlp_swiglu_f64(const uint16_t *X, int64_t x_rows, const int64_t *rows, int64_t R,
                            const uint16_t *Wg, const uint16_t *bg, const uint16_t *Wu,
                            const uint16_t *bu, const uint16_t *W2, const uint16_t *b2, int64_t H,
                            int64_t F, int32_t k, double *Z, double *Y) {
    if (!X || !Wg || !bg || !Wu || !bu || !W2 || !b2 || !Z || H <= 0 || F <= 0 || k <= 0 || R < 0)
        return -1;
    if (F % k != 0) return -1;
    const int64_t f = F / k;
    int failed = 0;

#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)f);
        double *au = (double *)malloc(sizeof(double) * (size_t)f);
        double *part = (double *)malloc(sizeof(double) * (size_t)H);
        double *zsum = (double *)malloc(sizeof(double) * (size_t)H);
        if (!ag || !au || !part || !zsum) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < R; ++r) {
                const int64_t m = rows ? rows[r] : r;
                if (m < 0 || m >= x_rows) {
#pragma omp atomic write
                    failed = 1;
                    continue;
                }
                const uint16_t *x = X + m * H;
                for (int64_t n = 0; n < H; ++n) zsum[n] = 0.0;

                for (int32_t i = 0; i < k; ++i) {
                    const int64_t j0 = (int64_t)i * f;
                    /* column shard i of the gate and of the up projection */
                    for (int64_t jj = 0; jj < f; ++jj) ag[jj] = au[jj] = 0.0;
                    for (int64_t h = 0; h < H; ++h) {
                        const double xh = widen_bf16(x[h]);
                        const uint16_t *wg = Wg + h * F + j0;
                        const uint16_t *wu = Wu + h * F + j0;
                        for (int64_t jj = 0; jj < f; ++jj) {
                            ag[jj] += xh * widen_bf16(wg[jj]);
                            au[jj] += xh * widen_bf16(wu[jj]);
                        }
                    }
                    for (int64_t jj = 0; jj < f; ++jj) {
                        const double g = ag[jj] + widen_bf16(bg[j0 + jj]);
                        const double u = au[jj] + widen_bf16(bu[j0 + jj]);
                        ag[jj] = oracle_silu(g) * u;
                        if (Y) Y[r * F + j0 + jj] = ag[jj];
                    }
                    /* row shard i of W2, then the all-reduce (shard order) */
                    for (int64_t n = 0; n < H; ++n) part[n] = 0.0;
                    for (int64_t jj = 0; jj < f; ++jj) {
                        const double y = ag[jj];
                        const uint16_t *w = W2 + (j0 + jj) * H;
                        for (int64_t n = 0; n < H; ++n) part[n] += y * widen_bf16(w[n]);
                    }
                    for (int64_t n = 0; n < H; ++n) zsum[n] += part[n];
                }
                for (int64_t n = 0; n < H; ++n) Z[r * H + n] = zsum[n] + widen_bf16(b2[n]);
            }
        }
        free(ag);
        free(au);
        free(part);
        free(zsum);
    }
    return failed ? -1 : 0;
}

/*
 * The steps either side of the block inside a Transformer layer: the layer adds the MLP's
 * output to its input, x = x + mlp(x) (AI大模型分布式训练 §3.4, TransformerBlock.forward), and
 * LayerNorm normalises each token's full hidden vector before the block (大模型分布式并行策略详解
 * §4.2: LayerNorm needs the whole hidden state; AI大模型分布式训练 §4.2: sequence parallelism
 * splits LayerNorm along the tokens, which are independent).
 * Reading: the pre-LayerNorm sub-layer Z = X + MLP(LN(X)) with the standard LayerNorm
 *   LN(x)_h = (x_h - mu) / sqrt(var + eps) * gamma_h + beta_h,
 *   mu = (1/H) sum_h x_h,  var = (1/H) sum_h (x_h - mu)^2   (biased variance)
 * and MLP = the GeLU block above (k shards, sum over shards, + b2).
 *   Xn  out or NULL, double [R][H]: LN(X) of the selected rows
 */
int oracle_block_f64(const uint16_t *X, int64_t x_rows, const int64_t *rows, int64_t R,
                     const uint16_t *gamma, const uint16_t *beta, double eps,
                     const uint16_t *W1, const uint16_t *b1, const uint16_t *W2,
                     const uint16_t *b2, int64_t H, int64_t F, int32_t k, double *Z, double *Xn) {
    if (!X || !gamma || !beta || !W1 || !b1 || !W2 || !b2 || !Z || H <= 0 || F <= 0 || k <= 0 ||
        R < 0 || eps < 0.0)
        return -1;
    if (F % k != 0) return -1;
    const int64_t f = F / k;
    int failed = 0;

#pragma omp parallel
    {
        double *xn = (double *)malloc(sizeof(double) * (size_t)H);
        double *acc = (double *)malloc(sizeof(double) * (size_t)f);
        double *part = (double *)malloc(sizeof(double) * (size_t)H);
        double *zsum = (double *)malloc(sizeof(double) * (size_t)H);
        if (!xn || !acc || !part || !zsum) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < R; ++r) {
                const int64_t m = rows ? rows[r] : r;
                if (m < 0 || m >= x_rows) {
#pragma omp atomic write
                    failed = 1;
                    continue;
                }
                const uint16_t *x = X + m * H;

                /* LayerNorm of the token's hidden vector */
                double mu = 0.0;
                for (int64_t h = 0; h < H; ++h) mu += widen_bf16(x[h]);
                mu /= (double)H;
                double var = 0.0;
                for (int64_t h = 0; h < H; ++h) {
                    const double d = widen_bf16(x[h]) - mu;
                    var += d * d;
                }
                var /= (double)H;
                const double inv = 1.0 / sqrt(var + eps);
                for (int64_t h = 0; h < H; ++h) {
                    xn[h] = (widen_bf16(x[h]) - mu) * inv * widen_bf16(gamma[h]) + widen_bf16(beta[h]);
                    if (Xn) Xn[r * H + h] = xn[h];
                }

                /* the block on LN(x) */
                for (int64_t n = 0; n < H; ++n) zsum[n] = 0.0;
                for (int32_t i = 0; i < k; ++i) {
                    const int64_t j0 = (int64_t)i * f;
                    for (int64_t jj = 0; jj < f; ++jj) acc[jj] = 0.0;
                    for (int64_t h = 0; h < H; ++h) {
                        const double xh = xn[h];
                        const uint16_t *w = W1 + h * F + j0;
                        for (int64_t jj = 0; jj < f; ++jj) acc[jj] += xh * widen_bf16(w[jj]);
                    }
                    for (int64_t jj = 0; jj < f; ++jj)
                        acc[jj] = oracle_gelu(acc[jj] + widen_bf16(b1[j0 + jj]));
                    for (int64_t n = 0; n < H; ++n) part[n] = 0.0;
                    for (int64_t jj = 0; jj < f; ++jj) {
                        const double y = acc[jj];
                        const uint16_t *w = W2 + (j0 + jj) * H;
                        for (int64_t n = 0; n < H; ++n) part[n] += y * widen_bf16(w[n]);
                    }
                    for (int64_t n = 0; n < H; ++n) zsum[n] += part[n];
                }
                /* residual: the sub-layer's input plus the block's output */
                for (int64_t n = 0; n < H; ++n)
                    Z[r * H + n] = widen_bf16(x[n]) + (zsum[n] + widen_bf16(b2[n]));
            }
        }
        free(xn);
        free(acc);
        free(part);
        free(zsum);
    }
    return failed ? -1 : 0;
}

/*
 * The two parallel linear layers on their own, as the pages' tensor-parallel attention uses
 * them (AI大模型分布式训练 §2.3: the Q/K/V projection is a ColumnParallelLinear, the output
 * projection a RowParallelLinear followed by the All-Reduce; the heads are split into k
 * groups, one per shard). W is [K][N] (Y = X W), b is [N].
 *   kind 0, column-parallel: shard i owns columns [i f, (i+1) f), f = N / k;
 *           out[m, i f + j] = b[i f + j] + sum_h X[m, h] W[h, i f + j]
 *   kind 1, row-parallel:    shard i owns rows [i f, (i+1) f), f = K / k, and the input
 *           columns with them; out[m, n] = b[n] + sum_i ( sum_{j<f} X[m, i f + j] W[i f + j, n] )
 *           (each shard's partial first, then the sum over shards in shard order, then b once)
 */
int oracle_linear_f64(int32_t kind, const uint16_t *X, int64_t x_rows, const int64_t *rows,
                      int64_t R, const uint16_t *W, const uint16_t *b, int64_t K, int64_t N,
                      int32_t k, double *out) {
    if (!X || !W || !b || !out || K <= 0 || N <= 0 || k <= 0 || R < 0) return -1;
    if (kind != 0 && kind != 1) return -1;
    if ((kind == 0 && N % k != 0) || (kind == 1 && K % k != 0)) return -1;
    int failed = 0;

#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *part = (double *)malloc(sizeof(double) * (size_t)N);
        if (!acc || !part) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < R; ++r) {
                const int64_t m = rows ? rows[r] : r;
                if (m < 0 || m >= x_rows) {
#pragma omp atomic write
                    failed = 1;
                    continue;
                }
                const uint16_t *x = X + m * K;
                if (kind == 0) {
                    const int64_t f = N / k;
                    for (int32_t i = 0; i < k; ++i) {
                        const int64_t j0 = (int64_t)i * f;
                        for (int64_t jj = 0; jj < f; ++jj) acc[jj] = 0.0;
                        for (int64_t h = 0; h < K; ++h) {
                            const double xh = widen_bf16(x[h]);
                            const uint16_t *w = W + h * N + j0;
                            for (int64_t jj = 0; jj < f; ++jj) acc[jj] += xh * widen_bf16(w[jj]);
                        }
                        for (int64_t jj = 0; jj < f; ++jj)
                            out[r * N + j0 + jj] = acc[jj] + widen_bf16(b[j0 + jj]);
                    }
                } else {
                    const int64_t f = K / k;
                    for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
                    for (int32_t i = 0; i < k; ++i) {
                        const int64_t j0 = (int64_t)i * f;
                        for (int64_t n = 0; n < N; ++n) part[n] = 0.0;
                        for (int64_t jj = 0; jj < f; ++jj) {
                            const double xj = widen_bf16(x[j0 + jj]);
                            const uint16_t *w = W + (j0 + jj) * N;
                            for (int64_t n = 0; n < N; ++n) part[n] += xj * widen_bf16(w[n]);
                        }
                        for (int64_t n = 0; n < N; ++n) acc[n] += part[n];
                    }
                    for (int64_t n = 0; n < N; ++n) out[r * N + n] = acc[n] + widen_bf16(b[n]);
                }
            }
        }
        free(acc);
        free(part);
    }
    return failed ? -1 : 0;
}

/*
 * Backward pass of the block (the pages note that the backward pass repeats the same split
 * and needs its own All-Reduce: 分布式训练系列第四篇 §4.2-4.3; AI大模型分布式训练 §2.4 counts an
 * All-Reduce in the forward and one in the backward of each block). Given the upstream
 * gradient dZ [M, H] of Z = sum_i GeLU(X W1_i + b1_i) W2_i + b2:
 *   A   = X W1 + b1                      pre-activation   [M, F]
 *   dY  = dZ W2^T                        per column shard [M, F]
 *   dA  = dY * GeLU'(A),  GeLU'(a) = Phi(a) + a phi(a),  phi(a) = exp(-a^2 / 2) / sqrt(2 pi)
 *   dX  = sum_i dA_i W1_i^T              (the backward All-Reduce: a sum over shards)
 *   dW1 = X^T dA,   db1 = sum_m dA[m, :]
 *   dW2 = Y^T dZ,   db2 = sum_m dZ[m, :],   Y = GeLU(A)
 * Sums in index order (over shards last for dX). All outputs are double; dW1 [H][F],
 * dW2 [F][H]; any output pointer may be NULL to skip it.
 */
double oracle_gelu_grad(double a) {
    const double inv_sqrt_2pi = 0.39894228040143267794; /* 1 / sqrt(2 pi) */
    return 0.5 * (1.0 + erf(a / sqrt(2.0))) + a * inv_sqrt_2pi * exp(-0.5 * a * a);
}

int oracle_backward_f64(const uint16_t *X, const uint16_t *W1, const uint16_t *b1,
                        const uint16_t *W2, const uint16_t *dZ, int64_t M, int64_t H, int64_t F,
                        int32_t k, double *dX, double *dW1, double *db1, double *dW2,
                        double *db2) {
    if (!X || !W1 || !b1 || !W2 || !dZ || M <= 0 || H <= 0 || F <= 0 || k <= 0) return -1;
    if (F % k != 0) return -1;
    const int64_t f = F / k;
    double *A = (double *)malloc(sizeof(double) * (size_t)(M * F));
    double *dA = (double *)malloc(sizeof(double) * (size_t)(M * F));
    if (!A || !dA) {
        free(A);
        free(dA);
        return -1;
    }
    /* forward pre-activation and dA, row by row */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        double *a = A + m * F;
        for (int64_t j = 0; j < F; ++j) a[j] = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            const double xh = widen_bf16(X[m * H + h]);
            for (int64_t j = 0; j < F; ++j) a[j] += xh * widen_bf16(W1[h * F + j]);
        }
        for (int64_t j = 0; j < F; ++j) a[j] += widen_bf16(b1[j]);
        /* dY[m, j] = sum_n dZ[m, n] W2[j, n], then dA = dY * GeLU'(A) */
        for (int64_t j = 0; j < F; ++j) {
            double dy = 0.0;
            for (int64_t n = 0; n < H; ++n) dy += widen_bf16(dZ[m * H + n]) * widen_bf16(W2[j * H + n]);
            dA[m * F + j] = dy * oracle_gelu_grad(a[j]);
        }
    }
    if (dX) {
        /* dX[m, h] = sum_i sum_{j in shard i} dA[m, j] W1[h, j]: each shard's partial, then the sum */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t h = 0; h < H; ++h) {
                double total = 0.0;
                for (int32_t i = 0; i < k; ++i) {
                    double part = 0.0;
                    for (int64_t jj = 0; jj < f; ++jj)
                        part += dA[m * F + i * f + jj] * widen_bf16(W1[h * F + i * f + jj]);
                    total += part;
                }
                dX[m * H + h] = total;
            }
        }
    }
    if (dW1) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t j = 0; j < F; ++j) {
                double acc = 0.0;
                for (int64_t m = 0; m < M; ++m) acc += widen_bf16(X[m * H + h]) * dA[m * F + j];
                dW1[h * F + j] = acc;
            }
    }
    if (db1) {
        for (int64_t j = 0; j < F; ++j) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += dA[m * F + j];
            db1[j] = acc;
        }
    }
    if (dW2) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t j = 0; j < F; ++j)
            for (int64_t n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int64_t m = 0; m < M; ++m)
                    acc += oracle_gelu(A[m * F + j]) * widen_bf16(dZ[m * H + n]);
                dW2[j * H + n] = acc;
            }
    }
    if (db2) {
        for (int64_t n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += widen_bf16(dZ[m * H + n]);
            db2[n] = acc;
        }
    }
    free(A);
    free(dA);
    return 0;
}

/*
 * Backward pass of the gated block. The pages split gate_up_proj by columns and down_proj by
 * rows (大模型分布式优化技术（一） §5.1; AI大模型分布式训练 §6.1), and the backward pass repeats
 * the forward's split with one more sum over shards (分布式训练系列第四篇 §4.2-4.3; AI大模型分布式训练
 * §2.4). Given dZ [M, H] of Z = sum_i (SiLU(G_i) * U_i) W2_i + b2, by the chain rule:
 *   G   = X Wg + bg,   U = X Wu + bu                     pre-activations [M, F]
 *   dY  = dZ W2^T                                        per column shard [M, F]
 *   dU  = dY * SiLU(G)
 *   dG  = dY * U * SiLU'(G),  SiLU'(g) = s (1 + g (1 - s)),  s = 1 / (1 + exp(-g))
 *   dX  = sum_i (dG_i Wg_i^T + dU_i Wu_i^T)             (the backward All-Reduce)
 *   dWg = X^T dG, dbg = sum_m dG[m, :];  dWu = X^T dU, dbu = sum_m dU[m, :]
 *   dW2 = Y^T dZ, db2 = sum_m dZ[m, :],  Y = SiLU(G) * U
 * Sums in index order; for dX, shard i's gate part then its up part, then the sum over
 * shards. All outputs are double; dWg, dWu [H][F], dW2 [F][H]; any output may be NULL.
 */
double oracle_silu_grad(double g) {
    const double s = 1.0 / (1.0 + exp(-g));
    return s * (1.0 + g * (1.0 - s));
}

int oracle_swiglu_backward_f64(const uint16_t *X, const uint16_t *Wg, const uint16_t *bg,
                               const uint16_t *Wu, const uint16_t *bu, const uint16_t *W2,
                               const uint16_t *dZ, int64_t M, int64_t H, int64_t F, int32_t k,
                               double *dX, double *dWg, double *dbg, double *dWu, double *dbu,
                               double *dW2, double *db2) {
    if (!X || !Wg || !bg || !Wu || !bu || !W2 || !dZ || M <= 0 || H <= 0 || F <= 0 || k <= 0)
        return -1;
    if (F % k != 0) return -1;
    const int64_t f = F / k;
    const size_t n = (size_t)(M * F);
    double *G = (double *)malloc(sizeof(double) * n);
    double *U = (double *)malloc(sizeof(double) * n);
    double *dG = (double *)malloc(sizeof(double) * n);
    double *dU = (double *)malloc(sizeof(double) * n);
    if (!G || !U || !dG || !dU) {
        free(G);
        free(U);
        free(dG);
        free(dU);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        double *g = G + m * F, *u = U + m * F;
        for (int64_t j = 0; j < F; ++j) g[j] = u[j] = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            const double xh = widen_bf16(X[m * H + h]);
            for (int64_t j = 0; j < F; ++j) {
                g[j] += xh * widen_bf16(Wg[h * F + j]);
                u[j] += xh * widen_bf16(Wu[h * F + j]);
            }
        }
        for (int64_t j = 0; j < F; ++j) {
            g[j] += widen_bf16(bg[j]);
            u[j] += widen_bf16(bu[j]);
        }
        for (int64_t j = 0; j < F; ++j) {
            double dy = 0.0;
            for (int64_t c = 0; c < H; ++c) dy += widen_bf16(dZ[m * H + c]) * widen_bf16(W2[j * H + c]);
            dU[m * F + j] = dy * oracle_silu(g[j]);
            dG[m * F + j] = dy * u[j] * oracle_silu_grad(g[j]);
        }
    }
    if (dX) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t h = 0; h < H; ++h) {
                double total = 0.0;
                for (int32_t i = 0; i < k; ++i) {
                    double part = 0.0;
                    for (int64_t jj = 0; jj < f; ++jj)
                        part += dG[m * F + i * f + jj] * widen_bf16(Wg[h * F + i * f + jj]);
                    for (int64_t jj = 0; jj < f; ++jj)
                        part += dU[m * F + i * f + jj] * widen_bf16(Wu[h * F + i * f + jj]);
                    total += part;
                }
                dX[m * H + h] = total;
            }
        }
    }
    if (dWg || dWu) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t j = 0; j < F; ++j) {
                double ag = 0.0, au = 0.0;
                for (int64_t m = 0; m < M; ++m) {
                    const double xh = widen_bf16(X[m * H + h]);
                    ag += xh * dG[m * F + j];
                    au += xh * dU[m * F + j];
                }
                if (dWg) dWg[h * F + j] = ag;
                if (dWu) dWu[h * F + j] = au;
            }
    }
    for (int64_t j = 0; j < F && (dbg || dbu); ++j) {
        double ag = 0.0, au = 0.0;
        for (int64_t m = 0; m < M; ++m) {
            ag += dG[m * F + j];
            au += dU[m * F + j];
        }
        if (dbg) dbg[j] = ag;
        if (dbu) dbu[j] = au;
    }
    if (dW2) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t j = 0; j < F; ++j)
            for (int64_t c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int64_t m = 0; m < M; ++m)
                    acc += oracle_silu(G[m * F + j]) * U[m * F + j] * widen_bf16(dZ[m * H + c]);
                dW2[j * H + c] = acc;
            }
    }
    if (db2) {
        for (int64_t c = 0; c < H; ++c) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += widen_bf16(dZ[m * H + c]);
            db2[c] = acc;
        }
    }
    free(G);
    free(U);
    free(dG);
    free(dU);
    return 0;
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
