/*
 * oracle.c -- plain, slow, unsharded CPU reference for the tensor-parallel
 * MLP block and the vocabulary-parallel cross-entropy.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
 * loads or calls this file; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg do. It shares no code, header or constant with
 * the CUDA library.
 *
 * Arithmetic: every input arrives as float64 (the callers widen the exact
 * bf16 or fp32 values that the GPU also reads); every sum, product, exp, log
 * and erf is done in double precision, in the plain order of the definition.
 * The matrix products are written out as loops; the only parallelism is an
 * OpenMP split over independent output rows, which does not change any sum.
 *
 * Layout: row-major everywhere. X, Z, dX, dZ, H, dH are [T, h]; A, dA are
 * [h, f]; B, dB are [f, h]; U, Y are [T, f]; E, dE are [v_pad, h].
 *
 * Sources (page title, then section):
 *   [MF]  "Tensor Parallelism and Pipeline Parallelism: Mathematical
 *         Foundations of Megatron-LM 1D Slicing ..." (llms.blog):
 *         "Column-Parallel Linear Layer", "Row-Parallel Linear Layer",
 *         "Conjugate Communication Operators".
 *   [LIT] "LIT-022: Megatron-LM: Training Multi-Billion Parameter Language
 *         Models Using Model Parallelism" (anthology digest): "Key takeaways".
 *   [LEC] "Cutting a Model Into Pieces" (lecture 3): "Megatron-LM: cutting
 *         inside the layer".
 *   [DEP] "Megatron-LM, in depth" (aicassindra): "Failure modes".
 *   [70B] "Distributed tensor parallelism: scale fine-tuning of 70B-parameter
 *         LLMs with Megatron-LM" (mohashari.github.io): "The Mechanics of
 *         Tensor Parallelism (TP) in Megatron-LM", "The MLP Block", "The
 *         Multi-Head Attention Block".
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - GeLU is the exact erf form x * Phi(x); its derivative Phi(x) + x phi(x).
 *   - The row-parallel bias bB is added once, after the shard sum.
 *   - The backward is the chain rule of the forward; f* sums the per-shard
 *     input gradients, g* hands the same dZ to every shard.
 *   - Cross-entropy is the textbook softmax cross-entropy over the real ids
 *     [0, v_valid); padded ids take no part in the max or the sum of exps
 *     and get a zero gradient.
 *   - The gradient returned is that of grad_scale * sum_t loss_t.
 *   - Swish in the SwiGLU block is x * sigmoid(x) (beta = 1); the first
 *     weight W1 = [W_gate | W_up] is one [h, 2f] matrix, gate columns first.
 *   - The fused QKV weight is laid out by key/value head groups: for each KV
 *     head g, the query heads that share it, then K_g, then V_g, so that a
 *     contiguous column split into t blocks hands each shard whole heads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* GeLU(x) = x * Phi(x), Phi the standard normal CDF written with erf.
 * [LIT] key takeaways (GeLU between the two GEMMs); [LEC] Y = GeLU(XA). */
double oracle_gelu(double x)
{
    return x * 0.5 * (1.0 + erf(x / sqrt(2.0)));
}

/* d/dx [x Phi(x)] = Phi(x) + x phi(x), phi the standard normal density. */
double oracle_gelu_grad(double x)
{
    double Phi = 0.5 * (1.0 + erf(x / sqrt(2.0)));
    double phi = exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
    return Phi + x * phi;
}

/* ------------------------------------------------------------------------ */
/* MLP forward, unsharded: U = X A + bA, Y = GeLU(U), Z = Y B + bB.
 * [LEC] Y = GeLU(X A), Z = Y B. bA, bB may be NULL (zero). U, Y, Z may be
 * NULL when the caller does not want them. */
void oracle_mlp_forward(int64_t T, int64_t h, int64_t f,
                        const double *X, const double *A, const double *bA,
                        const double *B, const double *bB,
                        double *U, double *Y, double *Z)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        double *u = (double *)malloc(sizeof(double) * (size_t)f);
        double *y = (double *)malloc(sizeof(double) * (size_t)f);
        for (int64_t j = 0; j < f; j++)
            u[j] = bA ? bA[j] : 0.0;
        for (int64_t k = 0; k < h; k++) {
            double x = X[t * h + k];
            for (int64_t j = 0; j < f; j++)
                u[j] += x * A[k * f + j];
        }
        for (int64_t j = 0; j < f; j++)
            y[j] = oracle_gelu(u[j]);
        if (Z) {
            for (int64_t n = 0; n < h; n++)
                Z[t * h + n] = bB ? bB[n] : 0.0;
            for (int64_t j = 0; j < f; j++) {
                double yj = y[j];
                for (int64_t n = 0; n < h; n++)
                    Z[t * h + n] += yj * B[j * h + n];
            }
        }
        if (U) memcpy(U + t * f, u, sizeof(double) * (size_t)f);
        if (Y) memcpy(Y + t * f, y, sizeof(double) * (size_t)f);
        free(u);
        free(y);
    }
}

/* MLP backward, unsharded, by the chain rule of oracle_mlp_forward for the
 * upstream gradient dZ:
 *   dB = Y^T dZ,  dbB = sum_t dZ,  dY = dZ B^T,  dU = dY (.) GeLU'(U),
 *   dA = X^T dU,  dbA = sum_t dU,  dX = dU A^T.
 * The oracle recomputes U and Y itself from X, A, bA. Any output may be NULL.
 */
void oracle_mlp_backward(int64_t T, int64_t h, int64_t f,
                         const double *X, const double *A, const double *bA,
                         const double *B, const double *dZ,
                         double *dX, double *dA, double *dbA,
                         double *dB, double *dbB)
{
    double *U = (double *)malloc(sizeof(double) * (size_t)(T * f));
    double *Y = (double *)malloc(sizeof(double) * (size_t)(T * f));
    double *dU = (double *)malloc(sizeof(double) * (size_t)(T * f));
    oracle_mlp_forward(T, h, f, X, A, bA, B, NULL, U, Y, NULL);

    int64_t t, j, k, n;
    /* dY = dZ B^T, then dU = dY (.) GeLU'(U) */
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        for (int64_t jj = 0; jj < f; jj++) {
            double acc = 0.0;
            for (int64_t nn = 0; nn < h; nn++)
                acc += dZ[t * h + nn] * B[jj * h + nn];
            dU[t * f + jj] = acc * oracle_gelu_grad(U[t * f + jj]);
        }
    }
    if (dX) {
        /* dX = dU A^T */
#pragma omp parallel for schedule(static)
        for (t = 0; t < T; t++) {
            for (int64_t kk = 0; kk < h; kk++) {
                double acc = 0.0;
                for (int64_t jj = 0; jj < f; jj++)
                    acc += dU[t * f + jj] * A[kk * f + jj];
                dX[t * h + kk] = acc;
            }
        }
    }
    if (dA) {
        /* dA = X^T dU */
#pragma omp parallel for schedule(static)
        for (k = 0; k < h; k++) {
            for (int64_t jj = 0; jj < f; jj++)
                dA[k * f + jj] = 0.0;
            for (int64_t tt = 0; tt < T; tt++) {
                double x = X[tt * h + k];
                for (int64_t jj = 0; jj < f; jj++)
                    dA[k * f + jj] += x * dU[tt * f + jj];
            }
        }
    }
    if (dB) {
        /* dB = Y^T dZ */
#pragma omp parallel for schedule(static)
        for (j = 0; j < f; j++) {
            for (int64_t nn = 0; nn < h; nn++)
                dB[j * h + nn] = 0.0;
            for (int64_t tt = 0; tt < T; tt++) {
                double y = Y[tt * f + j];
                for (int64_t nn = 0; nn < h; nn++)
                    dB[j * h + nn] += y * dZ[tt * h + nn];
            }
        }
    }
    if (dbA) {
        for (j = 0; j < f; j++) {
            double acc = 0.0;
            for (t = 0; t < T; t++)
                acc += dU[t * f + j];
            dbA[j] = acc;
        }
    }
    if (dbB) {
        for (n = 0; n < h; n++) {
            double acc = 0.0;
            for (t = 0; t < T; t++)
                acc += dZ[t * h + n];
            dbB[n] = acc;
        }
    }
    free(U);
    free(Y);
    free(dU);
}

/* Selected columns j of the weight gradients, from the same definitions:
 * dA[:, j] = X^T dU[:, j], dbA[j] = sum_t dU[t, j], dB[j, :] = Y[:, j]^T dZ,
 * with U[:, j] = X A[:, j] + bA[j], dU[:, j] = (dZ B[j, :]^T) (.) GeLU'(U[:, j]).
 * Column j needs only O(T h) work, which makes full-size spot checks cheap.
 * Outputs: dA_cols [h][ncols], dbA_cols [ncols], dB_rows [ncols][h]. */
void oracle_mlp_backward_cols(int64_t T, int64_t h, int64_t f,
                              const double *X, const double *A, const double *bA,
                              const double *B, const double *dZ,
                              int64_t ncols, const int64_t *cols,
                              double *dA_cols, double *dbA_cols, double *dB_rows)
{
    int64_t c;
#pragma omp parallel for schedule(dynamic)
    for (c = 0; c < ncols; c++) {
        int64_t j = cols[c];
        double *a = (double *)malloc(sizeof(double) * (size_t)h);   /* A[:, j] */
        double *u = (double *)malloc(sizeof(double) * (size_t)T);
        double *du = (double *)malloc(sizeof(double) * (size_t)T);
        double *da = (double *)calloc((size_t)h, sizeof(double));
        double *db = (double *)calloc((size_t)h, sizeof(double));
        for (int64_t k = 0; k < h; k++)
            a[k] = A[k * f + j];
        for (int64_t t = 0; t < T; t++) {
            double acc = bA ? bA[j] : 0.0;
            for (int64_t k = 0; k < h; k++)
                acc += X[t * h + k] * a[k];
            u[t] = acc;
            double dy = 0.0;
            for (int64_t n = 0; n < h; n++)
                dy += dZ[t * h + n] * B[j * h + n];
            du[t] = dy * oracle_gelu_grad(acc);
        }
        double sb = 0.0;
        for (int64_t t = 0; t < T; t++)
            sb += du[t];
        dbA_cols[c] = sb;
        /* dA[k, j] = sum_t X[t, k] du[t] and dB[j, n] = sum_t Y[t, j] dZ[t, n],
         * each sum taken over t in order */
        for (int64_t t = 0; t < T; t++) {
            double y = oracle_gelu(u[t]);
            for (int64_t k = 0; k < h; k++)
                da[k] += X[t * h + k] * du[t];
            for (int64_t n = 0; n < h; n++)
                db[n] += y * dZ[t * h + n];
        }
        for (int64_t k = 0; k < h; k++)
            dA_cols[k * ncols + c] = da[k];
        memcpy(dB_rows + c * h, db, sizeof(double) * (size_t)h);
        free(a);
        free(u);
        free(du);
        free(da);
        free(db);
    }
}

/* dbB = sum_t dZ[t, :] -- the row-parallel bias gradient on its own, the same
 * definition oracle_mlp_backward uses. Out: dbB [h]. */
void oracle_bias_grad(int64_t T, int64_t h, const double *dZ, double *dbB)
{
    for (int64_t n = 0; n < h; n++) {
        double acc = 0.0;
        for (int64_t t = 0; t < T; t++)
            acc += dZ[t * h + n];
        dbB[n] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* The sharded restatement of the same block, for t shards, written the way
 * the pages partition it. [MF] "Column-Parallel Linear Layer": A = [A_1 ..
 * A_t] by columns, Y_i = GeLU(X A_i) per shard with no exchange; [MF]
 * "Row-Parallel Linear Layer": B = [B_1; ..; B_t] by rows, Z_i = Y_i B_i and
 * Z = sum_i Z_i (the forward operator g); bias bA split with A's columns, bB
 * added once after the sum. The backward follows [MF] "Conjugate
 * Communication Operators": g* passes dZ unchanged to every shard, each shard
 * forms its own dB_i, dU_i, dA_i and partial dX_i, and f* sums the dX_i.
 * Used only to pin that the partition reproduces the unsharded block.
 * Requires f % t == 0. */
void oracle_mlp_sharded(int64_t T, int64_t h, int64_t f, int t,
                        const double *X, const double *A, const double *bA,
                        const double *B, const double *bB, const double *dZ,
                        double *Z, double *dX, double *dA, double *dB)
{
    int64_t fs = f / t;
    double *Zi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *dXi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *Ai = (double *)malloc(sizeof(double) * (size_t)(h * fs));
    double *bAi = (double *)malloc(sizeof(double) * (size_t)fs);
    double *Bi = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    double *dAi = (double *)malloc(sizeof(double) * (size_t)(h * fs));
    double *dBi = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    for (int64_t e = 0; e < T * h; e++) {
        Z[e] = 0.0;
        dX[e] = 0.0;
    }
    for (int i = 0; i < t; i++) {
        /* shard i's slices: columns [i fs, (i+1) fs) of A and bA, rows of B */
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++)
                Ai[k * fs + j] = A[k * f + (int64_t)i * fs + j];
        for (int64_t j = 0; j < fs; j++)
            bAi[j] = bA ? bA[(int64_t)i * fs + j] : 0.0;
        memcpy(Bi, B + (int64_t)i * fs * h, sizeof(double) * (size_t)(fs * h));
        /* forward of shard i (partial Z_i, no bias), then g: Z += Z_i */
        oracle_mlp_forward(T, h, fs, X, Ai, bAi, Bi, NULL, NULL, NULL, Zi);
        for (int64_t e = 0; e < T * h; e++)
            Z[e] += Zi[e];
        /* backward of shard i under g* (dZ unchanged), then f*: dX += dX_i */
        oracle_mlp_backward(T, h, fs, X, Ai, bAi, Bi, dZ, dXi, dAi, NULL, dBi, NULL);
        for (int64_t e = 0; e < T * h; e++)
            dX[e] += dXi[e];
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++)
                dA[k * f + (int64_t)i * fs + j] = dAi[k * fs + j];
        memcpy(dB + (int64_t)i * fs * h, dBi, sizeof(double) * (size_t)(fs * h));
    }
    /* bB enters once, after the sum over shards */
    for (int64_t tt = 0; tt < T; tt++)
        for (int64_t n = 0; n < h; n++)
            Z[tt * h + n] += bB ? bB[n] : 0.0;
    free(Zi);
    free(dXi);
    free(Ai);
    free(bAi);
    free(Bi);
    free(dAi);
    free(dBi);
}

/* ------------------------------------------------------------------------ */
/* Softmax cross-entropy over the logits l = H E^T, unsharded. [LIT] key
 * takeaways: the logit GEMM is fused with the cross-entropy loss. For token
 * t over the real ids j < v_valid:
 *   lse_t  = log sum_j exp(l_tj)        (written with the max subtracted)
 *   loss_t = lse_t - l_{t, target_t}
 *   dl_tj  = grad_scale * (exp(l_tj - lse_t) - [j == target_t]),  0 for j >= v_valid
 *   dH = dl E,  dE = dl^T H  (rows j >= v_valid of dE are zero).
 * loss, lse: [T]. dH [T, h] and dE [v_pad, h] may be NULL. A target outside
 * [0, v_valid) makes the loss of that token NaN. */
void oracle_ce(int64_t T, int64_t h, int64_t v_pad, int64_t v_valid,
               const double *H, const double *E, const int32_t *targets,
               double grad_scale, double *loss, double *lse,
               double *dH, double *dE)
{
    double *dl = NULL;
    if (dE)
        dl = (double *)malloc(sizeof(double) * (size_t)(T * v_valid));
    int64_t t;
#pragma omp parallel for schedule(dynamic)
    for (t = 0; t < T; t++) {
        double *l = (double *)malloc(sizeof(double) * (size_t)v_valid);
        for (int64_t j = 0; j < v_valid; j++) {
            double acc = 0.0;
            for (int64_t k = 0; k < h; k++)
                acc += H[t * h + k] * E[j * h + k];
            l[j] = acc;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < v_valid; j++)
            if (l[j] > m) m = l[j];
        double S = 0.0;
        for (int64_t j = 0; j < v_valid; j++)
            S += exp(l[j] - m);
        double L = m + log(S);
        int32_t y = targets[t];
        int ok = (y >= 0 && (int64_t)y < v_valid);
        lse[t] = L;
        loss[t] = ok ? L - l[y] : NAN;
        if (dH || dE) {
            for (int64_t j = 0; j < v_valid; j++)
                l[j] = grad_scale * (exp(l[j] - L) - (j == (int64_t)y ? 1.0 : 0.0));
            if (dH) {
                for (int64_t k = 0; k < h; k++)
                    dH[t * h + k] = 0.0;
                for (int64_t j = 0; j < v_valid; j++) {
                    double d = l[j];
                    for (int64_t k = 0; k < h; k++)
                        dH[t * h + k] += d * E[j * h + k];
                }
            }
            if (dE)
                memcpy(dl + t * v_valid, l, sizeof(double) * (size_t)v_valid);
        }
        free(l);
    }
    if (dE) {
        int64_t j;
#pragma omp parallel for schedule(static)
        for (j = 0; j < v_pad; j++) {
            for (int64_t k = 0; k < h; k++)
                dE[j * h + k] = 0.0;
            if (j >= v_valid) continue;
            for (int64_t tt = 0; tt < T; tt++) {
                double d = dl[tt * v_valid + j];
                for (int64_t k = 0; k < h; k++)
                    dE[j * h + k] += d * H[tt * h + k];
            }
        }
        free(dl);
    }
}

/* The vocabulary-parallel form of the same loss, written the way the digest
 * describes the fusion ([LIT] key takeaways): E is split by rows into t shards
 * of v_pad / t ids; shard i computes its own logits and reduces them, per
 * token, to three numbers -- its max m_i over its real ids, its sum
 * s_i = sum exp(l - m_i), and the target logit if it owns the target. Only
 * these per-token numbers are combined:
 *   m = max_i m_i,  S = sum_i s_i exp(m_i - m),  loss = m + log S - tau.
 * A shard holding only padded ids has m_i = -inf, s_i = 0 and takes no part.
 * Outputs: m_shard, s_shard [t][T], tau [T], loss [T]. */
void oracle_ce_sharded(int64_t T, int64_t h, int64_t v_pad, int64_t v_valid, int t,
                       const double *H, const double *E, const int32_t *targets,
                       double *m_shard, double *s_shard, double *tau, double *loss)
{
    int64_t vs = v_pad / t;
    int64_t tok;
#pragma omp parallel for schedule(dynamic)
    for (tok = 0; tok < T; tok++) {
        double *l = (double *)malloc(sizeof(double) * (size_t)vs);
        int32_t y = targets[tok];
        tau[tok] = NAN;
        for (int i = 0; i < t; i++) {
            int64_t lo = (int64_t)i * vs, hi = lo + vs;
            if (hi > v_valid) hi = v_valid; /* padded ids are not logits */
            double m = -INFINITY, s = 0.0;
            for (int64_t j = lo; j < hi; j++) {
                double acc = 0.0;
                for (int64_t k = 0; k < h; k++)
                    acc += H[tok * h + k] * E[j * h + k];
                l[j - lo] = acc;
                if (acc > m) m = acc;
            }
            for (int64_t j = lo; j < hi; j++)
                s += exp(l[j - lo] - m);
            if ((int64_t)y >= lo && (int64_t)y < hi)
                tau[tok] = l[y - lo];
            m_shard[(int64_t)i * T + tok] = m;
            s_shard[(int64_t)i * T + tok] = s;
        }
        double M = -INFINITY;
        for (int i = 0; i < t; i++)
            if (m_shard[(int64_t)i * T + tok] > M) M = m_shard[(int64_t)i * T + tok];
        double S = 0.0;
        for (int i = 0; i < t; i++) {
            double si = s_shard[(int64_t)i * T + tok];
            if (si > 0.0)
                S += si * exp(m_shard[(int64_t)i * T + tok] - M);
        }
        loss[tok] = M + log(S) - tau[tok];
        free(l);
    }
}

/* ------------------------------------------------------------------------ */
/* The SwiGLU variant of the block. [70B] "The MLP Block":
 *   MLP(x) = (Swish(x W_gate) (.) (x W_up)) W_down,
 * W_gate and W_up split by columns (column-parallel), W_down by rows
 * (row-parallel) with the partial products summed. Biases are optional and,
 * as in the GeLU block, the row-parallel bias enters once.
 * Layout: W1 = [W_gate | W_up] is [h, 2f] (gate columns 0..f-1, up columns
 * f..2f-1), b1 [2f]; W2 = W_down is [f, h], b2 [h]; GU = [G | Up] is [T, 2f]
 * with G = X W_gate + b_gate and Up = X W_up + b_up; Y = Swish(G) (.) Up is
 * [T, f]; Z = Y W2 + b2 is [T, h]. */

/* Swish(x) = x sigmoid(x) = x / (1 + e^{-x}). */
double oracle_swish(double x)
{
    return x / (1.0 + exp(-x));
}

/* d/dx [x sigmoid(x)] = sigmoid(x) + x sigmoid(x) (1 - sigmoid(x)). */
double oracle_swish_grad(double x)
{
    double s = 1.0 / (1.0 + exp(-x));
    return s + x * s * (1.0 - s);
}

/* Forward, unsharded. GU, Y, Z may be NULL; b1, b2 may be NULL (zero). */
void oracle_swiglu_forward(int64_t T, int64_t h, int64_t f,
                           const double *X, const double *W1, const double *b1,
                           const double *W2, const double *b2,
                           double *GU, double *Y, double *Z)
{
    int64_t f2 = 2 * f;
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        double *gu = (double *)malloc(sizeof(double) * (size_t)f2);
        double *y = (double *)malloc(sizeof(double) * (size_t)f);
        for (int64_t j = 0; j < f2; j++)
            gu[j] = b1 ? b1[j] : 0.0;
        for (int64_t k = 0; k < h; k++) {
            double x = X[t * h + k];
            for (int64_t j = 0; j < f2; j++)
                gu[j] += x * W1[k * f2 + j];
        }
        for (int64_t j = 0; j < f; j++)
            y[j] = oracle_swish(gu[j]) * gu[f + j];
        if (Z) {
            for (int64_t n = 0; n < h; n++)
                Z[t * h + n] = b2 ? b2[n] : 0.0;
            for (int64_t j = 0; j < f; j++) {
                double yj = y[j];
                for (int64_t n = 0; n < h; n++)
                    Z[t * h + n] += yj * W2[j * h + n];
            }
        }
        if (GU) memcpy(GU + t * f2, gu, sizeof(double) * (size_t)f2);
        if (Y) memcpy(Y + t * f, y, sizeof(double) * (size_t)f);
        free(gu);
        free(y);
    }
}

/* Backward, unsharded, by the chain rule of oracle_swiglu_forward:
 *   dW2 = Y^T dZ,  db2 = sum_t dZ,  dY = dZ W2^T,
 *   dG = dY (.) Up (.) Swish'(G),  dUp = dY (.) Swish(G),  dGU = [dG | dUp],
 *   dW1 = X^T dGU,  db1 = sum_t dGU,  dX = dGU W1^T.
 * G, Up and Y are recomputed from X, W1, b1. Any output may be NULL. */
void oracle_swiglu_backward(int64_t T, int64_t h, int64_t f,
                            const double *X, const double *W1, const double *b1,
                            const double *W2, const double *dZ,
                            double *dX, double *dW1, double *db1,
                            double *dW2, double *db2)
{
    int64_t f2 = 2 * f;
    double *GU = (double *)malloc(sizeof(double) * (size_t)(T * f2));
    double *Y = (double *)malloc(sizeof(double) * (size_t)(T * f));
    double *dGU = (double *)malloc(sizeof(double) * (size_t)(T * f2));
    oracle_swiglu_forward(T, h, f, X, W1, b1, W2, NULL, GU, Y, NULL);

    int64_t t, j, k, n;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        for (int64_t jj = 0; jj < f; jj++) {
            double dy = 0.0;
            for (int64_t nn = 0; nn < h; nn++)
                dy += dZ[t * h + nn] * W2[jj * h + nn];
            double g = GU[t * f2 + jj], u = GU[t * f2 + f + jj];
            dGU[t * f2 + jj] = dy * u * oracle_swish_grad(g);
            dGU[t * f2 + f + jj] = dy * oracle_swish(g);
        }
    }
    if (dX) {
#pragma omp parallel for schedule(static)
        for (t = 0; t < T; t++) {
            for (int64_t kk = 0; kk < h; kk++) {
                double acc = 0.0;
                for (int64_t jj = 0; jj < f2; jj++)
                    acc += dGU[t * f2 + jj] * W1[kk * f2 + jj];
                dX[t * h + kk] = acc;
            }
        }
    }
    if (dW1) {
#pragma omp parallel for schedule(static)
        for (k = 0; k < h; k++) {
            for (int64_t jj = 0; jj < f2; jj++)
                dW1[k * f2 + jj] = 0.0;
            for (int64_t tt = 0; tt < T; tt++) {
                double x = X[tt * h + k];
                for (int64_t jj = 0; jj < f2; jj++)
                    dW1[k * f2 + jj] += x * dGU[tt * f2 + jj];
            }
        }
    }
    if (dW2) {
#pragma omp parallel for schedule(static)
        for (j = 0; j < f; j++) {
            for (int64_t nn = 0; nn < h; nn++)
                dW2[j * h + nn] = 0.0;
            for (int64_t tt = 0; tt < T; tt++) {
                double y = Y[tt * f + j];
                for (int64_t nn = 0; nn < h; nn++)
                    dW2[j * h + nn] += y * dZ[tt * h + nn];
            }
        }
    }
    if (db1) {
        for (j = 0; j < f2; j++) {
            double acc = 0.0;
            for (t = 0; t < T; t++)
                acc += dGU[t * f2 + j];
            db1[j] = acc;
        }
    }
    if (db2) {
        for (n = 0; n < h; n++) {
            double acc = 0.0;
            for (t = 0; t < T; t++)
                acc += dZ[t * h + n];
            db2[n] = acc;
        }
    }
    free(GU);
    free(Y);
    free(dGU);
}

/* Selected columns j (0 <= j < f) of the SwiGLU weight gradients, from the
 * same definitions: the gate column j and the up column f + j of dW1 and db1,
 * and row j of dW2. O(T h) work per column, for full-size spot checks.
 * Outputs: dW1g_cols, dW1u_cols [h][ncols], db1g_cols, db1u_cols [ncols],
 * dW2_rows [ncols][h]. */
void oracle_swiglu_backward_cols(int64_t T, int64_t h, int64_t f,
                                 const double *X, const double *W1, const double *b1,
                                 const double *W2, const double *dZ,
                                 int64_t ncols, const int64_t *cols,
                                 double *dW1g_cols, double *dW1u_cols,
                                 double *db1g_cols, double *db1u_cols, double *dW2_rows)
{
    int64_t f2 = 2 * f;
    int64_t c;
#pragma omp parallel for schedule(dynamic)
    for (c = 0; c < ncols; c++) {
        int64_t j = cols[c];
        double *dg = (double *)malloc(sizeof(double) * (size_t)T);
        double *du = (double *)malloc(sizeof(double) * (size_t)T);
        double *y = (double *)malloc(sizeof(double) * (size_t)T);
        double *wg = (double *)calloc((size_t)h, sizeof(double));
        double *wu = (double *)calloc((size_t)h, sizeof(double));
        double *w2 = (double *)calloc((size_t)h, sizeof(double));
        for (int64_t t = 0; t < T; t++) {
            double g = b1 ? b1[j] : 0.0, u = b1 ? b1[f + j] : 0.0;
            for (int64_t k = 0; k < h; k++) {
                g += X[t * h + k] * W1[k * f2 + j];
                u += X[t * h + k] * W1[k * f2 + f + j];
            }
            double dy = 0.0;
            for (int64_t n = 0; n < h; n++)
                dy += dZ[t * h + n] * W2[j * h + n];
            dg[t] = dy * u * oracle_swish_grad(g);
            du[t] = dy * oracle_swish(g);
            y[t] = oracle_swish(g) * u;
        }
        double sg = 0.0, su = 0.0;
        for (int64_t t = 0; t < T; t++) {
            sg += dg[t];
            su += du[t];
        }
        db1g_cols[c] = sg;
        db1u_cols[c] = su;
        for (int64_t t = 0; t < T; t++) {
            for (int64_t k = 0; k < h; k++) {
                wg[k] += X[t * h + k] * dg[t];
                wu[k] += X[t * h + k] * du[t];
            }
            for (int64_t n = 0; n < h; n++)
                w2[n] += y[t] * dZ[t * h + n];
        }
        for (int64_t k = 0; k < h; k++) {
            dW1g_cols[k * ncols + c] = wg[k];
            dW1u_cols[k * ncols + c] = wu[k];
        }
        memcpy(dW2_rows + c * h, w2, sizeof(double) * (size_t)h);
        free(dg);
        free(du);
        free(y);
        free(wg);
        free(wu);
        free(w2);
    }
}

/* The SwiGLU block computed shard by shard, as [70B] "The MLP Block" lays
 * it out: shard i holds gate columns [i fs, (i+1) fs) and the same up
 * columns (f + i fs ...) of W1, and rows [i fs, (i+1) fs) of W2; it computes
 * Y_i = Swish(X W_gate,i) (.) (X W_up,i) and the partial Z_i = Y_i W2_i with
 * no exchange; Z = sum_i Z_i, then b2 once. Backward: every shard sees the
 * same dZ; the partial dX_i are summed. Requires f % t == 0. */
void oracle_swiglu_sharded(int64_t T, int64_t h, int64_t f, int t,
                           const double *X, const double *W1, const double *b1,
                           const double *W2, const double *b2, const double *dZ,
                           double *Z, double *dX, double *dW1, double *dW2)
{
    int64_t fs = f / t, f2 = 2 * f, fs2 = 2 * fs;
    double *Zi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *dXi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *W1i = (double *)malloc(sizeof(double) * (size_t)(h * fs2));
    double *b1i = (double *)malloc(sizeof(double) * (size_t)fs2);
    double *W2i = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    double *dW1i = (double *)malloc(sizeof(double) * (size_t)(h * fs2));
    double *dW2i = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    for (int64_t e = 0; e < T * h; e++) {
        Z[e] = 0.0;
        dX[e] = 0.0;
    }
    for (int i = 0; i < t; i++) {
        int64_t g0 = (int64_t)i * fs, u0 = f + (int64_t)i * fs;
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++) {
                W1i[k * fs2 + j] = W1[k * f2 + g0 + j];
                W1i[k * fs2 + fs + j] = W1[k * f2 + u0 + j];
            }
        for (int64_t j = 0; j < fs; j++) {
            b1i[j] = b1 ? b1[g0 + j] : 0.0;
            b1i[fs + j] = b1 ? b1[u0 + j] : 0.0;
        }
        memcpy(W2i, W2 + g0 * h, sizeof(double) * (size_t)(fs * h));
        oracle_swiglu_forward(T, h, fs, X, W1i, b1i, W2i, NULL, NULL, NULL, Zi);
        for (int64_t e = 0; e < T * h; e++)
            Z[e] += Zi[e];
        oracle_swiglu_backward(T, h, fs, X, W1i, b1i, W2i, dZ, dXi, dW1i, NULL, dW2i, NULL);
        for (int64_t e = 0; e < T * h; e++)
            dX[e] += dXi[e];
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++) {
                dW1[k * f2 + g0 + j] = dW1i[k * fs2 + j];
                dW1[k * f2 + u0 + j] = dW1i[k * fs2 + fs + j];
            }
        memcpy(dW2 + g0 * h, dW2i, sizeof(double) * (size_t)(fs * h));
    }
    for (int64_t tt = 0; tt < T; tt++)
        for (int64_t n = 0; n < h; n++)
            Z[tt * h + n] += b2 ? b2[n] : 0.0;
    free(Zi);
    free(dXi);
    free(W1i);
    free(b1i);
    free(W2i);
    free(dW1i);
    free(dW2i);
}

/* ------------------------------------------------------------------------ */
/* The two primitives of the 70B page ("The Mechanics of Tensor Parallelism
 * (TP) in Megatron-LM"): ColumnParallelLinear and RowParallelLinear. Both
 * compute the plain linear layer Y = X W + b, X [T, n_in], W [n_in, n_out],
 * b [n_out] (NULL: zero); they differ in which dimension of W the shards
 * split and so in where the shard sum falls. */
void oracle_linear_forward(int64_t T, int64_t n_in, int64_t n_out,
                           const double *X, const double *W, const double *b, double *Y)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; t++) {
        for (int64_t j = 0; j < n_out; j++)
            Y[t * n_out + j] = b ? b[j] : 0.0;
        for (int64_t k = 0; k < n_in; k++) {
            double x = X[t * n_in + k];
            for (int64_t j = 0; j < n_out; j++)
                Y[t * n_out + j] += x * W[k * n_out + j];
        }
    }
}

/* Backward of Y = X W + b for upstream dY: dX = dY W^T, dW = X^T dY,
 * db = sum_t dY. Any output may be NULL. */
void oracle_linear_backward(int64_t T, int64_t n_in, int64_t n_out,
                            const double *X, const double *W, const double *dY,
                            double *dX, double *dW, double *db)
{
    int64_t t, k, j;
    if (dX) {
#pragma omp parallel for schedule(static)
        for (t = 0; t < T; t++) {
            for (int64_t kk = 0; kk < n_in; kk++) {
                double acc = 0.0;
                for (int64_t jj = 0; jj < n_out; jj++)
                    acc += dY[t * n_out + jj] * W[kk * n_out + jj];
                dX[t * n_in + kk] = acc;
            }
        }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (k = 0; k < n_in; k++) {
            for (int64_t jj = 0; jj < n_out; jj++)
                dW[k * n_out + jj] = 0.0;
            for (int64_t tt = 0; tt < T; tt++) {
                double x = X[tt * n_in + k];
                for (int64_t jj = 0; jj < n_out; jj++)
                    dW[k * n_out + jj] += x * dY[tt * n_out + jj];
            }
        }
    }
    if (db) {
        for (j = 0; j < n_out; j++) {
            double acc = 0.0;
            for (t = 0; t < T; t++)
                acc += dY[t * n_out + j];
            db[j] = acc;
        }
    }
}

/* The same layer computed shard by shard. mode 0 (column-parallel, [MF]
 * "Column-Parallel Linear Layer"): W = [W_1 .. W_t] by columns, each shard
 * forms its own columns Y_i = X W_i + b_i with no exchange; in the backward
 * each shard's partial dX_i = dY_i W_i^T is summed (f*). mode 1
 * (row-parallel, "Row-Parallel Linear Layer"): W = [W_1; ..; W_t] by rows and
 * X by the matching columns, Z_i = X_i W_i, Y = sum_i Z_i (g), then b once;
 * in the backward every shard sees dY (g*) and forms its own columns of dX,
 * dX_i = dY W_i^T. dW_i = X_i^T dY_i in both. Requires the split dimension to
 * divide by t. */
void oracle_linear_sharded(int64_t T, int64_t n_in, int64_t n_out, int t, int mode,
                           const double *X, const double *W, const double *b, const double *dY,
                           double *Y, double *dX, double *dW)
{
    int64_t in_s = mode == 0 ? n_in : n_in / t;
    int64_t out_s = mode == 0 ? n_out / t : n_out;
    double *Xi = (double *)malloc(sizeof(double) * (size_t)(T * in_s));
    double *Wi = (double *)malloc(sizeof(double) * (size_t)(in_s * out_s));
    double *bi = (double *)malloc(sizeof(double) * (size_t)out_s);
    double *dYi = (double *)malloc(sizeof(double) * (size_t)(T * out_s));
    double *Yi = (double *)malloc(sizeof(double) * (size_t)(T * out_s));
    double *dXi = (double *)malloc(sizeof(double) * (size_t)(T * in_s));
    double *dWi = (double *)malloc(sizeof(double) * (size_t)(in_s * out_s));
    for (int64_t e = 0; e < T * n_out; e++)
        Y[e] = 0.0;
    for (int64_t e = 0; e < T * n_in; e++)
        dX[e] = 0.0;
    for (int i = 0; i < t; i++) {
        int64_t r0 = mode == 0 ? 0 : (int64_t)i * in_s;   /* first row of W_i, first column of X_i */
        int64_t c0 = mode == 0 ? (int64_t)i * out_s : 0;  /* first column of W_i */
        for (int64_t tt = 0; tt < T; tt++)
            for (int64_t k = 0; k < in_s; k++)
                Xi[tt * in_s + k] = X[tt * n_in + r0 + k];
        for (int64_t k = 0; k < in_s; k++)
            for (int64_t j = 0; j < out_s; j++)
                Wi[k * out_s + j] = W[(r0 + k) * n_out + c0 + j];
        for (int64_t j = 0; j < out_s; j++)
            bi[j] = (mode == 0 && b) ? b[c0 + j] : 0.0;  /* the row-parallel bias enters after the sum */
        for (int64_t tt = 0; tt < T; tt++)
            for (int64_t j = 0; j < out_s; j++)
                dYi[tt * out_s + j] = dY[tt * n_out + c0 + j];
        oracle_linear_forward(T, in_s, out_s, Xi, Wi, bi, Yi);
        oracle_linear_backward(T, in_s, out_s, Xi, Wi, dYi, dXi, dWi, NULL);
        for (int64_t tt = 0; tt < T; tt++) {
            for (int64_t j = 0; j < out_s; j++)
                Y[tt * n_out + c0 + j] += Yi[tt * out_s + j];     /* column: placement; row: g */
            for (int64_t k = 0; k < in_s; k++)
                dX[tt * n_in + r0 + k] += dXi[tt * in_s + k];     /* column: f*; row: placement */
        }
        for (int64_t k = 0; k < in_s; k++)
            for (int64_t j = 0; j < out_s; j++)
                dW[(r0 + k) * n_out + c0 + j] = dWi[k * out_s + j];
    }
    if (mode == 1 && b)
        for (int64_t tt = 0; tt < T; tt++)
            for (int64_t j = 0; j < n_out; j++)
                Y[tt * n_out + j] += b[j];
    free(Xi);
    free(Wi);
    free(bi);
    free(dYi);
    free(Yi);
    free(dXi);
    free(dWi);
}

/* Column of the fused QKV projection [70B] "The Multi-Head Attention Block"
 * holding element j (0 <= j < d) of head `head` of kind 0 (query), 1 (key) or
 * 2 (value), for n_q query heads sharing n_kv key/value heads of width d.
 * Columns are grouped by key/value head g: the n_q / n_kv query heads of
 * group g, then K_g, then V_g, each group (n_q / n_kv + 2) d wide. */
int64_t oracle_qkv_column(int kind, int64_t head, int64_t j, int64_t n_q, int64_t n_kv, int64_t d)
{
    int64_t qpg = n_q / n_kv;              /* query heads per group */
    int64_t gw = (qpg + 2) * d;            /* group width */
    if (kind == 0)
        return (head / qpg) * gw + (head % qpg) * d + j;
    return head * gw + (qpg + kind - 1) * d + j;
}

/* ------------------------------------------------------------------------ */
/* Sequence parallelism, [MF] "Sequence Parallelism": outside the tensor-
 * parallel region each of the t ranks holds one sequence chunk, rows
 * [r T/t, (r+1) T/t), of the activations. The block is entered by an
 * all-gather of the X chunks into the full sequence and left by a
 * reduce-scatter: rank r receives, for its own rows only, the sum over the
 * shards of the row-parallel partials Z_i (then bB). The backward mirrors
 * it: an all-gather of the dZ chunks, each shard's own backward over the
 * full sequence, and a reduce-scatter of the partial dX_i into dX chunks.
 * X_chunks, dZ_chunks, Z_chunks and dX_chunks are t arrays of [T/t, h];
 * dA [h, f], dB [f, h]. Requires T % t == 0 and f % t == 0. */
void oracle_mlp_seq_parallel(int64_t T, int64_t h, int64_t f, int t,
                             const double *const *X_chunks, const double *A, const double *bA,
                             const double *B, const double *bB, const double *const *dZ_chunks,
                             double *const *Z_chunks, double *const *dX_chunks, double *dA, double *dB)
{
    int64_t rows = T / t, fs = f / t;
    double *X = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *dZ = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *Zi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *dXi = (double *)malloc(sizeof(double) * (size_t)(T * h));
    double *Ai = (double *)malloc(sizeof(double) * (size_t)(h * fs));
    double *bAi = (double *)malloc(sizeof(double) * (size_t)fs);
    double *Bi = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    double *dAi = (double *)malloc(sizeof(double) * (size_t)(h * fs));
    double *dBi = (double *)malloc(sizeof(double) * (size_t)(fs * h));
    /* all-gather: chunk r fills rows [r rows, (r+1) rows) */
    for (int r = 0; r < t; r++) {
        memcpy(X + (int64_t)r * rows * h, X_chunks[r], sizeof(double) * (size_t)(rows * h));
        memcpy(dZ + (int64_t)r * rows * h, dZ_chunks[r], sizeof(double) * (size_t)(rows * h));
    }
    for (int r = 0; r < t; r++)
        for (int64_t e = 0; e < rows * h; e++) {
            Z_chunks[r][e] = 0.0;
            dX_chunks[r][e] = 0.0;
        }
    for (int i = 0; i < t; i++) {
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++)
                Ai[k * fs + j] = A[k * f + (int64_t)i * fs + j];
        for (int64_t j = 0; j < fs; j++)
            bAi[j] = bA ? bA[(int64_t)i * fs + j] : 0.0;
        memcpy(Bi, B + (int64_t)i * fs * h, sizeof(double) * (size_t)(fs * h));
        oracle_mlp_forward(T, h, fs, X, Ai, bAi, Bi, NULL, NULL, NULL, Zi);
        oracle_mlp_backward(T, h, fs, X, Ai, bAi, Bi, dZ, dXi, dAi, NULL, dBi, NULL);
        /* reduce-scatter: rank r adds shard i's partial for its own rows */
        for (int r = 0; r < t; r++)
            for (int64_t e = 0; e < rows * h; e++) {
                Z_chunks[r][e] += Zi[(int64_t)r * rows * h + e];
                dX_chunks[r][e] += dXi[(int64_t)r * rows * h + e];
            }
        for (int64_t k = 0; k < h; k++)
            for (int64_t j = 0; j < fs; j++)
                dA[k * f + (int64_t)i * fs + j] = dAi[k * fs + j];
        memcpy(dB + (int64_t)i * fs * h, dBi, sizeof(double) * (size_t)(fs * h));
    }
    for (int r = 0; r < t; r++)
        for (int64_t rr = 0; rr < rows; rr++)
            for (int64_t n = 0; n < h; n++)
                Z_chunks[r][rr * h + n] += bB ? bB[n] : 0.0;
    free(X);
    free(dZ);
    free(Zi);
    free(dXi);
    free(Ai);
    free(bAi);
    free(Bi);
    free(dAi);
    free(dBi);
}
