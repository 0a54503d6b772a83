/*
 * cm_oracle.c -- fp64 CPU oracle for the decomposed collective matmul.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * It computes the plain definitions that the decomposition reaches exactly
 * ("Overlap Communication with Dependent Computation via Decomposition in
 * Large Deep Learning Models", section "Why it works": gathering and summing
 * are linear maps, so the decomposed loop reaches the monolithic result
 * exactly):
 *
 *   AllGather -> GEMM:   Y_r = concat_j(X_j) @ W_r            for every rank r
 *                        (section "The idea", AllGather -> Einsum paragraph;
 *                         "Hiding Tensor-Parallel Collectives", section 2)
 *   GEMM -> ReduceScatter: Y_o = (sum_r X_r @ W_r)[rows of bucket o]
 *                        (section "The idea", Einsum -> ReduceScatter
 *                         paragraph; "Hiding Tensor-Parallel Collectives",
 *                         section 4: rank i's output shard adds up what
 *                         every rank contributed to those rows)
 *
 * Arithmetic: bf16 inputs are decoded bit-exactly to double; every output
 * element is a sequential sum over the contraction index k = 0..K-1 in
 * double; the ReduceScatter sum runs over r = 0..N-1 in that order.  There is
 * no blocking or reordering.  OpenMP parallelises over output rows only,
 * which does not change any element's arithmetic.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact bf16 -> double: a bf16 value is the top half of an IEEE float. */
static inline double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Weight element W[k][j] of a [K][n] operand stored either row-major [K][n]
 * (layout 0, "kn") or transposed [n][K] (layout 1, "nk"). */
static inline double w_at(const uint16_t *w, int layout, int64_t K, int64_t n,
                          int64_t k, int64_t j) {
    return layout == 0 ? bf16_to_f64(w[k * n + j]) : bf16_to_f64(w[j * K + k]);
}

/* One output row of a plain GEMM: out[j] = sum_k a[k] * W[k][j], k ascending.
 * Both loop orders below add the same products in the same order (starting
 * from 0.0, k = 0, 1, ..., K-1) for every j; only the memory walk differs. */
static void row_times_w(const uint16_t *a, const uint16_t *w, int layout,
                        int64_t K, int64_t n, double *out) {
    if (layout == 0) {                 /* W rows contiguous: sweep k outside */
        for (int64_t j = 0; j < n; ++j) out[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double ak = bf16_to_f64(a[k]);
            for (int64_t j = 0; j < n; ++j) out[j] += ak * w_at(w, layout, K, n, k, j);
        }
    } else {                           /* W columns contiguous: dot products */
        for (int64_t j = 0; j < n; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += bf16_to_f64(a[k]) * w_at(w, layout, K, n, k, j);
            out[j] = s;
        }
    }
}

/* Plain GEMM C[M][n] = A[M][K] @ W[K][n] in fp64 (A row-major bf16 bits). */
void cm_oracle_gemm(int64_t M, int64_t K, int64_t n, const uint16_t *a,
                    const uint16_t *w, int w_layout, double *c) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        row_times_w(a + i * K, w, w_layout, K, n, c + i * n);
}

/*
 * AllGather -> GEMM, sampled rows.
 * x: [N][m][K] (shard j = rows j*m..j*m+m-1 of the gathered X), w: N weight
 * shards each [K][n] (layout 0) or [n][K] (layout 1).
 * For t < count: out[t][:] = Y_{ranks[t]}[rows[t], :] where rows[t] indexes
 * the gathered X (0 <= rows[t] < N*m).
 */
void cm_oracle_ag_gemm_rows(int N, int64_t m, int64_t K, int64_t n,
                            const uint16_t *x, const uint16_t *w, int w_layout,
                            int64_t count, const int32_t *ranks,
                            const int64_t *rows, double *out) {
    (void)N;
    (void)m;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t *xrow = x + rows[t] * K;          /* concat_j X_j, row rows[t] */
        const uint16_t *wr = w + (int64_t)ranks[t] * K * n;
        row_times_w(xrow, wr, w_layout, K, n, out + t * n);
    }
}

/* AllGather -> GEMM, every output: y [N][N*m][n]. */
void cm_oracle_ag_gemm(int N, int64_t m, int64_t K, int64_t n,
                       const uint16_t *x, const uint16_t *w, int w_layout,
                       double *y) {
    const int64_t rows_per_rank = (int64_t)N * m;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < N; ++r)
        for (int64_t i = 0; i < rows_per_rank; ++i)
            row_times_w(x + i * K, w + (int64_t)r * K * n, w_layout, K, n,
                        y + ((int64_t)r * rows_per_rank + i) * n);
}

/*
 * GEMM -> ReduceScatter, sampled rows.
 * x: [N][M][k] (X_r), w: N shards each [k][n] (layout 0) or [n][k] (layout 1).
 * Bucket o owns rows o*(M/N) .. o*(M/N)+M/N-1 of the reduced output.
 * out[t][:] = sum_{r=0..N-1} X_r[owners[t]*(M/N) + rows[t], :] @ W_r.
 */
void cm_oracle_gemm_rs_rows(int N, int64_t M, int64_t k, int64_t n,
                            const uint16_t *x, const uint16_t *w, int w_layout,
                            int64_t count, const int32_t *owners,
                            const int64_t *rows, double *out) {
    const int64_t Mb = M / N;
#pragma omp parallel
    {
        double *tmp = (double *)malloc((size_t)n * sizeof(double)); /* one partial row */
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < count; ++t) {
            const int64_t grow = (int64_t)owners[t] * Mb + rows[t];
            double *o = out + t * n;
            for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
            for (int r = 0; r < N; ++r) {
                row_times_w(x + ((int64_t)r * M + grow) * k,
                            w + (int64_t)r * k * n, w_layout, k, n, tmp);
                for (int64_t j = 0; j < n; ++j) o[j] += tmp[j];
            }
        }
        free(tmp);
    }
}

/* GEMM -> ReduceScatter, every output: y [N][M/N][n]. */
void cm_oracle_gemm_rs(int N, int64_t M, int64_t k, int64_t n,
                       const uint16_t *x, const uint16_t *w, int w_layout,
                       double *y) {
    /* Bucket o is rows o*(M/N).. of the reduced sum, so y [N][M/N][n] is the
     * reduced sum [M][n] in row order: global row g lands at y + g*n. */
#pragma omp parallel
    {
        double *tmp = (double *)malloc((size_t)n * sizeof(double)); /* one partial row */
#pragma omp for schedule(dynamic, 1)
        for (int64_t g = 0; g < M; ++g) {
            double *o = y + g * n;
            for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
            for (int r = 0; r < N; ++r) {
                row_times_w(x + ((int64_t)r * M + g) * k, w + (int64_t)r * k * n,
                            w_layout, k, n, tmp);
                for (int64_t j = 0; j < n; ++j) o[j] += tmp[j];
            }
        }
        free(tmp);
    }
    (void)N;
}

/*
 * Weight gradient of the column-parallel layer whose forward is the
 * AllGather -> GEMM above.  "Tensor Parallelism > Communication Patterns":
 * the gradient of a column-parallel weight shard is computed locally from the
 * full input; "Hiding Tensor-Parallel Collectives", section 7: that full input
 * is an AllGather the data-gradient GEMM does not need (bulk overlap).  With
 * W_r stored [n][K] (Y_r[t][i] = sum_k X_all[t][k] * W_r[i][k]):
 *
 *   dW_r[i][k] = sum over tokens t = 0 .. N*m-1 of dY_r[t][i] * X_all[t][k],
 *   X_all = concat_j(X_j), t ascending.
 *
 * x: [N][m][K], dy: [N][N*m][n], rows (r, i) sampled by `ranks`/`rows`;
 * out: [count][K].
 */
void cm_oracle_wgrad_rows(int N, int64_t m, int64_t K, int64_t n,
                          const uint16_t *x, const uint16_t *dy, int64_t count,
                          const int32_t *ranks, const int64_t *rows, double *out) {
    const int64_t T = (int64_t)N * m;            /* tokens: concat_j(X_j) rows */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < count; ++s) {
        const int r = ranks[s];
        const int64_t i = rows[s];
        double *o = out + s * K;
        for (int64_t k = 0; k < K; ++k) o[k] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double d = bf16_to_f64(dy[((int64_t)r * T + t) * n + i]);
            const uint16_t *xt = x + t * K;      /* row t of X_all (shards are contiguous) */
            for (int64_t k = 0; k < K; ++k) o[k] += d * bf16_to_f64(xt[k]);
        }
    }
}

/* Every row of every rank's weight gradient: out [N][n][K]. */
void cm_oracle_wgrad(int N, int64_t m, int64_t K, int64_t n,
                     const uint16_t *x, const uint16_t *dy, double *out) {
    const int64_t count = (int64_t)N * n;
    int32_t *ranks = (int32_t *)malloc((size_t)count * sizeof(int32_t));
    int64_t *rows = (int64_t *)malloc((size_t)count * sizeof(int64_t));
    for (int64_t s = 0; s < count; ++s) {
        ranks[s] = (int32_t)(s / n);
        rows[s] = s % n;
    }
    cm_oracle_wgrad_rows(N, m, K, n, x, dy, count, ranks, rows, out);
    free(ranks);
    free(rows);
}

/* Threads OpenMP will use (reported next to the CPU timings). */
int cm_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
