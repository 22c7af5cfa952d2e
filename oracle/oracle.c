/*
 * oracle.c -- fp64 reference loops for the sharded-GEMM oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header or constant with the CUDA path.
 *
 * Every routine is the plain definition of a matrix product written as a
 * naive loop nest in double precision, with the contraction index running in
 * ascending order and no blocking, no reordering and no fused multiply-add
 * (the build passes -ffp-contract=off).  OpenMP only splits the independent
 * output rows across threads, which does not change any result.
 *
 * Definitions followed:
 *  - "MLX tensor parallelism guide", section 2.1 / 2.2: a linear layer with
 *    weight of shape (output_dims, input_dims) computes y = x @ W.T + b.
 *  - "ColossalAI 2D tensor parallel via SUMMA", SUMMA section: the linear
 *    layer Y = X A, with A laid out (K, N).
 */
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[j][k]   (y = x @ W.T) */
void orc_gemm_nt(int64_t M, int64_t N, int64_t K,
                 const double *A, int64_t lda,
                 const double *B, int64_t ldb,
                 double *C, int64_t ldc)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += A[i * lda + k] * B[j * ldb + k];
            C[i * ldc + j] = acc;
        }
    }
}

/* C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]   (Y = X A) */
void orc_gemm_nn(int64_t M, int64_t N, int64_t K,
                 const double *A, int64_t lda,
                 const double *B, int64_t ldb,
                 double *C, int64_t ldc)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += A[i * lda + k] * B[k * ldb + j];
            C[i * ldc + j] = acc;
        }
    }
}

/* Number of threads the loops above run on. */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
