// Host float64 linear algebra for the offline preparation of a DyRA layer
// (static fit, residual, R0, projection P). Own code: no LAPACK, no CUDA.
#pragma once
#include <cstddef>
#include <vector>

namespace dyra {
namespace fit {

// Run fn(i) for i in [0, n) on up to `threads` host threads (0 = hardware concurrency).
void parallel_for(int n, int threads, const void *ctx, void (*fn)(const void *ctx, int i));

// C[rows x cols] = A[rows x inner] * B[inner x cols] (row-major, optional transposes).
// transA: A is stored [inner x rows]; transB: B is stored [cols x inner].
void gemm(int rows, int cols, int inner, const double *A, bool transA, const double *B,
          bool transB, double *C, int threads);

// Eigen-decomposition of a symmetric n x n matrix (row-major, only read).
// evals: n values in descending order; evecs: n x n, row j = unit eigenvector of evals[j].
// Householder tridiagonalisation followed by implicit QL with Wilkinson shifts.
// Returns false if the QL iteration does not converge.
bool sym_eig(int n, const double *A, double *evals, double *evecs, int threads);

// Leading `count` singular triplets of W [d x m] (count <= min(d, m)), through the
// eigen-decomposition of the smaller Gram matrix. U [d x count] (columns = left vectors),
// S [count], Vt [count x m] (rows = right vectors).
bool top_svd(int d, int m, const double *W, int count, double *U, double *S, double *Vt,
             int threads);

// Cholesky of an SPD r x r matrix in place (lower triangle); false if not positive definite.
bool cholesky(int r, double *A);
// Solve (L L^T) X = B for X, B [r x ncols] row-major, in place.
void cholesky_solve(int r, const double *L, double *B, int ncols);
// Solve L^T X = B for X (L lower triangular from cholesky), B [r x ncols] row-major, in place.
void lower_transpose_solve(int r, const double *L, double *B, int ncols);

}  // namespace fit
}  // namespace dyra
