// Launch helpers of the non-GEMM kernels of the DyRA forward.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dyra {

// bf16 path, SPD solves (solve.cu)
// (G + ridge I)^-1 for r <= 64, and L~ = L (G + ridge I)^-1 written over the L columns
// [l0, l0 + r) of T [batch][n][ldT] (batch stride sTb elements); G^-1 also to Ginv (bf16).
cudaError_t launch_chol_apply(const float *G, int batch, int r, float ridge, __nv_bfloat16 *T,
                              int n, int ldT, int l0, long long sTb, __nv_bfloat16 *Ginv,
                              int *status, cudaStream_t s);
cudaError_t launch_ns_prep(const float *G, int batch, int r, float ridge, float *Gh, float *X0,
                           float *dinv, int *flags, cudaStream_t s);
cudaError_t launch_ns_finish(const float *X, const float *dinv, int batch, int r, const int *flags,
                             __nv_bfloat16 *Ginv, int *status, cudaStream_t s);

// fp32 path (f32_path.cu)
cudaError_t launch_sgemm(int batch, int M, int N, int K, const float *A, long long sAb,
                         long long sAi, long long sAk, const float *B, long long sBb, long long sBk,
                         long long sBj, float *C, long long sCb, long long sCi, long long sCj,
                         bool accumulate, const float *bias, cudaStream_t s);
cudaError_t launch_gram_f64(const float *T, int batch, int n, int ldT, int l0, int r,
                            long long sTb, double *G, cudaStream_t s);
cudaError_t launch_inverse_f64(const double *G, int batch, int r, double ridge, bool ns,
                               int ns_iters, double *Ginv, int *status, cudaStream_t s);
cudaError_t launch_apply_inverse(const double *Ginv, const float *B, int batch, int r, int m,
                                 float *R, cudaStream_t s);

}  // namespace dyra
