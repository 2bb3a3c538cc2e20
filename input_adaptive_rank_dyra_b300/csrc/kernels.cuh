// Launch helpers of the non-GEMM kernels of the DyRA forward.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dyra {

// bf16 path, SPD solves (solve.cu)
// C~ = (G + ridge I)^-1 C for r <= 64 (r % 4 == 0): G [batch][r][r] fp32, C given as
// C^T [batch][d][r] fp32, C~ to Cs [batch][r][d] bf16; G^-1 also to Ginv [batch][r][r] bf16.
cudaError_t launch_spd_solve(const float *G, int batch, int r, float ridge, const float *Ct,
                             int d, __nv_bfloat16 *Cs, __nv_bfloat16 *Ginv, int *status,
                             cudaStream_t s);
// Newton-Schulz start: dinv = diag(G + ridge I)^-1/2, Gh = D (G + ridge I) D,
// X0 = I / ||Gh||_inf; flags[b] marks a sample whose diagonal is not positive and finite.
cudaError_t launch_ns_prep(const float *G, int batch, int r, float ridge, float *Gh, float *X0,
                           float *dinv, int *flags, cudaStream_t s);
// G^-1 from the Newton-Schulz iterate: to Ginv (bf16) and G32 (fp32), both [batch][r][r].
cudaError_t launch_ns_finish(const float *X, const float *dinv, int batch, int r, const int *flags,
                             __nv_bfloat16 *Ginv, float *G32, int *status, cudaStream_t s);

// failure-path self-test (probe.cu): one CTA whose bounded mbarrier wait, limited to
// limit_ns, runs out on a barrier nothing arrives on; counted in status[1]
cudaError_t launch_bounded_wait_probe(int *status, unsigned long long limit_ns, cudaStream_t s);

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
