// Launch helpers of the non-GEMM kernels of the DyRA forward.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dyra {

// bf16 path, SPD solves (solve.cu)
// (G + ridge I)^-1 for r <= 64 (r % 4 == 0), one CTA per sample: G [batch][r][r] fp32 to
// Ginv32 (fp32) and Ginv (bf16), both [batch][r][r]; a sample that is not positive definite
// gets 0 and is counted in status[0].
cudaError_t launch_spd_invert(const float *G, int batch, int r, float ridge, float *Ginv32,
                              __nv_bfloat16 *Ginv, int *status, cudaStream_t s);
// C~ = G^-1 C for r <= 64: G^-1 from Ginv32, C given as C^T [batch][d][r] fp32, C~ to
// Cs [batch][r][d] bf16.
cudaError_t launch_spd_apply(const float *Ginv32, int batch, int r, const float *Ct, int d,
                             __nv_bfloat16 *Cs, cudaStream_t s);
// Newton-Schulz inverse of (G + ridge I) in one kernel (ns.cu), r <= 256, r % 8 == 0: the
// start (D = diag(G + ridge I)^-1/2, G_hat = D (G + ridge I) D, alpha = 1 / ||G_hat||_inf,
// E0 = I - alpha G_hat, X0 = alpha I, written to ex0), iters steps of X' = X + X E, E' = E E
// with the iterates in ex0 / ex1 ([batch][2r][r] fp32, [E ; X]), then G^-1 = D X D to G32
// (fp32) and Ginv (bf16). maps[i][0..1]: fp32 tensor maps of the E and X blocks of buffer i
// ([batch][r][r], row stride r, batch stride 2 r r, box {32, 128}). A sample whose diagonal
// is not positive and finite, or whose result is not finite, gets G^-1 = 0 and is counted in
// status[0]; bounded waits that gave up are counted in status[1].
cudaError_t launch_ns_fused(const CUtensorMap (&maps)[2][2], int batch, int r, int iters,
                            float ridge, const float *G, float *ex0, float *ex1, float *G32,
                            __nv_bfloat16 *Ginv, int *status, cudaStream_t s);

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
