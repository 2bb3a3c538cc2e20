// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward needs (G + lambda I)^-1 explicitly (bf16), which a tensor-core GEMM then
// applies to L (L G^-1). These kernels produce it from G = L^T L (fp32):
//   * r <= 64: Cholesky G = Lc Lc^T, W = Lc^-1, G^-1 = W^T W, all in fp32, one CTA of 256
//     threads per sample. The r x r matrix is padded to 64 x 64 with the identity; each
//     thread keeps 16 entries (row tid/4, columns tid%4 + 4k) in registers, and every
//     elimination step publishes one column (or row) through shared memory behind a single
//     barrier, so a step costs one barrier and 16 register FMAs.
//   * larger r: Newton-Schulz. ns_prep scales G symmetrically to unit diagonal and sets
//     X0 = I / ||G_hat||_inf; the iterations X <- X (2I - G_hat X) run as tf32 tensor-core
//     GEMMs (tc_gemm); ns_finish undoes the scaling.
// A sample whose pivot is not positive (or not finite) is counted in status[0] and gets
// G^-1 = 0, so its correction vanishes and its output is the static branch plus bias.
#include "kernels.cuh"

#include <cuda_bf16.h>

namespace dyra {

namespace {

constexpr int kCholMax = 64;

__global__ void __launch_bounds__(256)
    chol_inverse_kernel(const float *__restrict__ G, int r, float ridge,
                        __nv_bfloat16 *__restrict__ Ginv, int *status) {
  __shared__ float Lm[kCholMax][kCholMax + 1];   // Cholesky factor, later W = Lc^-1
  __shared__ float cbuf[2][kCholMax];            // column j of the trailing matrix
  __shared__ float rbuf[2][kCholMax];            // row j of W
  __shared__ int bad;
  const int tid = threadIdx.x, b = blockIdx.x;
  const int i = tid >> 2, p = tid & 3;           // row i, columns p + 4k
  const float *g = G + (size_t)b * r * r;
  float a[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int c = p + 4 * k;
    a[k] = (i < r && c < r) ? g[i * r + c] + (i == c ? ridge : 0.f) : (i == c ? 1.f : 0.f);
    Lm[i][c] = (i == c && i >= r) ? 1.f : 0.f;
  }
  if (tid == 0) bad = 0;
  if (p == 0) cbuf[0][i] = a[0];
  __syncthreads();
  bool mybad = false;
  // ---- Cholesky, right-looking on the unscaled trailing matrix (pivot d_j = A_jj)
  for (int j = 0; j < r; ++j) {
    const float *cb = cbuf[j & 1];
    float d = cb[j];
    if (!(d > 0.f) || !isfinite(d)) {
      mybad = true;
      d = 1.f;
    }
    const float li = cb[i];
    if (p == 0 && i >= j) Lm[i][j] = li * rsqrtf(d);
    if (i > j) {
      const float s = li / d;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (p + 4 * k > j) a[k] -= s * cb[p + 4 * k];
    }
    const int jn = j + 1;
    if (jn < r && p == (jn & 3)) {
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k == (jn >> 2)) v = a[k];
      cbuf[jn & 1][i] = v;
    }
    __syncthreads();
  }
  // ---- W = Lc^-1 by right-looking forward substitution on the identity
  float w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = (i == p + 4 * k) ? 1.f : 0.f;
  for (int j = 0; j < r; ++j) {
    if (i == j) {
      const float inv = 1.f / Lm[j][j];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        w[k] *= inv;
        rbuf[j & 1][p + 4 * k] = w[k];
      }
    }
    __syncthreads();
    if (i > j) {
      const float lij = Lm[i][j];
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] -= lij * rbuf[j & 1][p + 4 * k];
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 16; ++k) Lm[i][p + 4 * k] = w[k];
  if (mybad) atomicOr(&bad, 1);
  __syncthreads();
  // ---- G^-1 = W^T W (W lower triangular: rows t >= i contribute)
  if (i < r) {
    float s[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) s[k] = 0.f;
    for (int t = i; t < r; ++t) {
      const float wa = Lm[t][i];
#pragma unroll
      for (int k = 0; k < 16; ++k) s[k] += wa * Lm[t][p + 4 * k];
    }
    __nv_bfloat16 *out = Ginv + (size_t)b * r * r + (size_t)i * r;
    const bool zero = bad != 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int c = p + 4 * k;
      if (c < r) out[c] = __float2bfloat16_rn((zero || !isfinite(s[k])) ? 0.f : s[k]);
    }
  }
  if (tid == 0 && bad) atomicAdd(status, 1);
}

// Jacobi scaling and start of Newton-Schulz: dinv = diag(G + lambda I)^-1/2,
// G_hat = D (G + lambda I) D, X0 = I / max_i sum_j |G_hat_ij|.
__global__ void __launch_bounds__(256)
    ns_prep_kernel(const float *__restrict__ G, int r, float ridge, float *__restrict__ Gh,
                   float *__restrict__ X0, float *__restrict__ dinv, int *__restrict__ flags) {
  __shared__ float sd[256];
  __shared__ float red[256];
  __shared__ int bad;
  const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const float *g = G + (size_t)b * r * r;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int i = tid; i < r; i += nt) {
    const float gii = g[(size_t)i * r + i] + ridge;
    float v = 0.f;
    if (gii > 0.f && isfinite(gii)) v = rsqrtf(gii);
    else bad = 1;
    sd[i] = v;
  }
  __syncthreads();
  float mx = 0.f;
  for (int i = tid; i < r; i += nt) {
    float rs = 0.f;
    for (int j = 0; j < r; ++j) {
      float v = (g[(size_t)i * r + j] + (i == j ? ridge : 0.f)) * sd[i] * sd[j];
      if (bad) v = 0.f;
      Gh[(size_t)b * r * r + (size_t)i * r + j] = v;
      rs += fabsf(v);
    }
    mx = fmaxf(mx, rs);
  }
  red[tid] = mx;
  __syncthreads();
  for (int s = nt / 2; s > 0; s >>= 1) {
    if (tid < s) red[tid] = fmaxf(red[tid], red[tid + s]);
    __syncthreads();
  }
  const float alpha = (bad || !(red[0] > 0.f)) ? 0.f : 1.f / red[0];
  for (int t = tid; t < r * r; t += nt) {
    const int i = t / r, j = t % r;
    X0[(size_t)b * r * r + t] = (i == j) ? alpha : 0.f;
  }
  for (int i = tid; i < r; i += nt) dinv[(size_t)b * r + i] = bad ? 0.f : sd[i];
  if (tid == 0) flags[b] = bad;
}

__global__ void __launch_bounds__(256)
    ns_finish_kernel(const float *__restrict__ X, const float *__restrict__ dinv, int r,
                     const int *__restrict__ flags, __nv_bfloat16 *__restrict__ Ginv, int *status) {
  __shared__ int bad;
  const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) bad = flags[b];
  __syncthreads();
  for (int t = tid; t < r * r; t += nt) {
    const float v = X[(size_t)b * r * r + t];
    if (!isfinite(v)) bad = 1;
  }
  __syncthreads();
  const float *dv = dinv + (size_t)b * r;
  for (int t = tid; t < r * r; t += nt) {
    const int i = t / r, j = t % r;
    const float v = bad ? 0.f : X[(size_t)b * r * r + t] * dv[i] * dv[j];
    Ginv[(size_t)b * r * r + t] = __float2bfloat16_rn(v);
  }
  if (tid == 0 && bad) atomicAdd(status, 1);
}

}  // namespace

cudaError_t launch_chol_inverse(const float *G, int batch, int r, float ridge, __nv_bfloat16 *Ginv,
                                int *status, cudaStream_t s) {
  if (r > kCholMax) return cudaErrorInvalidValue;
  chol_inverse_kernel<<<batch, 256, 0, s>>>(G, r, ridge, Ginv, status);
  return cudaGetLastError();
}

cudaError_t launch_ns_prep(const float *G, int batch, int r, float ridge, float *Gh, float *X0,
                           float *dinv, int *flags, cudaStream_t s) {
  if (r > 256) return cudaErrorInvalidValue;
  ns_prep_kernel<<<batch, 256, 0, s>>>(G, r, ridge, Gh, X0, dinv, flags);
  return cudaGetLastError();
}

cudaError_t launch_ns_finish(const float *X, const float *dinv, int batch, int r, const int *flags,
                             __nv_bfloat16 *Ginv, int *status, cudaStream_t s) {
  ns_finish_kernel<<<batch, 256, 0, s>>>(X, dinv, r, flags, Ginv, status);
  return cudaGetLastError();
}

}  // namespace dyra
