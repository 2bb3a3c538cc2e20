// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward never forms R: since L R = (L G^-1) B with B = (L^T X) W_res, it rewrites
// the L columns of T as L~ = L G^-1 and lets the output GEMM multiply L~ by B. These kernels
// produce G^-1 from G = L^T L (fp32) and, for small r, apply it:
//   * r <= 64 (the Cholesky branch): chol_apply. Every CTA takes one sample and a block of
//     128 of its token rows. It inverts G + lambda I in place by Gauss-Jordan elimination
//     without pivoting -- for an SPD matrix the pivots are the successive Schur complements,
//     i.e. the squared diagonal of its Cholesky factor, so this is the Cholesky solve
//     organised as one elimination step per column -- with the r x r matrix padded to R x R
//     by the identity and held in registers (256 threads, R*R/256 entries each), one barrier
//     per step. It then multiplies its rows of L by the inverse (fp32 FMA) and writes L~
//     over them in T. CTAs of the first row block also store G^-1 (bf16).
//   * larger r: Newton-Schulz. ns_prep scales G symmetrically to unit diagonal and sets
//     X0 = I / ||G_hat||_inf; the iterations X <- X (2I - G_hat X) run as tf32 tensor-core
//     GEMMs (tc_gemm); ns_finish undoes the scaling; a bf16 tensor-core GEMM applies the
//     result to L.
// A sample with a pivot that is not positive (or not finite) is counted in status[0] and
// gets G^-1 = 0, so its correction vanishes and its output is the static branch plus bias.
#include "kernels.cuh"

#include <cuda_bf16.h>

namespace dyra {

namespace {

constexpr int kApplyRows = 128;   // token rows per chol_apply CTA

template <int R>
__global__ void __launch_bounds__(256)
    chol_apply_kernel(const float *__restrict__ G, int r, float ridge, __nv_bfloat16 *T, int n,
                      int ldT, int l0, long long sTb, __nv_bfloat16 *__restrict__ Ginv,
                      int *status) {
  constexpr int TPR = 256 / R;   // threads per matrix row
  constexpr int E = R / TPR;     // entries per thread: row i, columns p + TPR * e
  __shared__ float rowk[2][R];   // row k of the matrix before step k
  __shared__ float colk[2][R];   // column k of the matrix before step k
  __shared__ __align__(16) float Gi[R][R];
  const int tid = threadIdx.x, b = blockIdx.y;
  const int i = tid / TPR, p = tid % TPR;
  const float *g = G + (size_t)b * r * r;
  float a[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int c = p + TPR * e;
    a[e] = (i < r && c < r) ? g[i * r + c] + (i == c ? ridge : 0.f) : (i == c ? 1.f : 0.f);
  }
  if (i == 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) rowk[0][p + TPR * e] = a[e];
  }
  if (p == 0) colk[0][i] = a[0];
  __syncthreads();
  // Branch-free elimination step: every thread computes the pivot-row and the other-row
  // update and selects, so no warp diverges between the barriers.
  bool bad = false;
  for (int k = 0; k < r; ++k) {
    const int kb = k & 1;
    const float piv = rowk[kb][k];
    if (!(piv > 0.f) || !isfinite(piv)) bad = true;   // same decision in every thread
    const float inv = bad ? 0.f : __frcp_rn(piv);
    const bool prow = (i == k);
    const float f = prow ? 0.f : colk[kb][i] * inv;
    float rc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) rc[e] = rowk[kb][p + TPR * e];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool pcol = (p + TPR * e == k);
      const float v = prow ? a[e] * inv : fmaf(-f, rc[e], a[e]);
      a[e] = pcol ? (prow ? inv : -f) : v;
    }
    const int kn = k + 1;
    if (i == kn) {
#pragma unroll
      for (int e = 0; e < E; ++e) rowk[kn & 1][p + TPR * e] = a[e];
    }
    float v = a[0];
#pragma unroll
    for (int e = 1; e < E; ++e) v = (e == kn / TPR) ? a[e] : v;
    if (p == kn % TPR) colk[kn & 1][i] = v;
    __syncthreads();
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int c = p + TPR * e;
    const float v = (bad || !isfinite(a[e])) ? 0.f : a[e];
    Gi[i][c] = (i < r && c < r) ? v : 0.f;
  }
  if (blockIdx.x == 0 && i < r) {
    __nv_bfloat16 *out = Ginv + (size_t)b * r * r + (size_t)i * r;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = p + TPR * e;
      if (c < r) out[c] = __float2bfloat16_rn(bad ? 0.f : a[e]);
    }
  }
  if (blockIdx.x == 0 && tid == 0 && bad) atomicAdd(status, 1);
  __syncthreads();
  // L~ = L G^-1 for this CTA's rows: two threads per row, each producing R/2 columns
  const int row = blockIdx.x * kApplyRows + (tid >> 1);
  const int half = tid & 1;
  const bool active = row < n;   // the same for both threads of a pair
  __nv_bfloat16 *Lrow = T + (size_t)b * sTb + (size_t)(active ? row : 0) * ldT + l0;
  constexpr int H = R / 2;
  float acc[H];
#pragma unroll
  for (int c = 0; c < H; ++c) acc[c] = 0.f;
  if (active) {
    float x[R];
#pragma unroll
    for (int k = 0; k < R; k += 8) {
      if (k < r) {
        const uint4 w = *reinterpret_cast<const uint4 *>(Lrow + k);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f2 = __bfloat1622float2(h[j]);
          x[k + 2 * j] = f2.x;
          x[k + 2 * j + 1] = f2.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[k + j] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const float4 *gk = reinterpret_cast<const float4 *>(&Gi[k][half * H]);
#pragma unroll
      for (int c4 = 0; c4 < H / 4; ++c4) {
        const float4 gg = gk[c4];
        acc[4 * c4 + 0] = fmaf(x[k], gg.x, acc[4 * c4 + 0]);
        acc[4 * c4 + 1] = fmaf(x[k], gg.y, acc[4 * c4 + 1]);
        acc[4 * c4 + 2] = fmaf(x[k], gg.z, acc[4 * c4 + 2]);
        acc[4 * c4 + 3] = fmaf(x[k], gg.w, acc[4 * c4 + 3]);
      }
    }
  }
  // both threads of a pair (adjacent lanes) have read the whole row of L before either
  // overwrites its half of it
  __syncwarp();
  if (active) {
#pragma unroll
    for (int c = 0; c < H; c += 8) {
      const int col = half * H + c;
      if (col < r) {
        uint4 w;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          h[j] = __floats2bfloat162_rn(acc[c + 2 * j], acc[c + 2 * j + 1]);
        *reinterpret_cast<uint4 *>(Lrow + col) = w;
      }
    }
  }
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

cudaError_t launch_chol_apply(const float *G, int batch, int r, float ridge, __nv_bfloat16 *T,
                              int n, int ldT, int l0, long long sTb, __nv_bfloat16 *Ginv,
                              int *status, cudaStream_t s) {
  if (r > 64 || r % 8 || l0 % 8 || ldT % 8) return cudaErrorInvalidValue;
  if (batch <= 0 || n <= 0) return cudaSuccess;
  dim3 grid((n + kApplyRows - 1) / kApplyRows, batch);
  if (r <= 32)
    chol_apply_kernel<32><<<grid, 256, 0, s>>>(G, r, ridge, T, n, ldT, l0, sTb, Ginv, status);
  else
    chol_apply_kernel<64><<<grid, 256, 0, s>>>(G, r, ridge, T, n, ldT, l0, sTb, Ginv, status);
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
