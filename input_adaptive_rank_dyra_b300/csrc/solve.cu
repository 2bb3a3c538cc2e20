// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward never forms R: since L R = (L G^-1) B with B = (L^T X) W_res, it rewrites
// the L columns of T as L~ = L G^-1 and lets the output GEMM multiply L~ by B. These kernels
// produce G^-1 from G = L^T L (fp32) and, for small r, apply it:
//   * r <= 64 (the Cholesky branch): chol_apply. Every CTA takes one sample and a block of
//     128 of its token rows. It inverts G + lambda I in place by block Gauss-Jordan
//     elimination without pivoting, on 8 x 8 pivot blocks -- for an SPD matrix the pivot
//     blocks are SPD Schur complements, whose scalar pivots are the squared diagonal of the
//     Cholesky factor, so this is the Cholesky solve organised as r / 8 block steps -- with
//     the r x r matrix padded to R x R (R = 32 or 64) by the identity and double-buffered in
//     shared memory. It then multiplies its rows of L (staged in shared memory) by the
//     inverse (fp32 FMA) and writes L~ over them in T. CTAs of the first row block also
//     store G^-1 (bf16).
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

constexpr int kPivot = 8;       // pivot block of the block elimination

// threads of chol_apply: four matrix entries per thread
template <int R>
__host__ __device__ constexpr int apply_threads() { return R * R / 4; }

// In-place block Gauss-Jordan on the SPD matrix A = G + ridge I padded to R x R by the
// identity, in shared memory. For each pivot block K (kPivot columns starting at K0):
//   P = A[K][K]^-1 (8 x 8, SPD), RK = P A[K][:], CK = A[:][K] (before the step),
//   A[i][c] <- A[i][c] - CK[i][:] RK[:, c]   (i, c outside K),
//   A[i][K] <- -CK[i][:] P,  A[K][c] <- RK[:, c],  A[K][K] <- P.
// After R / kPivot steps A holds A^-1. Warp 0 forms P (two entries per lane, exchanged by
// shuffles) while the other threads copy CK; then every thread forms one entry of RK; then
// every thread rewrites its own entries of A. Three barriers per step.
template <int R>
__global__ void __launch_bounds__(apply_threads<R>())
    chol_apply_kernel(const float *__restrict__ G, int r, float ridge, __nv_bfloat16 *T, int n,
                      int ldT, int l0, long long sTb, __nv_bfloat16 *__restrict__ Ginv,
                      int *status) {
  constexpr int NT = apply_threads<R>();
  constexpr int E = R * R / NT;       // matrix entries per thread (4)
  __shared__ __align__(16) float A[R][R];
  __shared__ __align__(16) float RK[kPivot][R];
  __shared__ float CK[R][kPivot];
  __shared__ float Pm[kPivot][kPivot];
  __shared__ __align__(16) __nv_bfloat16 Ls[kApplyRows][R];   // this CTA's rows of L
  __shared__ int bad_s;
  const int tid = threadIdx.x, b = blockIdx.y, lane = tid & 31, warp = tid >> 5;
  const float *g = G + (size_t)b * r * r;
  // this CTA's rows of L, staged now (every read of L happens before any write below)
  const int row0 = blockIdx.x * kApplyRows;
  for (int t = tid; t < kApplyRows * (R / 8); t += NT) {
    const int rr = t / (R / 8), c8 = (t % (R / 8)) * 8;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + rr < n && c8 < r)
      w = *reinterpret_cast<const uint4 *>(T + (size_t)b * sTb + (size_t)(row0 + rr) * ldT + l0 + c8);
    *reinterpret_cast<uint4 *>(&Ls[rr][c8]) = w;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int idx = tid + NT * e, i = idx / R, c = idx % R;
    A[i][c] = (i < r && c < r) ? g[i * r + c] + (i == c ? ridge : 0.f) : (i == c ? 1.f : 0.f);
  }
  if (tid == 0) bad_s = 0;
  __syncthreads();
  const int steps = (r + kPivot - 1) / kPivot;
  for (int kb = 0; kb < steps; ++kb) {
    const int K0 = kb * kPivot;
    if (warp == 0) {
      // P = A[K][K]^-1: lane holds (x0, y) and (x0 + 4, y), x0 = lane / 8, y = lane % 8
      const int x0 = lane >> 3, y = lane & 7;
      float q0 = A[K0 + x0][K0 + y], q1 = A[K0 + x0 + 4][K0 + y];
      bool bad = false;
#pragma unroll
      for (int k = 0; k < kPivot; ++k) {
        const int src = ((k & 3) << 3);   // lanes holding row k, slot k >> 2
        const float piv = __shfl_sync(0xffffffffu, (k >> 2) ? q1 : q0, src + k);
        const float ky = __shfl_sync(0xffffffffu, (k >> 2) ? q1 : q0, src + y);   // A[k][y]
        const float xk0 = __shfl_sync(0xffffffffu, q0, (x0 << 3) + k);           // A[x0][k]
        const float xk1 = __shfl_sync(0xffffffffu, q1, (x0 << 3) + k);           // A[x0+4][k]
        if (!(piv > 0.f) || !isfinite(piv)) bad = true;
        const float inv = bad ? 0.f : __frcp_rn(piv);
        const float f0 = xk0 * inv, f1 = xk1 * inv;
        const float u0 = (x0 == k) ? ((y == k) ? inv : q0 * inv) : ((y == k) ? -f0 : fmaf(-f0, ky, q0));
        const float u1 = (x0 + 4 == k) ? ((y == k) ? inv : q1 * inv) : ((y == k) ? -f1 : fmaf(-f1, ky, q1));
        q0 = u0;
        q1 = u1;
      }
      Pm[x0][y] = q0;
      Pm[x0 + 4][y] = q1;
      if (bad && lane == 0) bad_s = 1;
    }
    // CK = A[:][K] before the step, by the warps other than warp 0
    for (int t = tid - 32; t >= 0 && t < R * kPivot; t += NT - 32)
      CK[t / kPivot][t % kPivot] = A[t / kPivot][K0 + t % kPivot];
    __syncthreads();
    // RK = P A[K][:] (one entry per thread)
    if (tid < kPivot * R) {
      const int x = tid / R, c = tid % R;
      float v = 0.f;
#pragma unroll
      for (int yy = 0; yy < kPivot; ++yy) v = fmaf(Pm[x][yy], A[K0 + yy][c], v);
      RK[x][c] = v;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int idx = tid + NT * e, i = idx / R, c = idx % R;
      const bool in_i = (unsigned)(i - K0) < (unsigned)kPivot;
      const bool in_c = (unsigned)(c - K0) < (unsigned)kPivot;
      float v;
      if (in_i) {
        v = in_c ? Pm[i - K0][c - K0] : RK[i - K0][c];
      } else if (in_c) {
        v = 0.f;
#pragma unroll
        for (int x = 0; x < kPivot; ++x) v = fmaf(-CK[i][x], Pm[x][c - K0], v);
      } else {
        v = A[i][c];
#pragma unroll
        for (int x = 0; x < kPivot; ++x) v = fmaf(-CK[i][x], RK[x][c], v);
      }
      A[i][c] = v;
    }
    __syncthreads();
  }
  const bool bad = bad_s != 0;
  if (blockIdx.x == 0) {
    for (int idx = tid; idx < r * r; idx += NT) {
      const int i = idx / r, c = idx % r;
      const float v = A[i][c];
      Ginv[(size_t)b * r * r + idx] = __float2bfloat16_rn((bad || !isfinite(v)) ? 0.f : v);
    }
    if (tid == 0 && bad) atomicAdd(status, 1);
  }
  // L~ = L G^-1 for this CTA's rows: TR threads per row, H columns each
  constexpr int TR = NT / kApplyRows, H = R / TR;
  const int rr = tid / TR, c0 = (tid % TR) * H;
  const int row = row0 + rr;
  if (row >= n || c0 >= r) return;
  float acc[H];
#pragma unroll
  for (int c = 0; c < H; ++c) acc[c] = 0.f;
  for (int k = 0; k < r; ++k) {
    const float xk = __bfloat162float(Ls[rr][k]);
    const float4 *gk = reinterpret_cast<const float4 *>(&A[k][c0]);
#pragma unroll
    for (int c4 = 0; c4 < H / 4; ++c4) {
      const float4 gg = gk[c4];
      acc[4 * c4 + 0] = fmaf(xk, gg.x, acc[4 * c4 + 0]);
      acc[4 * c4 + 1] = fmaf(xk, gg.y, acc[4 * c4 + 1]);
      acc[4 * c4 + 2] = fmaf(xk, gg.z, acc[4 * c4 + 2]);
      acc[4 * c4 + 3] = fmaf(xk, gg.w, acc[4 * c4 + 3]);
    }
  }
  if (bad) {
#pragma unroll
    for (int c = 0; c < H; ++c) acc[c] = 0.f;
  }
  __nv_bfloat16 *Lrow = T + (size_t)b * sTb + (size_t)row * ldT + l0;
#pragma unroll
  for (int c = 0; c < H; c += 8) {
    if (c0 + c < r) {
      uint4 w;
      __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        h[j] = __floats2bfloat162_rn(acc[c + 2 * j], acc[c + 2 * j + 1]);
      *reinterpret_cast<uint4 *>(Lrow + c0 + c) = w;
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
    chol_apply_kernel<32><<<grid, apply_threads<32>(), 0, s>>>(G, r, ridge, T, n, ldT, l0, sTb,
                                                              Ginv, status);
  else
    chol_apply_kernel<64><<<grid, apply_threads<64>(), 0, s>>>(G, r, ridge, T, n, ldT, l0, sTb,
                                                              Ginv, status);
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
