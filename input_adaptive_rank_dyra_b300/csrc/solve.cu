// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward solves before the residual product: C~ = G^-1 C with C = L^T X (read as
// the fp32 C^T [batch, d, r] that the Gram GEMM stores), so that the next GEMM forms R = C~ W_res directly and the output GEMM
// multiplies L itself. The solve then touches r x d values per sample whatever the token
// count.
//   * r <= 64 (the Cholesky branch): spd_solve. Every CTA takes one sample and 128 columns
//     of C. It inverts G + lambda I (padded to R x R, R = 32 or 64, by the identity) in place
//     by symmetric sweeps -- Gauss-Jordan without pivoting, whose pivots on an SPD matrix are
//     the squared diagonal of the Cholesky factor -- with the matrix spread over the CTA's
//     registers, then forms its columns of C~ (fp32 FMA). CTAs of the first column block also
//     store G^-1 (bf16).
//   * larger r: Newton-Schulz. ns_prep scales G symmetrically to unit diagonal and sets
//     X0 = I / ||G_hat||_inf; the iterations X <- X (2I - G_hat X) run as tf32 tensor-core
//     GEMMs (tc_gemm); ns_finish undoes the scaling; a bf16 tensor-core GEMM then forms
//     C~ = G^-1 C.
// A sample with a pivot that is not positive (or not finite) is counted in status[0] and
// gets G^-1 = 0 and C~ = 0, so its correction vanishes and its output is the static branch
// plus bias.
#include "kernels.cuh"

#include <cuda_bf16.h>

namespace dyra {

namespace {

constexpr int kSolveCols = 128;   // columns of C per spd_solve CTA

// Threads of spd_solve for the padded size R: each holds a BR x BC block of the matrix.
template <int R>
__host__ __device__ constexpr int solve_threads() { return R == 32 ? 128 : 256; }

// (G + ridge I)^-1 for one sample by in-place symmetric sweeps (Gauss-Jordan without
// pivoting; on an SPD matrix the pivots are the positive Schur complements that a Cholesky
// factorisation squares), then C~ = G^-1 C for kSolveCols columns of C. With s_i = a_ik / a_kk
// the sweep on pivot k is
//   a_ij -= s_i a_kj  (i, j != k),   a_ik = a_ki = s_i,   a_kk = -1 / a_kk,
// and after the sweeps on k = 0 .. r-1 the matrix holds -(G + ridge I)^-1. Every thread
// keeps its BR x BC block in registers; the pivot column (= pivot row, by symmetry) goes
// through a double-buffered shared-memory vector, so each sweep costs one barrier. The
// inverse then goes to shared memory and every thread forms rows of C~ for its column as
// dot products with broadcast rows of the inverse.
template <int R>
__global__ void __launch_bounds__(solve_threads<R>())
    spd_solve_kernel(const float *__restrict__ G, int r, float ridge,
                     const float *__restrict__ Ct, int d, __nv_bfloat16 *__restrict__ Cs,
                     __nv_bfloat16 *__restrict__ Ginv, int *status) {
  constexpr int NT = solve_threads<R>();
  constexpr int BR = R == 32 ? 2 : 4, BC = 4, QC = R / BC;
  static_assert((R / BR) * QC == NT, "thread blocks must tile the matrix");
  constexpr int TPC = NT / kSolveCols;   // threads per column in the apply
  __shared__ __align__(16) float colbuf[2][R];
  __shared__ __align__(16) float Ai[R][R + 4];
  const int tid = threadIdx.x, b = blockIdx.y;
  const int i0 = (tid / QC) * BR, j0 = (tid % QC) * BC;
  // this thread's column of C (row of C^T), loaded first so the loads overlap the sweeps
  const int col = blockIdx.x * kSolveCols + tid % kSolveCols;
  float x[R];
  {
    const float4 *cp = reinterpret_cast<const float4 *>(Ct + ((size_t)b * d + (col < d ? col : 0)) * r);
#pragma unroll
    for (int i4 = 0; i4 < R; i4 += 4) {
      const float4 v = (i4 < r && col < d) ? __ldg(cp + i4 / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[i4] = v.x;
      x[i4 + 1] = v.y;
      x[i4 + 2] = v.z;
      x[i4 + 3] = v.w;
    }
  }
  float a[BR][BC];
  const float *g = G + (size_t)b * r * r;
#pragma unroll
  for (int u = 0; u < BR; ++u)
#pragma unroll
    for (int v = 0; v < BC; ++v) {
      const int i = i0 + u, j = j0 + v;
      a[u][v] = (i < r && j < r) ? g[i * r + j] + (i == j ? ridge : 0.f) : (i == j ? 1.f : 0.f);
    }
  if (j0 == 0) {
#pragma unroll
    for (int u = 0; u < BR; ++u) colbuf[0][i0 + u] = a[u][0];
  }
  __syncthreads();
  bool bad = false;   // the same in every thread: every pivot is read from shared memory
  for (int k = 0; k < r; ++k) {
    const float *cur = colbuf[k & 1];
    const float piv = cur[k];
    if (!(piv > 0.f && piv < INFINITY)) bad = true;
    const float dinv = 1.f / piv;
    float ci[BR], cj[BC];
#pragma unroll
    for (int u = 0; u < BR; ++u) ci[u] = cur[i0 + u];
    {
      const float4 c4 = *reinterpret_cast<const float4 *>(cur + j0);
      cj[0] = c4.x;
      cj[1] = c4.y;
      cj[2] = c4.z;
      cj[3] = c4.w;
    }
#pragma unroll
    for (int u = 0; u < BR; ++u) {
      const float si = ci[u] * dinv;
#pragma unroll
      for (int v = 0; v < BC; ++v) a[u][v] = fmaf(-si, cj[v], a[u][v]);
    }
    if ((unsigned)(k - i0) < (unsigned)BR) {   // row k: a_kj = a_kj / a_kk
#pragma unroll
      for (int u = 0; u < BR; ++u)
        if (i0 + u == k) {
#pragma unroll
          for (int v = 0; v < BC; ++v) a[u][v] = cj[v] * dinv;
        }
    }
    if ((unsigned)(k - j0) < (unsigned)BC) {   // column k: a_ik = a_ik / a_kk; a_kk = -1 / a_kk
#pragma unroll
      for (int v = 0; v < BC; ++v)
        if (j0 + v == k) {
#pragma unroll
          for (int u = 0; u < BR; ++u) a[u][v] = (i0 + u == k) ? -dinv : ci[u] * dinv;
        }
    }
    const int kn = k + 1;   // the next pivot column, after this sweep
    if (kn < r && (unsigned)(kn - j0) < (unsigned)BC) {
      float *nxt = colbuf[kn & 1];
#pragma unroll
      for (int v = 0; v < BC; ++v)
        if (j0 + v == kn) {
#pragma unroll
          for (int u = 0; u < BR; ++u) nxt[i0 + u] = a[u][v];
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < BR; ++u)
#pragma unroll
    for (int v = 0; v < BC; ++v) Ai[i0 + u][j0 + v] = bad ? 0.f : -a[u][v];
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int t = tid; t < r * r; t += NT)
      Ginv[(size_t)b * r * r + t] = __float2bfloat16_rn(Ai[t / r][t % r]);
    if (tid == 0 && bad) atomicAdd(status, 1);
  }
  if (col >= d) return;
  // C~[i][col] = sum_j G^-1[i][j] C[j][col]; the TPC threads of a column split the rows
  __nv_bfloat16 *op = Cs + (size_t)b * r * d + col;
  for (int i = tid / kSolveCols; i < r; i += TPC) {
    const float4 *ar = reinterpret_cast<const float4 *>(&Ai[i][0]);
    float acc = 0.f;
#pragma unroll
    for (int j4 = 0; j4 < R / 4; ++j4) {
      const float4 w = ar[j4];
      acc = fmaf(w.x, x[4 * j4], acc);
      acc = fmaf(w.y, x[4 * j4 + 1], acc);
      acc = fmaf(w.z, x[4 * j4 + 2], acc);
      acc = fmaf(w.w, x[4 * j4 + 3], acc);
    }
    op[(size_t)i * d] = __float2bfloat16_rn(acc);
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
                     const int *__restrict__ flags, __nv_bfloat16 *__restrict__ Ginv,
                     float *__restrict__ G32, int *status) {
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
    G32[(size_t)b * r * r + t] = v;
  }
  if (tid == 0 && bad) atomicAdd(status, 1);
}

}  // namespace

cudaError_t launch_spd_solve(const float *G, int batch, int r, float ridge, const float *Ct,
                             int d, __nv_bfloat16 *Cs, __nv_bfloat16 *Ginv, int *status,
                             cudaStream_t s) {
  if (r <= 0 || r > 64 || r % 4 || d <= 0) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  dim3 grid((d + kSolveCols - 1) / kSolveCols, batch);
  if (r <= 32)
    spd_solve_kernel<32><<<grid, solve_threads<32>(), 0, s>>>(G, r, ridge, Ct, d, Cs, Ginv, status);
  else
    spd_solve_kernel<64><<<grid, solve_threads<64>(), 0, s>>>(G, r, ridge, Ct, d, Cs, Ginv, status);
  return cudaGetLastError();
}

cudaError_t launch_ns_prep(const float *G, int batch, int r, float ridge, float *Gh, float *X0,
                           float *dinv, int *flags, cudaStream_t s) {
  if (r > 256) return cudaErrorInvalidValue;
  ns_prep_kernel<<<batch, 256, 0, s>>>(G, r, ridge, Gh, X0, dinv, flags);
  return cudaGetLastError();
}

cudaError_t launch_ns_finish(const float *X, const float *dinv, int batch, int r, const int *flags,
                             __nv_bfloat16 *Ginv, float *G32, int *status, cudaStream_t s) {
  ns_finish_kernel<<<batch, 256, 0, s>>>(X, dinv, r, flags, Ginv, G32, status);
  return cudaGetLastError();
}

}  // namespace dyra
