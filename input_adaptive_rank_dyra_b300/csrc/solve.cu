// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward solves before the residual product: C~ = G^-1 C with C = L^T X (read as
// the fp32 C^T [batch, d, r] that the Gram GEMM stores), so that the next GEMM forms R = C~ W_res directly and the output GEMM
// multiplies L itself. The solve then touches r x d values per sample whatever the token
// count.
//   * r <= 64 (the Cholesky branch): spd_solve. Every CTA takes one sample and 128 columns
//     of C. It inverts G + lambda I (padded to R x R, R = 32 or 64, by the identity) in place
//     by block sweeps on 4 x 4 pivot blocks -- Gauss-Jordan without pivoting, whose scalar
//     pivots on an SPD matrix are the squared diagonal of the Cholesky factor -- with the
//     matrix spread over the CTA's registers, then forms its columns of C~ (fp32 FMA). CTAs
//     of the first column block also store G^-1 (bf16).
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

// Threads of spd_solve for the padded size R (the elimination uses (R / 4)^2 of them).
template <int R>
__host__ __device__ constexpr int solve_threads() { return R == 32 ? 128 : 256; }

// p = -(m^-1) of an SPD 4 x 4 block by four scalar sweeps; false if a pivot is not positive
// and finite.
__device__ __forceinline__ bool sweep4(const float (&m)[4][4], float (&p)[4][4]) {
  float w[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) w[i][j] = m[i][j];
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float dk = w[k][k];
    ok = ok && dk > 0.f && dk < INFINITY;
    const float di = 1.f / dk;
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = w[i][k];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[i][j] = fmaf(-c[i] * di, c[j], w[i][j]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[k][i] = c[i] * di;
      w[i][k] = c[i] * di;
    }
    w[k][k] = -di;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) p[i][j] = w[i][j];
  return ok;
}

// (G + ridge I)^-1 for one sample by in-place block sweeps on 4 x 4 pivot blocks (block
// Gauss-Jordan without pivoting; on an SPD matrix the pivot blocks are SPD Schur complements,
// whose scalar pivots are the squared diagonal of the Cholesky factor), then
// C~ = G^-1 C for kSolveCols columns of C. With K the pivot block, P = A_KK^-1 and
// S_i = A_iK P, one block sweep is
//   A_ij -= S_i A_Kj  (i, j outside K),  A_iK = S_i,  A_Kj = P A_Kj,  A_KK = -P,
// and after the sweeps over all blocks the matrix holds -(G + ridge I)^-1 (the identity
// padding up to R x R is never swept). Each of (R/4)^2 threads keeps one 4 x 4 block in
// registers. The pivot columns of the next step (rows of 4, = its pivot rows by symmetry) and
// the inverse of its pivot block, which the owner of that block forms after its update, go
// through double-buffered shared memory: one barrier per step, r / 4 steps. The inverse then
// goes to shared memory and every thread forms rows of C~ for its column as dot products with
// broadcast rows of the inverse.
template <int R>
__global__ void __launch_bounds__(solve_threads<R>())
    spd_solve_kernel(const float *__restrict__ G, int r, float ridge,
                     const float *__restrict__ Ct, int d, __nv_bfloat16 *__restrict__ Cs,
                     __nv_bfloat16 *__restrict__ Ginv, int *status) {
  constexpr int NT = solve_threads<R>();
  constexpr int Q = R / 4, NS = Q * Q;   // 4 x 4 blocks per side, elimination threads
  static_assert(NS <= NT, "every block needs a thread");
  constexpr int TPC = NT / kSolveCols;   // threads per column in the apply
  __shared__ __align__(16) float colbuf[2][R][4];   // the step's pivot columns A_iK
  __shared__ __align__(16) float pinv[2][4][4];     // P of the step
  __shared__ __align__(16) float Ai[R][R + 4];
  __shared__ int bad_s;
  const int tid = threadIdx.x, b = blockIdx.y;
  const bool el = tid < NS;   // takes part in the elimination
  const int i0 = (tid / Q) * 4, j0 = (tid % Q) * 4;
  // this thread's column of C (row of C^T), loaded first so the loads overlap the elimination
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
  float a[4][4];
  if (el) {
    const float *g = G + (size_t)b * r * r;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int i = i0 + u, j = j0 + v;
        a[u][v] = (i < r && j < r) ? g[i * r + j] + (i == j ? ridge : 0.f) : (i == j ? 1.f : 0.f);
      }
  }
  if (tid == 0) bad_s = 0;
  __syncthreads();
  if (el && j0 == 0) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4 *>(colbuf[0][i0 + u]) = make_float4(a[u][0], a[u][1], a[u][2], a[u][3]);
  }
  if (tid == 0) {   // owner of the first pivot block
    float p[4][4];
    if (!sweep4(a, p)) bad_s = 1;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) pinv[0][u][v] = -p[u][v];
  }
  __syncthreads();
  const int steps = r / 4;
  for (int kb = 0; kb < steps; ++kb) {
    const int k0 = kb * 4, cur = kb & 1;
    if (el) {
      float P[4][4], crow[4][4], ccol[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 pp = *reinterpret_cast<const float4 *>(pinv[cur][u]);
        const float4 cr = *reinterpret_cast<const float4 *>(colbuf[cur][i0 + u]);
        const float4 cc = *reinterpret_cast<const float4 *>(colbuf[cur][j0 + u]);
        P[u][0] = pp.x; P[u][1] = pp.y; P[u][2] = pp.z; P[u][3] = pp.w;
        crow[u][0] = cr.x; crow[u][1] = cr.y; crow[u][2] = cr.z; crow[u][3] = cr.w;
        ccol[u][0] = cc.x; ccol[u][1] = cc.y; ccol[u][2] = cc.z; ccol[u][3] = cc.w;
      }
      const bool rowsK = i0 == k0, colsK = j0 == k0;
      if (rowsK && colsK) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) a[u][v] = -P[u][v];
      } else if (rowsK) {   // A_Kj = P A_Kj = (A_jK P)^T
#pragma unroll
        for (int v = 0; v < 4; ++v)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float t = 0.f;
#pragma unroll
            for (int l = 0; l < 4; ++l) t = fmaf(ccol[v][l], P[l][u], t);
            a[u][v] = t;
          }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float S[4];   // S_i = A_iK P
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float t = 0.f;
#pragma unroll
            for (int l = 0; l < 4; ++l) t = fmaf(crow[u][l], P[l][m], t);
            S[m] = t;
          }
          if (colsK) {
#pragma unroll
            for (int v = 0; v < 4; ++v) a[u][v] = S[v];
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
#pragma unroll
              for (int m = 0; m < 4; ++m) a[u][v] = fmaf(-S[m], ccol[v][m], a[u][v]);
          }
        }
      }
      const int kn = k0 + 4;   // the next pivot block, after this step
      if (kn < r) {
        if (j0 == kn) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<float4 *>(colbuf[cur ^ 1][i0 + u]) =
                make_float4(a[u][0], a[u][1], a[u][2], a[u][3]);
        }
        if (i0 == kn && j0 == kn) {
          float p[4][4];
          if (!sweep4(a, p)) bad_s = 1;
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) pinv[cur ^ 1][u][v] = -p[u][v];
        }
      }
    }
    __syncthreads();
  }
  const bool bad = bad_s != 0;
  if (el) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) Ai[i0 + u][j0 + v] = bad ? 0.f : -a[u][v];
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int t = tid; t < r * r; t += NT)
      Ginv[(size_t)b * r * r + t] = __float2bfloat16_rn(Ai[t / r][t % r]);
    if (tid == 0 && bad) atomicAdd(status, 1);
  }
  if (col >= d) return;
  // C~[i][col] = sum_j G^-1[i][j] C[j][col]; the TPC threads of a column split the rows, four
  // independent partial sums per row
  __nv_bfloat16 *op = Cs + (size_t)b * r * d + col;
  for (int i = tid / kSolveCols; i < r; i += TPC) {
    const float4 *ar = reinterpret_cast<const float4 *>(&Ai[i][0]);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int j4 = 0; j4 < R / 4; ++j4) {
      const float4 w = ar[j4];
      s0 = fmaf(w.x, x[4 * j4], s0);
      s1 = fmaf(w.y, x[4 * j4 + 1], s1);
      s2 = fmaf(w.z, x[4 * j4 + 2], s2);
      s3 = fmaf(w.w, x[4 * j4 + 3], s3);
    }
    op[(size_t)i * d] = __float2bfloat16_rn((s0 + s1) + (s2 + s3));
  }
}

// Jacobi scaling and start of Newton-Schulz: dinv = diag(G + lambda I)^-1/2,
// G_hat = D (G + lambda I) D, X0 = I / max_i sum_j |G_hat_ij|. One CTA of kNsThreads per
// sample; a warp per row, so every load and store is coalesced and row sums are warp
// reductions.
constexpr int kNsThreads = 1024;

__global__ void __launch_bounds__(kNsThreads)
    ns_prep_kernel(const float *__restrict__ G, int r, float ridge, float *__restrict__ Gh,
                   float *__restrict__ X0, float *__restrict__ dinv, int *__restrict__ flags) {
  __shared__ float sd[256];
  __shared__ float red[kNsThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kNsThreads / 32;
  const float *g = G + (size_t)b * r * r;
  bool bad = false;
  if (tid < r) {
    const float gii = g[(size_t)tid * r + tid] + ridge;
    bad = !(gii > 0.f && gii < INFINITY);
    sd[tid] = bad ? 0.f : rsqrtf(gii);
  }
  bad = __syncthreads_or(bad) != 0;
  float mx = 0.f;
  for (int i = warp; i < r; i += NW) {
    float rs = 0.f;
    for (int j = lane; j < r; j += 32) {
      float v = (g[(size_t)i * r + j] + (i == j ? ridge : 0.f)) * sd[i] * sd[j];
      v = bad ? 0.f : v;
      Gh[(size_t)b * r * r + (size_t)i * r + j] = v;
      rs += fabsf(v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
    mx = fmaxf(mx, rs);
  }
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (warp == 0) {
    float m = red[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[0] = m;
  }
  __syncthreads();
  const float alpha = (bad || !(red[0] > 0.f)) ? 0.f : 1.f / red[0];
  for (int t = tid; t < r * r; t += kNsThreads) {
    const int i = t / r, j = t - i * r;
    X0[(size_t)b * r * r + t] = (i == j) ? alpha : 0.f;
  }
  if (tid < r) dinv[(size_t)b * r + tid] = bad ? 0.f : sd[tid];
  if (tid == 0) flags[b] = bad ? 1 : 0;
}

// G^-1 = D X_t D, to bf16 (workspace) and fp32 (operand of the apply GEMM). A sample whose
// iterate is not finite, or whose start was already flagged, gets G^-1 = 0.
__global__ void __launch_bounds__(kNsThreads)
    ns_finish_kernel(const float *__restrict__ X, const float *__restrict__ dinv, int r,
                     const int *__restrict__ flags, __nv_bfloat16 *__restrict__ Ginv,
                     float *__restrict__ G32, int *status) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const float *dv = dinv + (size_t)b * r;
  const size_t base = (size_t)b * r * r;
  bool bad = flags[b] != 0;
  for (int t = tid; t < r * r; t += kNsThreads) {
    const int i = t / r, j = t - i * r;
    const float x = X[base + t];
    bad = bad || !(fabsf(x) < INFINITY);
    const float v = x * dv[i] * dv[j];
    Ginv[base + t] = __float2bfloat16_rn(v);
    G32[base + t] = v;
  }
  if (__syncthreads_or(bad)) {   // rare: overwrite the sample with zeros
    for (int t = tid; t < r * r; t += kNsThreads) {
      Ginv[base + t] = __float2bfloat16_rn(0.f);
      G32[base + t] = 0.f;
    }
    if (tid == 0) atomicAdd(status, 1);
  }
}

}  // namespace

cudaError_t launch_spd_solve(const float *G, int batch, int r, float ridge, const float *Ct,
                             int d, __nv_bfloat16 *Cs, __nv_bfloat16 *Ginv, int *status,
                             cudaStream_t s) {
  if (r <= 0 || r > 64 || r % 4 || d <= 0) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  // a plain launch: the GEMM after it reads C~ through TMA only once this grid has completed
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
  ns_prep_kernel<<<batch, kNsThreads, 0, s>>>(G, r, ridge, Gh, X0, dinv, flags);
  return cudaGetLastError();
}

cudaError_t launch_ns_finish(const float *X, const float *dinv, int batch, int r, const int *flags,
                             __nv_bfloat16 *Ginv, float *G32, int *status, cudaStream_t s) {
  ns_finish_kernel<<<batch, kNsThreads, 0, s>>>(X, dinv, r, flags, Ginv, G32, status);
  return cudaGetLastError();
}

}  // namespace dyra
