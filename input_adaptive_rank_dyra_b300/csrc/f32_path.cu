// fp32 DyRA forward on CUDA cores. Used when the layer's dtype is fp32: tf32 tensor cores
// cannot hold a 1e-5 relative error, so every product here is an fp32 FFMA and the r x r
// least-squares system is solved in fp64.
//
// It follows the pages' order of operations literally ("DyRA：用输入相关的残差修正加速大模型的矩阵乘法",
// rank-r objective section; one-step section):
//   T = X [U | P]          (static projection X U and L = X P in one pass)
//   G = L^T L (fp64),  C = L^T X,  B = C W_res,  R = (G + lambda I)^-1 B (fp64 solve)
//   Y = (X U) V + b + L R
#include "kernels.cuh"

namespace dyra {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// C[b](i,j) = sum_k A[b](i,k) B[b](k,j) (+ C if accumulate) (+ bias[j]); generic strides.
__global__ void __launch_bounds__(256)
    sgemm_kernel(int M, int N, int K, const float *__restrict__ A, long long sAb, long long sAi,
                 long long sAk, const float *__restrict__ B, long long sBb, long long sBk,
                 long long sBj, float *__restrict__ C, long long sCb, long long sCi, long long sCj,
                 int accumulate, const float *__restrict__ bias) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int b = blockIdx.z;
  const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  A += b * sAb;
  B += b * sBb;
  C += b * sCb;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int t = threadIdx.x; t < TK * TM; t += 256) {
      const int kk = t / TM, ii = t % TM;
      const int gi = i0 + ii, gk = k0 + kk;
      As[kk][ii] = (gi < M && gk < K) ? A[gi * sAi + gk * sAk] : 0.f;
    }
    for (int t = threadIdx.x; t < TK * TN; t += 256) {
      const int kk = t / TN, jj = t % TN;
      const int gj = j0 + jj, gk = k0 + kk;
      Bs[kk][jj] = (gj < N && gk < K) ? B[gk * sBk + gj * sBj] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = As[kk][ty + 16 * u];
#pragma unroll
      for (int v = 0; v < 4; ++v) bv[v] = Bs[kk][tx + 16 * v];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int gi = i0 + ty + 16 * u;
    if (gi >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int gj = j0 + tx + 16 * v;
      if (gj >= N) continue;
      float val = acc[u][v];
      if (bias) val += bias[gj];
      float *dst = C + gi * sCi + gj * sCj;
      *dst = accumulate ? *dst + val : val;
    }
  }
}

// G[b] = L^T L in fp64; L = columns [l0, l0 + r) of T [n, ldT].
__global__ void gram_f64_kernel(const float *__restrict__ T, int n, int ldT, int l0, int r,
                                long long sTb, double *__restrict__ G) {
  const int b = blockIdx.y;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= r * r) return;
  const int i = t / r, j = t % r;
  const float *L = T + b * sTb + l0;
  double s = 0.0;
  for (int row = 0; row < n; ++row)
    s += (double)L[(size_t)row * ldT + i] * (double)L[(size_t)row * ldT + j];
  G[(size_t)b * r * r + t] = s;
}

// Explicit (G + lambda I)^-1 in fp64: Cholesky (or Newton-Schulz) then inverse. One CTA per
// sample, r <= 64.
__global__ void __launch_bounds__(64)
    inverse_f64_kernel(const double *__restrict__ G, int r, double ridge, int use_ns, int ns_iters,
                       double *__restrict__ Ginv, int *status) {
  __shared__ double A[64][65];
  __shared__ double Li[64][65];
  __shared__ int bad;
  const int b = blockIdx.x, tid = threadIdx.x;
  const double *g = G + (size_t)b * r * r;
  for (int t = tid; t < r * r; t += blockDim.x) A[t / r][t % r] = g[t] + ((t / r) == (t % r) ? ridge : 0.0);
  if (tid == 0) bad = 0;
  __syncthreads();
  double *out = Ginv + (size_t)b * r * r;
  if (!use_ns) {
    for (int j = 0; j < r; ++j) {
      if (tid == 0) {
        double ajj = A[j][j];
        if (!(ajj > 0.0) || !isfinite(ajj)) {
          bad = 1;
          ajj = 1.0;
        }
        A[j][j] = sqrt(ajj);
      }
      __syncthreads();
      for (int i = j + 1 + tid; i < r; i += blockDim.x) A[i][j] /= A[j][j];
      __syncthreads();
      const int w = r - j - 1;
      for (int t = tid; t < w * w; t += blockDim.x) {
        const int ii = j + 1 + t / w, cc = j + 1 + t % w;
        if (cc <= ii) A[ii][cc] -= A[ii][j] * A[cc][j];
      }
      __syncthreads();
    }
    for (int c = tid; c < r; c += blockDim.x)
      for (int i = 0; i < r; ++i) {
        double v = 0.0;
        if (i == c) v = 1.0 / A[i][i];
        else if (i > c) {
          double s = 0.0;
          for (int k = c; k < i; ++k) s += A[i][k] * Li[k][c];
          v = -s / A[i][i];
        }
        Li[i][c] = v;
      }
    __syncthreads();
    for (int t = tid; t < r * r; t += blockDim.x) {
      const int i = t / r, j = t % r;
      double s = 0.0;
      for (int k = (i > j ? i : j); k < r; ++k) s += Li[k][i] * Li[k][j];
      out[t] = bad ? 0.0 : s;
    }
  } else {
    // Newton-Schulz on the Jacobi-scaled matrix: X <- X (2I - G_hat X)
    __shared__ double d[64];
    __shared__ double alpha;
    for (int i = tid; i < r; i += blockDim.x) {
      const double a = A[i][i];
      if (!(a > 0.0) || !isfinite(a)) bad = 1;
      d[i] = (a > 0.0) ? 1.0 / sqrt(a) : 0.0;
    }
    __syncthreads();
    for (int t = tid; t < r * r; t += blockDim.x) A[t / r][t % r] *= d[t / r] * d[t % r];
    __syncthreads();
    if (tid == 0) {
      double mx = 0.0;
      for (int i = 0; i < r; ++i) {
        double s = 0.0;
        for (int j = 0; j < r; ++j) s += fabs(A[i][j]);
        mx = s > mx ? s : mx;
      }
      alpha = mx > 0.0 ? 1.0 / mx : 0.0;
    }
    __syncthreads();
    for (int t = tid; t < r * r; t += blockDim.x) Li[t / r][t % r] = (t / r == t % r) ? alpha : 0.0;
    __syncthreads();
    for (int it = 0; it < ns_iters; ++it) {
      // P = G_hat X  (kept in out[] as scratch), then X = 2X - X P
      for (int t = tid; t < r * r; t += blockDim.x) {
        const int i = t / r, j = t % r;
        double s = 0.0;
        for (int k = 0; k < r; ++k) s += A[i][k] * Li[k][j];
        out[t] = s;
      }
      __syncthreads();
      double nv[64];
      int cnt = 0;
      for (int t = tid; t < r * r; t += blockDim.x) {
        const int i = t / r, j = t % r;
        double s = 0.0;
        for (int k = 0; k < r; ++k) s += Li[i][k] * out[k * r + j];
        nv[cnt++] = 2.0 * Li[i][j] - s;
      }
      __syncthreads();
      cnt = 0;
      for (int t = tid; t < r * r; t += blockDim.x) Li[t / r][t % r] = nv[cnt++];
      __syncthreads();
    }
    for (int t = tid; t < r * r; t += blockDim.x) {
      const int i = t / r, j = t % r;
      const double v = Li[i][j] * d[i] * d[j];
      out[t] = (bad || !isfinite(v)) ? 0.0 : v;
    }
  }
  if (tid == 0 && bad) atomicAdd(status, 1);
}

// R[b][:, col] = Ginv[b] B[b][:, col], fp64 accumulation, fp32 output.
__global__ void apply_inverse_kernel(const double *__restrict__ Ginv, const float *__restrict__ Bm,
                                     int r, int m, float *__restrict__ R) {
  const int b = blockIdx.y;
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= m) return;
  const double *gi = Ginv + (size_t)b * r * r;
  const float *bb = Bm + (size_t)b * r * m;
  float *rr = R + (size_t)b * r * m;
  for (int i = 0; i < r; ++i) {
    double s = 0.0;
    for (int k = 0; k < r; ++k) s += gi[i * r + k] * (double)bb[(size_t)k * m + col];
    rr[(size_t)i * m + col] = (float)s;
  }
}

}  // namespace

cudaError_t launch_sgemm(int batch, int M, int N, int K, const float *A, long long sAb,
                         long long sAi, long long sAk, const float *B, long long sBb, long long sBk,
                         long long sBj, float *C, long long sCb, long long sCi, long long sCj,
                         bool accumulate, const float *bias, cudaStream_t s) {
  if (batch <= 0 || M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM, batch);
  sgemm_kernel<<<grid, 256, 0, s>>>(M, N, K, A, sAb, sAi, sAk, B, sBb, sBk, sBj, C, sCb, sCi, sCj,
                                    accumulate ? 1 : 0, bias);
  return cudaGetLastError();
}

cudaError_t launch_gram_f64(const float *T, int batch, int n, int ldT, int l0, int r,
                            long long sTb, double *G, cudaStream_t s) {
  dim3 grid((r * r + 127) / 128, batch);
  gram_f64_kernel<<<grid, 128, 0, s>>>(T, n, ldT, l0, r, sTb, G);
  return cudaGetLastError();
}

cudaError_t launch_inverse_f64(const double *G, int batch, int r, double ridge, bool ns,
                               int ns_iters, double *Ginv, int *status, cudaStream_t s) {
  if (r > 64) return cudaErrorInvalidValue;
  inverse_f64_kernel<<<batch, 64, 0, s>>>(G, r, ridge, ns ? 1 : 0, ns_iters, Ginv, status);
  return cudaGetLastError();
}

cudaError_t launch_apply_inverse(const double *Ginv, const float *B, int batch, int r, int m,
                                 float *R, cudaStream_t s) {
  dim3 grid((m + 127) / 128, batch);
  apply_inverse_kernel<<<grid, 128, 0, s>>>(Ginv, B, r, m, R);
  return cudaGetLastError();
}

}  // namespace dyra
