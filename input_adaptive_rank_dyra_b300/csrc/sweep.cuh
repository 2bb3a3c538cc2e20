// In-place inversion of one symmetric positive definite R x R matrix (R = 32 or 64) by block
// sweeps on 4 x 4 pivot blocks -- Gauss-Jordan without pivoting. On an SPD matrix the pivot
// blocks are SPD Schur complements, whose scalar pivots are the squared diagonal of the
// Cholesky factor ("DyRA" summary page 2.4: Cholesky for small r), so none is zero and no
// pivoting is needed. With K the pivot block, P = A_KK^-1 and S_i = A_iK P, one block sweep is
//   A_ij -= S_i A_Kj  (i, j outside K),  A_iK = S_i,  A_Kj = P A_Kj,  A_KK = -P,
// and after the sweeps over the first r / 4 blocks the matrix holds -A^-1 (identity padding up
// to R x R is never swept). Each of (R/4)^2 threads keeps one 4 x 4 block in registers; the
// pivot columns of the next step (= its pivot rows, by symmetry) and the inverse of its pivot
// block, which the owner of that block forms after its update, go through double-buffered
// shared memory: one barrier per step. Used by the standalone inversion kernel and by the
// epilogue of the fused Gram / solve GEMM.
#pragma once
#include <cstdint>

namespace dyra {
namespace sweep {

// Shared memory of one inversion.
template <int R>
struct alignas(16) Smem {
  float colbuf[2][R][4];   // the step's pivot columns A_iK, row i at cb_row<R>(i)
  float pinv[2][4][4];     // P of the step
  int bad;                 // a pivot was not positive and finite
};

// Position of row i of the pivot columns: rows with the same i % 4 are contiguous, so the 16-byte
// reads of one warp (rows 4k + u for every block column k, u fixed) hit distinct banks; with
// row i at position i the same reads were 8-way bank conflicts.
template <int R>
__device__ __forceinline__ int cb_row(int i) { return (i & 3) * (R / 4) + (i >> 2); }

// p = -(m^-1) of an SPD 4 x 4 block by four scalar sweeps; false if a pivot is not positive
// and finite. The four pivot reciprocals are the longest dependent chain of a step, so they
// use the hardware reciprocal (__fdividef, within 2 ulp) rather than IEEE division.
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
    const float di = __fdividef(1.f, dk);
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

// Sweeps over the first r / 4 pivot blocks (r % 4 == 0, r <= R). Thread `tid` (< (R/4)^2 takes
// part; others only meet the barriers) owns block (tid / (R/4), tid % (R/4)) in `a`, already
// loaded (padding: identity). `bar()` synchronises every thread that calls this function;
// all of them call it the same number of times. Returns true if every pivot was positive and
// finite; `a` then holds this thread's block of -A^-1.
template <int R, typename Bar>
__device__ __forceinline__ bool invert_blocks(float (&a)[4][4], int tid, int r, Smem<R> &sm,
                                              Bar bar) {
  constexpr int Q = R / 4;
  const bool el = tid < Q * Q;
  const int i0 = (tid / Q) * 4, j0 = (tid % Q) * 4;
  if (tid == 0) sm.bad = 0;
  bar();
  if (el && j0 == 0) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4 *>(sm.colbuf[0][cb_row<R>(i0 + u)]) =
          make_float4(a[u][0], a[u][1], a[u][2], a[u][3]);
  }
  if (tid == 0) {   // owner of the first pivot block
    float p[4][4];
    if (!sweep4(a, p)) sm.bad = 1;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) sm.pinv[0][u][v] = -p[u][v];
  }
  bar();
  const int steps = r / 4;
  for (int kb = 0; kb < steps; ++kb) {
    const int k0 = kb * 4, cur = kb & 1;
    if (el) {
      float P[4][4], crow[4][4], ccol[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 pp = *reinterpret_cast<const float4 *>(sm.pinv[cur][u]);
        const float4 cr = *reinterpret_cast<const float4 *>(sm.colbuf[cur][cb_row<R>(i0 + u)]);
        const float4 cc = *reinterpret_cast<const float4 *>(sm.colbuf[cur][cb_row<R>(j0 + u)]);
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
            *reinterpret_cast<float4 *>(sm.colbuf[cur ^ 1][cb_row<R>(i0 + u)]) =
                make_float4(a[u][0], a[u][1], a[u][2], a[u][3]);
        }
        if (i0 == kn && j0 == kn) {
          float p[4][4];
          if (!sweep4(a, p)) sm.bad = 1;
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) sm.pinv[cur ^ 1][u][v] = -p[u][v];
        }
      }
    }
    bar();
  }
  return sm.bad == 0;
}

}  // namespace sweep
}  // namespace dyra
