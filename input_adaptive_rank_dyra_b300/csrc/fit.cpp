// Host float64 linear algebra for the offline preparation of a DyRA layer.
//
// The offline step of the method ("DyRA：用输入相关的残差修正加速大模型的矩阵乘法", offline /
// online flow section; summary page Appendix B) needs a truncated SVD of W (low-rank
// static branch), rank-1 SVDs of blocks (Monarch) and the top right singular vectors of
// W_res (R0). All of them go through the symmetric eigen-decomposition below:
//   * Householder reduction to tridiagonal form (Golub & Van Loan, "Matrix Computations",
//     section 8.3.1), with the rank-2 updates spread over host threads;
//   * the implicit symmetric QL iteration with a Wilkinson shift (ibid. 8.3.3, QL variant)
//     on the tridiagonal matrix; its plane rotations are queued and applied in batches to
//     column strips of the eigenvector matrix so each strip stays in cache.
#include "fit.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace dyra {
namespace fit {

void parallel_for(int n, int threads, const void *ctx, void (*fn)(const void *ctx, int i)) {
  if (n <= 0) return;
  int hw = (int)std::thread::hardware_concurrency();
  if (hw <= 0) hw = 1;
  int t = threads > 0 ? threads : hw;
  t = std::min(t, n);
  if (t <= 1) {
    for (int i = 0; i < n; ++i) fn(ctx, i);
    return;
  }
  std::atomic<int> next(0);
  std::vector<std::thread> pool;
  pool.reserve(t);
  for (int w = 0; w < t; ++w) {
    pool.emplace_back([&]() {
      for (;;) {
        int i = next.fetch_add(1);
        if (i >= n) break;
        fn(ctx, i);
      }
    });
  }
  for (auto &th : pool) th.join();
}

// ------------------------------------------------------------------------------- GEMM

namespace {
struct GemmCtx {
  int rows, cols, inner;
  const double *A;   // [rows x inner]
  const double *B;   // [inner x cols]
  double *C;
  int col_blocks;
};

constexpr int kRB = 32, kCB = 512, kKB = 128;

// One (row block, column block) tile of C, accumulated over K in slabs.
void gemm_tile(const void *vctx, int t) {
  const GemmCtx &g = *static_cast<const GemmCtx *>(vctx);
  const int rb = t / g.col_blocks, cb = t % g.col_blocks;
  const int i0 = rb * kRB, i1 = std::min(g.rows, i0 + kRB);
  const int j0 = cb * kCB, j1 = std::min(g.cols, j0 + kCB);
  const int w = j1 - j0;
  for (int i = i0; i < i1; ++i) std::memset(g.C + (size_t)i * g.cols + j0, 0, sizeof(double) * w);
  for (int k0 = 0; k0 < g.inner; k0 += kKB) {
    const int k1 = std::min(g.inner, k0 + kKB);
    for (int i = i0; i < i1; ++i) {
      double *c = g.C + (size_t)i * g.cols + j0;
      const double *a = g.A + (size_t)i * g.inner;
      for (int k = k0; k < k1; ++k) {
        const double av = a[k];
        if (av == 0.0) continue;
        const double *b = g.B + (size_t)k * g.cols + j0;
        for (int j = 0; j < w; ++j) c[j] += av * b[j];
      }
    }
  }
}

struct TrCtx { const double *src; double *dst; int rows, cols; };
void transpose_rows(const void *vctx, int blk) {
  const TrCtx &c = *static_cast<const TrCtx *>(vctx);
  const int i0 = blk * 64, i1 = std::min(c.rows, i0 + 64);
  for (int j0 = 0; j0 < c.cols; j0 += 64) {
    const int j1 = std::min(c.cols, j0 + 64);
    for (int i = i0; i < i1; ++i)
      for (int j = j0; j < j1; ++j) c.dst[(size_t)j * c.rows + i] = c.src[(size_t)i * c.cols + j];
  }
}

std::vector<double> transposed(const double *src, int rows, int cols, int threads) {
  std::vector<double> dst((size_t)rows * cols);
  TrCtx c{src, dst.data(), rows, cols};
  parallel_for((rows + 63) / 64, threads, &c, transpose_rows);
  return dst;
}
}  // namespace

void gemm(int rows, int cols, int inner, const double *A, bool transA, const double *B,
          bool transB, double *C, int threads) {
  std::vector<double> at, bt;
  if (transA) {  // A stored [inner x rows]
    at = transposed(A, inner, rows, threads);
    A = at.data();
  }
  if (transB) {  // B stored [cols x inner]
    bt = transposed(B, cols, inner, threads);
    B = bt.data();
  }
  GemmCtx g{rows, cols, inner, A, B, C, (cols + kCB - 1) / kCB};
  parallel_for(((rows + kRB - 1) / kRB) * g.col_blocks, threads, &g, gemm_tile);
}

// --------------------------------------------------------------------- tridiagonalise

namespace {

struct Rank2Ctx {
  double *A;   // full symmetric storage, n x n
  int n, k0;   // trailing block starts at row/col k0
  const double *v, *q;
};

// A[i][j] -= 2 (v_i q_j + q_i v_j) on the trailing block (rows split across threads)
void rank2_rows(const void *vctx, int blk) {
  const Rank2Ctx &c = *static_cast<const Rank2Ctx *>(vctx);
  const int len = c.n - c.k0;
  const int i0 = blk * 32, i1 = std::min(len, i0 + 32);
  for (int i = i0; i < i1; ++i) {
    double *row = c.A + (size_t)(c.k0 + i) * c.n + c.k0;
    const double vi = 2.0 * c.v[i], qi = 2.0 * c.q[i];
    for (int j = 0; j < len; ++j) row[j] -= vi * c.q[j] + qi * c.v[j];
  }
}

struct SymvCtx {
  const double *A;
  int n, k0;
  const double *v;
  double *p;
};

void symv_rows(const void *vctx, int blk) {
  const SymvCtx &c = *static_cast<const SymvCtx *>(vctx);
  const int len = c.n - c.k0;
  const int i0 = blk * 32, i1 = std::min(len, i0 + 32);
  for (int i = i0; i < i1; ++i) {
    const double *row = c.A + (size_t)(c.k0 + i) * c.n + c.k0;
    double s = 0.0;
    for (int j = 0; j < len; ++j) s += row[j] * c.v[j];
    c.p[i] = s;
  }
}

struct ReflCtx {
  double *Q;    // n x n row-major
  int n, k0;    // reflector acts on rows/cols >= k0
  const double *v;
};

// Q[k0:, k0:] <- (I - 2 v v^T) Q[k0:, k0:], split over column blocks
void refl_cols(const void *vctx, int blk) {
  const ReflCtx &c = *static_cast<const ReflCtx *>(vctx);
  const int len = c.n - c.k0;
  const int j0 = blk * 64, j1 = std::min(len, j0 + 64);
  double acc[64];
  for (int j = j0; j < j1; ++j) acc[j - j0] = 0.0;
  for (int i = 0; i < len; ++i) {
    const double vi = c.v[i];
    if (vi == 0.0) continue;
    const double *row = c.Q + (size_t)(c.k0 + i) * c.n + c.k0;
    for (int j = j0; j < j1; ++j) acc[j - j0] += vi * row[j];
  }
  for (int i = 0; i < len; ++i) {
    const double vi = 2.0 * c.v[i];
    if (vi == 0.0) continue;
    double *row = c.Q + (size_t)(c.k0 + i) * c.n + c.k0;
    for (int j = j0; j < j1; ++j) row[j] -= vi * acc[j - j0];
  }
}

struct RotCtx {
  double *Zt;              // n x n, row j = current basis vector j (length n)
  int n;
  const int *idx;          // rotation acts on rows idx, idx+1
  const double *cs, *sn;
  int count;
};

// Apply the queued rotations, in order, to one 64-column strip of Zt.
void rot_strip(const void *vctx, int blk) {
  const RotCtx &c = *static_cast<const RotCtx *>(vctx);
  const int j0 = blk * 64, j1 = std::min(c.n, j0 + 64);
  for (int t = 0; t < c.count; ++t) {
    double *a = c.Zt + (size_t)c.idx[t] * c.n;
    double *b = a + c.n;
    const double cc = c.cs[t], ss = c.sn[t];
    for (int j = j0; j < j1; ++j) {
      const double f = b[j];
      b[j] = ss * a[j] + cc * f;
      a[j] = cc * a[j] - ss * f;
    }
  }
}

}  // namespace

bool sym_eig(int n, const double *Ain, double *evals, double *evecs, int threads) {
  if (n <= 0) return true;
  if (n == 1) {
    evals[0] = Ain[0];
    evecs[0] = 1.0;
    return true;
  }
  std::vector<double> A(Ain, Ain + (size_t)n * n);
  std::vector<double> diag(n), off(n, 0.0);        // off[i] couples i and i+1
  std::vector<double> V((size_t)n * n, 0.0);        // reflector k stored in row k (entries > k)
  std::vector<double> p(n), q(n);

  // Householder: for column k, zero A[k+2:, k] with H_k = I - 2 v v^T acting on indices > k.
  for (int k = 0; k < n - 2; ++k) {
    const int k0 = k + 1, len = n - k0;
    double norm2 = 0.0;
    for (int i = 0; i < len; ++i) norm2 += A[(size_t)(k0 + i) * n + k] * A[(size_t)(k0 + i) * n + k];
    const double x0 = A[(size_t)k0 * n + k];
    const double alpha = (x0 > 0 ? -1.0 : 1.0) * std::sqrt(norm2);
    double *v = &V[(size_t)k * n + k0];
    for (int i = 0; i < len; ++i) v[i] = A[(size_t)(k0 + i) * n + k];
    v[0] -= alpha;
    double vn = 0.0;
    for (int i = 0; i < len; ++i) vn += v[i] * v[i];
    diag[k] = A[(size_t)k * n + k];
    if (vn <= 1e-300) {          // column already reduced
      for (int i = 0; i < len; ++i) v[i] = 0.0;
      off[k] = x0;
      continue;
    }
    vn = 1.0 / std::sqrt(vn);
    for (int i = 0; i < len; ++i) v[i] *= vn;
    off[k] = alpha;
    // trailing block: A22 <- H A22 H = A22 - 2 v q^T - 2 q v^T, q = A22 v - (v^T A22 v) v
    SymvCtx sc{A.data(), n, k0, v, p.data()};
    parallel_for((len + 31) / 32, len > 256 ? threads : 1, &sc, symv_rows);
    double kk = 0.0;
    for (int i = 0; i < len; ++i) kk += v[i] * p[i];
    for (int i = 0; i < len; ++i) q[i] = p[i] - kk * v[i];
    Rank2Ctx rc{A.data(), n, k0, v, q.data()};
    parallel_for((len + 31) / 32, len > 256 ? threads : 1, &rc, rank2_rows);
  }
  diag[n - 2] = A[(size_t)(n - 2) * n + (n - 2)];
  diag[n - 1] = A[(size_t)(n - 1) * n + (n - 1)];
  off[n - 2] = A[(size_t)(n - 1) * n + (n - 2)];
  off[n - 1] = 0.0;

  // Q = H_0 H_1 ... H_{n-3}, accumulated from the inside out (only the trailing block of
  // each partial product is non-trivial).
  std::vector<double> Q((size_t)n * n, 0.0);
  for (int i = 0; i < n; ++i) Q[(size_t)i * n + i] = 1.0;
  for (int k = n - 3; k >= 0; --k) {
    const int k0 = k + 1, len = n - k0;
    ReflCtx fc{Q.data(), n, k0, &V[(size_t)k * n + k0]};
    parallel_for((len + 63) / 64, len > 256 ? threads : 1, &fc, refl_cols);
  }
  // Zt = Q^T: row j is column j of Q; QL rotations then mix adjacent rows of Zt.
  std::vector<double> &Zt = A;  // reuse storage
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) Zt[(size_t)j * n + i] = Q[(size_t)i * n + j];
  Q.clear();
  Q.shrink_to_fit();

  // Implicit QL with Wilkinson shift on (diag, off). An off-diagonal entry is negligible when
  // it is small against its two diagonal neighbours (relative accuracy for well-separated
  // eigenvalues) or against the whole tridiagonal matrix (a cluster of eigenvalues near zero,
  // e.g. the Gram matrix of a rank-deficient residual, has off-diagonal rounding noise of the
  // size eps * ||T|| that no relative test ever deflates).
  double tnorm = 0.0;
  for (int i = 0; i < n; ++i)
    tnorm = std::max(tnorm, std::fabs(diag[i]) + std::fabs(off[i]) + (i ? std::fabs(off[i - 1]) : 0.0));
  const double abs_tol = 4e-16 * tnorm;
  const int kQueue = 1 << 16;
  std::vector<int> ridx;
  std::vector<double> rc_, rs_;
  ridx.reserve(kQueue);
  rc_.reserve(kQueue);
  rs_.reserve(kQueue);
  auto flush = [&]() {
    if (ridx.empty()) return;
    RotCtx c{Zt.data(), n, ridx.data(), rc_.data(), rs_.data(), (int)ridx.size()};
    parallel_for((n + 63) / 64, n > 128 ? threads : 1, &c, rot_strip);
    ridx.clear();
    rc_.clear();
    rs_.clear();
  };
  for (int l = 0; l < n; ++l) {
    int iter = 0;
    for (;;) {
      int mm = l;
      for (; mm < n - 1; ++mm) {
        const double dd = std::fabs(diag[mm]) + std::fabs(diag[mm + 1]);
        if (std::fabs(off[mm]) <= 1e-16 * dd || std::fabs(off[mm]) <= abs_tol) break;
      }
      if (mm == l) break;
      if (++iter > 60) {
        flush();
        return false;
      }
      // shift: eigenvalue of the leading 2x2 block closest to diag[l]
      double g = (diag[l + 1] - diag[l]) / (2.0 * off[l]);
      double rr = std::hypot(g, 1.0);
      g = diag[mm] - diag[l] + off[l] / (g + (g >= 0 ? rr : -rr));
      double s = 1.0, c = 1.0, pp = 0.0;
      int i = mm - 1;
      bool early = false;
      for (; i >= l; --i) {
        double f = s * off[i];
        const double b = c * off[i];
        rr = std::hypot(f, g);
        off[i + 1] = rr;
        if (rr == 0.0) {
          diag[i + 1] -= pp;
          off[mm] = 0.0;
          early = true;
          break;
        }
        s = f / rr;
        c = g / rr;
        g = diag[i + 1] - pp;
        rr = (diag[i] - g) * s + 2.0 * c * b;
        pp = s * rr;
        diag[i + 1] = g + pp;
        g = c * rr - b;
        ridx.push_back(i);
        rc_.push_back(c);
        rs_.push_back(s);
        if ((int)ridx.size() >= kQueue) flush();
      }
      if (early && i >= l) continue;
      diag[l] -= pp;
      off[l] = g;
      off[mm] = 0.0;
    }
  }
  flush();

  // sort descending
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int a, int b) { return diag[a] > diag[b]; });
  for (int j = 0; j < n; ++j) {
    evals[j] = diag[order[j]];
    std::memcpy(evecs + (size_t)j * n, &Zt[(size_t)order[j] * n], sizeof(double) * n);
  }
  return true;
}

bool top_svd(int d, int m, const double *W, int count, double *U, double *S, double *Vt,
             int threads) {
  const int p = std::min(d, m);
  if (count > p || count < 0) return false;
  if (count == 0) return true;
  std::vector<double> H((size_t)p * p), ev(p), vec((size_t)p * p);
  if (d <= m) {
    gemm(d, d, m, W, false, W, true, H.data(), threads);        // W W^T
  } else {
    gemm(m, m, d, W, true, W, false, H.data(), threads);        // W^T W
  }
  if (!sym_eig(p, H.data(), ev.data(), vec.data(), threads)) return false;
  for (int j = 0; j < count; ++j) S[j] = std::sqrt(std::max(ev[j], 0.0));
  if (d <= m) {
    // vec rows = left vectors; V^T rows = u_j^T W / s_j
    for (int j = 0; j < count; ++j)
      for (int i = 0; i < d; ++i) U[(size_t)i * count + j] = vec[(size_t)j * d + i];
    gemm(count, m, d, vec.data(), false, W, false, Vt, threads);
    for (int j = 0; j < count; ++j) {
      const double inv = S[j] > 0 ? 1.0 / S[j] : 0.0;
      for (int i = 0; i < m; ++i) Vt[(size_t)j * m + i] *= inv;
    }
  } else {
    for (int j = 0; j < count; ++j)
      std::memcpy(Vt + (size_t)j * m, &vec[(size_t)j * m], sizeof(double) * m);
    // U = W V / s: U [d x count] = W [d x m] * Vt^T
    gemm(d, count, m, W, false, Vt, true, U, threads);
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < count; ++j) U[(size_t)i * count + j] *= (S[j] > 0 ? 1.0 / S[j] : 0.0);
  }
  return true;
}

bool cholesky(int r, double *A) {
  for (int j = 0; j < r; ++j) {
    double s = A[(size_t)j * r + j];
    for (int k = 0; k < j; ++k) s -= A[(size_t)j * r + k] * A[(size_t)j * r + k];
    if (!(s > 0.0) || !std::isfinite(s)) return false;
    const double ljj = std::sqrt(s);
    A[(size_t)j * r + j] = ljj;
    for (int i = j + 1; i < r; ++i) {
      double t = A[(size_t)i * r + j];
      for (int k = 0; k < j; ++k) t -= A[(size_t)i * r + k] * A[(size_t)j * r + k];
      A[(size_t)i * r + j] = t / ljj;
    }
  }
  return true;
}

void cholesky_solve(int r, const double *L, double *B, int ncols) {
  for (int col = 0; col < ncols; ++col) {
    for (int i = 0; i < r; ++i) {     // L y = b
      double t = B[(size_t)i * ncols + col];
      for (int k = 0; k < i; ++k) t -= L[(size_t)i * r + k] * B[(size_t)k * ncols + col];
      B[(size_t)i * ncols + col] = t / L[(size_t)i * r + i];
    }
    for (int i = r - 1; i >= 0; --i) {  // L^T x = y
      double t = B[(size_t)i * ncols + col];
      for (int k = i + 1; k < r; ++k) t -= L[(size_t)k * r + i] * B[(size_t)k * ncols + col];
      B[(size_t)i * ncols + col] = t / L[(size_t)i * r + i];
    }
  }
}

void lower_transpose_solve(int r, const double *L, double *B, int ncols) {
  for (int col = 0; col < ncols; ++col)
    for (int i = r - 1; i >= 0; --i) {
      double t = B[(size_t)i * ncols + col];
      for (int k = i + 1; k < r; ++k) t -= L[(size_t)k * r + i] * B[(size_t)k * ncols + col];
      B[(size_t)i * ncols + col] = t / L[(size_t)i * r + i];
    }
}

}  // namespace fit
}  // namespace dyra
