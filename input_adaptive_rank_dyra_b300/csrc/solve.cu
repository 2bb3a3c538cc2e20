// Per-sample SPD solves of the one-step ALS R-update, R = (L^T L + lambda I)^-1 (L^T X) W_res
// ("DyRA" summary page, 2.2 ridge; 2.4: Cholesky for small r, Newton-Schulz for larger r).
//
// The bf16 forward solves before the residual product: C~ = G^-1 C with C = L^T X (read as
// the fp32 C^T [batch, d, r] that the Gram GEMM stores), so that the next GEMM forms
// R = C~ W_res directly and the output GEMM multiplies L itself. The solve then touches r x d values per sample whatever the token
// count.
//   * r <= 64 (the Cholesky branch): spd_invert, one CTA per sample, inverts G + lambda I
//     (padded to R x R, R = 32 or 64, by the identity) in place by block sweeps on 4 x 4
//     pivot blocks -- Gauss-Jordan without pivoting, whose scalar pivots on an SPD matrix are
//     the squared diagonal of the Cholesky factor -- with the matrix spread over the CTA's
//     registers, and stores G^-1 (fp32 and bf16). spd_apply then forms C~ = G^-1 C in fp32 FMA, one CTA per sample and
//     128 columns of C, each thread a 4 x 8 block of the result.
//   * larger r: Newton-Schulz. ns_prep scales G symmetrically to unit diagonal and starts
//     from X0 = I / ||G_hat||_inf. The iteration X <- X (2I - G_hat X) runs in residual
//     form: with E = I - G_hat X (a polynomial in G_hat, like X), X (2I - G_hat X) = X (I + E)
//     and the next residual is E^2; ns_iterate (ns.cu) runs every iteration on tf32 tensor
//     cores and undoes the scaling in one kernel; a tf32 tensor-core GEMM then forms
//     C~ = G^-1 C.
// A sample with a pivot that is not positive (or not finite) is counted in status[0] and
// gets G^-1 = 0 and C~ = 0, so its correction vanishes and its output is the static branch
// plus bias.
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <mutex>

namespace dyra {

namespace {

constexpr int kSolveCols = 128;   // columns of C per spd_apply CTA

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
// whose scalar pivots are the squared diagonal of the Cholesky factor), one CTA per sample.
// With K the pivot block, P = A_KK^-1 and S_i = A_iK P, one block sweep is
//   A_ij -= S_i A_Kj  (i, j outside K),  A_iK = S_i,  A_Kj = P A_Kj,  A_KK = -P,
// and after the sweeps over all blocks the matrix holds -(G + ridge I)^-1 (the identity
// padding up to R x R is never swept). Each of (R/4)^2 threads keeps one 4 x 4 block in
// registers. The pivot columns of the next step (rows of 4, = its pivot rows by symmetry) and
// the inverse of its pivot block, which the owner of that block forms after its update, go
// through double-buffered shared memory: one barrier per step, r / 4 steps. The inverse goes
// to Ginv32 (fp32, read by spd_apply) and Ginv (bf16).
template <int R>
__global__ void __launch_bounds__((R / 4) * (R / 4))
    spd_invert_kernel(const float *__restrict__ G, int r, float ridge,
                      float *__restrict__ Ginv32, __nv_bfloat16 *__restrict__ Ginv, int *status) {
  constexpr int Q = R / 4;   // 4 x 4 blocks per side; one thread per block
  __shared__ __align__(16) float colbuf[2][R][4];   // the step's pivot columns A_iK
  __shared__ __align__(16) float pinv[2][4][4];     // P of the step
  __shared__ int bad_s;
  const int tid = threadIdx.x, b = blockIdx.x;
  const int i0 = (tid / Q) * 4, j0 = (tid % Q) * 4;
  // G comes from the previous kernel of the stream: nothing is read before this wait
  ptx::pdl_wait();
  float a[4][4];
  {
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
  if (j0 == 0) {
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
    {
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
  if (i0 < r && j0 < r) {   // r % 4 == 0: a block is inside r x r or outside it
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t row = (size_t)b * r * r + (size_t)(i0 + u) * r + j0;
      const float4 o = bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                           : make_float4(-a[u][0], -a[u][1], -a[u][2], -a[u][3]);
      *reinterpret_cast<float4 *>(Ginv32 + row) = o;
      Ginv[row] = __float2bfloat16_rn(o.x);
      Ginv[row + 1] = __float2bfloat16_rn(o.y);
      Ginv[row + 2] = __float2bfloat16_rn(o.z);
      Ginv[row + 3] = __float2bfloat16_rn(o.w);
    }
  }
  if (tid == 0 && bad) atomicAdd(status, 1);
  // the apply kernel may launch now (it waits for this grid to complete before reading)
  ptx::pdl_launch_dependents();
}

// Threads of spd_apply for the padded size R: R / 4 row groups x 16 column groups.
template <int R>
__host__ __device__ constexpr int apply_threads() { return (R / 4) * 16; }

template <int R>
__host__ __device__ constexpr uint32_t apply_smem() {
  return (uint32_t)(R * R + R * (kSolveCols + 4)) * 4u;
}

// C~ = G^-1 C for kSolveCols columns of one sample, fp32 FMA. G^-1 (fp32, from spd_invert;
// symmetric, so its row j is its column j) and the sample's C tile (read from the fp32
// C^T [batch, d, r] rows and transposed to [r][kSolveCols]) are staged in shared memory.
// Thread (ty, tx) forms rows 4 ty .. 4 ty + 3 and columns 8 tx .. 8 tx + 7 of the tile: each
// step over j reads 4 values of G^-1 and 8 of C (three 16-byte loads) for 32 FMAs. C~ is
// stored bf16 [batch, r, d] (rows of the next GEMM's K-major A operand), 16 bytes per row
// and thread.
template <int R>
__global__ void __launch_bounds__(apply_threads<R>())
    spd_apply_kernel(const float *__restrict__ Ginv32, int r, const float *__restrict__ Ct, int d,
                     __nv_bfloat16 *__restrict__ Cs) {
  constexpr int NT = apply_threads<R>();
  constexpr int LDC = kSolveCols + 4;   // row pitch of the transposed C tile (floats)
  extern __shared__ __align__(16) float apply_sm[];
  float *Gi = apply_sm;                 // [R][R]
  float *Ct_s = apply_sm + R * R;       // [R][LDC]: Ct_s[j][c] = C[j][col0 + c]
  const int tid = threadIdx.x, b = blockIdx.y;
  const int col0 = blockIdx.x * kSolveCols;
  // G^-1 and C come from earlier kernels of the stream: nothing is read before this wait
  ptx::pdl_wait();
  {
    // every load is issued before the first shared-memory store (one round trip)
    constexpr int GN = R * R / 4 / NT, CN = kSolveCols * (R / 4) / NT;
    const float *gi = Ginv32 + (size_t)b * r * r;
    float4 gv[GN];
#pragma unroll
    for (int k = 0; k < GN; ++k) {
      const int t = tid + k * NT, i = (4 * t) / R, j = (4 * t) % R;
      gv[k] = (i < r && j < r) ? __ldg(reinterpret_cast<const float4 *>(gi + (size_t)i * r + j))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // thread t takes column c = t % 128 and rows 4 (t / 128) .. + 3 of C, per pass
    const float *cp = Ct + (size_t)b * d * r;
    float4 cv[CN];
#pragma unroll
    for (int k = 0; k < CN; ++k) {
      const int t = tid + k * NT, cc = t % kSolveCols, j4 = 4 * (t / kSolveCols);
      const int col = col0 + cc;
      cv[k] = (col < d && j4 < r) ? __ldg(reinterpret_cast<const float4 *>(cp + (size_t)col * r + j4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < GN; ++k) {
      const int t = tid + k * NT, i = (4 * t) / R, j = (4 * t) % R;
      *reinterpret_cast<float4 *>(Gi + i * R + j) = gv[k];
    }
#pragma unroll
    for (int k = 0; k < CN; ++k) {
      const int t = tid + k * NT, cc = t % kSolveCols, j4 = 4 * (t / kSolveCols);
      Ct_s[(j4 + 0) * LDC + cc] = cv[k].x;
      Ct_s[(j4 + 1) * LDC + cc] = cv[k].y;
      Ct_s[(j4 + 2) * LDC + cc] = cv[k].z;
      Ct_s[(j4 + 3) * LDC + cc] = cv[k].w;
    }
  }
  __syncthreads();
  ptx::pdl_launch_dependents();
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][8];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[u][v] = 0.f;
#pragma unroll 4
  for (int j = 0; j < R; ++j) {
    const float4 g = *reinterpret_cast<const float4 *>(Gi + j * R + 4 * ty);
    const float4 c0 = *reinterpret_cast<const float4 *>(Ct_s + j * LDC + 8 * tx);
    const float4 c1 = *reinterpret_cast<const float4 *>(Ct_s + j * LDC + 8 * tx + 4);
    const float gv[4] = {g.x, g.y, g.z, g.w};
    const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(gv[u], cv[v], acc[u][v]);
  }
  const int cbase = col0 + 8 * tx;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = 4 * ty + u;
    if (i >= r) continue;
    __nv_bfloat16 *op = Cs + ((size_t)b * r + i) * d + cbase;
    if (cbase + 8 <= d) {   // d % 8 == 0: 16-byte aligned
      uint4 w;
      __nv_bfloat162 h;
      h = __floats2bfloat162_rn(acc[u][0], acc[u][1]); w.x = *reinterpret_cast<uint32_t *>(&h);
      h = __floats2bfloat162_rn(acc[u][2], acc[u][3]); w.y = *reinterpret_cast<uint32_t *>(&h);
      h = __floats2bfloat162_rn(acc[u][4], acc[u][5]); w.z = *reinterpret_cast<uint32_t *>(&h);
      h = __floats2bfloat162_rn(acc[u][6], acc[u][7]); w.w = *reinterpret_cast<uint32_t *>(&h);
      *reinterpret_cast<uint4 *>(op) = w;
    } else {
#pragma unroll
      for (int v = 0; v < 8; ++v)
        if (cbase + v < d) op[v] = __float2bfloat16_rn(acc[u][v]);
    }
  }
}

// Newton-Schulz start. A sample's r x r matrix is spread over a cluster of ceil(r / 32)
// CTAs of 32 warps: warp w of CTA c owns row 32 c + w, lane l the columns l, l + 32, ...
// (at most kNsPer values per thread, all loaded before any is used). The row-sum maximum
// goes through each CTA's shared memory and is read by the whole cluster through
// distributed shared memory.
constexpr int kNsThreads = 1024;
constexpr int kNsPer = 8;   // columns per lane: r <= 32 * kNsPer

__device__ __forceinline__ float ld_cluster_f32(const float *p, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];"
               : "=f"(v)
               : "r"(ptx::mapa_shared(ptx::smem_u32(p), rank))
               : "memory");
  return v;
}

// Jacobi scaling and start of Newton-Schulz in residual form: dinv = diag(G + lambda I)^-1/2,
// G_hat = D (G + lambda I) D, alpha = 1 / max_i sum_j |G_hat_ij| (the max taken over the
// cluster in a fixed order, so alpha is deterministic), and the iterate
// EX[b] = [E0 ; X0 ; Y0] = [I - alpha G_hat ; alpha I ; 2I - alpha G_hat] ([3r][r], fp32).
// A sample whose diagonal is not positive and finite gets alpha = 0: E0 = I and X0 = 0, so
// every iterate and its G^-1 stay 0.
__global__ void __launch_bounds__(kNsThreads)
    ns_prep_kernel(const float *__restrict__ G, int r, float ridge, float *__restrict__ EX,
                   float *__restrict__ dinv, int *__restrict__ flags) {
  __shared__ float sd[32 * kNsPer];
  __shared__ float red[32];
  __shared__ float cmax;
  const int c = blockIdx.x, b = blockIdx.y, nc = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = 32 * c + warp;   // this warp's row
  const float *g = G + (size_t)b * r * r;
  float v[kNsPer];
#pragma unroll
  for (int q = 0; q < kNsPer; ++q) {
    const int j = lane + 32 * q;
    v[q] = (i < r && j < r) ? __ldg(g + (size_t)i * r + j) : 0.f;
  }
  bool bad = false;
  if (tid < r) {
    const float gii = __ldg(g + (size_t)tid * r + tid) + ridge;
    bad = !(gii > 0.f && gii < INFINITY);
    sd[tid] = bad ? 0.f : rsqrtf(gii);
  }
  bad = __syncthreads_or(bad) != 0;   // every CTA of the sample sees the whole diagonal
  float rs = 0.f;
#pragma unroll
  for (int q = 0; q < kNsPer; ++q) {
    const int j = lane + 32 * q;
    float x = 0.f;
    if (i < r && j < r && !bad) x = (v[q] + (i == j ? ridge : 0.f)) * sd[i] * sd[j];
    v[q] = x;
    rs += fabsf(x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
  if (lane == 0) red[warp] = rs;
  __syncthreads();
  if (warp == 0) {
    float m = red[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) cmax = m;
  }
  ptx::cluster_sync_all();   // every CTA's cmax is written
  if (tid == 0) {
    float m = 0.f;
    for (int k = 0; k < nc; ++k) m = fmaxf(m, ld_cluster_f32(&cmax, (uint32_t)k));
    red[0] = m;
  }
  ptx::cluster_sync_all();   // no CTA leaves while a peer may still read its cmax
  const float alpha = (bad || !(red[0] > 0.f)) ? 0.f : 1.f / red[0];
  if (i < r) {
    float *E = EX + (size_t)b * 3 * r * r, *X = E + (size_t)r * r, *Y = X + (size_t)r * r;
#pragma unroll
    for (int q = 0; q < kNsPer; ++q) {
      const int j = lane + 32 * q;
      if (j < r) {
        const float e = (i == j ? 1.f : 0.f) - alpha * v[q];
        E[(size_t)i * r + j] = e;
        X[(size_t)i * r + j] = (i == j) ? alpha : 0.f;
        Y[(size_t)i * r + j] = (i == j ? 1.f : 0.f) + e;
      }
    }
  }
  if (c == 0 && tid < r) dinv[(size_t)b * r + tid] = bad ? 0.f : sd[tid];
  if (c == 0 && tid == 0) flags[b] = bad ? 1 : 0;
}

}  // namespace

namespace {

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel of the stream finishes; it reads nothing before its griddepcontrol.wait.
template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, uint32_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_spd_invert(const float *G, int batch, int r, float ridge, float *Ginv32,
                              __nv_bfloat16 *Ginv, int *status, cudaStream_t s) {
  if (r <= 0 || r > 64 || r % 4) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  if (r <= 32)
    return launch_pdl(spd_invert_kernel<32>, dim3(batch), dim3(64), 0u, s, G, r, ridge, Ginv32,
                      Ginv, status);
  return launch_pdl(spd_invert_kernel<64>, dim3(batch), dim3(256), 0u, s, G, r, ridge, Ginv32,
                    Ginv, status);
}

cudaError_t launch_spd_apply(const float *Ginv32, int batch, int r, const float *Ct, int d,
                             __nv_bfloat16 *Cs, cudaStream_t s) {
  if (r <= 0 || r > 64 || r % 4 || d <= 0) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  if (d % 8) return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(spd_apply_kernel<32>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)apply_smem<32>());
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(spd_apply_kernel<64>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)apply_smem<64>());
  });
  if (attr_err != cudaSuccess) return attr_err;
  const dim3 grid((d + kSolveCols - 1) / kSolveCols, batch);
  if (r <= 32)
    return launch_pdl(spd_apply_kernel<32>, grid, dim3(apply_threads<32>()), apply_smem<32>(), s,
                      Ginv32, r, Ct, d, Cs);
  return launch_pdl(spd_apply_kernel<64>, grid, dim3(apply_threads<64>()), apply_smem<64>(), s,
                    Ginv32, r, Ct, d, Cs);
}

namespace {

// Launch configuration of the Newton-Schulz helpers: a cluster of ceil(r / 32) CTAs per sample.
cudaLaunchConfig_t ns_config(int batch, int r, cudaStream_t s, cudaLaunchAttribute *attr) {
  const unsigned nc = (unsigned)((r + 31) / 32);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc, (unsigned)batch, 1);
  cfg.blockDim = dim3(kNsThreads, 1, 1);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_ns_prep(const float *G, int batch, int r, float ridge, float *EX, float *dinv,
                           int *flags, cudaStream_t s) {
  if (r <= 0 || r > 32 * kNsPer) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = ns_config(batch, r, s, attr);
  return cudaLaunchKernelEx(&cfg, ns_prep_kernel, G, r, ridge, EX, dinv, flags);
}


}  // namespace dyra
