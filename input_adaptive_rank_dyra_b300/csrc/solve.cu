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
//     registers, and stores G^-1 (fp32 and bf16). The R-update of the forward runs the same sweeps in the epilogue of
//     its Gram GEMM; this kernel serves the L-update of further ALS iterations. spd_apply then forms C~ = G^-1 C in fp32 FMA, one CTA per sample and
//     128 columns of C, each thread a 4 x 8 block of the result.
//   * larger r: Newton-Schulz (ns.cu): one cluster kernel scales G symmetrically to unit
//     diagonal, starts from X0 = I / ||G_hat||_inf and runs X <- X (2I - G_hat X) in
//     residual form (E = I - G_hat X, X' = X + X E, E' = E E) on tf32 tensor cores, then
//     undoes the scaling; a tf32 tensor-core GEMM then forms C~ = G^-1 C.
// A sample with a pivot that is not positive (or not finite) is counted in status[0] and
// gets G^-1 = 0 and C~ = 0, so its correction vanishes and its output is the static branch
// plus bias.
#include "kernels.cuh"
#include "ptx.cuh"
#include "sweep.cuh"

#include <cuda_bf16.h>
#include <mutex>

namespace dyra {

namespace {

constexpr int kSolveCols = 128;   // columns of C per spd_apply CTA

// (G + ridge I)^-1 for one sample, one CTA of (R/4)^2 threads: the block sweeps of
// sweep::invert_blocks with the matrix in registers, one barrier per 4 x 4 pivot block. The
// inverse goes to Ginv32 (fp32, read by spd_apply) and Ginv (bf16).
template <int R>
__global__ void __launch_bounds__((R / 4) * (R / 4))
    spd_invert_kernel(const float *__restrict__ G, int r, float ridge,
                      float *__restrict__ Ginv32, __nv_bfloat16 *__restrict__ Ginv, int *status) {
  constexpr int Q = R / 4;
  __shared__ sweep::Smem<R> sm;
  const int tid = threadIdx.x, b = blockIdx.x;
  const int i0 = (tid / Q) * 4, j0 = (tid % Q) * 4;
  // the apply kernel may start launching (it waits for this grid to finish before reading)
  ptx::pdl_launch_dependents();
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
        a[u][v] = (i < r && j < r) ? __ldcg(g + (size_t)i * r + j) + (i == j ? ridge : 0.f)
                                   : (i == j ? 1.f : 0.f);
      }
  }
  const bool bad = !sweep::invert_blocks<R>(a, tid, r, sm, []() { __syncthreads(); });
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
  // the next kernel may start launching (it waits for this grid to finish before reading)
  ptx::pdl_launch_dependents();
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
      gv[k] = (i < r && j < r) ? __ldcg(reinterpret_cast<const float4 *>(gi + (size_t)i * r + j))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // thread t takes column c = t % 128 and rows 4 (t / 128) .. + 3 of C, per pass
    const float *cp = Ct + (size_t)b * d * r;
    float4 cv[CN];
#pragma unroll
    for (int k = 0; k < CN; ++k) {
      const int t = tid + k * NT, cc = t % kSolveCols, j4 = 4 * (t / kSolveCols);
      const int col = col0 + cc;
      cv[k] = (col < d && j4 < r) ? __ldcg(reinterpret_cast<const float4 *>(cp + (size_t)col * r + j4))
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

}  // namespace dyra
