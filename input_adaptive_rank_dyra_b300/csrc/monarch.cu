// Monarch static branch of the bf16 DyRA forward: the stride permutation between the two
// block-diagonal factors (the factors themselves run on the tcgen05 GEMM engine).
#include "monarch.cuh"
#include "ptx.cuh"

namespace dyra {

namespace {

// One warp per row: lane a reads Z[row][a*nb .. a*nb + nb) (nb contiguous values, the
// warp reads the row coalesced), then for each c the nb lanes write Zp[row][c*nb + a],
// nb consecutive elements. Every lane has read its values before any lane writes.
template <int NB>
__global__ void __launch_bounds__(256) monarch_permute_kernel(__nv_bfloat16 *T, long long rows,
                                                              int ldT) {
  const int lane = threadIdx.x & 31;
  const long long warp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  // the next kernel may start launching (it waits for this grid to finish before reading)
  ptx::pdl_launch_dependents();
  // T comes from the previous kernels of the stream: nothing is read before this wait
  ptx::pdl_wait();
  for (long long row = warp; row < rows; row += nwarps) {
    __nv_bfloat16 *z = T + row * ldT;
    __nv_bfloat16 v[NB];
    if (lane < NB) {
#pragma unroll
      for (int c = 0; c < NB; c += 8) {
        const uint4 w = __ldcg(reinterpret_cast<const uint4 *>(z + lane * NB + c));
        const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&w);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[c + j] = h[j];
      }
    }
    __syncwarp();
    if (lane < NB) {
#pragma unroll
      for (int c = 0; c < NB; ++c) z[c * NB + lane] = v[c];
    }
    __syncwarp();
  }
}

}  // namespace

bool monarch_supported(int d, int m, int nb, int r) {
  if (nb != 8 && nb != 16 && nb != 32) return false;
  if (d != nb * nb || m != nb * nb) return false;
  if (256 % nb) return false;
  if (d % 256) return false;   // whole 256-column tiles in both stages
  return r > 0 && r % 8 == 0 && r <= 256;
}

cudaError_t launch_monarch_permute(__nv_bfloat16 *T, long long rows, int ldT, int nb,
                                   cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (ldT % 8) return cudaErrorInvalidValue;
  long long blocks = (rows + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  // programmatic stream serialization: the kernel may start while the previous one finishes
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (nb) {
    case 8: return cudaLaunchKernelEx(&cfg, monarch_permute_kernel<8>, T, rows, ldT);
    case 16: return cudaLaunchKernelEx(&cfg, monarch_permute_kernel<16>, T, rows, ldT);
    case 32: return cudaLaunchKernelEx(&cfg, monarch_permute_kernel<32>, T, rows, ldT);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dyra
