// Monarch static branch of the bf16 DyRA forward (summary page Appendix B; blog section on
// structured methods: block-diagonal factor, stride permutation, block-diagonal factor).
//
// With nb blocks, W_hat[(a,i),(c,j)] = B1[a][i,c] B2[c][a,j]. The forward computes
//   Z[:, a*nb + c]  = sum_i X[:, a*nb + i] B1[a][i][c]        (block-diagonal, tcgen05)
//   Zp[:, c*nb + a] = Z[:, a*nb + c]                           (stride permutation)
//   Y[:, c*nb + j] += sum_a Zp[:, c*nb + a] B2[c][a][j]       (block-diagonal, tcgen05)
// Supported shapes: square blocks, d = m = nb * nb, nb a multiple of 8 dividing 256, so a
// 256-column tile of either stage contracts with exactly 256 input columns.
#pragma once
#include <cstddef>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dyra {

bool monarch_supported(int d, int m, int nb, int r);

// In place, for every row of T [rows][ldT] (the first nb * nb columns):
// T[row][c * nb + a] <- T[row][a * nb + c]  (the stride permutation between the factors).
cudaError_t launch_monarch_permute(__nv_bfloat16 *T, long long rows, int ldT, int nb,
                                   cudaStream_t s);

}  // namespace dyra
