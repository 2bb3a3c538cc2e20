// Monarch static branch of the bf16 DyRA forward (W_hat = blockdiag(B1) . stride
// permutation . blockdiag(B2), summary page Appendix B).
#pragma once
#include <cstddef>
#include <string>
#include <cuda_runtime.h>

namespace dyra {

bool monarch_supported(int d, int m, int nb, int r);

}  // namespace dyra
