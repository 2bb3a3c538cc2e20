// Monarch static branch of the bf16 DyRA forward.
#include "monarch.cuh"

namespace dyra {

bool monarch_supported(int, int, int, int) { return false; }

}  // namespace dyra
