// Explicit instantiations: the fused kernel with the fold, add2 present, N = 1..6.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_A()
}  // namespace attnres
