// Explicit instantiations: the fused kernel with the fold, add2 absent, N = 7..12.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_D()
}  // namespace attnres
