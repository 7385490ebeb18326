// Explicit instantiations: the fused kernel with the fold, add2 present, N = 7..12.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_B()
}  // namespace attnres
