// Explicit instantiations: the fused kernel with the fold, add2 absent, N = 1..6.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_C()
}  // namespace attnres
