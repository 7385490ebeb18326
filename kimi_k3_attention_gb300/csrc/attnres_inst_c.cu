// Explicit instantiations of the fused kernel: add2 = false, N = 1..6.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_INSTANTIATE(1, false)
ATTNRES_INSTANTIATE(2, false)
ATTNRES_INSTANTIATE(3, false)
ATTNRES_INSTANTIATE(4, false)
ATTNRES_INSTANTIATE(5, false)
ATTNRES_INSTANTIATE(6, false)
}  // namespace attnres
