// Explicit instantiations of the fused kernel: add2 = true, N = 1..6.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_INSTANTIATE(1, true)
ATTNRES_INSTANTIATE(2, true)
ATTNRES_INSTANTIATE(3, true)
ATTNRES_INSTANTIATE(4, true)
ATTNRES_INSTANTIATE(5, true)
ATTNRES_INSTANTIATE(6, true)
}  // namespace attnres
