// Explicit instantiations of the fused kernel: add2 = false, N = 7..12.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_INSTANTIATE(7, false)
ATTNRES_INSTANTIATE(8, false)
ATTNRES_INSTANTIATE(9, false)
ATTNRES_INSTANTIATE(10, false)
ATTNRES_INSTANTIATE(11, false)
ATTNRES_INSTANTIATE(12, false)
}  // namespace attnres
