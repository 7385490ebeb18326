// Explicit instantiations of the fused kernel: add2 = true, N = 7..12.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_INSTANTIATE(7, true)
ATTNRES_INSTANTIATE(8, true)
ATTNRES_INSTANTIATE(9, true)
ATTNRES_INSTANTIATE(10, true)
ATTNRES_INSTANTIATE(11, true)
ATTNRES_INSTANTIATE(12, true)
}  // namespace attnres
