// Explicit instantiations: deep banks, N = 19..24 (split shape; with and without the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_G()
}  // namespace attnres
