// Explicit instantiations: deep banks, N = 25..31 (split shape; with and without the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_H()
}  // namespace attnres
