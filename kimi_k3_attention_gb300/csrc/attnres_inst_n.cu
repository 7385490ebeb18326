// Explicit instantiations: FP16 tensors with deep banks, N = 25..31 (split
// and deep streaming shapes; with and without the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_N()
}  // namespace attnres
