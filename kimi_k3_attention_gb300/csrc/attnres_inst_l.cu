// Explicit instantiations: FP16 tensors with deep banks, N = 13..18 (split
// and deep streaming shapes; with and without the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_L()
}  // namespace attnres
