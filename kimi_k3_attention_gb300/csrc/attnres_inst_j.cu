// Explicit instantiations: FP16 tensors, N = 7..12 (split and streaming shapes; with and without
// the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_J()
}  // namespace attnres
