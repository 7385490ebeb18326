// Explicit instantiations: FP16 tensors, N = 0..6 (split and streaming shapes; with and without
// the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_I()
}  // namespace attnres
