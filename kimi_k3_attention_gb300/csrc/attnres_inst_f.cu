// Explicit instantiations: deep banks, N = 13..18 (split shape; with and without the fold).
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_F()
}  // namespace attnres
