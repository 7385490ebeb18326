// Explicit instantiations: N = 0 with the fold (every shape; with no
// snapshots yet the mixture has the prefix as its only source), the
// attention-residual + RMSNorm alone for N = 0..12, and the standalone fold
// kernel.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_UNIT_E()
}  // namespace attnres
