// Explicit instantiations of the attention-residual + RMSNorm alone (no
// fold), N = 0..12, of every variant at N = 0 (no snapshots yet: the mixture
// has the prefix as its only source), and of the standalone fold kernel.
#include "attnres_launch.cuh"

namespace attnres {
ATTNRES_INSTANTIATE(0, true)
ATTNRES_INSTANTIATE(0, false)
ATTNRES_INSTANTIATE_NOFOLD(0)
ATTNRES_INSTANTIATE_NOFOLD(1)
ATTNRES_INSTANTIATE_NOFOLD(2)
ATTNRES_INSTANTIATE_NOFOLD(3)
ATTNRES_INSTANTIATE_NOFOLD(4)
ATTNRES_INSTANTIATE_NOFOLD(5)
ATTNRES_INSTANTIATE_NOFOLD(6)
ATTNRES_INSTANTIATE_NOFOLD(7)
ATTNRES_INSTANTIATE_NOFOLD(8)
ATTNRES_INSTANTIATE_NOFOLD(9)
ATTNRES_INSTANTIATE_NOFOLD(10)
ATTNRES_INSTANTIATE_NOFOLD(11)
ATTNRES_INSTANTIATE_NOFOLD(12)
template cudaError_t launch_tail_add<true>(const uint4*, const uint4*, const uint4*, uint4*,
                                           long long, int, bool, cudaStream_t);
template cudaError_t launch_tail_add<false>(const uint4*, const uint4*, const uint4*, uint4*,
                                            long long, int, bool, cudaStream_t);
}  // namespace attnres
