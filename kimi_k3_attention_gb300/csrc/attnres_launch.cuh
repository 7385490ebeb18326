// Host-side launch of one instantiation of the fused kernel, and the
// explicit-instantiation macro used by the attnres_inst_*.cu units.
#pragma once

#include <atomic>

#include "attnres_kernel.cuh"

namespace attnres {

constexpr int kMaxDevices = 64;

// The compiled shapes of the kernel.
//   split:  8 columns per thread, up to 256 threads (a cluster of CTAs per token)
//   stream: 8 columns per thread, up to 224 threads, registers capped so
//           that three CTAs fit an SM (many tokens in flight at large M)
//   cta:    16 columns per thread, up to 448 threads (one CTA per token)
constexpr int kSplitVPT = 1, kSplitMaxT = 256, kSplitMinB = 1;
constexpr int kStreamVPT = 1, kStreamMaxT = 224, kStreamMinB = 3;
constexpr int kCtaVPT = 2, kCtaMaxT = 448, kCtaMinB = 1;

template <int N, bool ADD2, int VPT, int MAXT, int MINB>
cudaError_t launch_fused(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                         cudaStream_t s) {
  auto kern = attnres_fused_kernel<N, ADD2, VPT, MAXT, MINB>;
  // Cluster sizes above 8 need an opt-in per function and device.
  static std::atomic<unsigned char> opted[kMaxDevices];
  if (cluster > 8) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      opted[dev].store(1, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

#define ATTNRES_INSTANTIATE(N, ADD2)                                                       \
  template cudaError_t launch_fused<N, ADD2, kSplitVPT, kSplitMaxT, kSplitMinB>(             \
      const Params&, dim3, int, int, bool, cudaStream_t);                                    \
  template cudaError_t launch_fused<N, ADD2, kStreamVPT, kStreamMaxT, kStreamMinB>(          \
      const Params&, dim3, int, int, bool, cudaStream_t);                                    \
  template cudaError_t launch_fused<N, ADD2, kCtaVPT, kCtaMaxT, kCtaMinB>(                   \
      const Params&, dim3, int, int, bool, cudaStream_t);

}  // namespace attnres
