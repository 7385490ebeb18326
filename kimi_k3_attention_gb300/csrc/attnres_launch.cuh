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

template <int N, int MODE, int VPT, int MAXT, int MINB>
cudaError_t launch_fused(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                         cudaStream_t s) {
  auto kern = attnres_fused_kernel<N, MODE, VPT, MAXT, MINB>;
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

// The persistent pipelined kernel: up to 256 threads, STAGES tokens in the
// shared-memory ring (STAGES - 1 in flight while one is reduced).
constexpr int kPipeMaxT = 256, kPipeMinB = 1;

inline int pipe_rows(int N, bool add2) { return N + (add2 ? 3 : 2); }

inline size_t pipe_smem_bytes(int N, bool add2, int threads, int stages) {
  return static_cast<size_t>(stages) * pipe_rows(N, add2) * threads * 16u;
}

// Launch the pipelined kernel with a grid of grid.y clusters; grid.y == 0
// asks for as many clusters as can be resident at once (capped at M).
template <int N, bool ADD2, int STAGES>
cudaError_t launch_pipe(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                        cudaStream_t s) {
  auto kern = attnres_pipe_kernel<N, ADD2, kPipeMaxT, kPipeMinB, STAGES>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const size_t smem = pipe_smem_bytes(N, ADD2, threads, STAGES);
  // Raise the dynamic shared-memory limit (and opt in to large clusters)
  // once per device; the limit only grows.
  static std::atomic<int> smem_set[kMaxDevices];
  static std::atomic<unsigned char> opted[kMaxDevices];
  if (static_cast<int>(smem) > smem_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    smem_set[dev].store(static_cast<int>(smem), std::memory_order_release);
  }
  if (cluster > 8 && !opted[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    opted[dev].store(1, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
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
  if (grid.y == 0) {
    // Resident clusters for this (threads, cluster, shared memory), cached
    // per device for the last configuration asked.
    static std::atomic<long long> cache[kMaxDevices];
    const long long key = (static_cast<long long>(threads) << 8 | cluster) << 20 | static_cast<long long>(smem >> 4);
    long long c = cache[dev].load(std::memory_order_acquire);
    int clusters = 0;
    if (c != 0 && (c >> 16) == key) {
      clusters = static_cast<int>(c & 0xffff);
    } else {
      cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      if (clusters > 0xffff) clusters = 0xffff;
      cache[dev].store(key << 16 | clusters, std::memory_order_release);
    }
    grid.y = static_cast<unsigned>(clusters < p.M ? clusters : p.M);
  }
  if (grid.y > 65535u) grid.y = 65535u;
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), grid.y, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// The standalone fold over M*H/8 chunks: 256-thread CTAs, at most 8 per SM
// worth of grid (grid-stride beyond that).
template <bool ADD2>
cudaError_t launch_tail_add(const uint4* prefix, const uint4* add, const uint4* add2,
                            uint4* new_prefix, long long chunks, int sms, bool pdl,
                            cudaStream_t s) {
  const long long want = (chunks + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attnres_tail_add_kernel<ADD2>, prefix, add, add2, new_prefix,
                            chunks);
}

#define ATTNRES_INSTANTIATE_PIPE(N, ADD2)                                                    \
  template cudaError_t launch_pipe<N, ADD2, 2>(const Params&, dim3, int, int, bool,          \
                                               cudaStream_t);                                \
  template cudaError_t launch_pipe<N, ADD2, 3>(const Params&, dim3, int, int, bool,          \
                                               cudaStream_t);                                \
  template cudaError_t launch_pipe<N, ADD2, 4>(const Params&, dim3, int, int, bool,          \
                                               cudaStream_t);

#define ATTNRES_INSTANTIATE(N, ADD2)                                                       \
  template cudaError_t launch_fused<N, ADD2 ? kFoldAdd2 : kFoldAdd, kSplitVPT, kSplitMaxT,     \
                                    kSplitMinB>(const Params&, dim3, int, int, bool,         \
                                                cudaStream_t);                               \
  template cudaError_t launch_fused<N, ADD2 ? kFoldAdd2 : kFoldAdd, kStreamVPT, kStreamMaxT,   \
                                    kStreamMinB>(const Params&, dim3, int, int, bool,        \
                                                 cudaStream_t);                              \
  template cudaError_t launch_fused<N, ADD2 ? kFoldAdd2 : kFoldAdd, kCtaVPT, kCtaMaxT,         \
                                    kCtaMinB>(const Params&, dim3, int, int, bool,           \
                                              cudaStream_t);                                 \
  ATTNRES_INSTANTIATE_PIPE(N, ADD2)

// The attention-residual + RMSNorm alone (no fold): split and streaming shapes.
#define ATTNRES_INSTANTIATE_NOFOLD(N)                                                        \
  template cudaError_t launch_fused<N, kNoFold, kSplitVPT, kSplitMaxT, kSplitMinB>(          \
      const Params&, dim3, int, int, bool, cudaStream_t);                                    \
  template cudaError_t launch_fused<N, kNoFold, kStreamVPT, kStreamMaxT, kStreamMinB>(       \
      const Params&, dim3, int, int, bool, cudaStream_t);

}  // namespace attnres
