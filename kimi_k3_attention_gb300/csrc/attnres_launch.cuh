// Host-side launch of one instantiation of the fused kernel, and the
// explicit-instantiation macro used by the attnres_inst_*.cu units.
#pragma once

#include <atomic>
#include <cmath>

#include "attnres_kernel.cuh"

namespace attnres {

constexpr int kMaxDevices = 64;

// The compiled shapes of the kernel.
//   split:  8 columns per thread, up to 256 threads (a cluster of CTAs per token)
//   stream: 8 columns per thread, up to 224 threads, registers capped so
//           that several CTAs fit an SM (many tokens in flight at large M;
//           stream_minb); deep banks have their own streaming shape (below)
//   cta:    16 columns per thread, up to 448 threads (one CTA per token)
constexpr int kSplitVPT = 1, kSplitMaxT = 256, kSplitMinB = 1;
// split2: the split shape with registers capped so that two CTAs of up to
// 256 threads share an SM (the next call's CTAs can be resident while this
// call runs, under programmatic dependent launch)
constexpr int kSplit2MinB = 2;
constexpr int kStreamVPT = 1, kStreamMaxT = 224;
// The streaming shape's registers and where a token's rows live.  With R
// rows per token (bank, prefix and addends: stream_rows), registers are
// capped at 56 (five CTAs of 224 threads, nine of 128, per SM) up to 6 rows
// and at 72 (four of 224, seven of 128) beyond, and up to 11 rows stay in
// registers, 11 of 12-13 and 12 of 14-15: the bank rows past that are
// copied into the thread's own slots of shared memory (HybridSources), which
// keeps the register allocation free of spills.  GB300, M = 8192, add2,
// against every row in registers at 72 registers (80 from 13 rows on): N = 1
// +5 %, N = 3 +4 %, N = 9 +1 %, N = 10 +3 %, N = 11 +1 %, N = 12 +2 %
// (6.71-6.73 TB/s, about the copy peak); 56 registers beyond 6 rows and
// fewer rows in registers spilled or lost 1-35 %.
constexpr int stream_rows(int n, int mode) {
  return n + (mode == kFoldAdd2 ? 3 : mode == kFoldAdd ? 2 : 1);
}
constexpr int stream_reg_rows(int r) { return r <= 11 ? r : r <= 13 ? 11 : 12; }
constexpr int stream_minb(int n, int mode) { return stream_rows(n, mode) <= 6 ? 5 : 4; }
constexpr int stream_nr(int n, int mode) {
  return n - (stream_rows(n, mode) - stream_reg_rows(stream_rows(n, mode)));
}
// Dispatch's MINB for the streaming shape: stream_minb and stream_nr of each
// (N, mode); the other shapes keep every row in registers.
constexpr int kStreamMinB = 0;
constexpr int minb_of(int minb, int n, int mode) { return minb != 0 ? minb : stream_minb(n, mode); }
constexpr int nr_of(int minb, int n, int mode) { return minb != 0 ? n : stream_nr(n, mode); }
constexpr int kCtaVPT = 2, kCtaMaxT = 448, kCtaMinB = 1;

// Every shape is compiled for N <= kShallowMaxN.  Deeper banks (up to
// ATTNRES_MAX_N) have the split shape and a streaming shape of their own:
// up to 128 threads, registers capped so that deep_minb(N) CTAs share an SM,
// and bank rows deep_nr(N)..N-1 held in shared memory instead of registers.
// GB300, M = 8192, swept per N over the cap (4-8 CTAs per SM) and the rows
// kept in registers (4..N): up to 14 snapshots every row in registers at
// 96 registers (5 CTAs); 15..17 snapshots rows 14.. in shared memory at 96
// registers (N = 16: 5.75 TB/s against 5.28 with every row in registers and
// 5.45 with rows 8.. and 7 CTAs; N = 17: 5.77 against 5.54); 18..22 every row
// in registers at 128 registers (4 CTAs; 96 registers spill 20-36 bytes and
// lose 3-7 %); from 23 on rows 16.. in shared memory at 128 registers.
// 4.9-6.5 TB/s over N = 13..31, against 3.3-4.1 TB/s uncapped.
constexpr int kDeepStreamMaxT = 128;
constexpr int deep_minb(int n) { return n <= 17 ? 5 : 4; }
constexpr int deep_nr(int n) { return (n >= 15 && n <= 17) ? 14 : n >= 23 ? 16 : n; }

// Clusters that fit the device at once for launch configuration cfg (its
// block size, dynamic shared memory and cluster attribute), cached per
// device for the last (threads, cluster, shared memory) asked.
template <class Kern>
cudaError_t resident_clusters(Kern kern, cudaLaunchConfig_t cfg, int dev, int cluster,
                              std::atomic<long long>* cache, int* clusters) {
  const long long key = (static_cast<long long>(cfg.blockDim.x) << 8 | cluster) << 20 |
                        static_cast<long long>(cfg.dynamicSmemBytes >> 4);
  const long long c = cache[dev].load(std::memory_order_acquire);
  if (c != 0 && (c >> 16) == key) {
    *clusters = static_cast<int>(c & 0xffff);
    return cudaSuccess;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (n > 0xffff) n = 0xffff;
  cache[dev].store(key << 16 | n, std::memory_order_release);
  *clusters = n;
  return cudaSuccess;
}

// The automatic grid of a walk over M tokens when R clusters fit the GPU at
// once (grid_tokens 0 for the streaming shapes).  Walking clusters take about
// L = sqrt(2 M / R) tokens each and the last T = R L / 2 clusters one token
// each (TokenWalk).  Clusters start in grid order as slots free up, so the
// walks end spread over about L tokens' time, and the T one-token clusters,
// started last, fill the slots that finish early.  Every cluster costs a
// start (its first token is not prefetched): L minimises the clusters per
// slot, M / (L R) + L / 2.  GB300, N = 12, against 10 clusters per SM each
// walking an equal share (one cluster per token below 1520 tokens): +2 % at
// M = 8192 and 16384, +5 % at 4096, +7..11 % at 256..2048; every cell of a
// sweep of (M - T) / L and T around this choice within 1 % of the best.
// L < 2: one cluster per token.
inline void walk_grid(int M, int R, unsigned* gy, int* tail) {
  const long long L = std::llround(std::sqrt(2.0 * M / (R > 0 ? R : 1)));
  if (L < 2) {
    *gy = static_cast<unsigned>(M < 65535 ? M : 65535);
    *tail = 0;
    return;
  }
  long long T = (static_cast<long long>(R) * L + 1) / 2;
  if (T > M / 2) T = M / 2;
  if (T > 32767) T = 32767;
  long long walkers = (M - T + L - 1) / L;
  if (walkers + T > 65535) walkers = 65535 - T;
  *gy = static_cast<unsigned>(walkers + T);
  *tail = static_cast<int>(T);
}

// The launch parameters of TokenWalk for a grid of gy clusters (p.tail set,
// 0 <= tail < gy <= M when tail > 0).
inline void set_walk(Params& p, unsigned gy) {
  p.walkers = static_cast<int>(gy) - p.tail;
  p.walk_end = p.M - p.tail;
}

template <int N, int MODE, int VPT, int MAXT, int MINB, int DT, int NR>
cudaError_t launch_fused(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                         cudaStream_t s) {
  auto kern = attnres_fused_kernel<N, MODE, VPT, MAXT, MINB, DT, NR>;
  // Cluster sizes above 8 need an opt-in per function and device, and so
  // does dynamic shared memory above the default limit (the limit set only
  // grows).
  static std::atomic<unsigned char> opted[kMaxDevices];
  static std::atomic<int> smem_set[kMaxDevices];
  const int dyn = (N - NR) * threads * 16;
  if (cluster > 8 || dyn > 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (cluster > 8 && !opted[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      opted[dev].store(1, std::memory_order_release);
    }
    if (dyn > smem_set[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
      if (e != cudaSuccess) return e;
      smem_set[dev].store(dyn, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  // bank rows NR..N-1 in shared memory
  cfg.dynamicSmemBytes = static_cast<size_t>(N - NR) * threads * 16u;
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
  Params q = p;
  if (grid.y == 0) {
    // size the walk from the clusters that fit at once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    static std::atomic<long long> cache[kMaxDevices];
    int clusters = 0;
    e = resident_clusters(kern, cfg, dev, cluster, cache, &clusters);
    if (e != cudaSuccess) return e;
    walk_grid(p.M, clusters, &cfg.gridDim.y, &q.tail);
  }
  set_walk(q, cfg.gridDim.y);
  return cudaLaunchKernelEx(&cfg, kern, q);
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
    static std::atomic<long long> cache[kMaxDevices];
    int clusters = 0;
    e = resident_clusters(kern, cfg, dev, cluster, cache, &clusters);
    if (e != cudaSuccess) return e;
    grid.y = static_cast<unsigned>(clusters < p.M ? clusters : p.M);
  }
  if (grid.y > 65535u) grid.y = 65535u;
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), grid.y, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// The standalone fold over M*H/8 chunks: 256-thread CTAs, at most 8 per SM
// worth of grid (grid-stride beyond that).
template <bool ADD2, int DT>
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
  return cudaLaunchKernelEx(&cfg, attnres_tail_add_kernel<ADD2, DT>, prefix, add, add2, new_prefix,
                            chunks);
}

// The access-pattern kernel: one thread per chunk of the CTA's columns, a
// cluster of `cluster` CTAs per token, grid.y clusters walking the tokens.
template <int N>
cudaError_t launch_pattern(const Params& p, dim3 grid, int threads, int cluster, cudaStream_t s) {
  auto kern = attnres_pattern_kernel<N>;
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
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  Params q = p;
  if (grid.y == 0) {
    // the fused kernel's automatic walk, sized for this kernel
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    static std::atomic<long long> cache[kMaxDevices];
    int clusters = 0;
    e = resident_clusters(kern, cfg, dev, cluster, cache, &clusters);
    if (e != cudaSuccess) return e;
    walk_grid(p.M, clusters, &cfg.gridDim.y, &q.tail);
  }
  set_walk(q, cfg.gridDim.y);
  return cudaLaunchKernelEx(&cfg, kern, q);
}

// Instantiations.  Each attnres_inst_*.cu unit expands its share with DEF
// empty (explicit instantiation definitions, where the kernels are
// compiled); the API unit expands all of them with DEF = extern, so that it
// compiles no kernel itself.
#define ATTNRES_FUSED(DEF, N, MODE, VPT, MAXT, MINB)                                      \
  DEF template cudaError_t launch_fused<N, MODE, VPT, MAXT, MINB>(const Params&, dim3, int, \
                                                                  int, bool, cudaStream_t);

#define ATTNRES_FUSED_DT(DEF, N, MODE, VPT, MAXT, MINB, DT)                                \
  DEF template cudaError_t launch_fused<N, MODE, VPT, MAXT, MINB, DT>(const Params&, dim3, int, \
                                                                      int, bool, cudaStream_t);

#define ATTNRES_FUSED_NR(DEF, N, MODE, VPT, MAXT, MINB, DT, NR)                              \
  DEF template cudaError_t launch_fused<N, MODE, VPT, MAXT, MINB, DT, NR>(                      \
      const Params&, dim3, int, int, bool, cudaStream_t);

#define ATTNRES_PIPE(DEF, N, ADD2, STAGES)                                          \
  DEF template cudaError_t launch_pipe<N, ADD2, STAGES>(const Params&, dim3, int, int, bool, \
                                                        cudaStream_t);

// N <= 12 with the fold (add2 present or not): every shape.
#define ATTNRES_INSTANTIATE(DEF, N, ADD2)                                                   \
  ATTNRES_FUSED(DEF, N, ADD2 ? kFoldAdd2 : kFoldAdd, kSplitVPT, kSplitMaxT, kSplitMinB)     \
  ATTNRES_FUSED(DEF, N, ADD2 ? kFoldAdd2 : kFoldAdd, kSplitVPT, kSplitMaxT, kSplit2MinB)    \
  ATTNRES_FUSED_NR(DEF, N, ADD2 ? kFoldAdd2 : kFoldAdd, kStreamVPT, kStreamMaxT,           \
                   stream_minb(N, ADD2 ? kFoldAdd2 : kFoldAdd), kBF16,                      \
                   stream_nr(N, ADD2 ? kFoldAdd2 : kFoldAdd))                               \
  ATTNRES_FUSED(DEF, N, ADD2 ? kFoldAdd2 : kFoldAdd, kCtaVPT, kCtaMaxT, kCtaMinB)           \
  ATTNRES_PIPE(DEF, N, ADD2, 2)                                                             \
  ATTNRES_PIPE(DEF, N, ADD2, 3)                                                             \
  ATTNRES_PIPE(DEF, N, ADD2, 4)

// The attention-residual + RMSNorm alone (no fold), N <= 12: split and
// streaming shapes.
#define ATTNRES_INSTANTIATE_NOFOLD(DEF, N)                               \
  ATTNRES_FUSED(DEF, N, kNoFold, kSplitVPT, kSplitMaxT, kSplitMinB)      \
  ATTNRES_FUSED_NR(DEF, N, kNoFold, kStreamVPT, kStreamMaxT, stream_minb(N, kNoFold), kBF16, \
                   stream_nr(N, kNoFold))

// Deep banks, 13 <= N <= 31: the split shape and the deep streaming shape,
// with the fold (add2 present or not) and without, for element format DT.
#define ATTNRES_INSTANTIATE_DEEP_DT(DEF, N, DT)                                               \
  ATTNRES_FUSED_DT(DEF, N, kFoldAdd2, kSplitVPT, kSplitMaxT, kSplitMinB, DT)                  \
  ATTNRES_FUSED_DT(DEF, N, kFoldAdd, kSplitVPT, kSplitMaxT, kSplitMinB, DT)                   \
  ATTNRES_FUSED_DT(DEF, N, kNoFold, kSplitVPT, kSplitMaxT, kSplitMinB, DT)                    \
  ATTNRES_FUSED_NR(DEF, N, kFoldAdd2, kStreamVPT, kDeepStreamMaxT, deep_minb(N), DT, deep_nr(N)) \
  ATTNRES_FUSED_NR(DEF, N, kFoldAdd, kStreamVPT, kDeepStreamMaxT, deep_minb(N), DT, deep_nr(N))  \
  ATTNRES_FUSED_NR(DEF, N, kNoFold, kStreamVPT, kDeepStreamMaxT, deep_minb(N), DT, deep_nr(N))
#define ATTNRES_INSTANTIATE_DEEP(DEF, N) ATTNRES_INSTANTIATE_DEEP_DT(DEF, N, kBF16)
#define ATTNRES_INSTANTIATE_DEEP_FP16(DEF, N) ATTNRES_INSTANTIATE_DEEP_DT(DEF, N, kFP16)

// FP16 tensors, N <= 12: the split and streaming shapes, with the fold
// (add2 present or not) and without.
#define ATTNRES_INSTANTIATE_FP16(DEF, N)                                               \
  ATTNRES_FUSED_DT(DEF, N, kFoldAdd2, kSplitVPT, kSplitMaxT, kSplitMinB, kFP16)        \
  ATTNRES_FUSED_DT(DEF, N, kFoldAdd, kSplitVPT, kSplitMaxT, kSplitMinB, kFP16)         \
  ATTNRES_FUSED_DT(DEF, N, kNoFold, kSplitVPT, kSplitMaxT, kSplitMinB, kFP16)          \
  ATTNRES_FUSED_NR(DEF, N, kFoldAdd2, kStreamVPT, kStreamMaxT, stream_minb(N, kFoldAdd2), kFP16, \
                   stream_nr(N, kFoldAdd2))                                                  \
  ATTNRES_FUSED_NR(DEF, N, kFoldAdd, kStreamVPT, kStreamMaxT, stream_minb(N, kFoldAdd), kFP16,   \
                   stream_nr(N, kFoldAdd))                                                   \
  ATTNRES_FUSED_NR(DEF, N, kNoFold, kStreamVPT, kStreamMaxT, stream_minb(N, kNoFold), kFP16,     \
                   stream_nr(N, kNoFold))

#define ATTNRES_TAIL_ADD(DEF, ADD2, DT)                                                      \
  DEF template cudaError_t launch_tail_add<ADD2, DT>(const uint4*, const uint4*, const uint4*,  \
                                                     uint4*, long long, int, bool, cudaStream_t);
#define ATTNRES_INSTANTIATE_TAIL_ADD(DEF)                                    \
  ATTNRES_TAIL_ADD(DEF, true, kBF16) ATTNRES_TAIL_ADD(DEF, false, kBF16)     \
  ATTNRES_TAIL_ADD(DEF, true, kFP16) ATTNRES_TAIL_ADD(DEF, false, kFP16)

#define ATTNRES_PATTERN(DEF, N) \
  DEF template cudaError_t launch_pattern<N>(const Params&, dim3, int, int, cudaStream_t);
#define ATTNRES_INSTANTIATE_PATTERN(DEF)                                                       \
  ATTNRES_PATTERN(DEF, 0) ATTNRES_PATTERN(DEF, 1) ATTNRES_PATTERN(DEF, 2) ATTNRES_PATTERN(DEF, 3) \
  ATTNRES_PATTERN(DEF, 4) ATTNRES_PATTERN(DEF, 5) ATTNRES_PATTERN(DEF, 6) ATTNRES_PATTERN(DEF, 7) \
  ATTNRES_PATTERN(DEF, 8) ATTNRES_PATTERN(DEF, 9) ATTNRES_PATTERN(DEF, 10)                      \
  ATTNRES_PATTERN(DEF, 11) ATTNRES_PATTERN(DEF, 12)

// Which unit defines what.
#define ATTNRES_UNIT_A(DEF)                                                             \
  ATTNRES_INSTANTIATE(DEF, 1, true) ATTNRES_INSTANTIATE(DEF, 2, true)                   \
  ATTNRES_INSTANTIATE(DEF, 3, true) ATTNRES_INSTANTIATE(DEF, 4, true)                   \
  ATTNRES_INSTANTIATE(DEF, 5, true) ATTNRES_INSTANTIATE(DEF, 6, true)
#define ATTNRES_UNIT_B(DEF)                                                             \
  ATTNRES_INSTANTIATE(DEF, 7, true) ATTNRES_INSTANTIATE(DEF, 8, true)                   \
  ATTNRES_INSTANTIATE(DEF, 9, true) ATTNRES_INSTANTIATE(DEF, 10, true)                  \
  ATTNRES_INSTANTIATE(DEF, 11, true) ATTNRES_INSTANTIATE(DEF, 12, true)
#define ATTNRES_UNIT_C(DEF)                                                             \
  ATTNRES_INSTANTIATE(DEF, 1, false) ATTNRES_INSTANTIATE(DEF, 2, false)                 \
  ATTNRES_INSTANTIATE(DEF, 3, false) ATTNRES_INSTANTIATE(DEF, 4, false)                 \
  ATTNRES_INSTANTIATE(DEF, 5, false) ATTNRES_INSTANTIATE(DEF, 6, false)
#define ATTNRES_UNIT_D(DEF)                                                             \
  ATTNRES_INSTANTIATE(DEF, 7, false) ATTNRES_INSTANTIATE(DEF, 8, false)                 \
  ATTNRES_INSTANTIATE(DEF, 9, false) ATTNRES_INSTANTIATE(DEF, 10, false)                \
  ATTNRES_INSTANTIATE(DEF, 11, false) ATTNRES_INSTANTIATE(DEF, 12, false)
#define ATTNRES_UNIT_E(DEF)                                                             \
  ATTNRES_INSTANTIATE(DEF, 0, true) ATTNRES_INSTANTIATE(DEF, 0, false)                  \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 0) ATTNRES_INSTANTIATE_NOFOLD(DEF, 1)                 \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 2) ATTNRES_INSTANTIATE_NOFOLD(DEF, 3)                 \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 4) ATTNRES_INSTANTIATE_NOFOLD(DEF, 5)                 \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 6) ATTNRES_INSTANTIATE_NOFOLD(DEF, 7)                 \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 8) ATTNRES_INSTANTIATE_NOFOLD(DEF, 9)                 \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 10) ATTNRES_INSTANTIATE_NOFOLD(DEF, 11)               \
  ATTNRES_INSTANTIATE_NOFOLD(DEF, 12) ATTNRES_INSTANTIATE_TAIL_ADD(DEF)               \
  ATTNRES_INSTANTIATE_PATTERN(DEF)
#define ATTNRES_UNIT_F(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP(DEF, 13) ATTNRES_INSTANTIATE_DEEP(DEF, 14)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 15) ATTNRES_INSTANTIATE_DEEP(DEF, 16)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 17) ATTNRES_INSTANTIATE_DEEP(DEF, 18)
#define ATTNRES_UNIT_G(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP(DEF, 19) ATTNRES_INSTANTIATE_DEEP(DEF, 20)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 21) ATTNRES_INSTANTIATE_DEEP(DEF, 22)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 23) ATTNRES_INSTANTIATE_DEEP(DEF, 24)
#define ATTNRES_UNIT_H(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP(DEF, 25) ATTNRES_INSTANTIATE_DEEP(DEF, 26)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 27) ATTNRES_INSTANTIATE_DEEP(DEF, 28)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 29) ATTNRES_INSTANTIATE_DEEP(DEF, 30)                   \
  ATTNRES_INSTANTIATE_DEEP(DEF, 31)
#define ATTNRES_UNIT_L(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 13) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 14)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 15) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 16)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 17) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 18)
#define ATTNRES_UNIT_M(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 19) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 20)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 21) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 22)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 23) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 24)
#define ATTNRES_UNIT_N(DEF)                                                             \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 25) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 26)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 27) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 28)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 29) ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 30)         \
  ATTNRES_INSTANTIATE_DEEP_FP16(DEF, 31)
#define ATTNRES_UNIT_I(DEF)                                                             \
  ATTNRES_INSTANTIATE_FP16(DEF, 0) ATTNRES_INSTANTIATE_FP16(DEF, 1)                     \
  ATTNRES_INSTANTIATE_FP16(DEF, 2) ATTNRES_INSTANTIATE_FP16(DEF, 3)                     \
  ATTNRES_INSTANTIATE_FP16(DEF, 4) ATTNRES_INSTANTIATE_FP16(DEF, 5)                     \
  ATTNRES_INSTANTIATE_FP16(DEF, 6)
#define ATTNRES_UNIT_J(DEF)                                                             \
  ATTNRES_INSTANTIATE_FP16(DEF, 7) ATTNRES_INSTANTIATE_FP16(DEF, 8)                     \
  ATTNRES_INSTANTIATE_FP16(DEF, 9) ATTNRES_INSTANTIATE_FP16(DEF, 10)                    \
  ATTNRES_INSTANTIATE_FP16(DEF, 11) ATTNRES_INSTANTIATE_FP16(DEF, 12)

}  // namespace attnres
