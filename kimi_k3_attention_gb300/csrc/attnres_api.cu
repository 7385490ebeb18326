// C ABI of the fused AttnRes + add2 + RMSNorm epilogue: argument validation,
// choice of launch configuration, dispatch to the compiled instantiations.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/attnres.h"
#include "attnres_launch.cuh"

namespace attnres {

// The kernels are compiled in the attnres_inst_*.cu units only.
ATTNRES_UNIT_A(extern)
ATTNRES_UNIT_B(extern)
ATTNRES_UNIT_C(extern)
ATTNRES_UNIT_D(extern)
ATTNRES_UNIT_E(extern)
ATTNRES_UNIT_F(extern)
ATTNRES_UNIT_G(extern)
ATTNRES_UNIT_H(extern)
ATTNRES_UNIT_I(extern)
ATTNRES_UNIT_J(extern)
ATTNRES_UNIT_L(extern)
ATTNRES_UNIT_M(extern)
ATTNRES_UNIT_N(extern)

namespace {

thread_local int g_last_cuda_error = 0;

// Status word written by the kernels (bit 0: an exchange wait timed out),
// one per device that loads the library.
__device__ unsigned int g_device_status;

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 ok, 2 wrong architecture
  std::atomic<int> sms{0};
  std::atomic<unsigned int*> status{nullptr};
};
DeviceInfo g_dev[kMaxDevices];

// Exchange-wait limit and the test hook that makes every exchange expect
// bytes that never come (see attnres_debug_exchange).
constexpr long long kDefaultWaitNs = 200LL * 1000 * 1000;
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<unsigned int> g_extra_tx{0};

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return ATTNRES_ERR_CUDA;
}

// Compute capability 10.3 (GB300) and SM count of the current device.
int current_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTNRES_ERR_DEVICE;
  DeviceInfo& d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, count = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda(e);
    d.sms.store(count, std::memory_order_relaxed);
    st = (major == 10 && minor == 3) ? 1 : 2;
    if (st == 1) {
      // The device address of this device's status word, taken with the
      // device current (the host-side symbol is not a device address).
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_device_status)) != cudaSuccess) return fail_cuda(e);
      d.status.store(static_cast<unsigned int*>(ptr), std::memory_order_relaxed);
    }
    d.state.store(st, std::memory_order_release);
  }
  if (st != 1) return ATTNRES_ERR_DEVICE;
  *sms = d.sms.load(std::memory_order_relaxed);
  return ATTNRES_OK;
}

unsigned int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_dev[dev].status.load(std::memory_order_relaxed);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// One call of the op, whichever entry point it came through.
struct Args {
  const void* prefix;
  const void* add;
  const void* add2;
  const void* bank;
  const void* w;
  const void* gamma;
  float eps;
  void* out;
  void* new_prefix;
  void* h_out;
  int M, N, H;
  bool fold;
  int dtype;  // ATTNRES_DTYPE_*
};

int validate_shape(int M, int N, int H) {
  if (M < 1 || N < 0 || N > ATTNRES_MAX_N || H < 8 || H > ATTNRES_MAX_H || (H % 8) != 0)
    return ATTNRES_ERR_SHAPE;
  return ATTNRES_OK;
}

int validate(const Args& a) {
  if (a.dtype != ATTNRES_DTYPE_BF16 && a.dtype != ATTNRES_DTYPE_FP16) return ATTNRES_ERR_DTYPE;
  if (!a.prefix || (a.N > 0 && !a.bank) || !a.w || !a.gamma || !a.out) return ATTNRES_ERR_NULL;
  if (a.fold && (!a.add || !a.new_prefix)) return ATTNRES_ERR_NULL;
  int st = validate_shape(a.M, a.N, a.H);
  if (st != ATTNRES_OK) return st;
  if (!(a.eps > 0.f) || !isfinite(a.eps)) return ATTNRES_ERR_EPS;
  const void* add = a.fold ? a.add : nullptr;
  const void* add2 = a.fold ? a.add2 : nullptr;
  const void* np = a.fold ? a.new_prefix : nullptr;
  if (misaligned(a.prefix) || (add && misaligned(add)) || (add2 && misaligned(add2)) ||
      (a.bank && misaligned(a.bank)) || misaligned(a.w) || misaligned(a.gamma) || misaligned(a.out) ||
      (np && misaligned(np)) || (a.h_out && misaligned(a.h_out)))
    return ATTNRES_ERR_ALIGN;
  const size_t R = static_cast<size_t>(a.M) * static_cast<size_t>(a.H) * 2u;
  const size_t B = R * static_cast<size_t>(a.N);
  const size_t V = static_cast<size_t>(a.H) * 2u;
  const void* ins[6] = {a.prefix, add, add2, a.N > 0 ? a.bank : nullptr, a.w, a.gamma};
  const size_t insz[6] = {R, add ? R : 0, add2 ? R : 0, B, V, V};
  // out and h_out overlap nothing; new_prefix overlaps no input except being
  // exactly prefix (in-place carry-on)
  const void* outs[3] = {a.out, a.h_out, np};
  for (int o = 0; o < 3; ++o) {
    if (!outs[o]) continue;
    for (int i = 0; i < 6; ++i) {
      if (o == 2 && i == 0 && np == a.prefix) continue;
      if (overlaps(outs[o], R, ins[i], insz[i])) return ATTNRES_ERR_ALIAS;
    }
    for (int q = o + 1; q < 3; ++q)
      if (outs[q] && overlaps(outs[o], R, outs[q], R)) return ATTNRES_ERR_ALIAS;
  }
  return ATTNRES_OK;
}

int round_up32(int x) { return (x + 31) & ~31; }

// Dynamic shared memory the pipelined ring may take: the 227 KB a CTA can
// hold, less the kernel's static exchange buffers and a little slack.
constexpr size_t kPipeSmemMax = 227 * 1024 - sizeof(Exchange<1>) - 1024;

// Fill every zero field of *c for (M, N, H) on a device with `sms` SMs, then
// check the result.  bf16_fold: the call folds BF16 tensors (the shapes
// compiled for that case only may be chosen).  Returns ATTNRES_OK or
// ATTNRES_ERR_CONFIG.
// Cluster size per token of the register-capped split shape (variant 5) at
// H = 7168 for M = 17..28, the fastest of 4..8 CTAs in same-box sweeps on
// GB300 (graphs of back-to-back calls, warm and cold), taken for tokens of
// at least 9 rows (bank, prefix, addends); tokens with fewer rows, and 29 to
// 32 tokens, keep about 128 / M CTAs (4 from 29 tokens on: 7-8 CTAs were
// within 0.05 us of it there, faster or slower depending on the run).  The
// sizes that fill 120-140 SMs win below 26 tokens; from there on the calls
// whose CTAs come close to every SM (6 CTAs from 24 tokens, 5 from 29) lose
// 0.3-0.8 us, presumably to clusters placed on SMs that already hold one of
// the same call, and 8 CTAs (two per SM on most SMs) are fastest.  N = 12:
// M = 26-28 2.95-2.97 us against 3.09-3.14 for 5 CTAs; M = 17-18 2.69-2.71
// against 2.81-2.82 for 7-8.
constexpr int kSplit2Cluster[12] = {4, 4, 6, 6, 6, 6, 6, 5, 5, 8, 8, 8};

int resolve(int M, int N, bool add2, int H, attnres_config* c, bool bf16_fold) {
  const int H8 = H / 8;
  auto min_cluster = [&](int maxt) {
    int cl = 1;
    while (cl <= 16 && round_up32((H8 + cl - 1) / cl) > maxt) ++cl;
    return cl;
  };
  // Deep banks (more than kShallowMaxN snapshots) have variants 2 and 3
  // only, and a streaming shape of their own.
  const bool deep = N > kShallowMaxN;
  if (deep && (c->variant == 1 || c->variant == 4)) return ATTNRES_ERR_CONFIG;
  const int stream_maxt = deep ? kDeepStreamMaxT : kStreamMaxT;
  if (c->variant == 0) {
    // Measured on GB300 at H = 7168 (the cluster sizes below are for that
    // H and scale with it): up to 32 tokens, a cluster of about 128 / M CTAs
    // (clamped to 4..8) per token keeps ~128 CTAs per call, one per SM; from
    // 17 tokens on, with the fold on BF16 tensors, registers capped so that
    // the next call's CTAs fit beside them (0.05-0.16 us faster there, the
    // same below), and the cluster size from kSplit2Cluster; up to 48
    // tokens, 8 CTAs of 112 columns (three fit an SM, still one wave); then
    // the register-capped shape, 4 CTAs of 224 columns up to 96 tokens and
    // 7 CTAs of 128 columns beyond, where many tokens are in flight on every
    // SM.  Deep banks: up to 32 tokens the
    // same clusters (4 CTAs from 8 tokens on once N >= 24, where a token's
    // rows are many), beyond that their streaming shape, 7 CTAs of 128
    // columns (the split shape's CTAs hold too many registers to share an
    // SM).
    int ref;
    if (M <= 32) {
      c->variant = (M >= 17 && bf16_fold && !deep) ? 5 : 2;
      ref = (128 + M / 2) / M;
      ref = ref < 4 ? 4 : (ref > 8 ? 8 : ref);
      if (c->variant == 5 && M <= 28 && N + (add2 ? 3 : 2) >= 9) ref = kSplit2Cluster[M - 17];
      if (N >= 24 && M >= 8) ref = 4;
    } else if (deep) {
      c->variant = 3;
      ref = 7;
    } else if (M <= 48) {
      c->variant = 2;
      ref = 8;
    } else if (M <= 96) {
      c->variant = 3;
      ref = 4;
    } else {
      c->variant = 3;
      ref = 7;
    }
    if (c->cluster == 0) {
      const int lo = min_cluster(c->variant == 3 ? stream_maxt : kSplitMaxT);
      int cl = (ref * H8 + 448) / 896;
      c->cluster = cl < lo ? lo : (cl > 16 ? 16 : cl);
    }
  }
  if (deep && c->variant == 5) return ATTNRES_ERR_CONFIG;
  if (c->variant == 1) {
    if (c->cluster == 0) c->cluster = 1;
    if (c->cluster != 1) return ATTNRES_ERR_CONFIG;
    const int need = round_up32((H8 + kCtaVPT - 1) / kCtaVPT);
    if (c->threads == 0) c->threads = need;
    if (c->threads < need || c->threads > kCtaMaxT || (c->threads % 32) != 0)
      return ATTNRES_ERR_CONFIG;
  } else if (c->variant == 2 || c->variant == 3 || c->variant == 5) {
    const int maxt = (c->variant == 3) ? stream_maxt : kSplitMaxT;
    if (c->cluster == 0) c->cluster = min_cluster(maxt);
    if (c->cluster < 1 || c->cluster > 16) return ATTNRES_ERR_CONFIG;
    const int cpc = (H8 + c->cluster - 1) / c->cluster;
    const int need = round_up32(cpc);
    if (c->threads == 0) c->threads = need;
    if (c->threads < need || c->threads > maxt || (c->threads % 32) != 0)
      return ATTNRES_ERR_CONFIG;
  } else if (c->variant == 4) {
    if (c->cluster == 0) c->cluster = min_cluster(kPipeMaxT);
    if (c->cluster < 1 || c->cluster > 16) return ATTNRES_ERR_CONFIG;
    const int cpc = (H8 + c->cluster - 1) / c->cluster;
    const int need = round_up32(cpc);
    if (c->threads == 0) c->threads = need;
    if (c->threads < need || c->threads > kPipeMaxT || (c->threads % 32) != 0)
      return ATTNRES_ERR_CONFIG;
    if (c->stages == 0) {
      // the deepest ring that still lets two CTAs share an SM (228 KB of
      // shared memory per SM, 1 KB of it reserved per CTA), else the
      // deepest that fits one
      c->stages = 4;
      while (c->stages > 2 &&
             2 * (pipe_smem_bytes(N, add2, c->threads, c->stages) + sizeof(Exchange<1>) + 1024) >
                 228 * 1024)
        --c->stages;
      if (2 * (pipe_smem_bytes(N, add2, c->threads, c->stages) + sizeof(Exchange<1>) + 1024) >
          228 * 1024) {
        c->stages = 4;
        while (c->stages > 2 && pipe_smem_bytes(N, add2, c->threads, c->stages) > kPipeSmemMax)
          --c->stages;
      }
    }
    if (c->stages < 2 || c->stages > 4 ||
        pipe_smem_bytes(N, add2, c->threads, c->stages) > kPipeSmemMax)
      return ATTNRES_ERR_CONFIG;
    // grid_tokens 0 stays 0: the launcher sizes the grid to the resident
    // clusters.
    if (c->grid_tokens < 0 || c->grid_tokens > 65535) return ATTNRES_ERR_CONFIG;
    if (c->tail_tokens != 0) return ATTNRES_ERR_CONFIG;
  } else {
    return ATTNRES_ERR_CONFIG;
  }
  if (c->variant != 4) {
    if (c->stages != 0) return ATTNRES_ERR_CONFIG;
    if (c->tail_tokens < 0) return ATTNRES_ERR_CONFIG;
    // The register-capped shapes (variant 3) keep grid_tokens 0: the launcher
    // sizes a walk from the clusters that fit at once (walk_grid; with M
    // below about R, one cluster per token).  GB300, M = 8192, N = 12,
    // against grids of clusters that each walk an equal share: 10 per SM
    // 6.44 TB/s, 6 or 14 per SM 6.37, only the resident clusters 3.7.
    if (c->grid_tokens == 0 && c->variant != 3) c->grid_tokens = M < 65535 ? M : 65535;
    if (c->grid_tokens == 0) {
      if (c->tail_tokens != 0) return ATTNRES_ERR_CONFIG;
    } else {
      if (c->grid_tokens < 1 || c->grid_tokens > 65535) return ATTNRES_ERR_CONFIG;
      // the streaming shape only; the walking clusters need a token each
      if (c->tail_tokens > 0 &&
          (c->variant != 3 || c->tail_tokens >= c->grid_tokens || c->grid_tokens > M))
        return ATTNRES_ERR_CONFIG;
    }
  }
  if (c->pdl < -1 || c->pdl > 1) return ATTNRES_ERR_CONFIG;
  if (c->pdl == 0) c->pdl = 1;
  if (c->prefetch < -1 || c->prefetch > 15) return ATTNRES_ERR_CONFIG;
  if (c->prefetch == 0) {
    const bool fused = c->variant == 2 || c->variant == 3 || c->variant == 5;
    c->prefetch = (fused && M <= 96) ? 1 : 0;
    if (fused && M <= 32) c->prefetch |= 8;   // the decode window
    if (fused && c->grid_tokens < M) c->prefetch |= 4;   // clusters walk tokens
    if (c->prefetch == 0) c->prefetch = -1;
  }
  if (c->prefetch > 0 && c->variant != 2 && c->variant != 3 && c->variant != 5)
    return ATTNRES_ERR_CONFIG;
  return ATTNRES_OK;
}

template <int VPT, int MAXT, int MINB>
cudaError_t dispatch(int N, bool add2, const Params& p, dim3 g, int t, int c, bool pdl,
                     cudaStream_t s) {
#define ATTNRES_CASE(n)                                                                  \
  case n:                                                                                \
    return add2 ? launch_fused<n, kFoldAdd2, VPT, MAXT, minb_of(MINB, n, kFoldAdd2), kBF16, \
                               nr_of(MINB, n, kFoldAdd2)>(p, g, t, c, pdl, s)              \
                : launch_fused<n, kFoldAdd, VPT, MAXT, minb_of(MINB, n, kFoldAdd), kBF16,   \
                               nr_of(MINB, n, kFoldAdd)>(p, g, t, c, pdl, s);
  switch (N) {
    ATTNRES_CASE(0)
    ATTNRES_CASE(1) ATTNRES_CASE(2) ATTNRES_CASE(3) ATTNRES_CASE(4)
    ATTNRES_CASE(5) ATTNRES_CASE(6) ATTNRES_CASE(7) ATTNRES_CASE(8)
    ATTNRES_CASE(9) ATTNRES_CASE(10) ATTNRES_CASE(11) ATTNRES_CASE(12)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

template <int VPT, int MAXT, int MINB>
cudaError_t dispatch_nofold(int N, const Params& p, dim3 g, int t, int c, bool pdl,
                            cudaStream_t s) {
#define ATTNRES_CASE(n) \
  case n:               \
    return launch_fused<n, kNoFold, VPT, MAXT, minb_of(MINB, n, kNoFold), kBF16,          \
                        nr_of(MINB, n, kNoFold)>(p, g, t, c, pdl, s);
  switch (N) {
    ATTNRES_CASE(0)
    ATTNRES_CASE(1) ATTNRES_CASE(2) ATTNRES_CASE(3) ATTNRES_CASE(4)
    ATTNRES_CASE(5) ATTNRES_CASE(6) ATTNRES_CASE(7) ATTNRES_CASE(8)
    ATTNRES_CASE(9) ATTNRES_CASE(10) ATTNRES_CASE(11) ATTNRES_CASE(12)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

template <int N, bool ADD2>
cudaError_t dispatch_pipe_stages(int stages, const Params& p, dim3 g, int t, int c, bool pdl,
                                 cudaStream_t s) {
  switch (stages) {
    case 2: return launch_pipe<N, ADD2, 2>(p, g, t, c, pdl, s);
    case 3: return launch_pipe<N, ADD2, 3>(p, g, t, c, pdl, s);
    case 4: return launch_pipe<N, ADD2, 4>(p, g, t, c, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

// FP16 tensors (N <= 12): the split or the streaming shape.
template <int VPT, int MAXT, int MINB>
cudaError_t dispatch_fp16(int N, int mode, const Params& p, dim3 g, int t, int c, bool pdl,
                          cudaStream_t s) {
#define ATTNRES_CASE(n)                                                                    \
  case n:                                                                                  \
    return mode == kFoldAdd2                                                               \
               ? launch_fused<n, kFoldAdd2, VPT, MAXT, minb_of(MINB, n, kFoldAdd2), kFP16,    \
                              nr_of(MINB, n, kFoldAdd2)>(p, g, t, c, pdl, s)               \
           : mode == kFoldAdd                                                              \
               ? launch_fused<n, kFoldAdd, VPT, MAXT, minb_of(MINB, n, kFoldAdd), kFP16,      \
                              nr_of(MINB, n, kFoldAdd)>(p, g, t, c, pdl, s)                \
               : launch_fused<n, kNoFold, VPT, MAXT, minb_of(MINB, n, kNoFold), kFP16,        \
                              nr_of(MINB, n, kNoFold)>(p, g, t, c, pdl, s);
  switch (N) {
    ATTNRES_CASE(0)
    ATTNRES_CASE(1) ATTNRES_CASE(2) ATTNRES_CASE(3) ATTNRES_CASE(4)
    ATTNRES_CASE(5) ATTNRES_CASE(6) ATTNRES_CASE(7) ATTNRES_CASE(8)
    ATTNRES_CASE(9) ATTNRES_CASE(10) ATTNRES_CASE(11) ATTNRES_CASE(12)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

// Deep banks: the split shape (STREAM false) or the deep streaming shape,
// with or without the fold, element format DT.
template <int N, bool STREAM, int DT>
cudaError_t launch_deep(int mode, const Params& p, dim3 g, int t, int c, bool pdl,
                        cudaStream_t s) {
  constexpr int VPT = STREAM ? kStreamVPT : kSplitVPT;
  constexpr int MAXT = STREAM ? kDeepStreamMaxT : kSplitMaxT;
  constexpr int MINB = STREAM ? deep_minb(N) : kSplitMinB;
  constexpr int NR = STREAM ? deep_nr(N) : N;
  return mode == kFoldAdd2 ? launch_fused<N, kFoldAdd2, VPT, MAXT, MINB, DT, NR>(p, g, t, c, pdl, s)
         : mode == kFoldAdd ? launch_fused<N, kFoldAdd, VPT, MAXT, MINB, DT, NR>(p, g, t, c, pdl, s)
                            : launch_fused<N, kNoFold, VPT, MAXT, MINB, DT, NR>(p, g, t, c, pdl, s);
}

template <bool STREAM, int DT>
cudaError_t dispatch_deep(int N, int mode, const Params& p, dim3 g, int t, int c, bool pdl,
                          cudaStream_t s) {
#define ATTNRES_CASE(n) \
  case n:               \
    return launch_deep<n, STREAM, DT>(mode, p, g, t, c, pdl, s);
  switch (N) {
    ATTNRES_CASE(13) ATTNRES_CASE(14) ATTNRES_CASE(15) ATTNRES_CASE(16)
    ATTNRES_CASE(17) ATTNRES_CASE(18) ATTNRES_CASE(19) ATTNRES_CASE(20)
    ATTNRES_CASE(21) ATTNRES_CASE(22) ATTNRES_CASE(23) ATTNRES_CASE(24)
    ATTNRES_CASE(25) ATTNRES_CASE(26) ATTNRES_CASE(27) ATTNRES_CASE(28)
    ATTNRES_CASE(29) ATTNRES_CASE(30) ATTNRES_CASE(31)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

cudaError_t dispatch_pipe(int N, bool add2, int stages, const Params& p, dim3 g, int t, int c,
                          bool pdl, cudaStream_t s) {
#define ATTNRES_CASE(n)                                                              \
  case n:                                                                            \
    return add2 ? dispatch_pipe_stages<n, true>(stages, p, g, t, c, pdl, s)          \
                : dispatch_pipe_stages<n, false>(stages, p, g, t, c, pdl, s);
  switch (N) {
    ATTNRES_CASE(0)
    ATTNRES_CASE(1) ATTNRES_CASE(2) ATTNRES_CASE(3) ATTNRES_CASE(4)
    ATTNRES_CASE(5) ATTNRES_CASE(6) ATTNRES_CASE(7) ATTNRES_CASE(8)
    ATTNRES_CASE(9) ATTNRES_CASE(10) ATTNRES_CASE(11) ATTNRES_CASE(12)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

int run(const Args& a, const attnres_config* cfg, cudaStream_t s) {
  int st = validate(a);
  if (st != ATTNRES_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != ATTNRES_OK) return st;
  const bool has_add2 = a.fold && a.add2 != nullptr;
  attnres_config c = cfg ? *cfg : attnres_config{0, 0, 0, 0, 0, 0, 0, 0};
  if ((st = resolve(a.M, a.N, has_add2, a.H, &c, a.fold && a.dtype == ATTNRES_DTYPE_BF16)) !=
      ATTNRES_OK)
    return st;
  // the attention-residual alone and FP16 tensors exist in the two fused
  // shapes only
  if ((!a.fold || a.dtype == ATTNRES_DTYPE_FP16) && c.variant != 2 && c.variant != 3)
    return ATTNRES_ERR_CONFIG;

  Params p;
  p.prefix = static_cast<const uint4*>(a.prefix);
  p.add = static_cast<const uint4*>(a.fold ? a.add : nullptr);
  p.add2 = static_cast<const uint4*>(has_add2 ? a.add2 : nullptr);
  p.bank = static_cast<const uint4*>(a.bank);
  p.w = static_cast<const uint4*>(a.w);
  p.gamma = static_cast<const uint4*>(a.gamma);
  p.out = static_cast<uint4*>(a.out);
  p.new_prefix = static_cast<uint4*>(a.fold ? a.new_prefix : nullptr);
  p.h_out = static_cast<uint4*>(a.h_out);
  p.M = a.M;
  p.H8 = a.H / 8;
  p.bank_stride = static_cast<long long>(a.M) * p.H8;
  p.cpc = (p.H8 + c.cluster - 1) / c.cluster;
  p.eps = a.eps;
  p.inv_h = 1.0f / static_cast<float>(a.H);
  p.status = device_status_ptr();
  p.wait_ns = static_cast<unsigned long long>(g_wait_ns.load(std::memory_order_relaxed));
  p.extra_tx = g_extra_tx.load(std::memory_order_relaxed);
  p.prefetch = c.prefetch > 0 ? c.prefetch : 0;
  p.tail = c.tail_tokens;   // grid_tokens 0: set by the launcher

  const dim3 grid(static_cast<unsigned>(c.cluster), static_cast<unsigned>(c.grid_tokens), 1);
  const bool pdl = c.pdl >= 0;
  cudaError_t e;
  const int mode = !a.fold ? kNoFold : has_add2 ? kFoldAdd2 : kFoldAdd;
  const bool fp16 = a.dtype == ATTNRES_DTYPE_FP16;
  if (a.N > kShallowMaxN && c.variant == 2)
    e = fp16 ? dispatch_deep<false, kFP16>(a.N, mode, p, grid, c.threads, c.cluster, pdl, s)
             : dispatch_deep<false, kBF16>(a.N, mode, p, grid, c.threads, c.cluster, pdl, s);
  else if (a.N > kShallowMaxN)
    e = fp16 ? dispatch_deep<true, kFP16>(a.N, mode, p, grid, c.threads, c.cluster, pdl, s)
             : dispatch_deep<true, kBF16>(a.N, mode, p, grid, c.threads, c.cluster, pdl, s);
  else if (fp16 && c.variant == 2)
    e = dispatch_fp16<kSplitVPT, kSplitMaxT, kSplitMinB>(a.N, mode, p, grid, c.threads, c.cluster,
                                                         pdl, s);
  else if (fp16)
    e = dispatch_fp16<kStreamVPT, kStreamMaxT, kStreamMinB>(a.N, mode, p, grid, c.threads,
                                                            c.cluster, pdl, s);
  else if (!a.fold && c.variant == 2)
    e = dispatch_nofold<kSplitVPT, kSplitMaxT, kSplitMinB>(a.N, p, grid, c.threads, c.cluster, pdl, s);
  else if (!a.fold)
    e = dispatch_nofold<kStreamVPT, kStreamMaxT, kStreamMinB>(a.N, p, grid, c.threads, c.cluster,
                                                              pdl, s);
  else if (c.variant == 1)
    e = dispatch<kCtaVPT, kCtaMaxT, kCtaMinB>(a.N, has_add2, p, grid, c.threads, 1, pdl, s);
  else if (c.variant == 2)
    e = dispatch<kSplitVPT, kSplitMaxT, kSplitMinB>(a.N, has_add2, p, grid, c.threads, c.cluster,
                                                    pdl, s);
  else if (c.variant == 5)
    e = dispatch<kSplitVPT, kSplitMaxT, kSplit2MinB>(a.N, has_add2, p, grid, c.threads, c.cluster,
                                                     pdl, s);
  else if (c.variant == 3)
    e = dispatch<kStreamVPT, kStreamMaxT, kStreamMinB>(a.N, has_add2, p, grid, c.threads,
                                                       c.cluster, pdl, s);
  else
    e = dispatch_pipe(a.N, has_add2, c.stages, p, grid, c.threads, c.cluster, pdl, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTNRES_OK;
}

Args make_args(const void* prefix, const void* add, const void* add2, const void* bank,
               const void* w, const void* gamma, float eps, void* out, void* new_prefix,
               void* h_out, int M, int N, int H, bool fold, int dtype = ATTNRES_DTYPE_BF16) {
  Args a;
  a.prefix = prefix;
  a.add = add;
  a.add2 = add2;
  a.bank = bank;
  a.w = w;
  a.gamma = gamma;
  a.eps = eps;
  a.out = out;
  a.new_prefix = new_prefix;
  a.h_out = h_out;
  a.M = M;
  a.N = N;
  a.H = H;
  a.fold = fold;
  a.dtype = dtype;
  return a;
}

}  // namespace
}  // namespace attnres

using namespace attnres;

extern "C" int attnres_add_rmsnorm_ex(const void* prefix, const void* add, const void* add2,
                                      const void* bank, const void* w, const void* gamma,
                                      float eps, void* out, void* new_prefix, int M, int N,
                                      int H, attnres_stream_t stream,
                                      const attnres_config* cfg) {
  return run(make_args(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, nullptr, M, N, H,
                       true),
             cfg, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attnres_add_rmsnorm(const void* prefix, const void* add, const void* add2,
                                   const void* bank, const void* w, const void* gamma, float eps,
                                   void* out, void* new_prefix, int M, int N, int H,
                                   attnres_stream_t stream) {
  return attnres_add_rmsnorm_ex(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, M, N, H,
                                stream, nullptr);
}

extern "C" int attnres_add_rmsnorm_f16(const void* prefix, const void* add, const void* add2,
                                       const void* bank, const void* w, const void* gamma,
                                       float eps, void* out, void* new_prefix, int M, int N, int H,
                                       attnres_stream_t stream) {
  return run(make_args(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, nullptr, M, N, H,
                       true, ATTNRES_DTYPE_FP16),
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attnres_add_rmsnorm_tap(const void* prefix, const void* add, const void* add2,
                                       const void* bank, const void* w, const void* gamma,
                                       float eps, void* out, void* new_prefix, void* h_out, int M,
                                       int N, int H, attnres_stream_t stream) {
  if (!h_out) return ATTNRES_ERR_NULL;
  return run(make_args(prefix, add, add2, bank, w, gamma, eps, out, new_prefix, h_out, M, N, H,
                       true),
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attnres_rmsnorm(const void* prefix, const void* bank, const void* w,
                               const void* gamma, float eps, void* out, int M, int N, int H,
                               attnres_stream_t stream) {
  return run(make_args(prefix, nullptr, nullptr, bank, w, gamma, eps, out, nullptr, nullptr, M, N,
                       H, false),
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attnres_launch(const attnres_args* args, const attnres_config* cfg,
                              attnres_stream_t stream) {
  if (!args) return ATTNRES_ERR_NULL;
  return run(make_args(args->prefix, args->add, args->add2, args->bank, args->w, args->gamma,
                       args->eps, args->out, args->new_prefix, args->h_out, args->M, args->N,
                       args->H, args->fold != 0, args->dtype),
             cfg, reinterpret_cast<cudaStream_t>(stream));
}

namespace attnres {
namespace {

int tail_add(const void* prefix, const void* add, const void* add2, void* new_prefix, int M,
             int H, int dtype, attnres_stream_t stream) {
  if (!prefix || !add || !new_prefix) return ATTNRES_ERR_NULL;
  if (M < 1 || H < 8 || H > ATTNRES_MAX_H || (H % 8) != 0) return ATTNRES_ERR_SHAPE;
  if (misaligned(prefix) || misaligned(add) || (add2 && misaligned(add2)) || misaligned(new_prefix))
    return ATTNRES_ERR_ALIGN;
  const size_t R = static_cast<size_t>(M) * static_cast<size_t>(H) * 2u;
  if ((new_prefix != prefix && overlaps(new_prefix, R, prefix, R)) || overlaps(new_prefix, R, add, R) ||
      overlaps(new_prefix, R, add2, add2 ? R : 0))
    return ATTNRES_ERR_ALIAS;
  int sms = 0;
  int st = current_device(&sms);
  if (st != ATTNRES_OK) return st;
  const long long chunks = static_cast<long long>(M) * (H / 8);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint4* p4 = static_cast<const uint4*>(prefix);
  const uint4* a4 = static_cast<const uint4*>(add);
  const uint4* b4 = static_cast<const uint4*>(add2);
  uint4* n4 = static_cast<uint4*>(new_prefix);
  cudaError_t e;
  if (dtype == ATTNRES_DTYPE_FP16)
    e = add2 ? launch_tail_add<true, kFP16>(p4, a4, b4, n4, chunks, sms, true, s)
             : launch_tail_add<false, kFP16>(p4, a4, b4, n4, chunks, sms, true, s);
  else
    e = add2 ? launch_tail_add<true, kBF16>(p4, a4, b4, n4, chunks, sms, true, s)
             : launch_tail_add<false, kBF16>(p4, a4, b4, n4, chunks, sms, true, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTNRES_OK;
}

}  // namespace
}  // namespace attnres

extern "C" int attnres_tail_add(const void* prefix, const void* add, const void* add2,
                                void* new_prefix, int M, int H, attnres_stream_t stream) {
  return tail_add(prefix, add, add2, new_prefix, M, H, ATTNRES_DTYPE_BF16, stream);
}

extern "C" int attnres_tail_add_f16(const void* prefix, const void* add, const void* add2,
                                    void* new_prefix, int M, int H, attnres_stream_t stream) {
  return tail_add(prefix, add, add2, new_prefix, M, H, ATTNRES_DTYPE_FP16, stream);
}

namespace attnres {
namespace {

cudaError_t dispatch_pattern(int N, const Params& p, dim3 g, int t, int c, cudaStream_t s) {
#define ATTNRES_CASE(n) \
  case n:               \
    return launch_pattern<n>(p, g, t, c, s);
  switch (N) {
    ATTNRES_CASE(0)
    ATTNRES_CASE(1) ATTNRES_CASE(2) ATTNRES_CASE(3) ATTNRES_CASE(4)
    ATTNRES_CASE(5) ATTNRES_CASE(6) ATTNRES_CASE(7) ATTNRES_CASE(8)
    ATTNRES_CASE(9) ATTNRES_CASE(10) ATTNRES_CASE(11) ATTNRES_CASE(12)
    default:
      return cudaErrorInvalidValue;
  }
#undef ATTNRES_CASE
}

}  // namespace
}  // namespace attnres

extern "C" int attnres_access_pattern(const void* prefix, const void* add, const void* add2,
                                      const void* bank, void* out, void* new_prefix, int M, int N,
                                      int H, attnres_stream_t stream) {
  if (!add2) return ATTNRES_ERR_NULL;
  if (N > kShallowMaxN) return ATTNRES_ERR_SHAPE;
  // the same checks as the fused call (w and gamma are not read: stand-ins)
  Args a = make_args(prefix, add, add2, bank, prefix, prefix, 1.0f, out, new_prefix, nullptr, M,
                     N, H, true);
  int st = validate(a);
  if (st != ATTNRES_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != ATTNRES_OK) return st;
  attnres_config c = {0, 0, 0, 0, 0, 0, 0, 0};
  if ((st = resolve(M, N, true, H, &c, true)) != ATTNRES_OK) return st;
  if (c.threads > kPatternMaxT) return ATTNRES_ERR_CONFIG;
  Params p = {};
  p.prefix = static_cast<const uint4*>(prefix);
  p.add = static_cast<const uint4*>(add);
  p.add2 = static_cast<const uint4*>(add2);
  p.bank = static_cast<const uint4*>(bank);
  p.out = static_cast<uint4*>(out);
  p.new_prefix = static_cast<uint4*>(new_prefix);
  p.M = M;
  p.H8 = H / 8;
  p.bank_stride = static_cast<long long>(M) * p.H8;
  p.cpc = (p.H8 + c.cluster - 1) / c.cluster;
  p.prefetch = c.prefetch > 0 ? c.prefetch : 0;
  const dim3 grid(static_cast<unsigned>(c.cluster), static_cast<unsigned>(c.grid_tokens), 1);
  cudaError_t e = dispatch_pattern(N, p, grid, c.threads, c.cluster,
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTNRES_OK;
}

extern "C" int attnres_plan(int M, int N, int H, int has_add2, attnres_config* plan) {
  if (!plan) return ATTNRES_ERR_NULL;
  if (validate_shape(M, N, H) != ATTNRES_OK) return ATTNRES_ERR_SHAPE;
  int sms = 0;
  int st = current_device(&sms);
  if (st != ATTNRES_OK) return st;
  attnres_config c = {0, 0, 0, 0, 0, 0, 0, 0};
  if ((st = resolve(M, N, has_add2 != 0, H, &c, true)) != ATTNRES_OK) return st;
  *plan = c;
  return ATTNRES_OK;
}

extern "C" int attnres_plan_host(int M, int N, int H, int has_add2, attnres_config* plan) {
  if (!plan) return ATTNRES_ERR_NULL;
  if (validate_shape(M, N, H) != ATTNRES_OK) return ATTNRES_ERR_SHAPE;
  attnres_config c = {0, 0, 0, 0, 0, 0, 0, 0};
  const int st = resolve(M, N, has_add2 != 0, H, &c, true);
  if (st != ATTNRES_OK) return st;
  *plan = c;
  return ATTNRES_OK;
}

extern "C" const char* attnres_status_string(int status) {
  switch (status) {
    case ATTNRES_OK: return "ok";
    case ATTNRES_ERR_NULL: return "a required pointer is NULL";
    case ATTNRES_ERR_SHAPE: return "unsupported shape: need M >= 1, 0 <= N <= 31, 8 <= H <= 16384, H % 8 == 0";
    case ATTNRES_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case ATTNRES_ERR_ALIAS: return "out overlaps a tensor, or new_prefix overlaps an input other than prefix";
    case ATTNRES_ERR_EPS: return "eps must be finite and > 0";
    case ATTNRES_ERR_CUDA: return "a CUDA runtime call failed (see attnres_last_cuda_error)";
    case ATTNRES_ERR_DEVICE: return "the current device is not a compute capability 10.3 GPU";
    case ATTNRES_ERR_CONFIG: return "invalid launch configuration";
    case ATTNRES_ERR_DTYPE: return "unsupported element type: BF16 or FP16";
    default: return "unknown status";
  }
}

extern "C" int attnres_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int attnres_device_status(unsigned int* bits, int clear) {
  if (!bits) return ATTNRES_ERR_NULL;
  int sms = 0;
  int st = current_device(&sms);
  if (st != ATTNRES_OK) return st;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return fail_cuda(e);
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ATTNRES_OK;
}

extern "C" int attnres_debug_exchange(int extra_bytes, long long wait_ns) {
  if (extra_bytes < 0 || extra_bytes > 4096 || wait_ns < 0 || wait_ns > 10LL * 1000 * 1000 * 1000)
    return ATTNRES_ERR_CONFIG;
  g_extra_tx.store(static_cast<unsigned int>(extra_bytes), std::memory_order_relaxed);
  g_wait_ns.store(wait_ns == 0 ? kDefaultWaitNs : wait_ns, std::memory_order_relaxed);
  return ATTNRES_OK;
}

extern "C" int attnres_version(void) { return 200; }
