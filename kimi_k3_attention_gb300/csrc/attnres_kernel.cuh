// Device code of the fused AttnRes + add2 + RMSNorm epilogue (sm_103a).
//
// One token is processed by a thread-block cluster of C CTAs (C = 1 is a
// single CTA).  CTA c of the cluster owns a contiguous slice of the token's
// H/8 sixteen-byte chunks; every thread owns VPT chunks of every source row
// and keeps them in registers from the single HBM read to the final store:
//
//   load    prefix, add, add2, bank[0..N-1] chunks: 16-byte vector loads
//           straight to registers (attnres_fused_kernel; a cluster may walk
//           several tokens (TokenWalk) and ask L2 for the next one's rows
//           while it reduces the current one), or cp.async copies into a per-thread
//           shared-memory ring several tokens ahead (attnres_pipe_kernel,
//           persistent)
//   fold    new_prefix = bf16(prefix + bf16(add + add2)), each addition
//           the exact sum rounded once to BF16: the bits of the float32
//           round-to-nearest additions of TensorRT-LLM PR #20546 ("Op"),
//           written as paired BF16 additions in PTX (add.rn.bf16x2, which
//           has no flush-to-zero form, so no fast-math flag can flush
//           subnormal sums); FP16 tensors round to FP16 (Fmt<kFP16>)
//   stats   ss_i = sum v^2 and d_i = w.v for the N+1 sources, one pass of
//           mixed-precision FMAs (16-bit operands, float32 accumulators)
//   R1      2(N+1) partial sums: warp transpose-reduction (one per group of
//           up to 16 sources, see Sums), CTA sum in shared
//           memory, then every CTA stores its totals into the shared memory
//           of every CTA of the cluster with st.async (one warp per receiving
//           CTA in the latency shapes), each store counted on the receiver's
//           mbarrier, which the receiver waits on
//   softmax logits and softmax from the cluster totals in a fixed order:
//           evaluated by every warp redundantly (latency and deep shapes: all
//           warps of all CTAs agree bitwise, no barrier), or by one warp and
//           read by the others after a CTA barrier (the streaming shapes of
//           up to 12 snapshots); the latency shapes keep the weights
//           unnormalised, e_i = exp(l_i - max l), and apply their sum in r_h
//   mix     h = sum_i alpha_i v_i from registers (no second read)
//   R2      sum h^2: warp reduction, st.async to every CTA, mbarrier wait
//           (the latency shapes first add their warps' sums in the CTA and
//           send one float per CTA)
//   out     bf16(h * rsqrt(mean(h^2) + eps) * gamma) (FP16 for FP16 tensors)
//           and new_prefix stored
//
// Every reduction has a fixed order, so results are deterministic.  Waits:
// the CTA barrier, one cluster barrier per kernel (arrive when the exchange
// mbarriers are set up, wait before the first remote store; every thread of
// every CTA reaches both on the same path), cp.async.wait_group (completes
// with its copies), griddepcontrol.wait (completes with the previous grid),
// and the exchange mbarriers, whose waits are bounded in time: on expiry the
// kernel sets a bit in the library's status word, stops waiting, writes NaN
// in place of the outputs that depend on the exchange, and stays resident
// for the same bound before exiting.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

struct Params {
  const uint4* prefix;
  const uint4* add;
  const uint4* add2;
  const uint4* bank;
  const uint4* w;
  const uint4* gamma;
  uint4* out;
  uint4* new_prefix;      // unused when the kernel does not fold
  uint4* h_out;           // optional 16-bit copy of the mixture h (NULL: none)
  long long bank_stride;  // chunks between snapshots: M * H8
  int M;
  int H8;                 // 16-byte chunks per row: H / 8
  int cpc;                // chunks owned by one CTA of the cluster
  float eps;
  float inv_h;            // 1 / H
  unsigned int* status;   // library status word of this device (bit 0: a wait timed out)
  unsigned long long wait_ns;  // limit of every exchange wait
  unsigned int extra_tx;  // test hook: bytes every exchange expects beyond what is sent
  int prefetch;           // bit 0: warm L2 with the first token's rows before
                          // waiting on the previous kernel; bit 1: also let the
                          // next kernel be scheduled at once; bit 2: while a
                          // token is reduced, warm L2 with the next token's rows;
                          // bit 3: before waiting, read a word of every 128-byte
                          // line of the first token's rows
  int tail;               // the last `tail` clusters of the grid take one
                          // token each (see TokenWalk); 0 = none
  int walkers;            // set by the launcher: gridDim.y - tail
  int walk_end;           // set by the launcher: M - tail
};

// The tokens one cluster handles.  With tail == 0, cluster c takes c,
// c + G, c + 2G, ... (G = gridDim.y).  With tail = T > 0 the first G - T
// clusters walk tokens [0, M - T) with stride G - T and the last T clusters
// take one token each, M - T + (c - (G - T)): clusters are started in grid
// order, so the short ones come last and fill the SMs that the long walks
// leave idle at the end.  The host keeps 0 <= T < G <= M.  Written with the
// launch parameters only, so that the walk holds no registers beyond the
// token index.  PLAIN (the latency shapes, which the host never gives a
// tail) takes c, c + G, ... straight from the grid: their first loads wait
// on no parameter read (GB300, decode: 0.02-0.09 us per call).
template <bool PLAIN>
struct TokenWalk {
  // the first token of cluster c (blockIdx.y)
  static __host__ __device__ __forceinline__ int first(const Params& p, int c) {
    if constexpr (PLAIN) return c;
    return c < p.walkers ? c : p.walk_end + (c - p.walkers);
  }
  // the token a cluster takes after m in a grid of G clusters (gridDim.y),
  // or M when it has none
  static __host__ __device__ __forceinline__ int next(const Params& p, int m, int G) {
    if constexpr (PLAIN) return m + G;
    const int n = m + p.walkers;
    return (m < p.walk_end && n < p.walk_end) ? n : p.M;
  }
};

// Every shape is compiled for up to kShallowMaxN snapshots; deeper banks
// (up to 31) have shapes of their own (attnres_launch.cuh).
constexpr int kShallowMaxN = 12;

// What a launch does with the prefix sum.
//   kFoldAdd:  new_prefix = bf16(prefix + add)            (no second addend)
//   kFoldAdd2: new_prefix = bf16(prefix + bf16(add + add2))
//   kNoFold:   the prefix itself is the last source; no addends, no
//              new_prefix (the attention-residual + RMSNorm alone)
constexpr int kFoldAdd = 0, kFoldAdd2 = 1, kNoFold = 2;

// Status bits written by the kernels.
constexpr unsigned int kStatusWaitTimeout = 1u;

constexpr unsigned FULL = 0xffffffffu;

// Threads per CTA of the access-pattern kernel (at most).
constexpr int kPatternMaxT = 256;

// ---------------------------------------------------------------- PTX helpers

// Global loads.  Each is volatile with a memory clobber, so the compiler
// keeps it after griddep_wait(): under programmatic dependent launch the
// data may be written by the previous kernel on the stream.
//   ld_stream: a row chunk, read once, not kept in L1, coherent (plain
//              ld.global: the prefix may be overwritten in place by the
//              same call, and on GB300 this form decodes slightly faster
//              than the non-coherent one)
//   ld_keep:   small read-only vectors (w, gamma), cached
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

// One 32-bit word through L2 only (never allocated in L1).
__device__ __forceinline__ uint32_t ld_l2_word(const void* p) {
  uint32_t r;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_keep(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

__device__ __forceinline__ void st_out(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// float32 fused multiply-add and multiply, round to nearest even, subnormal
// inputs and results kept.  Written in PTX so that a fast-math build (which
// turns the compiler's own float32 arithmetic into .ftz forms) cannot flush
// the mixture of tiny sources to zero.
__device__ __forceinline__ float fma_rn(float a, float b, float c) {
  float r;
  asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two float32 in one 64-bit register (lo in the low half), and the packed
// fused multiply-add acc = a * b + acc on both halves, each rounded to
// nearest even with subnormals kept.
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ void fma_rn_x2(unsigned long long& acc, unsigned long long a,
                                          unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// Both halves: a * b, each rounded to nearest even, subnormals kept.
__device__ __forceinline__ unsigned long long mul_rn_x2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float add_rn(float a, float b) {
  float r;
  asm("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float mul_rn(float a, float b) {
  float r;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Element formats of the tensors: BF16 (the model's) and FP16.  For each,
// the 16-bit halves of a 32-bit word unpacked to exact float32 (`lo` is the
// low half), two float32 packed into one word with one rounding to nearest
// even each (no .ftz: subnormal results are kept), and the per-source sums
// of a word's two lanes: ss += x*x, d += w*x, each a float32 FMA rounded
// once.  The products of two BF16 or two FP16 values are exact in float32,
// so the mixed-precision FMA (16-bit operands, float32 accumulator) gives
// the same bits as unpacking both operands and using fma.rn.f32, without
// the unpacking instructions.
constexpr int kBF16 = 0, kFP16 = 1;

template <int DT>
struct Fmt;

template <>
struct Fmt<kBF16> {
  static constexpr uint32_t kNaN2 = 0x7FC07FC0u;   // a quiet NaN in both lanes
  // integer moves only
  static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
  static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  static __device__ __forceinline__ void stats(uint32_t x, uint32_t w, float& ss, float& d) {
    asm("{\n .reg .b16 xl, xh, wl, wh;\n mov.b32 {xl, xh}, %2;\n mov.b32 {wl, wh}, %3;\n"
        " fma.rn.f32.bf16 %0, xl, xl, %0;\n fma.rn.f32.bf16 %1, wl, xl, %1;\n"
        " fma.rn.f32.bf16 %0, xh, xh, %0;\n fma.rn.f32.bf16 %1, wh, xh, %1;\n}"
        : "+f"(ss), "+f"(d)
        : "r"(x), "r"(w));
  }
  // a + b on both lanes, the exact sum rounded once to BF16 (nearest even,
  // subnormals kept)
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
};

template <>
struct Fmt<kFP16> {
  static constexpr uint32_t kNaN2 = 0x7E007E00u;   // a quiet NaN in both lanes
  // FP16 subnormals are normal float32 values: the conversion is exact
  static __device__ __forceinline__ float lo(uint32_t u) {
    float r;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, l;\n}" : "=f"(r) : "r"(u));
    return r;
  }
  static __device__ __forceinline__ float hi(uint32_t u) {
    float r;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, h;\n}" : "=f"(r) : "r"(u));
    return r;
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  static __device__ __forceinline__ void stats(uint32_t x, uint32_t w, float& ss, float& d) {
    asm("{\n .reg .b16 xl, xh, wl, wh;\n mov.b32 {xl, xh}, %2;\n mov.b32 {wl, wh}, %3;\n"
        " fma.rn.f32.f16 %0, xl, xl, %0;\n fma.rn.f32.f16 %1, wl, xl, %1;\n"
        " fma.rn.f32.f16 %0, xh, xh, %0;\n fma.rn.f32.f16 %1, wh, xh, %1;\n}"
        : "+f"(ss), "+f"(d)
        : "r"(x), "r"(w));
  }
  // a + b on both lanes, the exact sum rounded once to FP16 (nearest even,
  // subnormals kept: no .ftz)
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
};

// Element e (0..7) of a 16-byte chunk as float32.
template <int DT>
__device__ __forceinline__ float elem(const uint4& v, int e) {
  const uint32_t u = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return (e & 1) ? Fmt<DT>::hi(u) : Fmt<DT>::lo(u);
}

// One 32-bit word (two lanes) of the fold.  The pages' arithmetic is a
// float32 round-to-nearest addition rounded to the element format (BF16 or
// FP16).  The sum of two 16-bit values is exact in float32 unless it
// overflows or needs more than 24 significant bits, and rounding a float32
// result to a format of p <= 11 bits gives the correctly rounded sum
// whenever 24 >= 2p + 2 (double rounding is innocuous).  So the paired
// 16-bit addition, which rounds the exact sum once, gives the same bits
// (subnormals and signed zeros included) in one instruction per pair.
template <bool ADD2, int DT>
__device__ __forceinline__ uint32_t fold_word(uint32_t p, uint32_t a, uint32_t a2) {
  using F = Fmt<DT>;
  const uint32_t s = ADD2 ? F::add(a, a2) : a;
  return F::add(p, s);
}

template <bool ADD2, int DT>
__device__ __forceinline__ uint4 fold_chunk(const uint4& p, const uint4& a, const uint4& a2) {
  uint4 r;
  r.x = fold_word<ADD2, DT>(p.x, a.x, a2.x);
  r.y = fold_word<ADD2, DT>(p.y, a.y, a2.y);
  r.z = fold_word<ADD2, DT>(p.z, a.z, a2.z);
  r.w = fold_word<ADD2, DT>(p.w, a.w, a2.w);
  return r;
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Ask L2 to fetch `bytes` (a multiple of 16) from a 16-byte aligned global
// address.  A hint only: L2 is coherent, so a prefetch issued before an
// earlier kernel's writes have landed cannot make a later load stale.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the same shared-memory location (given as a
// shared::cta address) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// ---- mbarrier and remote-store primitives of the cluster exchange

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the other CTAs of the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and expect `tx` bytes of remote stores in the current phase.
__device__ __forceinline__ void mbar_arm(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` to complete, for at most `limit_ns`.
static __device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                               unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Store one float into another CTA's shared memory and count its 4 bytes
// on that CTA's mbarrier (both addresses are shared::cluster addresses).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr),
               "f"(v), "r"(bar)
               : "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy, bypassing L1 (Ampere-style asynchronous copy).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}


// XOR-butterfly sums: every lane ends with the same bits, because each step
// adds the same two operands (in either order) in every lane of a pair.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// The maximum over the warp in one instruction (sm_100 family); NaN lanes
// are ignored, as by fmaxf.
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// Transpose-reduction of KP (a power of two <= 32) values per lane across the
// warp with KP-1 + (5 - log2 KP) shuffles.  Afterwards lane l holds the warp
// total of value index l >> (5 - log2 KP); lanes sharing an index agree.
template <int KP>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[KP], int lane) {
#pragma unroll
  for (int half = KP / 2, o = 16; half >= 1; half >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float give = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, give, o);
    }
  }
  float r = v[0];
  constexpr int LOGKP = (KP >= 32) ? 5 : (KP >= 16) ? 4 : (KP >= 8) ? 3 : (KP >= 4) ? 2 : 1;
  // lanes that differ only in the low 5 - log2(KP) bits hold partial sums of
  // the same index: finish them with plain butterfly steps
  constexpr int FIRST = (LOGKP < 5) ? (1 << (4 - LOGKP)) : 0;
#pragma unroll
  for (int o = FIRST; o > 0; o >>= 1) r += __shfl_xor_sync(FULL, r, o);
  return r;
}

template <int K>
struct Pow2 {
  static constexpr int value = K <= 2 ? 2 : K <= 4 ? 4 : K <= 8 ? 8 : K <= 16 ? 16 : 32;
  static constexpr int log2 = K <= 2 ? 1 : K <= 4 ? 2 : K <= 8 ? 3 : K <= 16 ? 4 : 5;
};

// The 2(N+1) sums of a token (ss_i, d_i for every source, in source order)
// are reduced in groups of up to 16 sources, one warp transpose-reduction of
// at most 32 values each: one group for N <= 15, two for N <= 31.  Group g
// is padded to KP<g> values; `total` floats per CTA cross the cluster.
template <int N>
struct Sums {
  static constexpr int S = N + 1;
  static constexpr int K = 2 * S;
  static constexpr int G = (K + 31) / 32;
  static constexpr int K0 = K < 32 ? K : 32;
  static constexpr int K1 = K - K0;
  static constexpr int KP0 = Pow2<K0>::value;
  static constexpr int KP1 = K1 > 0 ? Pow2<K1>::value : 0;
  static constexpr int SH0 = 5 - Pow2<K0>::log2;
  static constexpr int SH1 = 5 - Pow2<(K1 > 0 ? K1 : 1)>::log2;
  static constexpr int total = KP0 + KP1;
  static_assert(G <= 2, "at most 31 bank snapshots");
};

// ---------------------------------------------------------------- per token

// Shared memory of the per-token reductions.
//   red:  per-warp partials of R1 (local)
//   xin1: R1 totals pushed by each CTA of the cluster (st.async), by rank
//   xin2: per-warp sums of h^2 pushed by each CTA, index rank * warps + warp
//         (latency shapes: one CTA sum each, index rank; their per-warp sums
//         of h^2 are kept locally in xin2[128..143], which no CTA stores to)
//   bar1, bar2: mbarriers counting the bytes of xin1 / xin2 of one token
// Protocol per token k (phase parity k & 1 on both mbarriers):
//   R1: warp 0 of every CTA stores its Sums<N>::total totals into
//       xin1[rank] of every CTA with st.async (the latency shapes: warp c
//       into CTA c); every thread waits on bar1; thread 0 then re-arms
//       bar1 for token k+1.  The next write into red follows, in every warp,
//       the token's R2: after R2's CTA barrier in the latency shapes (which
//       every sending warp reaches after its sends), else after the R1 wait,
//       which needs warp 0's own store, made after its reads of red.
//   R2: lane c of every warp stores the warp's sum of h^2 into CTA c (the
//       latency shapes: lane c of warp 0 stores the CTA's sum, formed from
//       the warps' sums after a CTA barrier); every thread waits on bar2;
//       thread 0 re-arms bar2.
// A peer's next store into xin1 (token k+1) needs this CTA's R2(k) stores,
// which follow this CTA's reads of xin1(k) and its re-arm of bar1; its next
// store into xin2 needs this CTA's R1(k+1) stores, which follow the reads of
// xin2(k) and the re-arm of bar2.  So slots are never overwritten early, no
// phase can complete while a local thread still waits on the previous one,
// and the transaction count never runs ahead of its arming.  No CTA reads
// another's shared memory, so there is no barrier at exit.
template <int G>
struct alignas(16) Exchange {
  float red[16][32 * G];   // up to 16 warps (448-thread CTAs have 14)
  float xin1[16][32 * G];  // up to 16 CTAs per cluster
  float xin2[256];         // 16 CTAs x 16 warps
  float alpha[32 * G];     // softmax weights (shapes where one warp evaluates it)
  unsigned long long bar1;
  unsigned long long bar2;
};

struct Thread {
  int lane, warp, nwarps;
  uint32_t crank, csize;
  uint32_t phase;   // parity of the current token's exchange phase
  bool failed;      // an exchange wait timed out: stop waiting, report it
};

// Bytes each CTA expects per token: kp (Sums<N>::total) totals from every
// CTA (R1) and one float per warp of every CTA (R2), or one per CTA where
// the CTA sums its warps first (CTA_R2: the latency shapes).
__device__ __forceinline__ uint32_t r1_bytes(int kp, const Thread& t, const Params& p) {
  return static_cast<uint32_t>(kp) * t.csize * 4u + p.extra_tx;
}
template <bool CTA_R2>
__device__ __forceinline__ uint32_t r2_bytes(const Thread& t, const Params& p) {
  return (CTA_R2 ? 1u : static_cast<uint32_t>(t.nwarps)) * t.csize * 4u + p.extra_tx;
}

// Once per kernel, before the first exchange: thread 0 initialises and arms
// both mbarriers; the start of the cluster handshake (arrive now, wait
// before the first remote store) both publishes them and guarantees every
// CTA of the cluster runs.
template <int KP, bool CTA_R2, int G>
__device__ __forceinline__ void exchange_init(Exchange<G>& x, const Thread& t, const Params& p) {
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&x.bar1), 1);
    mbar_init(smem_u32(&x.bar2), 1);
    mbar_arm(smem_u32(&x.bar1), r1_bytes(KP, t, p));
    mbar_arm(smem_u32(&x.bar2), r2_bytes<CTA_R2>(t, p));
    fence_mbar_init();
  }
  cluster_arrive_relaxed();
}

__device__ __forceinline__ void exchange_wait(uint32_t bar, Thread& t, const Params& p) {
  if (t.failed || mbar_try_wait(bar, t.phase)) return;
  if (!mbar_wait_bounded(bar, t.phase, p.wait_ns)) {
    t.failed = true;
    atomicOr(p.status, kStatusWaitTimeout);
  }
}

// After a timed-out wait a peer may still be storing into this CTA's shared
// memory: stay resident (bounded) before exiting.
__device__ __forceinline__ void exchange_exit(const Thread& t, const Params& p) {
  if (!t.failed) return;
  const unsigned long long t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < p.wait_ns) {
  }
}

// Where a token's sources live between the two passes over them.
//   RegSources:  all N+1 chunks in registers (loaded once from HBM).
//   SmemSources: the N bank chunks in this thread's own slots of the
//                shared-memory ring, read once per pass; the updated prefix
//                in registers.
template <int N, int VPT>
struct RegSources {
  uint4 (&v)[N + 1][VPT];
  __device__ __forceinline__ uint4 get(int i, int k) const { return v[i][k]; }
  __device__ __forceinline__ void set_new_prefix(int k, const uint4& u) { v[N][k] = u; }
  __device__ __forceinline__ uint4 new_prefix(int k) const { return v[N][k]; }
  // Keep only the packed 16-bit words alive across the reductions: without
  // this the compiler reuses the unpacked floats of the first pass in the
  // mixture and holds twice the registers.
  __device__ __forceinline__ void fence() {
#pragma unroll
    for (int i = 0; i <= N; ++i)
#pragma unroll
      for (int k = 0; k < VPT; ++k)
        asm volatile("" : "+r"(v[i][k].x), "+r"(v[i][k].y), "+r"(v[i][k].z), "+r"(v[i][k].w));
  }
};

// Deep banks in the streaming shape: bank[0..NR-1] and the updated prefix in
// registers, bank[NR..N-1] in this thread's own slots of a shared-memory
// area (cp.async copies, read twice: sums, then mixture).
template <int N, int NR>
struct HybridSources {
  uint4 (&v)[NR + 1][1];   // bank[0..NR-1]; index NR holds the updated prefix
  uint32_t slot0;          // shared address of this thread's bank[NR] slot
  uint32_t step;           // bytes between consecutive rows
  bool ok;
  __device__ __forceinline__ uint4 get(int i, int) const {
    if (i < NR) return v[i][0];
    if (i == N) return v[NR][0];
    return ok ? lds16(slot0 + static_cast<uint32_t>(i - NR) * step) : make_uint4(0, 0, 0, 0);
  }
  __device__ __forceinline__ void set_new_prefix(int, const uint4& u) { v[NR][0] = u; }
  __device__ __forceinline__ uint4 new_prefix(int) const { return v[NR][0]; }
  __device__ __forceinline__ void fence() {
#pragma unroll
    for (int i = 0; i <= NR; ++i)
      asm volatile("" : "+r"(v[i][0].x), "+r"(v[i][0].y), "+r"(v[i][0].z), "+r"(v[i][0].w));
  }
};

template <int N>
struct SmemSources {
  uint32_t bank0;     // shared address of this thread's bank[0] slot
  uint32_t step;      // bytes between consecutive rows of a stage
  bool ok;
  uint4 np;
  __device__ __forceinline__ uint4 get(int i, int) const {
    if (i == N) return np;
    return ok ? lds16(bank0 + static_cast<uint32_t>(i) * step) : make_uint4(0, 0, 0, 0);
  }
  __device__ __forceinline__ void set_new_prefix(int, const uint4& u) { np = u; }
  __device__ __forceinline__ uint4 new_prefix(int) const { return np; }
  __device__ __forceinline__ void fence() {}
};

// Sums of squares and dot products with w of sources I0..I1-1 over this
// thread's chunks: part[2(i - I0)] = ss_i, part[2(i - I0) + 1] = d_i, the
// rest of the KP slots zero.
template <int VPT, int DT, class Src>
__device__ __forceinline__ void source_stats(const Src& src, int i, const uint4 (&wv)[VPT],
                                             float& ss, float& d) {
  ss = 0.f;
  d = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const uint4 u = src.get(i, k);
    Fmt<DT>::stats(u.x, wv[k].x, ss, d);
    Fmt<DT>::stats(u.y, wv[k].y, ss, d);
    Fmt<DT>::stats(u.z, wv[k].z, ss, d);
    Fmt<DT>::stats(u.w, wv[k].w, ss, d);
  }
}

template <int I0, int I1, int KP, int VPT, int DT, class Src>
__device__ __forceinline__ void source_sums(const Src& src, const uint4 (&wv)[VPT],
                                            float (&part)[KP]) {
#pragma unroll
  for (int i = I0; i < I1; ++i) {
    float ss = 0.f, d = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const uint4 u = src.get(i, k);
      Fmt<DT>::stats(u.x, wv[k].x, ss, d);
      Fmt<DT>::stats(u.y, wv[k].y, ss, d);
      Fmt<DT>::stats(u.z, wv[k].z, ss, d);
      Fmt<DT>::stats(u.w, wv[k].w, ss, d);
    }
    part[2 * (i - I0)] = ss;
    part[2 * (i - I0) + 1] = d;
  }
#pragma unroll
  for (int i = 2 * (I1 - I0); i < KP; ++i) part[i] = 0.f;
}

// The sums of sources I0..I1-1 (32 partials, padded with zeros) reduced over
// the warp: the result of source_sums followed by warp_transpose_reduce<32>,
// bit for bit, with the first transpose step (which pairs partial i with
// partial i + 16, i.e. source I0 + s with source I0 + 8 + s) taken as each
// upper source's sums are formed, so that 16 partials and the pair in hand
// are live instead of 32 beside the rows of every source.  The first group
// of the deep banks' sums uses it: their shapes spill much less (N = 24, 12
// rows in registers, 96 registers: 4 bytes against 40); the shallow shapes
// spill a little more with it, and keep the plain order.
template <int I0, int I1, int VPT, int DT, class Src>
__device__ __forceinline__ float sums_reduce_folded(const Src& src, const uint4 (&wv)[VPT], int lane) {
  constexpr int LO_END = I1 < I0 + 8 ? I1 : I0 + 8;
  float v[16];
  source_sums<I0, LO_END, 16, VPT, DT>(src, wv, v);
  const bool upper = (lane & 16) != 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    float b[2] = {0.f, 0.f};
    if (I0 + 8 + s < I1) source_stats<VPT, DT>(src, I0 + 8 + s, wv, b[0], b[1]);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 2 * s + j;
      const float give = upper ? v[i] : b[j];
      const float keep = upper ? b[j] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, give, 16);
    }
  }
  // the remaining steps of warp_transpose_reduce<32>
#pragma unroll
  for (int half = 8, o = 8; half >= 1; half >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float give = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, give, o);
    }
  }
  return v[0];
}

// Everything after the loads for one token: fold, sums, both exchanges,
// softmax, mixture, and the two stores.  pr/ad/ad2 are the token's prefix and
// addend chunks, src gives the bank chunks (and receives the updated prefix),
// wv the pseudo-query chunks; masked chunks (ok false) are zeros and store
// nothing.  LAT (the latency shapes) adds the R2 partials in every lane
// instead of with shuffles: the same bits, a shorter dependent chain.
template <int N, int MODE, int VPT, int DT, bool LAT, bool SMX, class Src>
__device__ __forceinline__ void token_epilogue(const Params& p, Exchange<Sums<N>::G>& x, Thread& t,
                                               size_t row, const int (&jj)[VPT],
                                               const bool (&ok)[VPT], const uint4 (&wv)[VPT],
                                               const uint4 (&gv)[VPT],
                                               const uint4 (&pr)[VPT], const uint4 (&ad)[VPT],
                                               const uint4 (&ad2)[VPT], Src& src, bool& first) {
  using SL = Sums<N>;
  constexpr int S = SL::S;             // sources: bank[0..N-1], new prefix
  constexpr int S0 = S < 16 ? S : 16;  // sources of the first group
  const int lane = t.lane, warp = t.warp;

  // ---- fold.  The latency shapes store the updated prefix at once, so that
  // the store has drained by the end of the call; the streaming shapes
  // store it at the end with the output (GB300: within noise there).
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    src.set_new_prefix(k, MODE == kNoFold ? pr[k] : fold_chunk<MODE == kFoldAdd2, DT>(pr[k], ad[k], ad2[k]));
    if constexpr (LAT && MODE != kNoFold)
      if (ok[k]) st_out(p.new_prefix + row + jj[k], src.new_prefix(k));
  }

  // ---- per-source sums of squares and dot products with w, and R1: warp
  // transpose-reduction per group, CTA sum, st.async to every CTA
  float wt0, wt1 = 0.f;
  if constexpr (SL::G == 1) {
    float part0[SL::KP0];
    source_sums<0, S0, SL::KP0, VPT, DT>(src, wv, part0);
    src.fence();
    wt0 = warp_transpose_reduce<SL::KP0>(part0, lane);
  } else {
    static_assert(SL::KP0 == 32, "the second group exists only beside a full first one");
    wt0 = sums_reduce_folded<0, S0, VPT, DT>(src, wv, lane);
    float part1[SL::KP1 > 0 ? SL::KP1 : 1];
    source_sums<16, S, (SL::KP1 > 0 ? SL::KP1 : 1), VPT, DT>(src, wv, part1);
    src.fence();
    wt1 = warp_transpose_reduce<SL::KP1>(part1, lane);
  }
  if ((lane & ((1 << SL::SH0) - 1)) == 0) x.red[warp][lane >> SL::SH0] = wt0;
  if constexpr (SL::G == 2)
    if ((lane & ((1 << SL::SH1) - 1)) == 0) x.red[warp][32 + (lane >> SL::SH1)] = wt1;
  __syncthreads();
  const uint32_t bar1 = smem_u32(&x.bar1), bar2 = smem_u32(&x.bar2);
  // The first remote store of the kernel waits for every CTA of the cluster
  // to run and to have set up its mbarriers (see exchange_init).
  if (first) {
    cluster_wait();
    first = false;
  }
  // Warp 0 forms the CTA's totals and stores them into every CTA; in the
  // latency shapes warps 0..C-1 each form them (the same additions in the
  // same order) and warp c stores into CTA c (GB300, same-box A/B: -0.01 to
  // -0.06 us on 15 of 16 decode shapes, M = 32, N = 12 unchanged).
  if (LAT ? static_cast<uint32_t>(warp) < t.csize : warp == 0) {
#pragma unroll
    for (int g = 0; g < SL::G; ++g) {
      const int kp = g == 0 ? SL::KP0 : SL::KP1;
      if (lane < kp) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w)
          if (w < t.nwarps) s += x.red[w][32 * g + lane];
        const uint32_t a = smem_u32(&x.xin1[t.crank][32 * g + lane]);
        if (LAT) {
          for (uint32_t c = warp; c < t.csize; c += t.nwarps)
            st_async_f32(dsmem_map(a, c), s, dsmem_map(bar1, c));
        } else {
          for (uint32_t c = 0; c < t.csize; ++c) st_async_f32(dsmem_map(a, c), s, dsmem_map(bar1, c));
        }
      }
    }
  }
  exchange_wait(bar1, t, p);
  if (threadIdx.x == 0 && !t.failed) mbar_arm(bar1, r1_bytes(SL::total, t, p));  // next token
  // ---- cluster totals, logits and softmax (in one warp: lane i < S returns
  // the weight of source i)
  auto softmax = [&]() -> float {
    // cluster totals: lane l of tot[g] holds sum 32 g + l
    float tot[SL::G];
#pragma unroll
    for (int g = 0; g < SL::G; ++g) {
      const int kp = g == 0 ? SL::KP0 : SL::KP1;
      tot[g] = 0.f;
      if (lane < kp) {
#pragma unroll
        for (uint32_t c = 0; c < 16; ++c)
          if (c < t.csize) tot[g] += x.xin1[c][32 * g + lane];
      }
    }

    // logits and softmax, lane i < S holds source i (sums 2i and 2i + 1 sit
    // in group i / 16 at lanes (2i) mod 32 and (2i + 1) mod 32)
    float ss_i = __shfl_sync(FULL, tot[0], (2 * lane) & 31);
    float d_i = __shfl_sync(FULL, tot[0], (2 * lane + 1) & 31);
    if constexpr (SL::G == 2) {
      const float ss1 = __shfl_sync(FULL, tot[SL::G - 1], (2 * lane) & 31);
      const float d1 = __shfl_sync(FULL, tot[SL::G - 1], (2 * lane + 1) & 31);
      if (lane >= 16) {
        ss_i = ss1;
        d_i = d1;
      }
    }
    const float logit = (lane < S) ? rsqrtf(__fmaf_rn(ss_i, p.inv_h, p.eps)) * d_i : -INFINITY;
    // up to 16 sources sit in lanes 0..15: reduce over 16 lanes, else 32
    const float mx = S <= 16 ? half_warp_max(logit) : warp_max(logit);
    const float ex = (lane < S) ? __expf(logit - mx) : 0.f;
    const float den = S <= 16 ? half_warp_sum(ex) : warp_sum(ex);
    return ex / den;
  };
  float alpha[S];
  float den = 1.f;   // latency shapes: the sum of the unnormalised weights
  if constexpr (SMX) {
    // the streaming shapes of up to 12 snapshots: one warp evaluates the
    // softmax, the others read the weights after a CTA barrier (its next
    // write follows the next token's R1 barrier, which every warp passes
    // after these reads).  GB300, same-box A/B: M = 8192 +1..3 % at
    // N = 1..9 and FP16 N = 12, BF16 N = 12 unchanged, M = 96 +4 %; with the
    // four to seven CTAs per SM of the deep shapes the barrier cost 14-19 %,
    // so those keep every warp evaluating it (as do the latency shapes,
    // where it would add a barrier to the critical path).
    if (warp == 0) {
      const float alpha_l = softmax();
      if (lane < S) x.alpha[lane] = alpha_l;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < S; ++i) alpha[i] = x.alpha[i];
  } else if constexpr (LAT) {
    // Every warp evaluates it, with the shortest dependent chain in front of
    // the mixture: lane i reads the pair (ss_i, d_i) of each CTA (the same
    // additions, in the same order, as the totals above), the maximum is one
    // redux.sync, and the mixture takes e_i = exp(l_i - max) while the sum
    // of the e_i is formed beside it.  With h' = sum_i e_i v_i = den * h,
    // RMSNorm(h) = h' * rsqrt(mean(h'^2) + eps * den^2) exactly, so den
    // enters only r_h (and the tap's h = h' / den).  GB300, graphs of
    // back-to-back calls, same-box A/B: -0.05 to -0.12 us on every decode
    // shape (M <= 32, N = 1..12); out differs from the normalised form in
    // a few elements by one BF16 ulp.
    float ss_i = 0.f, d_i = 0.f;
    if (lane < S) {
#pragma unroll
      for (uint32_t c = 0; c < 16; ++c)
        if (c < t.csize) {
          const float2 f = *reinterpret_cast<const float2*>(&x.xin1[c][2 * lane]);
          ss_i += f.x;
          d_i += f.y;
        }
    }
    const float logit = (lane < S) ? rsqrtf(__fmaf_rn(ss_i, p.inv_h, p.eps)) * d_i : -INFINITY;
    const float mx = redux_max(logit);
    const float ex = (lane < S) ? __expf(logit - mx) : 0.f;
    den = warp_sum(ex);   // lanes >= S add zeros: the same bits in every lane
#pragma unroll
    for (int i = 0; i < S; ++i) alpha[i] = __shfl_sync(FULL, ex, i);
  } else {
    // every warp evaluates it from identical totals in identical order:
    // bit-identical weights everywhere, no barrier
    const float alpha_l = softmax();
#pragma unroll
    for (int i = 0; i < S; ++i) alpha[i] = __shfl_sync(FULL, alpha_l, i);
  }

  // ---- mixture h = sum_i alpha_i v_i, and sum h^2
  float h[VPT][8];
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if constexpr (VPT == 1) {
      // packed float32x2 arithmetic (each lane a mul.rn / fma.rn.f32: the
      // same bits as the scalar form, half the instructions; GB300,
      // M = 8192, N = 12: +2 % bandwidth for the FMAs)
      unsigned long long h2[4];
      {
        const uint4 u = src.get(0, k);
        const unsigned long long a2 = pack_f32x2(alpha[0], alpha[0]);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
          h2[q2] = mul_rn_x2(a2, pack_f32x2(Fmt<DT>::lo(w4[q2]), Fmt<DT>::hi(w4[q2])));
      }
#pragma unroll
      for (int i = 1; i < S; ++i) {
        const uint4 u = src.get(i, k);
        const unsigned long long a2 = pack_f32x2(alpha[i], alpha[i]);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
          fma_rn_x2(h2[q2], a2, pack_f32x2(Fmt<DT>::lo(w4[q2]), Fmt<DT>::hi(w4[q2])));
      }
      // sum of squares: even and odd columns in the two lanes, then added
      unsigned long long q2 = pack_f32x2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) fma_rn_x2(q2, h2[j], h2[j]);
      float qe, qo;
      unpack_f32x2(q2, qe, qo);
      q = add_rn(qe, qo);
#pragma unroll
      for (int q2i = 0; q2i < 4; ++q2i) unpack_f32x2(h2[q2i], h[k][2 * q2i], h[k][2 * q2i + 1]);
    } else {
      // two chunks per thread: the packed form costs more registers than it
      // saves instructions
      {
        const uint4 u = src.get(0, k);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[k][e] = mul_rn(alpha[0], elem<DT>(u, e));
      }
#pragma unroll
      for (int i = 1; i < S; ++i) {
        const uint4 u = src.get(i, k);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[k][e] = fma_rn(alpha[i], elem<DT>(u, e), h[k][e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) q = fma_rn(h[k][e], h[k][e], q);
    }
  }

  // ---- R2: warp sum, lane c stores it into CTA c, every warp sums all
  // warps of all CTAs in one fixed order.  The latency shapes add the warps'
  // sums in the CTA first (a CTA barrier) and send one float per CTA: GB300,
  // same-box A/B, -0.02 to -0.08 us on every decode shape against 4-8 floats
  // per CTA and 16-32 partials summed in every lane
  q = warp_sum(q);
  if constexpr (LAT) {
    // the warps' sums in xin2[128..] rather than in a member of their own:
    // 64 more bytes of static shared memory cost the N = 12 streaming
    // shapes 1-2 % (GB300, same-box A/B)
    float* red2 = &x.xin2[128];
    if (lane == 0) red2[warp] = q;
    __syncthreads();
    if (warp == 0) {
      float sq = 0.f;
#pragma unroll
      for (int w = 0; w < 16; ++w)
        if (w < t.nwarps) sq += red2[w];
      if (static_cast<uint32_t>(lane) < t.csize)
        st_async_f32(dsmem_map(smem_u32(&x.xin2[t.crank]), lane), sq, dsmem_map(bar2, lane));
    }
  } else {
    if (static_cast<uint32_t>(lane) < t.csize)
      st_async_f32(dsmem_map(smem_u32(&x.xin2[t.crank * t.nwarps + warp]), lane), q,
                   dsmem_map(bar2, lane));
  }
  exchange_wait(bar2, t, p);
  if (threadIdx.x == 0 && !t.failed) mbar_arm(bar2, r2_bytes<LAT>(t, p));  // next token
  t.phase ^= 1u;
  float qq = 0.f;
  if constexpr (LAT) {
    // every lane adds the CTAs' sums in rank order
#pragma unroll
    for (uint32_t c = 0; c < 16; ++c)
      if (c < t.csize) qq += x.xin2[c];
  } else {
    const int nw_total = static_cast<int>(t.csize) * t.nwarps;
    for (int idx = lane; idx < nw_total; idx += 32) qq += x.xin2[idx];
    qq = warp_sum(qq);
  }
  const float rh = rsqrtf(__fmaf_rn(qq, p.inv_h, LAT ? p.eps * (den * den) : p.eps));

  // ---- outputs (after a timed-out exchange wait the sums are partial: out
  // and h_out are written as NaN, so that no wrong value passes as a
  // result; new_prefix does not depend on the exchange and stays exact)
  const uint4 nan4 = make_uint4(Fmt<DT>::kNaN2, Fmt<DT>::kNaN2, Fmt<DT>::kNaN2, Fmt<DT>::kNaN2);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if (ok[k]) {
      if (MODE != kNoFold && !LAT) st_out(p.new_prefix + row + jj[k], src.new_prefix(k));
      if (p.h_out != nullptr) {
        // the latency shapes hold h' = den * h
        const float hs = LAT ? 1.f / den : 1.f;
        uint4 hv;
        hv.x = Fmt<DT>::pack(h[k][0] * hs, h[k][1] * hs);
        hv.y = Fmt<DT>::pack(h[k][2] * hs, h[k][3] * hs);
        hv.z = Fmt<DT>::pack(h[k][4] * hs, h[k][5] * hs);
        hv.w = Fmt<DT>::pack(h[k][6] * hs, h[k][7] * hs);
        st_out(p.h_out + row + jj[k], t.failed ? nan4 : hv);
      }
      // (h * r_h) * gamma, two lanes per instruction, each product rounded
      const unsigned long long rh2 = pack_f32x2(rh, rh);
      const uint32_t g4[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
      uint32_t o4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned long long v2 =
            mul_rn_x2(mul_rn_x2(pack_f32x2(h[k][2 * j], h[k][2 * j + 1]), rh2),
                      pack_f32x2(Fmt<DT>::lo(g4[j]), Fmt<DT>::hi(g4[j])));
        float lo, hi;
        unpack_f32x2(v2, lo, hi);
        o4[j] = Fmt<DT>::pack(lo, hi);
      }
      const uint4 o = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      st_out(p.out + row + jj[k], t.failed ? nan4 : o);
    }
  }
}


__device__ __forceinline__ Thread thread_info() {
  Thread t;
  t.lane = threadIdx.x & 31;
  t.warp = threadIdx.x >> 5;
  t.nwarps = blockDim.x >> 5;
  t.crank = cluster_ctarank();
  t.csize = cluster_nctarank();
  t.phase = 0;
  t.failed = false;
  return t;
}

// ---------------------------------------------------------------- kernels

// Loads straight to registers; each cluster handles the tokens of its
// TokenWalk.  DT is the element format of every tensor.
// NR < N keeps bank rows NR..N-1 in shared memory instead (HybridSources;
// one column chunk per thread).
template <int N, int MODE, int VPT, int MAXT, int MINB, int DT = kBF16, int NR = N>
__global__ void __launch_bounds__(MAXT, MINB) attnres_fused_kernel(const Params p) {
  constexpr bool HYB = NR < N;
  static_assert(!HYB || VPT == 1, "shared-memory rows take one chunk per thread");
  // the latency shapes (split, split with two CTAs per SM, one CTA per
  // token): at most a few warps per SM, latency rather than issue bound
  constexpr bool LAT = (MINB <= 2) && (MAXT >= 256);
  // one warp evaluates the softmax: the streaming shapes of up to 12 snapshots
  constexpr bool SMX = !LAT && N <= kShallowMaxN;
  __shared__ Exchange<Sums<N>::G> x;
  extern __shared__ __align__(16) uint4 hyb[];   // [N - NR][blockDim.x] when HYB
  Thread t = thread_info();
  using Walk = TokenWalk<LAT>;
  const int m0 = Walk::first(p, static_cast<int>(blockIdx.y));
  const int c0 = static_cast<int>(t.crank) * p.cpc;
  const int cend = min(c0 + p.cpc, p.H8);
  int jj[VPT];
  bool ok[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    jj[k] = c0 + static_cast<int>(threadIdx.x) + k * static_cast<int>(blockDim.x);
    ok[k] = jj[k] < cend;
  }

  // Latency regime: let the next kernel on the stream be scheduled at once
  // (it still waits for this grid to finish before touching memory), and
  // start pulling this CTA's slice of its first token into L2 while the
  // previous kernel finishes.
  if (p.prefetch & 2) griddep_launch_dependents();
  if (p.prefetch & 1) {
    const int rows = N + (MODE == kNoFold ? 1 : MODE == kFoldAdd ? 2 : 3) + 2;
    // (a hint: with fewer threads than rows, the last rows go without)
    if (static_cast<int>(threadIdx.x) < rows && cend > c0 && m0 < p.M) {
      const int r = threadIdx.x;
      const size_t off = static_cast<size_t>(m0) * p.H8 + c0;
      const uint32_t bytes = static_cast<uint32_t>(cend - c0) * 16u;
      const uint4* src = r < N ? p.bank + r * p.bank_stride + off
                       : r == N ? p.prefix + off
                       : r == N + 1 && MODE != kNoFold ? p.add + off
                       : r == N + 2 && MODE == kFoldAdd2 ? p.add2 + off
                       : r == rows - 2 ? p.w + c0 : p.gamma + c0;
      prefetch_l2(src, bytes);
    }
  }
  // Distributed shared memory may be written only once every CTA of the
  // cluster runs and has set up its mbarriers: set them up and arrive, wait
  // just before the first remote store.  In the latency regime this happens
  // here, overlapping the previous kernel's tail (shared memory only); in the
  // streaming regime after the first token's loads are issued, so that the
  // set-up does not delay them.
  const bool early_init = p.prefetch != 0;
  if (early_init && m0 < p.M) exchange_init<Sums<N>::total, LAT>(x, t, p);
  // Latency regime, bit 3: before the wait, read one 32-bit word of every
  // 128-byte line of this CTA's first-token rows (through L2 only, never
  // allocated in L1).  On GB300 lines an SM has read are served to it faster
  // afterwards than lines only prefetched into L2: cold decode calls gain
  // 0.25-0.35 us, warm ones up to 0.15 us (M <= 16).  The words are
  // combined and tested here, before the wait, so that the reads complete
  // before it (a read whose value is used only after the wait may be moved
  // past it); a test that can never be true keeps them.  The values are
  // discarded, and the loads after the wait see the previous kernel's writes.
  if constexpr (VPT == 1 && !HYB) {
    if ((p.prefetch & 8) && m0 < p.M && ok[0] && (jj[0] & 7) == 0) {
      const size_t off = static_cast<size_t>(m0) * p.H8 + jj[0];
      constexpr int WROWS = N + (MODE == kNoFold ? 1 : MODE == kFoldAdd ? 2 : 3);
      uint32_t acc = 0;
#pragma unroll
      for (int r = 0; r < WROWS; ++r)
        acc ^= ld_l2_word(r < N ? p.bank + r * p.bank_stride + off
                          : r == N ? p.prefix + off : r == N + 1 ? p.add + off : p.add2 + off);
      if (acc == 0x9e3779b9u && p.M < 0) atomicOr(p.status, 0u);   // never taken (M >= 1)
    }
  }
  // Programmatic dependent launch: this grid may have been scheduled while
  // the previous kernel on the stream was still running; wait for it to
  // complete (and its writes to be visible) before reading its outputs.
  // Without the launch attribute this returns at once.
  griddep_wait();

  uint4 wv[VPT], gv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    wv[k] = ok[k] ? ld_keep(p.w + jj[k]) : make_uint4(0, 0, 0, 0);
    gv[k] = ok[k] ? ld_keep(p.gamma + jj[k]) : make_uint4(0, 0, 0, 0);
  }

  bool first = true;
  for (int m = m0; m < p.M; m = Walk::next(p, m, static_cast<int>(gridDim.y))) {
    const size_t row = static_cast<size_t>(m) * p.H8;
    uint4 v[NR + 1][VPT];
    uint4 pr[VPT], ad[VPT], ad2[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      pr[k] = ok[k] ? ld_stream(p.prefix + row + jj[k]) : z;
      ad[k] = (MODE != kNoFold && ok[k]) ? ld_stream(p.add + row + jj[k]) : z;
      ad2[k] = (MODE == kFoldAdd2 && ok[k]) ? ld_stream(p.add2 + row + jj[k]) : z;
#pragma unroll
      for (int i = 0; i < NR; ++i)
        v[i][k] = ok[k] ? ld_stream(p.bank + i * p.bank_stride + row + jj[k]) : z;
    }
    const uint32_t hyb0 = smem_u32(hyb) + threadIdx.x * 16u;
    const uint32_t hstep = blockDim.x * 16u;
    if constexpr (HYB) {
      if (ok[0]) {
#pragma unroll
        for (int i = NR; i < N; ++i)
          cp_async16(hyb0 + static_cast<uint32_t>(i - NR) * hstep, p.bank + i * p.bank_stride + row + jj[0]);
      }
      cp_async_commit();
    }
    // While this token is reduced, let L2 fetch this CTA's rows of the next
    // token it will take: the requests keep HBM busy during the reductions
    // and the next loads hit L2.
    if ((p.prefetch & 4) && Walk::next(p, m, static_cast<int>(gridDim.y)) < p.M) {
      constexpr int rows = N + (MODE == kNoFold ? 1 : MODE == kFoldAdd ? 2 : 3);
      if (static_cast<int>(threadIdx.x) < rows && cend > c0) {
        const int r = threadIdx.x;
        const size_t off = static_cast<size_t>(Walk::next(p, m, static_cast<int>(gridDim.y))) * p.H8 + c0;
        const uint4* src = r < N ? p.bank + r * p.bank_stride + off
                         : r == N ? p.prefix + off
                         : r == N + 1 ? p.add + off : p.add2 + off;
        prefetch_l2(src, static_cast<uint32_t>(cend - c0) * 16u);
      }
    }
    // Let the next kernel on the stream be scheduled once every CTA of this
    // grid is past its first loads; it still waits for this grid to finish.
    if (m == m0) griddep_launch_dependents();
    if (!early_init && m == m0) exchange_init<Sums<N>::total, LAT>(x, t, p);
    if constexpr (HYB) {
      cp_async_wait<0>();   // this thread's own slots: no barrier needed
      HybridSources<N, NR> src{v, hyb0, hstep, ok[0]};
      token_epilogue<N, MODE, VPT, DT, LAT, SMX>(p, x, t, row, jj, ok, wv, gv, pr, ad, ad2, src, first);
    } else {
      RegSources<N, VPT> src{v};
      token_epilogue<N, MODE, VPT, DT, LAT, SMX>(p, x, t, row, jj, ok, wv, gv, pr, ad, ad2, src, first);
    }
  }
  exchange_exit(t, p);
}

// Persistent streaming kernel: each cluster walks tokens blockIdx.y +
// k * gridDim.y; every thread copies its own chunk of each source row of the
// token STAGES-1 steps ahead into its private slots of a shared-memory ring
// (cp.async), so HBM reads stay in flight through the reductions of the
// current token.  The bank chunks are read from the ring once per pass (sums,
// then mixture) instead of being held in registers, which keeps the kernel
// small enough for several CTAs per SM.  A thread only ever reads slots it
// filled itself, so the ring needs no barrier beyond cp.async.wait_group.
template <int N, bool ADD2, int MAXT, int MINB, int STAGES>
__global__ void __launch_bounds__(MAXT, MINB) attnres_pipe_kernel(const Params p) {
  constexpr int ROWS = N + (ADD2 ? 3 : 2);   // prefix, add, [add2], bank[0..N-1]
  extern __shared__ uint4 ring[];             // [STAGES][ROWS][blockDim.x]
  __shared__ Exchange<Sums<N>::G> x;
  Thread t = thread_info();
  const int c0 = static_cast<int>(t.crank) * p.cpc;
  const int cend = min(c0 + p.cpc, p.H8);
  const int jj1 = c0 + static_cast<int>(threadIdx.x);
  const int jj[1] = {jj1};
  const bool ok[1] = {jj1 < cend};
  const uint32_t ring0 = smem_u32(ring) + threadIdx.x * 16u;
  const uint32_t row_step = blockDim.x * 16u;
  const uint32_t stage_step = ROWS * row_step;

  exchange_init<Sums<N>::total, false>(x, t, p);
  griddep_wait();
  const uint4 wv[1] = {ok[0] ? ld_keep(p.w + jj1) : make_uint4(0, 0, 0, 0)};
  const uint4 gv[1] = {ok[0] ? ld_keep(p.gamma + jj1) : make_uint4(0, 0, 0, 0)};

  auto issue = [&](int m, int stage) {
    if (m < p.M && ok[0]) {
      const size_t off = static_cast<size_t>(m) * p.H8 + jj1;
      uint32_t d = ring0 + stage * stage_step;
      cp_async16(d, p.prefix + off);
      d += row_step;
      cp_async16(d, p.add + off);
      d += row_step;
      if (ADD2) {
        cp_async16(d, p.add2 + off);
        d += row_step;
      }
#pragma unroll
      for (int i = 0; i < N; ++i, d += row_step) cp_async16(d, p.bank + i * p.bank_stride + off);
    }
    cp_async_commit();  // an empty group keeps the group count uniform
  };

  const int G = gridDim.y;
  const int m0 = blockIdx.y;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) issue(m0 + s * G, s);
  griddep_launch_dependents();

  bool first = true;
  int stage = 0;
  for (int m = m0; m < p.M; m += G) {
    const int ahead = (stage + STAGES - 1) % STAGES;
    issue(m + (STAGES - 1) * G, ahead);
    cp_async_wait<STAGES - 1>();
    uint4 pr[1], ad[1], ad2[1];
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint32_t a = ring0 + stage * stage_step;
    pr[0] = ok[0] ? lds16(a) : z;
    a += row_step;
    ad[0] = ok[0] ? lds16(a) : z;
    a += row_step;
    ad2[0] = z;
    if (ADD2) {
      ad2[0] = ok[0] ? lds16(a) : z;
      a += row_step;
    }
    SmemSources<N> src{a, row_step, ok[0], z};
    token_epilogue<N, ADD2 ? kFoldAdd2 : kFoldAdd, 1, kBF16, false, false>(p, x, t, static_cast<size_t>(m) * p.H8, jj,
                                                     ok, wv, gv, pr, ad, ad2, src, first);
    stage = (stage + 1 == STAGES) ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  if (first) cluster_wait();  // a cluster with no token still pairs its arrive
  exchange_exit(t, p);
}

// The standalone fold: new_prefix = bf16(prefix + bf16(add + add2)) (or
// bf16(prefix + add)) over n 16-byte chunks, grid-stride, 16-byte vectors.
// The addition that the fused kernel replaces; kept for comparison.
// new_prefix may be prefix itself (in place): prefix is read with a
// coherent load, and neither pointer is marked restrict.
template <bool ADD2, int DT>
__global__ void __launch_bounds__(256) attnres_tail_add_kernel(const uint4* prefix,
                                                               const uint4* __restrict__ add,
                                                               const uint4* __restrict__ add2,
                                                               uint4* new_prefix,
                                                               long long n) {
  griddep_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const uint4 a2 = ADD2 ? ld_stream(add2 + i) : make_uint4(0, 0, 0, 0);
    st_out(new_prefix + i, fold_chunk<ADD2, DT>(ld_stream(prefix + i), ld_stream(add + i), a2));
  }
  griddep_launch_dependents();
}

// The access pattern of the streaming fused kernel without its arithmetic:
// the same grid of clusters walking tokens, the same 16-byte loads of every
// row chunk (prefix, add, add2, bank[0..N-1]), the same next-token L2
// prefetch and the same two 16-byte stores per chunk, but no fold, sums,
// exchanges or mixture: new_prefix receives the prefix chunk and out the XOR
// of all loaded chunks (which keeps every load live).  A measurement of how
// fast this GPU serves the fused kernel's traffic, not a result.
template <int N>
__global__ void __launch_bounds__(kPatternMaxT) attnres_pattern_kernel(const Params p) {
  const int c0 = static_cast<int>(cluster_ctarank()) * p.cpc;
  const int cend = min(c0 + p.cpc, p.H8);
  const int j = c0 + static_cast<int>(threadIdx.x);
  const bool ok = j < cend;
  griddep_wait();
  const int G = static_cast<int>(gridDim.y);
  for (int m = TokenWalk<false>::first(p, static_cast<int>(blockIdx.y)); m < p.M;
       m = TokenWalk<false>::next(p, m, G)) {
    const size_t row = static_cast<size_t>(m) * p.H8;
    uint4 v[N + 3];
    const uint4 z = make_uint4(0, 0, 0, 0);
    v[0] = ok ? ld_stream(p.prefix + row + j) : z;
    v[1] = ok ? ld_stream(p.add + row + j) : z;
    v[2] = ok ? ld_stream(p.add2 + row + j) : z;
#pragma unroll
    for (int i = 0; i < N; ++i) v[3 + i] = ok ? ld_stream(p.bank + i * p.bank_stride + row + j) : z;
    if ((p.prefetch & 4) && TokenWalk<false>::next(p, m, G) < p.M) {
      constexpr int rows = N + 3;
      if (static_cast<int>(threadIdx.x) < rows && cend > c0) {
        const int r = threadIdx.x;
        const size_t off = static_cast<size_t>(TokenWalk<false>::next(p, m, G)) * p.H8 + c0;
        const uint4* src = r < N ? p.bank + r * p.bank_stride + off
                         : r == N ? p.prefix + off : r == N + 1 ? p.add + off : p.add2 + off;
        prefetch_l2(src, static_cast<uint32_t>(cend - c0) * 16u);
      }
    }
    griddep_launch_dependents();
    uint4 x = v[0];
#pragma unroll
    for (int i = 1; i < N + 3; ++i) {
      x.x ^= v[i].x;
      x.y ^= v[i].y;
      x.z ^= v[i].z;
      x.w ^= v[i].w;
    }
    if (ok) {
      st_out(p.new_prefix + row + j, v[0]);
      st_out(p.out + row + j, x);
    }
  }
}

// Host-side launchers of one instantiation (defined in attnres_launch.cuh).
template <int N, int MODE, int VPT, int MAXT, int MINB, int DT = kBF16, int NR = N>
cudaError_t launch_fused(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                         cudaStream_t s);
template <int N, bool ADD2, int STAGES>
cudaError_t launch_pipe(const Params& p, dim3 grid, int threads, int cluster, bool pdl,
                        cudaStream_t s);
template <bool ADD2, int DT>
cudaError_t launch_tail_add(const uint4* prefix, const uint4* add, const uint4* add2,
                            uint4* new_prefix, long long chunks, int sms, bool pdl,
                            cudaStream_t s);
template <int N>
cudaError_t launch_pattern(const Params& p, dim3 grid, int threads, int cluster, cudaStream_t s);

}  // namespace attnres
