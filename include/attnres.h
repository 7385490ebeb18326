/*
 * attnres.h -- C ABI of the GB300 (sm_103a) fused AttnRes + add2 + RMSNorm
 * decode-layer epilogue.
 *
 * The operation, per token m of M (H columns, all tensors BF16):
 *
 *   1. Fold of the deferred MoE tail into the prefix sum.
 *        s          = bf16(add + add2)     (s = add when add2 is NULL)
 *        new_prefix = bf16(prefix + s)
 *      Both additions are float32 round-to-nearest-even with subnormals kept
 *      (no flush to zero); each result is rounded to BF16 to nearest even.
 *      This is bit for bit the result of the two BF16 tensor additions, and
 *      bit for bit the exact sum rounded once to BF16 (float32 holds the
 *      sum of two BF16 values closely enough that the second rounding never
 *      differs), which is how the kernels compute it.
 *      Defined in: TensorRT-LLM PR #20546 ("Kimi K3: fold the MoE-tail
 *      additions into the next attention-residual"), section "Op", the
 *      optional trailing layer_residual_add2 of attn_res_add_rmsnorm_fwd.
 *   2. Attention-residual depth mixture over the N bank snapshots
 *      v_0..v_{N-1} = bank[0..N-1, m, :] and the updated prefix
 *      v_N = new_prefix[m, :]:
 *        l_i   = w . RMSNorm(v_i) = (w . v_i) / sqrt(mean(v_i^2) + eps)
 *        alpha = softmax(l)
 *        h     = sum_i alpha_i v_i                   (float32)
 *   3. out = bf16( h / sqrt(mean(h^2) + eps) * gamma ), one final rounding.
 *      Steps 2-3 are the attention-residual + RMSNorm consumer that the same
 *      PR page names (sections "Description" and "Op"); the page does not
 *      write their math out, and the form above is the specification this
 *      library implements.
 *
 * Conventions shared by every entry point
 *   - Tensors are BF16 (FP16 for the _f16 entry point and dtype
 *     ATTNRES_DTYPE_FP16) stored as 16-bit words, row-major, contiguous, in
 *     device memory of the current CUDA device, each 16-byte aligned.
 *     [M,H] tensors have row stride H; the bank is [N,M,H] (snapshot-major:
 *     snapshot i of token m starts at element (i*M + m)*H).
 *   - The caller owns every buffer.  The library allocates nothing per call,
 *     keeps no pointer after the call returns, and needs no workspace.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     nothing is synchronised on the host.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and returns a negative status.  A failed launch returns
 *     ATTNRES_ERR_CUDA and attnres_last_cuda_error() holds the cudaError_t.
 *     No entry point aborts, traps or prints.
 *   - A failure inside a running kernel cannot be returned by the call (it
 *     is asynchronous).  The one the kernels detect is a CTA of a cluster
 *     waiting longer than a time limit (200 ms) for its peers' partial
 *     sums, which happens only if the GPU does not run the CTAs of a cluster
 *     together.  The kernel then finishes without hanging: the CTAs that
 *     gave up write NaN into their part of out (and h_out), new_prefix
 *     (which does not depend on the exchange) stays exact, and a bit is set
 *     that attnres_device_status() reports.  A caller that must not consume
 *     such outputs checks that status word after synchronising; when it is
 *     set, no out or h_out value of that call is to be trusted (a CTA that
 *     was itself the late one may finish on sums of several tokens without
 *     writing NaN).
 *   - Aliasing: new_prefix may be exactly prefix (in-place carry-on of the
 *     prefix sum) or any region that overlaps no input (e.g. bank slot N,
 *     which the call does not read).  out may overlap nothing.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     call, whatever the launch configuration of the same variant and cluster
 *     size; new_prefix is bit-identical across all configurations.
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* attnres_stream_t;

typedef enum {
  ATTNRES_OK = 0,
  ATTNRES_ERR_NULL = -1,    /* a required pointer is NULL                  */
  ATTNRES_ERR_SHAPE = -2,   /* M < 1, N not in [0,31], H not a multiple of 8
                               or H outside [8, 16384]                     */
  ATTNRES_ERR_ALIGN = -3,   /* a pointer is not 16-byte aligned            */
  ATTNRES_ERR_ALIAS = -4,   /* out overlaps a tensor, or new_prefix overlaps
                               an input other than exactly prefix          */
  ATTNRES_ERR_EPS = -5,     /* eps is not finite and > 0                   */
  ATTNRES_ERR_CUDA = -6,    /* a CUDA runtime call failed                  */
  ATTNRES_ERR_DEVICE = -7,  /* the current device is not compute 10.3      */
  ATTNRES_ERR_CONFIG = -8,  /* a forced launch configuration is invalid    */
  ATTNRES_ERR_DTYPE = -9    /* unknown element type                        */
} attnres_status;

/* Element type of every tensor of a call. */
#define ATTNRES_DTYPE_BF16 0
#define ATTNRES_DTYPE_FP16 1

#define ATTNRES_MAX_N 31   /* N = 0 is allowed */
#define ATTNRES_MAX_H 16384

/*
 * attnres_add_rmsnorm -- the fused epilogue (steps 1-3 above).
 *
 *   prefix      [M,H]   prefix sum before this layer (layer_residual)
 *   add         [M,H]   first deferred addend (routed MoE output)
 *   add2        [M,H]   second addend (shared-expert output) or NULL: with
 *                       NULL the fold is new_prefix = bf16(prefix + add)
 *   bank        [N,M,H] depth bank of snapshots, 0 <= N <= 31 (may be NULL
 *                       when N = 0)
 *   w           [H]     per-layer pseudo-query of the mixture
 *   gamma       [H]     RMSNorm weight of the output norm
 *   eps                 epsilon of both RMSNorms, finite and > 0
 *   out         [M,H]   output: RMSNorm(h) * gamma
 *   new_prefix  [M,H]   output: the updated prefix sum
 *   M, N, H             tokens, snapshots, hidden size (H = 7168 in the model)
 *   stream              CUDA stream of the launch
 *
 * N = 0 ("no snapshots yet", the first layer) is supported: the new prefix is
 * the only source, alpha = 1 and out = RMSNorm(new_prefix) * gamma; the PR
 * adds first and runs another path there.  13 <= N <= 31 ("N > 12", the
 * PR's other fallback) is fused here too, in variant 2 only; N > 31 is
 * rejected with ATTNRES_ERR_SHAPE (the sums of 32 sources fill two warp-wide
 * reductions).
 * The launch configuration is chosen from M, N, H and the presence of add2
 * (attnres_plan reports it).
 */
int attnres_add_rmsnorm(const void* prefix, const void* add, const void* add2,
                        const void* bank, const void* w, const void* gamma,
                        float eps, void* out, void* new_prefix,
                        int M, int N, int H, attnres_stream_t stream);

/*
 * Launch configuration, for tests and benchmarks that pin one.
 *   variant   0 = automatic (same as attnres_add_rmsnorm);
 *             1 = one CTA per token, 16 columns per thread (<= 448 threads);
 *             2 = a thread-block cluster of `cluster` CTAs per token, each
 *                 CTA owning a contiguous 1/cluster of the columns, 8 columns
 *                 per thread (<= 256 threads); the per-token sums are
 *                 exchanged through distributed shared memory;
 *             3 = as 2 with at most 224 threads and registers capped by the
 *                 rows a token has (bank, prefix and addends): at 56 (five
 *                 CTAs of 224 threads share an SM) up to 6 rows, else at 72
 *                 (four), with the bank rows past the first 11-12 rows in
 *                 the thread's own slots of shared memory;
 *             5 = as 2 with registers capped so that two CTAs of up to 256
 *                 threads share an SM (in back-to-back calls the next
 *                 call's CTAs can become resident, and prefetch, while this
 *                 call runs); the automatic choice from 17 to 32 tokens
 *                 when the call folds BF16 tensors and N <= 12, with 4 to
 *                 8 CTAs per token chosen per M (measured on GB300);
 *             Variants 1, 4 and 5 exist for N <= 12 only (variant 5 with
 *             the fold on BF16 tensors only).  For N > 12
 *             variant 3 takes at most 128 threads, registers capped so
 *             that four or five CTAs share an SM (at N = 15..17 with bank
 *             rows 14..N-1, from N = 23 on with rows 16..N-1, in dynamic
 *             shared memory).
 *             4 = persistent and pipelined (the large-M streaming kernel): a
 *                 grid of as many clusters as fit the GPU at once walks the
 *                 tokens; every thread copies its chunks of the token
 *                 `stages`-1 steps ahead into a shared-memory ring (cp.async),
 *                 so HBM reads continue during the reductions.
 *             All variants give bit-identical new_prefix; out is identical
 *             for the same variant family and cluster size.
 *   cluster   CTAs per token for variants 2, 3 and 5 (1..16); 0 = the
 *             smallest that fits the variant's thread limit.
 *   threads   threads per CTA, a multiple of 32 within the variant's limit;
 *             0 = the smallest count that covers the CTA's columns.
 *   grid_tokens  CTAs (clusters) along the token axis, each looping over
 *             tokens with this stride (see tail_tokens); 0 = sized when the
 *             kernel is launched for variants 3 and 4 (below), else
 *             min(M, 65535).  Variant 4: the clusters that fit the GPU at
 *             once.  Variant 3: with R clusters fitting at once, about
 *             sqrt(2M/R) + R sqrt(M/(2R)) clusters: the walking ones take
 *             about L = sqrt(2M/R) tokens each, the last R L / 2 one token
 *             each (clusters start in grid order, so the short ones fill
 *             the SMs that the walks leave idle at the end); with M below
 *             about R, one cluster per token.
 *   tail_tokens  variant 3 with grid_tokens > 0: the last tail_tokens
 *             clusters of the grid take one token each (the last tail_tokens
 *             tokens) and the other grid_tokens - tail_tokens walk the rest
 *             with that stride; needs tail_tokens < grid_tokens <= M.  0 =
 *             none (and chosen with the grid when grid_tokens is 0).  Must
 *             be 0 for the other variants.
 *   pdl       programmatic dependent launch: 1 = on, -1 = off, 0 = the
 *             default (on).  With it the kernel may be scheduled while the
 *             previous kernel on the stream is still running; it waits for
 *             that kernel to complete before its first global-memory access,
 *             so results are the same either way.
 *   stages    variant 4 only: tokens held by the shared-memory ring (2..4);
 *             0 = as many as fit 227 KB of shared memory.  Must be 0 for
 *             the other variants.
 *   prefetch  variants 2, 3 and 5, a bit mask: 1 = before waiting on the
 *             previous kernel (see pdl), ask L2 to fetch this CTA's rows of
 *             its first token; 2 = let the next kernel be scheduled at once;
 *             4 = while a token is reduced, ask L2 for the CTA's rows of the
 *             next token it takes (when clusters walk several tokens);
 *             8 = before waiting on the previous kernel, read one 32-bit
 *             word of every 128-byte line of this CTA's rows of its first
 *             token through L2 (values discarded, nothing allocated in L1):
 *             lines an SM has read reach it sooner than lines only
 *             prefetched; -1 = none; 0 = the default (1 up to 96 tokens, plus
 *             8 up to 32 tokens, plus 4 when the grid is smaller than M).
 *             These reads are hints to a coherent L2 and cannot change
 *             results.
 */
typedef struct {
  int variant;
  int cluster;
  int threads;
  int grid_tokens;
  int pdl;
  int stages;
  int prefetch;
  int tail_tokens;
} attnres_config;

/* The fused epilogue with a pinned configuration (cfg may be NULL = auto).
 * An unusable cfg returns ATTNRES_ERR_CONFIG without launching. */
int attnres_add_rmsnorm_ex(const void* prefix, const void* add, const void* add2,
                           const void* bank, const void* w, const void* gamma,
                           float eps, void* out, void* new_prefix,
                           int M, int N, int H, attnres_stream_t stream,
                           const attnres_config* cfg);

/*
 * attnres_add_rmsnorm_tap -- the fused epilogue that also writes the
 * pre-norm mixture: h_out[M,H] = bf16(h) (one rounding of the float32 h).
 * Layers whose hidden state is captured (speculative decoding) need that
 * tensor; with it they can take the fused path instead of adding first
 * (TensorRT-LLM PR #20546, section "Model": a capture layer declines the
 * fold because the tap needs the pre-norm mixture).  h_out must be non-NULL,
 * 16-byte aligned and overlap no other tensor.  Other arguments as above.
 */
int attnres_add_rmsnorm_tap(const void* prefix, const void* add, const void* add2,
                            const void* bank, const void* w, const void* gamma,
                            float eps, void* out, void* new_prefix, void* h_out,
                            int M, int N, int H, attnres_stream_t stream);

/*
 * attnres_add_rmsnorm_f16 -- attnres_add_rmsnorm on FP16 tensors (every
 * tensor FP16: 1 sign, 5 exponent, 10 mantissa bits): the same steps with
 * FP16 in place of BF16, s = fp16(add + add2), new_prefix = fp16(prefix + s)
 * (float32 additions, round to nearest even, FP16 subnormals kept, overflow
 * to infinity), out = fp16(h / sqrt(mean(h^2) + eps) * gamma).  The PR's
 * fused window is BF16 only (section "Model"); this is the same op for a
 * model kept in FP16.  0 <= N <= 31, as for BF16.  Variants 2 and 3 only
 * (attnres_launch with dtype ATTNRES_DTYPE_FP16 takes the tap and the
 * attention-residual alone too).
 */
int attnres_add_rmsnorm_f16(const void* prefix, const void* add, const void* add2,
                            const void* bank, const void* w, const void* gamma,
                            float eps, void* out, void* new_prefix,
                            int M, int N, int H, attnres_stream_t stream);

/*
 * attnres_rmsnorm -- the attention-residual + RMSNorm alone, without the
 * fold: the sources are bank[0..N-1, m] and prefix[m] itself; writes only
 * out.  This is the op the fused epilogue is measured against (section
 * "Performance": the fused op's cost over the attention-residual alone).
 */
int attnres_rmsnorm(const void* prefix, const void* bank, const void* w,
                    const void* gamma, float eps, void* out, int M, int N, int H,
                    attnres_stream_t stream);

/*
 * attnres_tail_add -- the standalone fold in one kernel:
 * new_prefix = bf16(prefix + bf16(add + add2)) (or bf16(prefix + add) when
 * add2 is NULL), elementwise over [M,H], both additions float32 round to
 * nearest even without flushing subnormals.  The single-kernel addition the
 * fused epilogue replaces (section "Performance").  new_prefix may be
 * exactly prefix; it may overlap no other input.
 */
int attnres_tail_add(const void* prefix, const void* add, const void* add2,
                     void* new_prefix, int M, int H, attnres_stream_t stream);

/*
 * attnres_tail_add_f16 -- attnres_tail_add on FP16 tensors:
 * new_prefix = fp16(prefix + fp16(add + add2)), each addition the exact sum
 * rounded once to FP16 (nearest even, subnormals kept, overflow to
 * infinity), which is bit for bit the float32 addition rounded to FP16.  The
 * comparator of attnres_add_rmsnorm_f16.  Same arguments and aliasing rules.
 */
int attnres_tail_add_f16(const void* prefix, const void* add, const void* add2,
                         void* new_prefix, int M, int H, attnres_stream_t stream);

/*
 * attnres_access_pattern -- a measurement aid, not part of the op: the
 * memory traffic of attnres_add_rmsnorm (both addends) without its
 * arithmetic.  It runs with the launch configuration attnres_add_rmsnorm
 * would choose for (M, N, H) -- the same clusters, grid, 16-byte loads of
 * prefix, add, add2 and bank[0..N-1], the same L2 prefetch of the next token
 * and the same two 16-byte stores per chunk -- but computes no fold, sums,
 * exchanges or mixture: new_prefix receives a copy of prefix and out the XOR
 * of the N+3 input rows (bit patterns).  The time of this call is the
 * ceiling the fused op's access pattern can reach on this GPU.
 * 0 <= N <= 12; add2 must be non-NULL; other rules as attnres_add_rmsnorm
 * (w and gamma are not needed).
 */
int attnres_access_pattern(const void* prefix, const void* add, const void* add2,
                           const void* bank, void* out, void* new_prefix,
                           int M, int N, int H, attnres_stream_t stream);

/* All arguments of one call, for attnres_launch. */
typedef struct {
  const void* prefix;
  const void* add;        /* fold != 0: required                          */
  const void* add2;       /* fold != 0: optional second addend             */
  const void* bank;
  const void* w;
  const void* gamma;
  float eps;
  void* out;
  void* new_prefix;       /* fold != 0: required                          */
  void* h_out;            /* optional mixture tap                          */
  int M, N, H;
  int fold;               /* 1: fused epilogue; 0: attention-residual alone */
  int dtype;              /* ATTNRES_DTYPE_BF16 or ATTNRES_DTYPE_FP16       */
} attnres_args;

/* Any of the calls above (the tail adds excepted) with a pinned
 * configuration (cfg may be NULL).  The attention-residual alone (fold = 0)
 * and FP16 tensors exist for variants 2 and 3 only; other variants return
 * ATTNRES_ERR_CONFIG. */
int attnres_launch(const attnres_args* args, const attnres_config* cfg,
                   attnres_stream_t stream);

/* The configuration attnres_add_rmsnorm would launch for (M, N, H) with
 * (has_add2 != 0) or without a second addend on the current device, written
 * to *plan with every field resolved (grid_tokens 0 for variants 3 and 4:
 * sized from the clusters that fit when the kernel is launched).  Returns a status; needs a CUDA device (it
 * reads the SM count). */
int attnres_plan(int M, int N, int H, int has_add2, attnres_config* plan);

/* The same choice computed on the host alone, without a CUDA device (the
 * choice depends on M, N, H and the second addend only; a launch still
 * checks that the current device is a compute capability 10.3 GPU).
 * Returns a status. */
int attnres_plan_host(int M, int N, int H, int has_add2, attnres_config* plan);

/* Static description of a status code; never NULL. */
const char* attnres_status_string(int status);

/* cudaError_t of the last failing CUDA call made by this thread inside the
 * library (0 if none). */
int attnres_last_cuda_error(void);

/* Status word the kernels of the current device write, for failures they
 * cannot return: bit 0 (ATTNRES_DEVICE_WAIT_TIMEOUT) is set when a CTA of a
 * cluster waited longer than the limit for its peers' partial sums (that
 * call wrote NaN into the outputs that depended on them).  Reads it into *bits (and zeroes it when
 * `clear` is non-zero).  Synchronous: waits for the device's work to finish.
 * No correct call sets a bit. */
#define ATTNRES_DEVICE_WAIT_TIMEOUT 1u
int attnres_device_status(unsigned int* bits, int clear);

/* Test hook for the failure path.  From the next launch on, every exchange
 * of partial sums expects `extra_bytes` (0..4096) more than its peers send,
 * so its waits expire after `wait_ns` (0 = the default of 200 ms, at most
 * 10 s); the kernel then sets ATTNRES_DEVICE_WAIT_TIMEOUT and finishes
 * without hanging.  (0, 0) restores normal operation.  Process-wide. */
int attnres_debug_exchange(int extra_bytes, long long wait_ns);

/* Library version: major * 10000 + minor * 100 + patch. */
int attnres_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */
