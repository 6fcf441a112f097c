/*
 * flce.h — fused linear cross-entropy for NVIDIA GB300 (sm_103a), C ABI.
 *
 * Computes the next-token cross-entropy of logits = hidden @ weight^T (plus an
 * optional bias, a logit scale and a final-logit soft cap), forward and
 * backward, without ever materialising the (tokens x vocab) logit matrix.
 *
 * The operation is the one described in TRL PR #6859 ("Add loss_type="cce", a
 * fused linear cross-entropy loaded from the Hub"):
 *   - "What it supports": optional lm_head bias, non-unit logit_scale, float32
 *     hidden states, final_logit_softcapping; the accuracy and entropy metrics
 *     come out of the same fused pass as the loss (a 4-tuple);
 *   - review by albertvillanova, list of things "verified", bullet 2: the
 *     chain is matmul with fp32 accumulation, then + bias, then * logit_scale,
 *     then soft cap c * tanh(x / c); the entropy is lse - sum(p * logit); the
 *     argmax is taken on the scaled, soft-capped logits;
 *   - same review, "Correctness" item 2: ignored targets only zero the
 *     per-token weight after the product; the weight gradient is d^T * hidden.
 * The per-token loss is always fp32 (Liger-Kernel PR #1574, Summary item 1),
 * and reduction 'none' scales each token's gradient by its own upstream
 * gradient (same PR, Summary item 2).
 *
 * Conventions shared by every call:
 *   - Every pointer argument except `problem` and `status` is a DEVICE pointer
 *     owned by the caller.  The library allocates no device or host memory and
 *     keeps no state between calls other than a per-device cache of the SM
 *     count and kernel attributes (and, for flce_forward_noalloc, the address
 *     of its static scratch array per CUDA context).
 *   - hidden, weight, dhidden, dweight and the workspace must be memory of
 *     the current device (its device memory, or managed memory): the tensor
 *     maps and the kernels address this GPU's memory only.  Host memory
 *     (pageable, pinned or registered) and another GPU's memory are refused
 *     with FLCE_ERR_INVALID_ARG before anything is enqueued.
 *   - Tensors are dense and row-major: hidden [N, D], weight [V, D], bias [V],
 *     targets [N] (int64), lse [N], dloss [1] or [N].
 *   - Every launch is enqueued on `stream` (0 = the legacy default stream) and
 *     is asynchronous; nothing synchronises the host except
 *     flce_read_device_status.  The GEMM kernels are launched with
 *     programmatic stream serialisation: one may start its set-up (shared
 *     memory, tensor memory) while the kernel before it on the stream is
 *     finishing, and it waits for that kernel to complete before it reads or
 *     writes global memory, so stream order is kept for every buffer.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     are returned as a status code; nothing is launched in that case.
 *   - Errors that depend on data (a target outside [0, V) that is not the
 *     ignore index, or a wait inside a kernel that gave up) are recorded in a
 *     status word at the start of the workspace; each flce_forward /
 *     flce_backward call clears that word first.  Read it with
 *     flce_read_device_status.
 *   - Results are deterministic: no floating-point atomics; every reduction
 *     runs in a fixed order.
 *   - Host threads may call at once (on their own streams and workspaces): the
 *     library's per-device caches are synchronised.  The flce_testing_* hooks
 *     are process-wide switches and are not.
 *   - flce_forward, flce_backward and flce_forward_backward enqueue only
 *     kernels and asynchronous memsets, so a step built from them can be
 *     captured into a CUDA graph once the device's one-time set-up has run
 *     (any earlier call on that device with the same problem), and replayed
 *     with the same pointers; replays give the eager results bit for bit.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (the runtime's cudaStream_t). */
typedef struct CUstream_st* flce_stream_t;

/* Element types of hidden, weight, bias and the gradients. */
enum { FLCE_F32 = 0, FLCE_BF16 = 1 };

/* Reduction of the per-token losses. */
enum { FLCE_RED_NONE = 0, FLCE_RED_SUM = 1, FLCE_RED_MEAN = 2 };

/* Bits of flce_problem.flags. */
enum {
  /*
   * Gather the tokens whose target is valid before any product, so that the
   * cost scales with the number of valid tokens instead of N (TRL PR #6859,
   * review "Correctness" item 2: gather before the call).  Loss, metrics and
   * gradients are unchanged (up to summation order); ignored tokens then get
   * lse = 0 and entropy = 0 instead of their values over the vocabulary, and a
   * zero dhidden row.
   */
  FLCE_FLAG_COMPACT_VALID = 1u,
  /*
   * Backward algorithm of flce_forward_backward (the other calls ignore these
   * two bits; setting both is FLCE_ERR_INVALID_ARG).  With neither bit the
   * library chooses from the problem's sizes alone, and
   * flce_workspace_size(problem, 2) follows the choice.
   *
   * FLCE_FLAG_BWD_RECOMPUTE: every logit tile is recomputed in the backward
   *   (TRL PR #6859, review "Correctness" item 2: the backward sweeps the
   *   vocabulary again per row).  8*N*V*D flops; the scratch is bounded (a
   *   bf16 gradient chunk of at most 1 GiB).
   * FLCE_FLAG_BWD_KEEP_LOGITS: token-chunked.  The tokens are cut into chunks
   *   of at most half of N (rounded up to 256 rows), whose kept logits stay
   *   within a 4 GiB budget; a batch of at most 256 tokens is one chunk, whose
   *   kept logits are at most 256 x V.  The forward product of a chunk keeps
   *   its fp32 logits in the workspace, and the chunk's logit gradient,
   *   dhidden rows and dweight / dbias contributions are formed from them
   *   before the next chunk starts (TRL PR #6863, opening section: token
   *   chunks whose logits come from a bf16 tensor-core product and are held
   *   in fp32).  6*N*V*D flops, at the price of about 6 bytes of scratch per
   *   logit of a chunk plus 4*V*(D + 1) bytes of fp32 dweight / dbias
   *   accumulators (not needed with one chunk).  With
   *   FLCE_FLAG_COMPACT_VALID the chunks cut the gathered valid tokens.
   */
  FLCE_FLAG_BWD_RECOMPUTE = 2u,
  FLCE_FLAG_BWD_KEEP_LOGITS = 4u,
  /*
   * fp32 operands at full single precision: an fp32 hidden state (and an fp32
   * head) is split into three bf16 terms, t0 = rn(x), t1 = rn(x - t0),
   * t2 = rn(x - t0 - t1), which sum to x exactly for |x| >= 2^-100 (below,
   * the lower terms are subnormal and lose bits); the logit product sums the
   * term products of total order <= 2 (3 products for fp32 hidden with a bf16
   * head, 6 with an fp32 head), so it carries the fp32 inputs' 24 bits into the
   * tensor cores' fp32 accumulation, whose own error (about K/16 units in the
   * last place of the accumulator) then dominates for long K.  Without it fp32
   * operands take two terms (about 16 bits: 2 products, or 3 with an fp32
   * head) in the logit products, and their leading term alone in the
   * gradient products dweight = G^T hidden and dhidden = G weight, whose
   * other operand G is rounded to bf16 (with this flag those take all three
   * terms).  No effect on bf16 operands.
   * (The pages' fp32 path: TRL PR #6859, review "verified" bullet 3, with the
   * head cast to the activations' dtype.)
   */
  FLCE_FLAG_FP32_FULL = 8u,
  /*
   * The head (and its bias) are frozen, as in the LoRA rows of TRL PR #6859's
   * Benchmark table, where only the adapters are trained: the backward forms
   * dhidden alone.  flce_backward and flce_forward_backward then take NULL for
   * dweight and dbias (a non-NULL pointer is FLCE_ERR_INVALID_ARG) and skip the
   * dweight products and the dbias sums: 2*N*V*D flops fewer, and the
   * workspace holds no fp32 dweight / dbias accumulators.  The bias, when
   * given, still enters the logits.  flce_forward ignores this bit.
   */
  FLCE_FLAG_FROZEN_HEAD = 16u
};

/* Status codes returned by every call (and stored in the device status word). */
enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,         /* null or non-local pointer, bad size or enum    */
  FLCE_ERR_UNSUPPORTED_DTYPE = 2,   /* e.g. fp32 weight                               */
  FLCE_ERR_DTYPE_MISMATCH = 3,      /* bf16 hidden with a non-bf16 weight              */
  FLCE_ERR_MISALIGNED = 4,          /* pointer not 16-byte aligned, D % 8 != 0         */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 5, /* workspace_bytes below flce_workspace_size       */
  FLCE_ERR_CUDA = 6,                /* a CUDA runtime call or launch failed            */
  FLCE_ERR_TARGET_OUT_OF_RANGE = 7, /* device: a target not in [0,V) nor ignore_index  */
  FLCE_ERR_TIMEOUT = 8,             /* device: a bounded in-kernel wait gave up         */
  FLCE_ERR_UNSUPPORTED_DEVICE = 9   /* current device is not sm_103                    */
};

/*
 * The problem description shared by the forward and the backward.
 *   n_tokens   N >= 0 (0 is allowed: empty batch)
 *   hidden     D, 8 <= D, D % 8 == 0 (16-byte rows for the tensor-memory copies)
 *   vocab      V >= 1
 *   hidden_dtype  FLCE_BF16 or FLCE_F32.  fp32 hidden is split on the device
 *                 into bf16 terms whose products are summed: two terms (about
 *                 16 bits of mantissa), or three with FLCE_FLAG_FP32_FULL.
 *   weight_dtype  FLCE_BF16, or FLCE_F32 with an fp32 hidden state (the head is
 *                 cast to the activations' dtype by the caller; TRL PR #6859
 *                 review, "verified" bullet 3).  bf16 hidden with an fp32
 *                 head is FLCE_ERR_DTYPE_MISMATCH.  An fp32 head is split on
 *                 the device into bf16 terms like an fp32 hidden state, and
 *                 dweight is then fp32.
 *   bias_dtype    FLCE_BF16 or FLCE_F32; ignored when bias is NULL.  The bias
 *                 is added in fp32 after the fp32-accumulated product.
 *   logit_scale   s (1.0f = identity)
 *   final_logit_softcapping  c; c <= 0 turns the soft cap off
 *   ignore_index  targets equal to it contribute nothing (usually -100)
 *   reduction     FLCE_RED_MEAN (divide by the number of valid tokens; 0 when
 *                 there are none), FLCE_RED_SUM or FLCE_RED_NONE.
 *   num_items_in_batch  0, or the count of valid tokens of a whole accumulated
 *                 batch: the mean then divides by it, in the forward and the
 *                 backward (TRL PR #6859 review, "Test coverage" item 10).
 *                 Finite and >= 0.
 *   flags         an OR of FLCE_FLAG_* bits, or 0.
 *   reserved      0.
 * (ABI version 2: num_items_in_batch, flags and reserved were added; version
 * 3: the two backward-algorithm flags.)
 */
typedef struct {
  int64_t n_tokens;
  int64_t hidden;
  int64_t vocab;
  int32_t hidden_dtype;
  int32_t weight_dtype;
  int32_t bias_dtype;
  int32_t reduction;
  float logit_scale;
  float final_logit_softcapping;
  int64_t ignore_index;
  double num_items_in_batch;  /* > 0: FLCE_RED_MEAN divides by it instead of n_valid */
  uint32_t flags;             /* FLCE_FLAG_* */
  uint32_t reserved;          /* must be 0 */
} flce_problem;

/*
 * Bytes of device workspace flce_forward (for_backward = 0), flce_backward
 * (for_backward = 1) or flce_forward_backward (for_backward = 2) needs for
 * `problem`, written to *bytes.  The size grows
 * with N * (number of vocabulary splits) for the forward and with
 * N * (vocabulary chunk) + N * D for the recompute backward, whose bf16
 * gradient chunk is at most 1 GiB; the token-chunked backward holds one token
 * chunk's logits (at most 4 GiB, or 256 x V for a batch of at most 256
 * tokens) and O(V * D + N * D) more.  It never grows with N * V.
 * The size is an upper bound that does not depend on the device, so the call
 * needs no GPU.  Returns FLCE_OK or the validation error of `problem`.
 */
FLCE_API int flce_workspace_size(const flce_problem* problem, int for_backward, size_t* bytes);

/*
 * Forward: TRL PR #6859, "What it supports" (the 4-tuple) and the review's
 * "verified" bullet 2 (logit chain, entropy identity, argmax on the final
 * logits).
 *   hidden   [N, D] in hidden_dtype, 16-byte aligned
 *   weight   [V, D] bf16, 16-byte aligned
 *   bias     [V] in bias_dtype, or NULL
 *   targets  [N] int64; ignore_index marks ignored tokens
 *   loss     fp32: [1] for mean / sum, [N] for none (0 at ignored tokens)
 *   lse      [N] fp32 log-sum-exp of the final logits of every token; the
 *            backward needs it unchanged
 *   entropy  [N] fp32 per-token entropy lse - sum(p * z), or NULL
 *   correct  [1] int64: valid tokens whose argmax (lowest index on ties)
 *            equals the target
 *   n_valid  [1] int64: tokens whose target is not ignore_index
 *   entropy_sum [1] fp32: sum of the per-token entropy over valid tokens
 *   workspace, workspace_bytes: at least flce_workspace_size(problem, 0),
 *            256-byte aligned; its first 4 bytes are the device status word
 */
FLCE_API int flce_forward(const flce_problem* problem, const void* hidden, const void* weight,
                 const void* bias, const int64_t* targets, float* loss, float* lse,
                 float* entropy, int64_t* correct, int64_t* n_valid, float* entropy_sum,
                 void* workspace, size_t workspace_bytes, flce_stream_t stream);

/*
 * Backward: TRL PR #6859 review, "Correctness" item 2 (d = w_n * (softmax -
 * onehot) with the per-row weight zero at ignored tokens; the weight gradient
 * is d^T * hidden) with the chain rule of the scale and soft cap, and
 * Liger-Kernel PR #1574, Summary item 2 (reduction 'none' multiplies row n by
 * dloss[n] once, in fp32, in registers).
 *   hidden, weight, bias, targets: as passed to flce_forward
 *   lse      [N] fp32 from flce_forward on the same inputs
 *   n_valid  [1] int64 from flce_forward (the mean's denominator)
 *   dloss    fp32 upstream gradient: [1] for mean / sum, [N] for none
 *   dhidden  [N, D] in hidden_dtype (written, not accumulated), 16-byte aligned
 *   dweight  [V, D] in weight_dtype (written, not accumulated), 16-byte aligned;
 *            NULL with FLCE_FLAG_FROZEN_HEAD (and only then)
 *   dbias    [V] in bias_dtype; must be NULL exactly when bias is NULL, and
 *            NULL with FLCE_FLAG_FROZEN_HEAD
 *   workspace, workspace_bytes: at least flce_workspace_size(problem, 1)
 * All-ignored batches produce exact zero gradients.
 */
FLCE_API int flce_backward(const flce_problem* problem, const void* hidden, const void* weight,
                  const void* bias, const int64_t* targets, const float* lse,
                  const int64_t* n_valid, const float* dloss, void* dhidden, void* dweight,
                  void* dbias, void* workspace, size_t workspace_bytes, flce_stream_t stream);

/*
 * Forward and backward in one call, for callers that know the upstream
 * gradient before the forward runs (a training step whose loss is used as is).
 * Same arguments and results as flce_forward followed by flce_backward with
 * `lse` and `n_valid` passed from one to the other.  With the recompute
 * backward (FLCE_FLAG_BWD_RECOMPUTE) the results are the same bit for bit; the
 * two halves share argument checks, planning, the fp32 hidden split and the
 * valid-token compaction, and their scratch shares one workspace of
 * flce_workspace_size(problem, 2) bytes.  With the token-chunked backward
 * (FLCE_FLAG_BWD_KEEP_LOGITS) every output is the same up to the order of the
 * fp32 sums: the vocabulary splits of the forward are planned per chunk, and
 * dhidden / dweight are summed over different partitions of the vocabulary /
 * the tokens.
 *   dloss    fp32 upstream gradient, [1] (mean / sum) or [N] (none), on the
 *            device before the call's work reaches the backward
 *   lse, n_valid: outputs of the forward half, read by the backward half
 */
FLCE_API int flce_forward_backward(const flce_problem* problem, const void* hidden, const void* weight,
                                   const void* bias, const int64_t* targets, const float* dloss, float* loss,
                                   float* lse, float* entropy, int64_t* correct, int64_t* n_valid,
                                   float* entropy_sum, void* dhidden, void* dweight, void* dbias, void* workspace,
                                   size_t workspace_bytes, flce_stream_t stream);

/*
 * Gradients computed before the upstream gradient is known, scaled once it is:
 * x[i] = rn(x[i] * *scale) in place, with an fp32 multiply and one rounding
 * (Liger-Kernel PR #1574, Summary item 2: the saved gradient scaled by the
 * upstream gradient in the backward).  A caller that runs
 * flce_forward_backward with dloss = 1 for a mean / sum loss (whose
 * gradients are linear in the scalar upstream gradient) scales dhidden,
 * dweight and dbias with it when the upstream gradient arrives.
 *   scale   device pointer to one fp32; when it holds exactly 1 the buffer is
 *           neither read nor written
 *   x, n    device buffer of n elements of `dtype` (FLCE_BF16 or FLCE_F32)
 * Asynchronous on `stream`.  Returns FLCE_OK, FLCE_ERR_INVALID_ARG,
 * FLCE_ERR_UNSUPPORTED_DTYPE or FLCE_ERR_CUDA.
 */
FLCE_API int flce_scale_gradient(const float* scale, void* x, int64_t n, int32_t dtype, flce_stream_t stream);

/*
 * Synchronises `stream`, then copies the device status word at the start of
 * `workspace` into *status (FLCE_OK or one of the FLCE_ERR_* device codes).
 * Returns FLCE_OK, FLCE_ERR_INVALID_ARG or FLCE_ERR_CUDA.
 */
FLCE_API int flce_read_device_status(const void* workspace, flce_stream_t stream, int* status);

/*
 * Forward without any allocation, for callers that cannot call cudaMalloc
 * (for example a plugin inside a host application that owns the device-memory
 * budget and gives its plugins no allocator, or latency-critical code that
 * cannot accept cudaMalloc's implicit device synchronisation).  The pages have
 * no counterpart: it is flce_forward with the same arguments minus the
 * workspace, whose scratch lives instead in a static device array of
 * FLCE_NOALLOC_SCRATCH_BYTES that each GPU loading the library holds until the
 * process exits.
 *   - Problems whose forward workspace (flce_workspace_size(problem, 0)) is
 *     larger than FLCE_NOALLOC_SCRATCH_BYTES are rejected with
 *     FLCE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  With bf16
 *     hidden states and a vocabulary of 16K or more that admits about 13K
 *     tokens (2.6 KB of split records per token); fp32 hidden states need
 *     4*N*D more bytes.
 *   - The first call in a CUDA context looks up the array's device address
 *     there (with the caller's device current) and caches it under the
 *     context's process-unique id, so a second context on the device, or the
 *     new one after cudaDeviceReset, looks it up again; make the first call
 *     before any stream capture.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - All calls share the one array, which keeps the last call's contents; the
 *     call clears what must start at zero.  Calls whose GPU work overlaps in
 *     time race on the array.
 *   - The caller holds no workspace, so flce_read_device_status cannot be
 *     used: a target outside [0, V) that is not ignore_index is still treated
 *     as ignored, but it is not reported.
 */
#define FLCE_NOALLOC_SCRATCH_BYTES (32u << 20)
FLCE_API int flce_forward_noalloc(const flce_problem* problem, const void* hidden, const void* weight,
                                  const void* bias, const int64_t* targets, float* loss, float* lse,
                                  float* entropy, int64_t* correct, int64_t* n_valid, float* entropy_sum,
                                  flce_stream_t stream);

/* Static English description of a status code (never NULL). */
FLCE_API const char* flce_status_string(int status);

/* Library ABI version (incremented on any signature change). */
FLCE_API int flce_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
