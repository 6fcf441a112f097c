/*
 * flce_testing.h — test hook of the fused linear cross-entropy library.
 *
 * Not part of the loss API: it exposes the library's tcgen05 GEMM core so that
 * each operand layout it uses (K-major and MN-major A and B, ragged tails) can
 * be checked in isolation.  The paper pages have no counterpart; the GEMM is
 * the "matmul with fp32 accumulation" step of the logit chain (TRL PR #6859,
 * review, "verified" bullet 2) and of the gradient products.
 *
 * C[m, n] = sum_k A(m, k) * B(n, k), bf16 inputs, fp32 accumulation and output.
 *   a_mn_major = 0: A is [M rows][K] with row stride lda (elements)
 *   a_mn_major = 1: A is [K rows][M] with row stride lda
 *   b_mn_major = 0: B is [N rows][K] with row stride ldb
 *   b_mn_major = 1: B is [K rows][N] with row stride ldb
 *   C is [M][N] fp32 with row stride ldc.
 * Device pointers, 16-byte aligned; lda, ldb multiples of 8, ldc of 4.
 * Asynchronous on `stream`.  Returns an FLCE_* status code.
 */
#ifndef FLCE_TESTING_H_
#define FLCE_TESTING_H_

#include "flce.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Process-wide override of two backward planning choices, for tests and tuning
 * sweeps (0 restores the automatic choice):
 *   chunk_cols  vocabulary columns per backward chunk (rounded up to 256)
 *   dh_ksplit   K splits of the dh product, 1..16
 * flce_workspace_size follows the override, so query it after setting.  Not
 * thread-safe with respect to calls in flight on other threads.
 */
FLCE_API int flce_testing_set_tuning(int64_t chunk_cols, int dh_ksplit);

/*
 * Process-wide choice of GEMM kernel, for tests and A/B timing: 0 automatic
 * (CTA pairs with 256-row tiles when there are at least 256 rows and enough
 * tiles, else single CTAs), 1 single-CTA kernel only, 2 CTA-pair kernel only.
 */
FLCE_API int flce_testing_set_gemm_mode(int mode);

/*
 * The plan the library makes for `problem` on a device with `num_sms` SMs, for
 * tests of the host-side planning; it needs no GPU.  for_backward as in
 * flce_workspace_size: 0 for flce_forward (only the fwd_* fields are set), 1
 * for flce_backward (the fwd_* fields describe flce_forward), 2 for
 * flce_forward_backward (with kept logits the forward runs per token chunk:
 * the fwd_* fields describe the first chunk).  The testing overrides above
 * apply.  Returns FLCE_OK, the validation error of `problem`,
 * or FLCE_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t keep_logits;       /* 1: token-chunked backward (6NVD); 0: recompute (8NVD) */
  int32_t dh_pair;           /* 1: the dh product runs on CTA pairs (256-row tiles) */
  int64_t token_chunk_rows;  /* keep_logits: tokens per chunk */
  int64_t vocab_chunk_cols;  /* recompute: columns of the G scratch (its row stride) */
  int64_t run_chunk_cols;    /* recompute: columns per chunk as run, at most vocab_chunk_cols */
  int64_t n_chunks;          /* chunks as run: token chunks, or vocabulary chunks */
  int32_t dh_ksplit_max;     /* fp32 dh slots in the workspace */
  int32_t dh_ksplit;         /* K splits of the dh product as run */
  int32_t fwd_pair;          /* 1: the forward logit product runs on CTA pairs */
  int32_t fwd_splits;        /* vocabulary splits of the forward (records per token) */
  int32_t fwd_tiles_per_split;  /* 256-column vocabulary tiles per split */
  int32_t reserved;          /* 0 */
} flce_testing_plan_info;
FLCE_API int flce_testing_plan(const flce_problem* problem, int for_backward, int num_sms,
                               flce_testing_plan_info* out);

/*
 * Process-wide override of the token-chunk size of the token-chunked backward
 * (FLCE_FLAG_BWD_KEEP_LOGITS), for tests and tuning: rows per chunk, rounded up
 * to 256 and capped at half of N rounded up to 256; 0 restores the automatic
 * size.  flce_workspace_size follows it.  Not thread-safe.
 */
FLCE_API int flce_testing_set_token_chunk(int64_t rows);

/* Kinds of launch recorded by the launch log. */
enum {
  FLCE_LAUNCH_FWD_LOGITS = 0,   /* forward logit GEMM + online statistics        */
  FLCE_LAUNCH_BWD_RECOMPUTE = 1,/* backward logit recompute + G                   */
  FLCE_LAUNCH_BWD_DWEIGHT = 2,  /* dW = G^T h                                     */
  FLCE_LAUNCH_BWD_DHIDDEN = 3,  /* dh += G W                                      */
  FLCE_LAUNCH_OTHER = 4,        /* split, merge, reduce, dbias, dh finalize        */
  FLCE_LAUNCH_BWD_LOGIT_GRAD = 5/* token-chunked backward: G from kept logits     */
};

/* One logged launch: two caller-created CUDA events (cudaEvent_t, timing
 * enabled) that the library records on the call's stream right before and
 * right after the kernel, and the kind of the kernel (written by the library). */
typedef struct {
  void* begin_event;
  void* end_event;
  int32_t kind;
  int32_t reserved;
} flce_launch_record;

/*
 * Profiling hook: while set, every kernel launch of flce_forward /
 * flce_backward is bracketed by the events of records[*count], its kind is
 * stored and *count is incremented, until *count reaches capacity.  Pass NULL
 * records to switch it off.  `records` and `count` are host memory owned by the
 * caller and must stay valid while the hook is set.  Not thread-safe.
 */
FLCE_API int flce_testing_set_launch_log(flce_launch_record* records, int32_t capacity, int32_t* count);

/* Number of kernels this process has launched through the library so far. */
FLCE_API int64_t flce_testing_launch_count(void);

FLCE_API int flce_testing_gemm(int a_mn_major, int b_mn_major, int64_t M, int64_t N, int64_t K, const void* A,
                      int64_t lda, const void* B, int64_t ldb, float* C, int64_t ldc, flce_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_TESTING_H_ */
