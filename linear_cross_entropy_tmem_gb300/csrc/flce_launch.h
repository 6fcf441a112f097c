// flce_launch.h — host-side launchers for the kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

// A and B operand maps; a1, a2, b1, b2 are the further bf16 terms of split
// fp32 operands (GemmSched::seg_maps picks the pair of each K segment).
struct TmaMaps {
  CUtensorMap a0, a1, a2, b0, b1, b2;
};

// Per-token merge of the split partials, with per-block partial sums.
struct BlockPartial {
  double loss;
  double entropy;
  long long correct;
  long long valid;
};

struct MergeParams {
  int64_t n_tokens, vocab;
  int32_t n_splits;
  int32_t reduction;
  int64_t ignore_index;
  const float *part_m, *part_s, *part_a, *part_best;
  const int32_t* part_idx;
  const float* z_target;
  const int64_t* targets;
  float* lse;
  float* entropy;     // nullable
  float* loss_tok;    // the loss output when reduction is 'none', else nullptr
  BlockPartial* blocks;
  const int32_t* row_map;    // compacted row -> output row, or nullptr
  const int32_t* row_count;  // rows at or past *row_count are skipped, or nullptr
  float* lse_compact;        // also write lse at the compacted row, or nullptr
};

struct ReduceParams {
  const BlockPartial* blocks;
  int32_t n_blocks;
  int32_t reduction;
  double num_items;   // > 0: the mean divides by it instead of the valid count
  float* loss;        // [1] for mean / sum
  int64_t* correct;
  int64_t* n_valid;
  float* entropy_sum;
};

constexpr int kMergeThreads = 256;  // threads per block of the merge: 8 warps, one token per warp at a time
constexpr int kMergeRows = 32;      // tokens per block of the merge = per BlockPartial

// GEMM launches.  `pair` selects the CTA-pair kernel (clusters of two CTAs,
// 256-row tiles); `num_sms` bounds the persistent grid (CTAs, or 2 x clusters).
cudaError_t launch_fwd_gemm(bool bias, bool softcap, bool pair, const TmaMaps& maps, const GemmSched& sc,
                            const FwdParams& p, int* status, int num_sms, cudaStream_t stream);
cudaError_t launch_grad_gemm(bool bias, bool softcap, bool pair, const TmaMaps& maps, const GemmSched& sc,
                             const GradParams& p, int* status, int num_sms, cudaStream_t stream);
cudaError_t launch_store_gemm(bool pair, const TmaMaps& maps, const GemmSched& sc, const StoreParams& p,
                              int* status, int num_sms, cudaStream_t stream);
cudaError_t launch_accum_gemm(bool pair, const TmaMaps& maps, const GemmSched& sc, const AccumParams& p,
                              int* status, int num_sms, cudaStream_t stream);

cudaError_t launch_zgrad(const ZGradParams& p, bool softcap, cudaStream_t stream);
// Under compaction, the valid rows of each token chunk of the kept-logits backward.
cudaError_t launch_chunk_rows(const int32_t* count, int64_t rows_per_chunk, int n_chunks, int32_t* out,
                              cudaStream_t stream);
// n_valid[0] = number of targets in [0, vocab) other than ignore_index (one block).
cudaError_t launch_count_valid(const int64_t* targets, int64_t n, int64_t vocab, int64_t ignore_index,
                               int64_t* n_valid, cudaStream_t stream);

// x (fp32, n % 4 == 0) -> bf16 terms t0 = rn(x), t1 = rn(x - t0) [, t2 = rn(x - t0 - t1)].
cudaError_t launch_split_f32(const float* x, uint16_t* t0, uint16_t* t1, uint16_t* t2, int64_t n, int grid,
                             cudaStream_t stream);
cudaError_t launch_fwd_merge(const MergeParams& p, int* status, cudaStream_t stream);
cudaError_t launch_fwd_reduce(const ReduceParams& p, cudaStream_t stream);
// x *= *scale in place (bf16 or fp32), skipped on the device when *scale == 1.
cudaError_t launch_scale(const float* scale, void* x, int64_t n, int x_f32, int grid, cudaStream_t stream);
// s[j] = sum over the m_tiles per-tile partials (tiles of rows_per_tile rows), in tile order; with
// an fp32 accumulator `acc` (else nullptr) s[j] is added to acc[j] when `accumulate`.  s goes to
// dbias in its dtype when `write_final` (or there is no accumulator), else to acc.  Under
// compaction only the tiles below *row_count rows were computed.
cudaError_t launch_dbias_reduce(const float* part, int64_t ldg, int m_tiles, int rows_per_tile, int64_t cols,
                                void* dbias, int bias_f32, const int32_t* row_count, float* acc, int accumulate,
                                int write_final, cudaStream_t stream);
cudaError_t launch_dh_finalize(const float* part, int64_t stride, int ksplit, int64_t rows, int64_t cols, void* out,
                               int out_f32, const int32_t* row_map, const int32_t* row_count, int grid,
                               cudaStream_t stream);
// Valid-token compaction: count, scan, gather (see CompactParams).
cudaError_t launch_compact(const CompactParams& p, int* status, int num_sms, cudaStream_t stream);

}  // namespace flce
