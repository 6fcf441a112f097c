// flce_internal.h — constants and parameter blocks shared by the host launcher
// and the sm_103a kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace flce {

// ---- GEMM tiling (one CTA per SM, warp-specialised) ------------------------
constexpr int kBM = 128;          // tile rows = TMEM lanes (tokens, or vocab rows for dW)
constexpr int kBN = 256;          // tile columns = TMEM columns of one accumulator
constexpr int kBK = 64;           // K per pipeline stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K of one tcgen05.mma.kind::f16
constexpr int kStages = 4;        // shared-memory ring depth
constexpr int kAccBufs = 2;       // TMEM accumulators (2 x 256 columns = all 512)
constexpr int kTmemCols = 512;

constexpr int kATileBytes = kBM * kBK * 2;         // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;         // 32 KB
constexpr int kMnAtomBytes = 64 * kBK * 2;         // 8 KB: 64 MN elements x 64 K rows
constexpr int kStageBytes = kATileBytes + kBTileBytes;

// CTA-pair (cta_group::2) tiles: each CTA holds its 128 rows of A and its half
// (128 of 256 columns) of B, so a stage is 32 KB per CTA and six fit.
constexpr int kPairRows = 2 * kBM;                  // tile rows per CTA pair
constexpr int kStagesPair = 6;
constexpr int kBHalfBytes = (kBN / 2) * kBK * 2;    // 16 KB
constexpr int kStagePairBytes = kATileBytes + kBHalfBytes;

// Two epilogue warpgroups work in ping-pong: group g owns TMEM accumulator g
// and processes every other tile, so each group has two mainloops' time per
// tile.  Within a group, warp w reads TMEM lane quarter w.
constexpr int kEpilogueGroups = kAccBufs;
constexpr int kEpilogueWarps = 4;                   // warps per group
constexpr int kEpilogueThreads = kEpilogueWarps * 32;
constexpr int kTmaWarp = kEpilogueGroups * kEpilogueWarps;  // warp 8
constexpr int kMmaWarp = kTmaWarp + 1;                      // warp 9
constexpr int kThreads = (kMmaWarp + 1) * 32;               // 320

constexpr int kEpiSmemGroupFloats = kEpilogueWarps * kBN;   // dbias column-sum staging per group
constexpr int kEpiSmemBytes = kEpilogueGroups * kEpiSmemGroupFloats * 4;
constexpr int kBarrierBytes = 256;
// Dynamic shared memory: alignment slack, the stage ring, the barriers padded
// to 1024 bytes, then the epilogue's own region (its 1024-aligned tail).
constexpr int kGemmSmemBase = 1024 + kStages * kStageBytes + 1024;
constexpr int kGemmPairSmemBase = 1024 + kStagesPair * kStagePairBytes + 1024;

constexpr int kMaxSegments = 6;   // fp32 x fp32 with three-term splits: 6 products

// A bounded wait inside a kernel gives up after this much wall time.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Device status codes (same values as the public FLCE_ERR_* codes).
constexpr int kStatusTargetOutOfRange = 7;
constexpr int kStatusTimeout = 8;

constexpr float kLog2e = 1.4426950408889634f;

// ---- Persistent tile schedule ----------------------------------------------
// Work is a list of units; CTA b takes units b, b + gridDim.x, ...  A unit is
// one m tile, a run of `n_per_unit` consecutive n tiles and one K split.
// Units are rasterised in groups of `group_m` m tiles so that CTAs running at
// the same time share operand tiles through L2.
struct GemmSched {
  int32_t m_tiles, n_tiles;
  int32_t k_blocks;       // 64-wide K blocks over the whole K range
  // K segments: products of bf16 terms of fp32 operands summed into one
  // accumulator.  Segment s (< nseg <= kMaxSegments) multiplies A map
  // (seg_maps >> 4s) & 3 by B map (seg_maps >> (4s + 2)) & 3.
  int32_t nseg;
  uint32_t seg_maps;
  int32_t ksplit;         // K splits per output tile
  int32_t kb_per_split;
  int32_t n_per_unit;
  int32_t n_units;        // ceil(n_tiles / n_per_unit)
  int32_t group_m;
  int32_t ks_outer;       // 0: within a group of m tiles the K split varies fastest after m; 1: the n unit does
  int32_t total_units;
  int32_t a_mn, b_mn;     // operand majorness: 0 = K-major, 1 = MN-major
  int32_t a_mn_off, a_k_off;   // coordinate offsets into the A tensor map
  int32_t b_mn_off, b_k_off;   // coordinate offsets into the B tensor map
  // Optional device-side limits (valid-token compaction): units whose first
  // row is at or past *m_limit are skipped, and the K range stops at *k_limit
  // elements.  nullptr = no limit.
  const int32_t* m_limit;
  const int32_t* k_limit;
};

// ---- Epilogue parameter blocks --------------------------------------------
// Epilogue TMA stores: each warp stages a 32 x 32 box (fp32 at most).
constexpr int kStoreStageBytes = 32 * 32 * 4;
// Forward: online per-token statistics over each unit's vocabulary range
// (one unit = one vocabulary split of one m tile).  Each epilogue group keeps
// its own statistics over the unit's tiles it processed and writes its own
// record: record r = split * kEpilogueGroups + group.
struct FwdParams {
  CUtensorMap z_map;      // kept logits [n_tokens][ldz] fp32, 32 x 32 boxes, 128-byte swizzle (with z_out)
  int64_t n_tokens, vocab;
  const void* bias;       // nullptr, bf16 or fp32 [V]
  int32_t bias_f32;
  int32_t bias_vec;       // bias is 16-byte aligned: load it as 16-byte vectors
  int32_t n_splits;
  float scale, softcap, inv_softcap;
  int64_t ignore_index;
  const int64_t* targets;
  // partials, [n_splits * kEpilogueGroups][n_tokens] each
  float* part_m;          // running max of z
  float* part_s;          // sum exp(z - m)
  float* part_a;          // sum exp(z - m) * z
  float* part_best;       // largest z
  int32_t* part_idx;      // its lowest vocabulary index
  float* z_target;        // [n_tokens] z at the target, written by the owning split
  float* z_out;           // token-chunked backward: every z, fp32 [n_tokens][ldz]; nullptr = not kept
  int64_t ldz;            // multiple of 32 and >= vocab rounded up to 32
};

// Backward recompute: G = w_n (softmax - onehot) * dz/dacc for one vocabulary
// chunk, written as bf16; optional per-m-tile column sums for dbias.
struct GradParams {
  int64_t n_tokens, vocab;
  int64_t v0;             // first vocabulary row of the chunk
  const void* bias;
  int32_t bias_f32;
  int32_t bias_vec;
  int32_t reduction;      // FLCE_RED_*
  float scale, softcap, inv_softcap;
  int64_t ignore_index;
  const int64_t* targets;
  const float* lse;
  const float* dloss;
  const int64_t* n_valid;
  float num_items;        // > 0: the mean divides by it instead of *n_valid
  uint16_t* g;            // bf16 [n_tokens][ldg]
  int64_t ldg;
  float* dbias_part;      // [m_tiles][ldg] or nullptr
};

// Token-chunked backward: G = w_n (e^(z - lse) - onehot) * dz/dx from the kept
// fp32 logits of one token chunk, as bf16, with per-128-row column sums for
// dbias.  Thread blocks cover kZGradRows rows x kZGradCols columns.
constexpr int kZGradThreads = 256;
constexpr int kZGradVec = 8;                               // columns per thread
constexpr int kZGradCols = kZGradThreads * kZGradVec;      // 2048
constexpr int kZGradRows = 32;     // rows per tile of a block = dbias partial granularity
constexpr int kTokenChunkAlign = 256;  // token chunks start on multiples of this (>= any GEMM tile height)
struct ZGradParams {
  int64_t rows, vocab;    // rows of this chunk
  // Under compaction: rows at or past *row_limit get G = 0 up to the next
  // multiple of kTokenChunkAlign (the GEMMs read that far) and nothing past it.
  const int32_t* row_limit;
  const float* z;         // [rows][ldz] fp32
  int64_t ldz;
  uint16_t* g;            // [rows][ldz] bf16
  int32_t reduction;
  float scale, softcap, inv_softcap;
  int64_t ignore_index;
  const int64_t* targets; // [rows]
  const float* lse;       // [rows]
  const float* dloss;     // [1] or [rows] (reduction none)
  const int64_t* n_valid; // [1] over the whole batch
  float num_items;
  float* dbias_part;      // [ceil(rows / kZGradRows)][ldz] or nullptr
};

// Plain store of the accumulator (dW, and the test GEMM), through TMA stores:
// each epilogue warp stages 32 rows x 128 bytes in shared memory
// (kStoreStageBytes per warp) and one lane copies the box out.
struct StoreParams {
  CUtensorMap out_map;    // [rows][cols] in the output dtype: fp32 boxes 32 x 32, bf16 boxes 32 x 64; 128-byte swizzle
  int64_t rows, cols;     // valid extent of the output
  int32_t out_f32;
};

// dh accumulation over vocabulary chunks and K splits.
struct AccumParams {
  int64_t rows, cols;
  float* part;            // [ksplit][rows][cols] fp32
  int64_t part_stride;    // elements between K-split slots
  int32_t accumulate;     // add the slot's previous value
  int32_t write_final;    // write `out` in its dtype instead of the slot (ksplit == 1)
  void* out;
  int32_t out_f32;
  const int32_t* row_map;   // compacted row -> output row, or nullptr
  const int32_t* row_count; // rows at or past *row_count are not written, or nullptr
};

// Valid-token compaction.
constexpr int kCompactBlock = 1024;  // rows per block of the count / gather kernels
struct CompactParams {
  int64_t n_tokens, hidden, vocab, ignore_index;
  const int64_t* targets;
  const void* hidden_in;   // [N][D] bf16 or fp32
  int32_t hidden_f32;
  int32_t* block_counts;   // [blocks]
  int32_t* block_offsets;  // [blocks]
  int32_t* count;          // [1] number of valid tokens
  int32_t* row_map;        // [N] compacted position -> original row
  int64_t* targets_out;    // [N] compacted targets (ignore_index past the count)
  uint16_t* hc;            // [N][D] bf16 compacted hidden (bf16 input), or first bf16 term (fp32 input)
  uint16_t* lo;            // [N][D] second bf16 term (fp32 input), else nullptr
  uint16_t* lo2;           // [N][D] third bf16 term (fp32 input split in three), else nullptr
  const float* lse_in;     // backward: [N] lse to compact, or nullptr
  float* lse_out;
  const float* dloss_in;   // backward, reduction none: [N] upstream grads to compact, or nullptr
  float* dloss_out;
  float* lse_default;      // forward: write 0 at ignored rows of these outputs (nullable)
  float* entropy_default;
  float* loss_default;
};

}  // namespace flce
