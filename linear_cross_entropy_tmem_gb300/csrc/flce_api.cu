// flce_api.cu — the C ABI: argument validation, workspace layout, tensor-map
// encoding, tile/split planning and the launch sequence of the forward and
// the backward.  Host code only; every step of the computation runs in the
// kernels of flce_fwd.cu and flce_bwd.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce.h"
#include "flce_launch.h"
#include "flce_testing.h"

#define FLCE_TRY(expr)               \
  do {                               \
    const int rc_ = (expr);          \
    if (rc_ != FLCE_OK) return rc_;  \
  } while (0)

namespace flce {
namespace {

constexpr int kAbiVersion = 3;
constexpr int kMaxSplits = 64;                     // forward vocabulary splits
// A batch of at most two CTA-pair tiles of tokens has too few m tiles for 64
// splits to fill the GPU; it may split the vocabulary further, so that the
// product runs on CTA pairs (which read each head tile once per pair instead
// of once per 128-row CTA).  Its split records stay small (<= 5 MB).
constexpr int kMaxSplitsSmall = 256;
constexpr int64_t kSmallBatchRows = 512;
constexpr int kMaxKSplit = 16;                     // dh K splits
constexpr size_t kGChunkBudget = size_t(1) << 30;  // bytes of the bf16 G chunk
// Token-chunked backward: bytes of the kept fp32 logits + bf16 G of one chunk,
// and the smallest hidden size for which the automatic choice keeps logits:
// below it the recompute's 2*D flops per logit cost less than the 6 bytes per
// logit of the extra pass over the kept logits (measured on GB300 at
// N = 16384, V = 151936: the recompute is faster at D = 1024, kept logits at
// D = 1152).
constexpr size_t kLogitChunkBudget = size_t(4) << 30;
constexpr int64_t kKeepLogitsMinHidden = 1152;
constexpr int kMaxDevices = 64;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
// Largest forward split count for a product over `rows` tokens.
int max_splits(int64_t rows) { return rows <= kSmallBatchRows ? kMaxSplitsSmall : kMaxSplits; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DeviceInfo {
  bool init = false;
  int index = 0;
  int num_sms = 0;
  int major = 0, minor = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FLCE_ERR_CUDA;
    d.index = dev;
    d.init = true;
  }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FLCE_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = d;
  if (d.major != 10 || d.minor != 3) return FLCE_ERR_UNSUPPORTED_DEVICE;
  return FLCE_OK;
}

// 2-D bf16 tensor map with 128-byte swizzle; out-of-range elements read as 0.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
             uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FLCE_OK : FLCE_ERR_CUDA;
}

// Output map of the TMA-store epilogue: [rows][cols] fp32 in 32 x 32 boxes or
// bf16 in 32 x 64 boxes, so that a box row is one 128-byte line, with the
// 128-byte swizzle.
int make_store_map(CUtensorMap* m, void* base, bool f32, uint64_t cols, uint64_t rows, uint64_t row_bytes) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {f32 ? 32u : 64u, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FLCE_OK : FLCE_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The operands the tensor maps and the products address (hidden, weight, the
// gradients, the workspace) must be memory of the current device: device
// memory of this GPU or managed memory.  Host memory (pageable, pinned or
// registered) and another GPU's memory are refused with FLCE_ERR_INVALID_ARG
// before anything is enqueued.  nullptr passes (the callers check presence).
int check_local(const DeviceInfo& dev, const void* p) {
  if (!p) return FLCE_OK;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return FLCE_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeManaged) return FLCE_OK;
  if (a.type == cudaMemoryTypeDevice && a.device == dev.index) return FLCE_OK;
  return FLCE_ERR_INVALID_ARG;
}
template <class... P>
int check_local(const DeviceInfo& dev, const void* p, P... rest) {
  FLCE_TRY(check_local(dev, p));
  return check_local(dev, rest...);
}

int validate(const flce_problem* p) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if (p->n_tokens < 0 || p->n_tokens > INT32_MAX - 256) return FLCE_ERR_INVALID_ARG;
  if (p->vocab < 1 || p->vocab > INT32_MAX - 256) return FLCE_ERR_INVALID_ARG;
  if (p->hidden < 8 || p->hidden > (int64_t(1) << 20)) return FLCE_ERR_INVALID_ARG;
  if (p->reduction < FLCE_RED_NONE || p->reduction > FLCE_RED_MEAN) return FLCE_ERR_INVALID_ARG;
  if (!std::isfinite(p->logit_scale) || !std::isfinite(p->final_logit_softcapping)) return FLCE_ERR_INVALID_ARG;
  if (p->hidden_dtype != FLCE_BF16 && p->hidden_dtype != FLCE_F32) return FLCE_ERR_UNSUPPORTED_DTYPE;
  if (p->weight_dtype != FLCE_BF16 && p->weight_dtype != FLCE_F32) return FLCE_ERR_UNSUPPORTED_DTYPE;
  if (p->weight_dtype == FLCE_F32 && p->hidden_dtype == FLCE_BF16) return FLCE_ERR_DTYPE_MISMATCH;
  if (!std::isfinite(p->num_items_in_batch) || p->num_items_in_batch < 0.0) return FLCE_ERR_INVALID_ARG;
  constexpr uint32_t kKnownFlags = FLCE_FLAG_COMPACT_VALID | FLCE_FLAG_BWD_RECOMPUTE | FLCE_FLAG_BWD_KEEP_LOGITS |
                                   FLCE_FLAG_FP32_FULL | FLCE_FLAG_FROZEN_HEAD;
  if ((p->flags & ~kKnownFlags) != 0 || p->reserved != 0) return FLCE_ERR_INVALID_ARG;
  if ((p->flags & FLCE_FLAG_BWD_RECOMPUTE) && (p->flags & FLCE_FLAG_BWD_KEEP_LOGITS)) return FLCE_ERR_INVALID_ARG;
  if (p->hidden % 8 != 0) return FLCE_ERR_MISALIGNED;
  return FLCE_OK;
}

bool compact(const flce_problem* p) { return (p->flags & FLCE_FLAG_COMPACT_VALID) != 0; }
// The head (and bias) are not trained: the backward forms dhidden only.
bool frozen(const flce_problem* p) { return (p->flags & FLCE_FLAG_FROZEN_HEAD) != 0; }

// bf16 terms the products read of each operand: 1 for bf16, 2 for fp32 (about
// 16 significant bits), 3 with FLCE_FLAG_FP32_FULL (all 24).
int term_count(int32_t dtype, const flce_problem* p) {
  if (dtype != FLCE_F32) return 1;
  return (p->flags & FLCE_FLAG_FP32_FULL) ? 3 : 2;
}
int h_terms(const flce_problem* p) { return term_count(p->hidden_dtype, p); }
int w_terms(const flce_problem* p) { return term_count(p->weight_dtype, p); }
// Terms of h (dW) or W (dh) the gradient products read.  G, their other
// operand, is rounded to bf16 (8 significant bits), so a second term of the
// fp32 operand (bits 9 to 16) buys no precision there: by default the
// gradient products take the leading term only, and all three terms only with
// FLCE_FLAG_FP32_FULL.
int grad_terms(int terms, const flce_problem* p) { return (p->flags & FLCE_FLAG_FP32_FULL) ? terms : 1; }
size_t weight_elem(const flce_problem* p) { return p->weight_dtype == FLCE_F32 ? 4 : 2; }

// K segments: (A term, B term) pairs packed for GemmSched::seg_maps.
uint32_t pack_segments(const int (*pairs)[2], int n) {
  uint32_t m = 0;
  for (int i = 0; i < n; ++i) m |= static_cast<uint32_t>(pairs[i][0] | (pairs[i][1] << 2)) << (4 * i);
  return m;
}
// Logit products sum_k h[n,k] W[v,k] over the bf16 terms: every h term with a
// bf16 head; with an fp32 head the term pairs of total order <= 1 (two-term
// splits: 3 products) or <= 2 (three-term splits: 6 products).  Every segment
// runs the whole K range into one accumulator, so the smallest products go
// first: their partial sums stay small, and the tensor cores' accumulation
// error (about one ulp of the accumulator per MMA step) is then that of the
// leading product alone.
int logit_segments(int nh, int nw, uint32_t* maps) {
  static const int kPairs2[3][2] = {{1, 0}, {0, 1}, {0, 0}};
  static const int kPairs3[6][2] = {{2, 0}, {1, 1}, {0, 2}, {1, 0}, {0, 1}, {0, 0}};
  static const int kHOnly[3][3][2] = {{{0, 0}}, {{1, 0}, {0, 0}}, {{2, 0}, {1, 0}, {0, 0}}};
  if (nw == 1) {
    *maps = pack_segments(kHOnly[nh - 1], nh);
    return nh;
  }
  if (nw == 2) {
    *maps = pack_segments(kPairs2, 3);
    return 3;
  }
  *maps = pack_segments(kPairs3, 6);
  return 6;
}
// Gradient products with G (one bf16 term) as A and the n terms of h or W as
// B, smallest first.
int b_term_segments(int n, uint32_t* maps) {
  n = std::max(1, std::min(n, 3));
  static const int kBOnly[3][3][2] = {{{0, 0}}, {{0, 1}, {0, 0}}, {{0, 2}, {0, 1}, {0, 0}}};
  *maps = pack_segments(kBOnly[n - 1], n);
  return n;
}

int check_bias_dtype(const flce_problem* p, const void* bias) {
  if (bias && p->bias_dtype != FLCE_BF16 && p->bias_dtype != FLCE_F32) return FLCE_ERR_UNSUPPORTED_DTYPE;
  return FLCE_OK;
}

// ---------------------------------------------------------------------------
// Workspace layout.  Sizes use upper bounds that do not depend on the SM
// count, so flce_workspace_size needs no device.
// ---------------------------------------------------------------------------
struct Layout {
  size_t status = 0;
  size_t h_term[3] = {0, 0, 0};  // bf16 terms of an fp32 hidden state
  size_t w_term[3] = {0, 0, 0};  // bf16 terms of an fp32 head
  size_t part_m = 0, part_s = 0, part_a = 0, part_best = 0, part_idx = 0, z_target = 0, blocks = 0;
  size_t g = 0, dbias_part = 0, dh_part = 0;
  // valid-token compaction
  size_t c_count = 0, c_blocks = 0, c_offsets = 0, c_map = 0, c_targets = 0, c_hidden = 0, c_lse = 0, c_dloss = 0;
  size_t total = 0;
  // backward geometry
  int64_t vc = 0;        // vocabulary chunk width (multiple of 256) = row stride of G
  int64_t n_chunks = 0;
  int ksplit_max = 1;
  bool need_dh_part = false;
  // token-chunked backward (flce_forward_backward keeping the logits)
  bool token = false;
  int64_t nc = 0;         // rows per token chunk (multiple of kTokenChunkAlign)
  int64_t n_tchunks = 0;
  int64_t ldz = 0;        // row stride of the kept logits and of G (elements)
  size_t z = 0, zg = 0, dw_acc = 0, dbias_acc = 0;
  size_t c_chunk_rows = 0;  // under compaction: valid rows of each token chunk
};

// Test/tuning overrides (flce_testing_set_tuning, flce_testing_set_gemm_mode); 0 = automatic.
std::atomic<int64_t> g_force_chunk_cols{0};
std::atomic<int> g_force_dh_ksplit{0};
std::atomic<int> g_gemm_mode{0};  // 0 automatic, 1 single-CTA kernel, 2 CTA-pair kernel
std::atomic<int64_t> g_force_token_rows{0};

// CTA pairs (256-row tiles) when there are at least 256 rows and enough units
// to give every cluster work; otherwise single CTAs (128-row tiles).
bool use_pair(int64_t m_rows, int64_t units_per_pair_row, int num_sms) {
  const int mode = g_gemm_mode.load();
  if (mode == 1) return false;
  if (mode == 2) return true;
  return m_rows >= kPairRows && cdiv(m_rows, kPairRows) * units_per_pair_row >= num_sms / 2;
}

int64_t chunk_width(int64_t n_tokens, int64_t vocab) {
  const int64_t forced = g_force_chunk_cols.load();
  if (forced > 0) return std::min(cdiv(forced, kBN) * kBN, cdiv(vocab, kBN) * kBN);
  const int64_t rows = std::max<int64_t>(1, n_tokens);
  int64_t vc_max = static_cast<int64_t>(kGChunkBudget / (static_cast<size_t>(rows) * 2));
  vc_max = std::max<int64_t>(kBN, vc_max / kBN * kBN);
  // At least two chunks whenever the vocabulary spans more than one tile, so
  // that the G scratch never holds the whole (tokens x vocab) matrix.
  const int64_t n_chunks = std::max<int64_t>(cdiv(vocab, vc_max), vocab > kBN ? 2 : 1);
  return cdiv(cdiv(vocab, n_chunks), kBN) * kBN;
}

// fp32 dh slots of the recompute backward (K splits of each chunk's dh
// product).  Small products split K to fill the GPU (at least 8 K blocks per
// split); mid-sized ones (up to 2048 128-row tiles) get up to 8 slots so that
// the run can even out the last wave of tiles (choose_recompute_ksplit).
int dh_ksplit_bound(int64_t n_tokens, int64_t hidden, int64_t vc) {
  const int forced = g_force_dh_ksplit.load();
  if (forced > 0) return std::min(forced, kMaxKSplit);
  const int64_t tiles = cdiv(n_tokens, kBM) * cdiv(hidden, kBN);
  const int64_t kb = cdiv(vc, kBK);
  const int64_t cap = tiles >= 128 ? std::min<int64_t>(8, cdiv(2048, tiles)) : kMaxKSplit;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cap, kb / 8)));
}

enum LayoutKind { kForward = 0, kBackward = 1, kFused = 2 };

// Backward algorithm of the fused call: keep the logits of token chunks
// (6NVD) or recompute them (8NVD).  Depends on the problem only, so that
// flce_workspace_size agrees with the call.  Keeping costs 6 bytes per logit
// where the recompute costs 2*D flops and another pass over the head, so the
// threshold on D holds for small batches too (at N <= 256 the recompute also
// re-reads the whole head for few tokens).
bool keep_logits(const flce_problem* p) {
  if (p->flags & FLCE_FLAG_BWD_RECOMPUTE) return false;
  if (p->flags & FLCE_FLAG_BWD_KEEP_LOGITS) return true;
  return p->hidden >= kKeepLogitsMinHidden;
}

int64_t logit_row_stride(int64_t vocab) { return cdiv(vocab, 32) * 32; }

// Rows per token chunk: as many as the logit budget allows, balanced over the
// chunks, at most half of N rounded up to kTokenChunkAlign (so that the kept
// logits never cover all tokens of a batch of more than kTokenChunkAlign).  A
// batch of at most kTokenChunkAlign tokens is one chunk of its own rows: its
// kept logits are bounded by kTokenChunkAlign * V, whatever N.
int64_t token_chunk_rows(int64_t n_tokens, int64_t vocab) {
  if (n_tokens <= kTokenChunkAlign) return std::max<int64_t>(kZGradRows, cdiv(n_tokens, kZGradRows) * kZGradRows);
  const int64_t cap = cdiv(cdiv(n_tokens, 2), kTokenChunkAlign) * kTokenChunkAlign;
  const int64_t forced = g_force_token_rows.load();
  if (forced > 0) return std::min(cap, cdiv(forced, kTokenChunkAlign) * kTokenChunkAlign);
  const size_t per_row = size_t(logit_row_stride(vocab)) * 6;
  const int64_t max_rows =
      std::max<int64_t>(kTokenChunkAlign, int64_t(kLogitChunkBudget / per_row) / kTokenChunkAlign * kTokenChunkAlign);
  const int64_t n_chunks = std::max<int64_t>(2, cdiv(n_tokens, max_rows));
  return std::min(cap, cdiv(cdiv(n_tokens, n_chunks), kTokenChunkAlign) * kTokenChunkAlign);
}

// K splits the token-chunked dh product may use (slots in the workspace).
int token_dh_ksplit_bound(int64_t nc, int64_t hidden) {
  const int forced = g_force_dh_ksplit.load();
  if (forced > 0) return std::min(forced, kMaxKSplit);
  const int64_t tiles = cdiv(nc, kBM) * cdiv(hidden, kBN);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxKSplit, cdiv(4096, tiles))));
}

template <class Take>
void take_terms(const flce_problem* p, Layout& L, Take& take) {
  const int th = h_terms(p), tw = w_terms(p);
  for (int i = 0; th > 1 && i < th; ++i) L.h_term[i] = take(size_t(p->n_tokens) * p->hidden * 2);
  for (int i = 0; tw > 1 && i < tw; ++i) L.w_term[i] = take(size_t(p->vocab) * p->hidden * 2);
}

// [status][hi, lo][forward records of one chunk][kept logits][G][dbias
// partials of one chunk's row tiles][fp32 dbias accumulator][fp32 dW
// accumulator][dh K-split slots].  With one chunk the two accumulators are
// not needed: dW and dbias are written straight from that chunk.
Layout make_token_layout(const flce_problem* p, bool has_bias) {
  Layout L;
  L.token = true;
  const int64_t N = p->n_tokens, D = p->hidden, V = p->vocab;
  size_t off = 256;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  take_terms(p, L, take);
  L.nc = token_chunk_rows(N, V);
  L.n_tchunks = cdiv(N, L.nc);
  L.ldz = logit_row_stride(V);
  if (compact(p)) {  // the chunks run over the compacted tokens
    const size_t blocks = size_t(cdiv(N, kCompactBlock));
    L.c_count = take(4);
    L.c_blocks = take(blocks * 4);
    L.c_offsets = take(blocks * 4);
    L.c_map = take(size_t(N) * 4);
    L.c_targets = take(size_t(N) * 8);
    if (p->hidden_dtype != FLCE_F32) L.c_hidden = take(size_t(N) * D * 2);
    L.c_lse = take(size_t(N) * 4);
    L.c_dloss = take(size_t(N) * 4);
    L.c_chunk_rows = take(size_t(L.n_tchunks) * 4);
  }
  const int64_t splits = std::min<int64_t>(max_splits(L.nc), cdiv(V, kBN)) * kEpilogueGroups;
  const size_t part = size_t(splits) * L.nc * 4;
  L.part_m = take(part);
  L.part_s = take(part);
  L.part_a = take(part);
  L.part_best = take(part);
  L.part_idx = take(part);
  L.z_target = take(size_t(L.nc) * 4);
  L.blocks = take(size_t(cdiv(N, kMergeRows)) * sizeof(BlockPartial));
  L.z = take(size_t(L.nc) * L.ldz * 4);
  L.zg = take(size_t(L.nc) * L.ldz * 2);
  const bool weight_grads = !frozen(p);  // a frozen head needs neither dW nor dbias scratch
  if (has_bias && weight_grads) L.dbias_part = take(size_t(cdiv(L.nc, kZGradRows)) * L.ldz * 4);
  if (has_bias && weight_grads && L.n_tchunks > 1) L.dbias_acc = take(size_t(L.ldz) * 4);
  if (weight_grads && L.n_tchunks > 1) L.dw_acc = take(size_t(V) * D * 4);
  L.ksplit_max = token_dh_ksplit_bound(L.nc, D);
  L.need_dh_part = L.ksplit_max > 1;
  if (L.need_dh_part) L.dh_part = take(size_t(L.ksplit_max) * L.nc * D * 4);
  L.total = off;
  return L;
}

// [status][hi, lo][compaction][forward region | backward region]; in the fused
// call the forward and backward regions overlap (the forward's scratch is dead
// before the backward starts, in stream order).
Layout make_layout(const flce_problem* p, int kind, bool has_bias) {
  if (kind == kFused && keep_logits(p)) return make_token_layout(p, has_bias);
  Layout L;
  const int64_t N = p->n_tokens, D = p->hidden, V = p->vocab;
  size_t off = 256;  // status word + padding
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  take_terms(p, L, take);
  if (compact(p)) {
    const size_t blocks = size_t(cdiv(N, kCompactBlock));
    L.c_count = take(4);
    L.c_blocks = take(blocks * 4);
    L.c_offsets = take(blocks * 4);
    L.c_map = take(size_t(N) * 4);
    L.c_targets = take(size_t(N) * 8);
    if (p->hidden_dtype != FLCE_F32) L.c_hidden = take(size_t(N) * D * 2);  // fp32 input compacts into its terms
    if (kind != kForward) {
      L.c_lse = take(size_t(N) * 4);
      L.c_dloss = take(size_t(N) * 4);
    }
  }
  const size_t region = off;
  size_t end = off;
  if (kind != kBackward) {
    const int64_t splits = std::min<int64_t>(max_splits(N), cdiv(V, kBN)) * kEpilogueGroups;
    const size_t part = size_t(splits) * N * 4;
    L.part_m = take(part);
    L.part_s = take(part);
    L.part_a = take(part);
    L.part_best = take(part);
    L.part_idx = take(part);
    L.z_target = take(size_t(N) * 4);
    L.blocks = take(size_t(cdiv(N, kMergeRows)) * sizeof(BlockPartial));
    end = std::max(end, off);
  }
  if (kind != kForward) {
    off = region;
    L.vc = chunk_width(N, V);
    L.n_chunks = cdiv(V, L.vc);
    L.ksplit_max = dh_ksplit_bound(N, D, L.vc);
    L.g = take(size_t(N) * L.vc * 2);
    if (has_bias && !frozen(p)) L.dbias_part = take(size_t(cdiv(N, kBM)) * L.vc * 4);
    L.need_dh_part = L.n_chunks > 1 || L.ksplit_max > 1;
    if (L.need_dh_part) L.dh_part = take(size_t(L.ksplit_max) * N * D * 4);
    end = std::max(end, off);
  }
  L.total = end;
  return L;
}

GemmSched base_sched(int64_t m_rows, int64_t n_cols, int64_t k, int nseg, uint32_t seg_maps, bool pair = false) {
  GemmSched s{};
  s.m_tiles = static_cast<int32_t>(cdiv(m_rows, pair ? kPairRows : kBM));
  s.n_tiles = static_cast<int32_t>(cdiv(n_cols, kBN));
  s.k_blocks = static_cast<int32_t>(cdiv(k, kBK));
  s.nseg = nseg;
  s.seg_maps = seg_maps;
  s.ksplit = 1;
  s.kb_per_split = s.k_blocks;
  s.n_per_unit = 1;
  s.n_units = s.n_tiles;
  s.group_m = 1;
  return s;
}

void finish_sched(GemmSched& s) {
  s.n_units = static_cast<int32_t>(cdiv(s.n_tiles, s.n_per_unit));
  s.group_m = std::max(1, std::min(s.group_m, s.m_tiles));
  s.total_units = s.m_tiles * s.n_units * s.ksplit;
}

// Forward vocabulary split: the split count (<= max_s) that best fills
// the SMs with equal units; ties go to fewer splits.
int choose_splits(int64_t m_tiles, int64_t n_tiles, int64_t max_splits, int num_sms, int* per_unit) {
  double best_eff = -1.0;
  int best_s = 1, best_per = static_cast<int>(n_tiles);
  const int64_t max_s = std::min<int64_t>(max_splits, n_tiles);
  for (int64_t s = 1; s <= max_s; ++s) {
    const int64_t per = cdiv(n_tiles, s);
    const int64_t splits = cdiv(n_tiles, per);
    if (splits != s) continue;
    const int64_t units = m_tiles * splits;
    const int64_t waves = cdiv(units, num_sms);
    const double eff = double(m_tiles * n_tiles) / double(waves * num_sms * per);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best_s = static_cast<int>(s);
      best_per = static_cast<int>(per);
    }
  }
  *per_unit = best_per;
  return best_s;
}

// The forward logit product over `rows` tokens: its kernel (CTA pairs or
// single CTAs) and its vocabulary splits.
struct FwdPlan {
  bool pair;
  int splits;
  int per_unit;  // vocabulary tiles per split
};
FwdPlan plan_forward(int64_t rows, int64_t V, int num_sms) {
  FwdPlan f;
  const int max_s = max_splits(rows);
  f.pair = use_pair(rows, std::min<int64_t>(max_s, cdiv(V, kBN)), num_sms);
  f.per_unit = 1;
  f.splits = choose_splits(cdiv(rows, f.pair ? kPairRows : kBM), cdiv(V, kBN), max_s,
                           f.pair ? num_sms / 2 : num_sms, &f.per_unit);
  return f;
}

int fail(cudaError_t e) { return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA; }

// Launch log (flce_testing_set_launch_log) and launch counter.
flce_launch_record* g_log = nullptr;
int32_t g_log_cap = 0;
int32_t* g_log_count = nullptr;
std::atomic<int64_t> g_launches{0};

// Runs `launch` (returning cudaError_t) on `st`, bracketed by logged events
// when the launch log is on; counts the launch.
template <class F>
int logged(int kind, cudaStream_t st, F&& launch) {
  flce_launch_record* rec = nullptr;
  if (g_log && g_log_count && *g_log_count < g_log_cap) rec = &g_log[*g_log_count];
  if (rec && cudaEventRecord(static_cast<cudaEvent_t>(rec->begin_event), st) != cudaSuccess) return FLCE_ERR_CUDA;
  const cudaError_t e = launch();
  if (e != cudaSuccess) return FLCE_ERR_CUDA;
  g_launches.fetch_add(1);
  if (rec) {
    if (cudaEventRecord(static_cast<cudaEvent_t>(rec->end_event), st) != cudaSuccess) return FLCE_ERR_CUDA;
    rec->kind = kind;
    ++*g_log_count;
  }
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" {

int flce_abi_version(void) { return kAbiVersion; }

const char* flce_status_string(int status) {
  switch (status) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_INVALID_ARG: return "invalid argument";
    case FLCE_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case FLCE_ERR_DTYPE_MISMATCH: return "hidden and weight dtypes do not match";
    case FLCE_ERR_MISALIGNED: return "misaligned pointer or hidden size not a multiple of 8";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FLCE_ERR_CUDA: return "CUDA runtime error";
    case FLCE_ERR_TARGET_OUT_OF_RANGE: return "a target is outside [0, vocab) and is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case FLCE_ERR_UNSUPPORTED_DEVICE: return "the current device is not an sm_103 GPU";
    default: return "unknown status";
  }
}

int flce_workspace_size(const flce_problem* problem, int for_backward, size_t* bytes) {
  if (!bytes) return FLCE_ERR_INVALID_ARG;
  FLCE_TRY(validate(problem));
  // The bias-dependent part is included whenever a bias could be passed.
  if (for_backward < 0 || for_backward > 2) return FLCE_ERR_INVALID_ARG;
  *bytes = make_layout(problem, for_backward, true).total;
  return FLCE_OK;
}

int flce_read_device_status(const void* workspace, flce_stream_t stream, int* status) {
  if (!workspace || !status) return FLCE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLCE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_CUDA;
  *status = v;
  return FLCE_OK;
}

}  // extern "C"

namespace flce {
namespace {

// Inputs of the products after the shared preparation: the bf16 view of the
// hidden states the GEMMs read, and (under compaction) the row count, row map
// and compacted per-token arrays.
struct Prep {
  bool h32 = false, cmp = false;
  int nh = 1, nw = 1;                          // bf16 terms of h and of W
  const void* h[3] = {nullptr, nullptr, nullptr};  // [N][D] bf16 (compacted under compaction)
  const void* w[3] = {nullptr, nullptr, nullptr};  // [V][D] bf16
  const int32_t* row_count = nullptr;
  const int32_t* row_map = nullptr;
  const int64_t* tgt = nullptr;
  float* c_lse = nullptr;
  const float* c_dloss = nullptr;
};

int prepare(const flce_problem* p, const Layout& L, const DeviceInfo& dev, uint8_t* ws, int* status,
            cudaStream_t st, const void* hidden, const void* weight, const int64_t* targets, const float* lse_in,
            const float* dloss, float* lse_def, float* ent_def, float* loss_def, Prep* out) {
  const int64_t N = p->n_tokens, D = p->hidden;
  Prep r;
  r.h32 = p->hidden_dtype == FLCE_F32;
  r.cmp = compact(p);
  r.tgt = targets;
  r.nh = h_terms(p);
  r.nw = w_terms(p);
  r.h[0] = hidden;
  r.w[0] = weight;
  uint16_t* ht[3] = {nullptr, nullptr, nullptr};
  for (int i = 0; r.nh > 1 && i < r.nh; ++i) ht[i] = reinterpret_cast<uint16_t*>(ws + L.h_term[i]);
  if (r.nw > 1) {  // fp32 head: its bf16 terms
    uint16_t* wt[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i < r.nw; ++i) wt[i] = reinterpret_cast<uint16_t*>(ws + L.w_term[i]);
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
      return launch_split_f32(static_cast<const float*>(weight), wt[0], wt[1], wt[2], p->vocab * D,
                              dev.num_sms * 4, st);
    }));
    for (int i = 0; i < r.nw; ++i) r.w[i] = wt[i];
  }
  const bool none = p->reduction == FLCE_RED_NONE;
  if (r.cmp) {
    CompactParams cp{};
    cp.n_tokens = N;
    cp.hidden = D;
    cp.vocab = p->vocab;
    cp.ignore_index = p->ignore_index;
    cp.targets = targets;
    cp.hidden_in = hidden;
    cp.hidden_f32 = r.h32;
    cp.block_counts = reinterpret_cast<int32_t*>(ws + L.c_blocks);
    cp.block_offsets = reinterpret_cast<int32_t*>(ws + L.c_offsets);
    cp.count = reinterpret_cast<int32_t*>(ws + L.c_count);
    cp.row_map = reinterpret_cast<int32_t*>(ws + L.c_map);
    cp.targets_out = reinterpret_cast<int64_t*>(ws + L.c_targets);
    cp.hc = r.h32 ? ht[0] : reinterpret_cast<uint16_t*>(ws + L.c_hidden);
    cp.lo = ht[1];
    cp.lo2 = ht[2];
    if (L.c_lse) {
      cp.lse_in = lse_in;
      cp.lse_out = reinterpret_cast<float*>(ws + L.c_lse);
      r.c_lse = cp.lse_out;
    }
    if (L.c_dloss && none && dloss) {
      cp.dloss_in = dloss;
      cp.dloss_out = reinterpret_cast<float*>(ws + L.c_dloss);
      r.c_dloss = cp.dloss_out;
    }
    cp.lse_default = lse_def;
    cp.entropy_default = ent_def;
    cp.loss_default = loss_def;
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_compact(cp, status, dev.num_sms, st); }));
    r.row_count = cp.count;
    r.row_map = cp.row_map;
    r.tgt = cp.targets_out;
    r.h[0] = cp.hc;
    for (int i = 1; i < r.nh; ++i) r.h[i] = ht[i];
  } else if (r.h32) {
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
      return launch_split_f32(static_cast<const float*>(hidden), ht[0], ht[1], ht[2], N * D, dev.num_sms * 4, st);
    }));
    for (int i = 0; i < r.nh; ++i) r.h[i] = ht[i];
  }
  *out = r;
  return FLCE_OK;
}

ReduceParams reduce_params(const flce_problem* p, const Layout& L, uint8_t* ws, float* loss, int64_t* correct,
                           int64_t* n_valid, float* entropy_sum) {
  ReduceParams rp{};
  rp.blocks = reinterpret_cast<BlockPartial*>(ws + L.blocks);
  rp.n_blocks = static_cast<int32_t>(cdiv(p->n_tokens, kMergeRows));
  rp.reduction = p->reduction;
  rp.num_items = p->num_items_in_batch;
  rp.loss = loss;
  rp.correct = correct;
  rp.n_valid = n_valid;
  rp.entropy_sum = entropy_sum;
  return rp;
}

// Tensor maps of the n bf16 terms of one operand ([outer][inner] rows of
// row_bytes, `offset` bytes into each term); unused slots repeat term 0.
int make_term_maps(CUtensorMap* m0, CUtensorMap* m1, CUtensorMap* m2, const void* const* terms, int n,
                   size_t offset, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                   uint32_t box_outer) {
  CUtensorMap* m[3] = {m0, m1, m2};
  for (int i = 0; i < 3; ++i) {
    if (i < n) {
      FLCE_TRY(make_map(m[i], static_cast<const uint8_t*>(terms[i]) + offset, inner, outer, row_bytes, box_inner,
                        box_outer));
    } else {
      *m[i] = *m[0];
    }
  }
  return FLCE_OK;
}

int run_forward(const flce_problem* p, const Layout& L, const DeviceInfo& dev, uint8_t* ws, int* status,
                cudaStream_t st, const void* bias, const Prep& pr, float* loss, float* lse,
                float* entropy, int64_t* correct, int64_t* n_valid, float* entropy_sum, float* lse_compact) {
  const int64_t N = p->n_tokens, D = p->hidden, V = p->vocab;
  const FwdPlan fpl = plan_forward(N, V, dev.num_sms);
  const bool pair = fpl.pair;
  TmaMaps maps;
  FLCE_TRY(make_term_maps(&maps.a0, &maps.a1, &maps.a2, pr.h, pr.nh, 0, D, N, D * 2, kBK, kBM));
  FLCE_TRY(make_term_maps(&maps.b0, &maps.b1, &maps.b2, pr.w, pr.nw, 0, D, V, D * 2, kBK, pair ? kBN / 2 : kBN));
  uint32_t seg_maps = 0;
  const int nseg = logit_segments(pr.nh, pr.nw, &seg_maps);
  GemmSched sc = base_sched(N, V, D, nseg, seg_maps, pair);
  const int splits = fpl.splits;
  sc.n_per_unit = fpl.per_unit;
  sc.group_m = pair ? 16 : 32;
  sc.m_limit = pr.row_count;
  finish_sched(sc);

  const bool softcap = p->final_logit_softcapping > 0.f;
  FwdParams fp{};
  fp.n_tokens = N;
  fp.vocab = V;
  fp.bias = bias;
  fp.bias_f32 = p->bias_dtype == FLCE_F32;
  fp.bias_vec = bias != nullptr && aligned(bias, 16);
  fp.n_splits = splits;
  fp.scale = p->logit_scale;
  fp.softcap = softcap ? p->final_logit_softcapping : 0.f;
  fp.inv_softcap = softcap ? 1.f / p->final_logit_softcapping : 0.f;
  fp.ignore_index = p->ignore_index;
  fp.targets = pr.tgt;
  fp.part_m = reinterpret_cast<float*>(ws + L.part_m);
  fp.part_s = reinterpret_cast<float*>(ws + L.part_s);
  fp.part_a = reinterpret_cast<float*>(ws + L.part_a);
  fp.part_best = reinterpret_cast<float*>(ws + L.part_best);
  fp.part_idx = reinterpret_cast<int32_t*>(ws + L.part_idx);
  fp.z_target = reinterpret_cast<float*>(ws + L.z_target);
  FLCE_TRY(logged(FLCE_LAUNCH_FWD_LOGITS, st, [&] {
    return launch_fwd_gemm(bias != nullptr, softcap, pair, maps, sc, fp, status, dev.num_sms, st);
  }));

  MergeParams mp{};
  mp.n_tokens = N;
  mp.vocab = V;
  mp.n_splits = splits * kEpilogueGroups;  // one record per split and epilogue group
  mp.reduction = p->reduction;
  mp.ignore_index = p->ignore_index;
  mp.part_m = fp.part_m;
  mp.part_s = fp.part_s;
  mp.part_a = fp.part_a;
  mp.part_best = fp.part_best;
  mp.part_idx = fp.part_idx;
  mp.z_target = fp.z_target;
  mp.targets = pr.tgt;
  mp.lse = lse;
  mp.entropy = entropy;
  mp.loss_tok = p->reduction == FLCE_RED_NONE ? loss : nullptr;
  mp.blocks = reinterpret_cast<BlockPartial*>(ws + L.blocks);
  mp.row_map = pr.row_map;
  mp.row_count = pr.row_count;
  mp.lse_compact = lse_compact;
  FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_merge(mp, status, st); }));
  const ReduceParams rp = reduce_params(p, L, ws, loss, correct, n_valid, entropy_sum);
  return logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_reduce(rp, st); });
}

// K splits of one token chunk's dh product: the fewest that fill the device's
// CTAs (or clusters) within 1 % of the best wave efficiency.
int choose_token_ksplit(int64_t tiles, int ctas, int bound) {
  if (g_force_dh_ksplit.load() > 0) return bound;
  double best = 0.0;
  std::vector<double> eff(bound + 1, 0.0);
  for (int k = 1; k <= bound; ++k) {
    const int64_t units = tiles * k;
    eff[k] = double(units) / double(cdiv(units, ctas) * ctas);
    best = std::max(best, eff[k]);
  }
  for (int k = 1; k <= bound; ++k)
    if (eff[k] >= best - 0.01) return k;
  return 1;
}

// K splits of the recompute backward's dh product.  Every split adds an fp32
// slot that each chunk reads and writes back in the epilogue, so the wave
// efficiency is weighed against 2 % per split (measured on the Gemma-like
// head: 3 splits 3.74 ms, 5 splits 4.3 ms, 1 split 3.9 ms per step).
int choose_recompute_ksplit(int64_t tiles, int ctas, int bound) {
  if (g_force_dh_ksplit.load() > 0) return bound;
  double best = -1.0;
  int best_k = 1;
  for (int k = 1; k <= bound; ++k) {
    const int64_t units = tiles * k;
    const double score = double(units) / double(cdiv(units, ctas) * ctas) * (1.0 - 0.02 * k);
    if (score > best + 1e-9) {
      best = score;
      best_k = k;
    }
  }
  return best_k;
}

// Column width of the recompute backward's vocabulary chunks, at most L.vc:
// the width with the least dW time plus per-chunk overhead.  A dW unit is one
// output tile over K = N, so a wave of units (one per CTA or CTA pair) takes
// cdiv(N, 64) k-blocks of MMA time either way; each chunk adds launches and
// tails worth about kChunkOverheadKBlocks k-blocks (~15 us; one 64-deep
// k-block of a pair's 256 x 256 tile is ~0.27 us at 1.9 GHz).  Widths down to
// half of L.vc are considered.
constexpr double kChunkOverheadKBlocks = 56.0;
int64_t recompute_chunk_cols(const Layout& L, int64_t N, int64_t D, int64_t V, int num_sms) {
  if (g_force_chunk_cols.load() > 0 || !L.need_dh_part) return L.vc;
  const int64_t max_t = L.vc / kBN, n_t = cdiv(D, kBN);
  const double wave = double(cdiv(N, kBK));
  double best = 0.0;
  int64_t best_t = max_t;
  for (int64_t t = max_t; t >= std::max<int64_t>(1, max_t / 2); --t) {
    double cost = 0.0;
    for (int64_t v0 = 0; v0 < V; v0 += t * kBN) {
      const int64_t width = std::min<int64_t>(t * kBN, V - v0);
      const bool pair = use_pair(width, n_t, num_sms);
      cost += wave * double(cdiv(cdiv(width, pair ? kPairRows : kBM) * n_t, pair ? num_sms / 2 : num_sms)) +
              kChunkOverheadKBlocks;
    }
    if (t == max_t || cost < best - 1e-9) {
      best = cost;
      best_t = t;
    }
  }
  return best_t * kBN;
}

// The dh product's kernel (CTA pairs or single CTAs), its CTA (or pair) count
// and its K split, for each backward algorithm.
struct DhPlan {
  bool pair;
  int ctas;
  int ksplit;
};
// A dh product with few output tiles splits K to fill the GPU, so the units
// per 256-row tile row count its K splits too (CTA pairs then read each W tile
// once per pair instead of once per 128-row CTA).
DhPlan plan_recompute_dh(const Layout& L, int64_t N, int64_t D, int num_sms) {
  DhPlan d;
  d.pair = use_pair(N, cdiv(D, kBN) * L.ksplit_max, num_sms);
  d.ctas = d.pair ? num_sms / 2 : num_sms;
  const int64_t tiles = cdiv(N, d.pair ? kPairRows : kBM) * cdiv(D, kBN);
  d.ksplit = L.ksplit_max > 1 ? choose_recompute_ksplit(tiles, d.ctas, L.ksplit_max) : 1;
  return d;
}
DhPlan plan_token_dh(const Layout& L, int64_t D, int num_sms) {
  DhPlan d;
  d.pair = use_pair(L.nc, cdiv(D, kBN) * L.ksplit_max, num_sms);
  d.ctas = d.pair ? num_sms / 2 : num_sms;
  d.ksplit = choose_token_ksplit(cdiv(L.nc, d.pair ? kPairRows : kBM) * cdiv(D, kBN), d.ctas, L.ksplit_max);
  return d;
}

int run_backward(const flce_problem* p, const Layout& L, const DeviceInfo& dev, uint8_t* ws, int* status,
                 cudaStream_t st, const void* bias, const Prep& pr, const float* lse_use,
                 const int64_t* n_valid, const float* dloss_use, void* dhidden, void* dweight, void* dbias) {
  const int64_t N = p->n_tokens, D = p->hidden, V = p->vocab;
  const bool h32 = pr.h32;
  const size_t bias_elem = p->bias_dtype == FLCE_F32 ? 4 : 2;
  if (pr.cmp) {  // ignored tokens get a zero dhidden row; the valid ones are written below
    FLCE_TRY(fail(cudaMemsetAsync(dhidden, 0, size_t(N) * D * (h32 ? 4 : 2), st)));
  }
  const bool softcap = p->final_logit_softcapping > 0.f;
  uint16_t* g = reinterpret_cast<uint16_t*>(ws + L.g);
  float* dbias_part = dbias ? reinterpret_cast<float*>(ws + L.dbias_part) : nullptr;  // none with a frozen head
  float* dh_part = L.need_dh_part ? reinterpret_cast<float*>(ws + L.dh_part) : nullptr;

  // Maps that do not change across chunks.
  const bool pair_rec = use_pair(N, cdiv(L.vc, kBN), dev.num_sms);
  TmaMaps rec;  // recompute: A = h terms (K-major), B = W terms (K-major)
  FLCE_TRY(make_term_maps(&rec.a0, &rec.a1, &rec.a2, pr.h, pr.nh, 0, D, N, D * 2, kBK, kBM));
  FLCE_TRY(make_term_maps(&rec.b0, &rec.b1, &rec.b2, pr.w, pr.nw, 0, D, V, D * 2, kBK, pair_rec ? kBN / 2 : kBN));
  uint32_t rec_segs = 0, dw_segs = 0, dh_segs = 0;
  const int rec_nseg = logit_segments(pr.nh, pr.nw, &rec_segs);
  const int dw_nseg = b_term_segments(grad_terms(pr.nh, p), &dw_segs);  // dW = G^T (sum of h terms)
  const int dh_nseg = b_term_segments(grad_terms(pr.nw, p), &dh_segs);  // dh = G (sum of W terms)
  TmaMaps hmn, wmn;  // MN-major views: h terms for dW, W terms for dh
  FLCE_TRY(make_term_maps(&hmn.b0, &hmn.b1, &hmn.b2, pr.h, pr.nh, 0, D, N, D * 2, 64, kBK));
  FLCE_TRY(make_term_maps(&wmn.b0, &wmn.b1, &wmn.b2, pr.w, pr.nw, 0, D, V, D * 2, 64, kBK));
  const size_t w_elem = weight_elem(p);

  // dh: CTA pairs or single CTAs, and the K split for this device (bounded by
  // the layout's slot count).
  const DhPlan dhp = plan_recompute_dh(L, N, D, dev.num_sms);
  const bool pair_dh = dhp.pair;
  const int dh_ctas = dhp.ctas;
  const int ksplit = dhp.ksplit;

  // Vocabulary chunks of at most L.vc columns (the G scratch keeps L.vc as its
  // row stride).
  const int64_t vcw = recompute_chunk_cols(L, N, D, V, dev.num_sms);
  const int64_t n_chunks = cdiv(V, vcw);
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t v0 = c * vcw;
    const int64_t width = std::min<int64_t>(vcw, V - v0);
    const bool first = c == 0, last = c == n_chunks - 1;

    // (1) recompute the logits of the chunk and form G (bf16) + dbias partials
    GemmSched s1 = base_sched(N, width, D, rec_nseg, rec_segs, pair_rec);
    s1.b_mn_off = static_cast<int32_t>(v0);
    s1.group_m = pair_rec ? 16 : 32;
    s1.m_limit = pr.row_count;
    finish_sched(s1);
    GradParams gp{};
    gp.n_tokens = N;
    gp.vocab = V;
    gp.v0 = v0;
    gp.bias = bias;
    gp.bias_f32 = p->bias_dtype == FLCE_F32;
    gp.bias_vec = bias != nullptr && aligned(bias, 16);
    gp.reduction = p->reduction;
    gp.scale = p->logit_scale;
    gp.softcap = softcap ? p->final_logit_softcapping : 0.f;
    gp.inv_softcap = softcap ? 1.f / p->final_logit_softcapping : 0.f;
    gp.ignore_index = p->ignore_index;
    gp.targets = pr.tgt;
    gp.lse = lse_use;
    gp.dloss = dloss_use;
    gp.n_valid = n_valid;
    gp.num_items = static_cast<float>(p->num_items_in_batch);
    gp.g = g;
    gp.ldg = L.vc;
    gp.dbias_part = dbias_part;
    FLCE_TRY(logged(FLCE_LAUNCH_BWD_RECOMPUTE, st, [&] {
      return launch_grad_gemm(bias != nullptr, softcap, pair_rec, rec, s1, gp, status, dev.num_sms, st);
    }));
    if (dbias) {
      FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
        return launch_dbias_reduce(dbias_part, L.vc, static_cast<int>(cdiv(N, kBM)), kBM, width,
                                   static_cast<uint8_t*>(dbias) + v0 * bias_elem,
                                   p->bias_dtype == FLCE_F32, pr.row_count, nullptr, 0, 1, st);
      }));
    }

    // (2) dW[v0 : v0+width] = G^T h    (A = G MN-major, B = h MN-major, K = N); none with a frozen head
    if (dweight) {
      TmaMaps mw;
      FLCE_TRY(make_map(&mw.a0, g, width, N, L.vc * 2, 64, kBK));
      mw.a1 = mw.a2 = mw.a0;
      mw.b0 = hmn.b0;
      mw.b1 = hmn.b1;
      mw.b2 = hmn.b2;
      const bool pair_dw = use_pair(width, cdiv(D, kBN), dev.num_sms);
      GemmSched s2 = base_sched(width, D, N, dw_nseg, dw_segs, pair_dw);
      s2.a_mn = 1;
      s2.b_mn = 1;
      s2.group_m = std::max(1, (pair_dw ? dev.num_sms / 2 : dev.num_sms) / std::max(1, s2.n_tiles));
      s2.k_limit = pr.row_count;
      finish_sched(s2);
      StoreParams sp{};
      sp.rows = width;
      sp.cols = D;
      sp.out_f32 = w_elem == 4 ? 1 : 0;
      FLCE_TRY(make_store_map(&sp.out_map, static_cast<uint8_t*>(dweight) + size_t(v0) * D * w_elem, w_elem == 4, D,
                              width, D * w_elem));
      FLCE_TRY(logged(FLCE_LAUNCH_BWD_DWEIGHT, st,
                      [&] { return launch_store_gemm(pair_dw, mw, s2, sp, status, dev.num_sms, st); }));
    }

    // (3) dh (+)= G W[v0 : v0+width]   (A = G K-major, B = W MN-major, K = width)
    TmaMaps mh;
    FLCE_TRY(make_map(&mh.a0, g, width, N, L.vc * 2, kBK, kBM));
    mh.a1 = mh.a2 = mh.a0;
    mh.b0 = wmn.b0;
    mh.b1 = wmn.b1;
    mh.b2 = wmn.b2;
    GemmSched s3 = base_sched(N, D, width, dh_nseg, dh_segs, pair_dh);
    s3.b_mn = 1;
    s3.b_k_off = static_cast<int32_t>(v0);
    s3.ksplit = ksplit;
    s3.kb_per_split = static_cast<int32_t>(cdiv(s3.k_blocks, ksplit));
    s3.group_m = std::max(1, dh_ctas / std::max(1, s3.n_tiles * ksplit));
    s3.m_limit = pr.row_count;
    finish_sched(s3);
    AccumParams ap{};
    ap.rows = N;
    ap.cols = D;
    ap.part = dh_part;
    ap.part_stride = N * D;
    ap.accumulate = first ? 0 : 1;
    ap.write_final = (ksplit == 1 && last) ? 1 : 0;
    ap.out = dhidden;
    ap.out_f32 = h32 ? 1 : 0;
    ap.row_map = pr.row_map;
    ap.row_count = pr.row_count;
    FLCE_TRY(logged(FLCE_LAUNCH_BWD_DHIDDEN, st,
                    [&] { return launch_accum_gemm(pair_dh, mh, s3, ap, status, dev.num_sms, st); }));
  }
  if (ksplit > 1) {
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
      return launch_dh_finalize(dh_part, N * D, ksplit, N, D, dhidden, h32 ? 1 : 0, pr.row_map, pr.row_count,
                                dev.num_sms * 4, st);
    }));
  }
  return FLCE_OK;
}

// Token-chunked forward + backward (FLCE_FLAG_BWD_KEEP_LOGITS).  Per chunk of
// L.nc tokens: the forward product keeps z (fp32), the merge gives lse and the
// per-token outputs, zgrad forms G and the dbias partials from the kept z, the
// chunk's dh rows come from one product over the whole vocabulary, and dW
// and dbias accumulate in fp32 across chunks (the last chunk writes the
// results in their dtypes; a single chunk writes them directly).
int run_fused_tokens(const flce_problem* p, const Layout& L, const DeviceInfo& dev, uint8_t* ws, int* status,
                     cudaStream_t st, const void* bias, const Prep& pr, const float* dloss,
                     float* loss, float* lse, float* entropy, int64_t* correct, int64_t* n_valid,
                     float* entropy_sum, void* dhidden, void* dweight, void* dbias) {
  const int64_t N = p->n_tokens, D = p->hidden, V = p->vocab;
  const bool h32 = pr.h32;
  const bool none = p->reduction == FLCE_RED_NONE;
  const bool softcap = p->final_logit_softcapping > 0.f;
  const size_t out_elem = h32 ? 4 : 2;
  float* z = reinterpret_cast<float*>(ws + L.z);
  uint16_t* g = reinterpret_cast<uint16_t*>(ws + L.zg);
  float* dw_acc = L.dw_acc ? reinterpret_cast<float*>(ws + L.dw_acc) : nullptr;
  float* dbias_part = dbias ? reinterpret_cast<float*>(ws + L.dbias_part) : nullptr;  // none with a frozen head
  float* dbias_acc = dbias && L.dbias_acc ? reinterpret_cast<float*>(ws + L.dbias_acc) : nullptr;
  float* dh_part = L.need_dh_part ? reinterpret_cast<float*>(ws + L.dh_part) : nullptr;
  BlockPartial* blocks = reinterpret_cast<BlockPartial*>(ws + L.blocks);
  // Under compaction the chunks cut the compacted tokens: chunk c holds
  // chunk_rows[c] of them (device-side), its outputs go through the row map,
  // and ignored tokens keep a zero dhidden row.
  int32_t* chunk_rows = pr.cmp ? reinterpret_cast<int32_t*>(ws + L.c_chunk_rows) : nullptr;
  if (pr.cmp) {
    FLCE_TRY(fail(cudaMemsetAsync(dhidden, 0, size_t(N) * D * out_elem, st)));
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
      return launch_chunk_rows(pr.row_count, L.nc, static_cast<int>(L.n_tchunks), chunk_rows, st);
    }));
  }

  // The mean's denominator is needed by the first chunk's gradient.
  if (p->reduction == FLCE_RED_MEAN && !(p->num_items_in_batch > 0.0)) {
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st,
                    [&] { return launch_count_valid(pr.tgt, N, V, p->ignore_index, n_valid, st); }));
  }
  TmaMaps wmn;  // W terms as the MN-major B operand of dh
  FLCE_TRY(make_term_maps(&wmn.b0, &wmn.b1, &wmn.b2, pr.w, pr.nw, 0, D, V, D * 2, 64, kBK));
  uint32_t logit_segs = 0, dw_segs = 0, dh_segs = 0;
  const int logit_nseg = logit_segments(pr.nh, pr.nw, &logit_segs);
  const int dw_nseg = b_term_segments(grad_terms(pr.nh, p), &dw_segs);
  const int dh_nseg = b_term_segments(grad_terms(pr.nw, p), &dh_segs);
  const size_t w_elem = weight_elem(p);
  const DhPlan dhp = plan_token_dh(L, D, dev.num_sms);
  const bool pair_dh = dhp.pair;
  const int ksplit = dhp.ksplit;
  const bool pair_dw = use_pair(V, cdiv(D, kBN), dev.num_sms);
  const int dw_ctas = pair_dw ? dev.num_sms / 2 : dev.num_sms;

  for (int64_t c = 0; c < L.n_tchunks; ++c) {
    const int64_t r0 = c * L.nc;
    const int64_t rows = std::min<int64_t>(L.nc, N - r0);
    const bool last = c == L.n_tchunks - 1;
    const size_t h_off = size_t(r0) * D * 2;  // the chunk's rows in every h term
    const int64_t* tgt = pr.tgt + r0;
    const int32_t* lim = pr.cmp ? chunk_rows + c : nullptr;      // valid rows of the chunk (device)
    const int32_t* rmap = pr.cmp ? pr.row_map + r0 : nullptr;   // chunk row -> token

    // (1) logits of the chunk: online statistics, and z kept in fp32
    const FwdPlan fpl = plan_forward(rows, V, dev.num_sms);
    const bool pair_f = fpl.pair;
    TmaMaps fm;
    FLCE_TRY(make_term_maps(&fm.a0, &fm.a1, &fm.a2, pr.h, pr.nh, h_off, D, rows, D * 2, kBK, kBM));
    FLCE_TRY(make_term_maps(&fm.b0, &fm.b1, &fm.b2, pr.w, pr.nw, 0, D, V, D * 2, kBK, pair_f ? kBN / 2 : kBN));
    GemmSched sf = base_sched(rows, V, D, logit_nseg, logit_segs, pair_f);
    const int splits = fpl.splits;
    sf.n_per_unit = fpl.per_unit;
    sf.group_m = pair_f ? 16 : 32;
    sf.m_limit = lim;
    finish_sched(sf);
    FwdParams fp{};
    fp.n_tokens = rows;
    fp.vocab = V;
    fp.bias = bias;
    fp.bias_f32 = p->bias_dtype == FLCE_F32;
    fp.bias_vec = bias != nullptr && aligned(bias, 16);
    fp.n_splits = splits;
    fp.scale = p->logit_scale;
    fp.softcap = softcap ? p->final_logit_softcapping : 0.f;
    fp.inv_softcap = softcap ? 1.f / p->final_logit_softcapping : 0.f;
    fp.ignore_index = p->ignore_index;
    fp.targets = tgt;
    fp.part_m = reinterpret_cast<float*>(ws + L.part_m);
    fp.part_s = reinterpret_cast<float*>(ws + L.part_s);
    fp.part_a = reinterpret_cast<float*>(ws + L.part_a);
    fp.part_best = reinterpret_cast<float*>(ws + L.part_best);
    fp.part_idx = reinterpret_cast<int32_t*>(ws + L.part_idx);
    fp.z_target = reinterpret_cast<float*>(ws + L.z_target);
    fp.z_out = z;
    fp.ldz = L.ldz;
    FLCE_TRY(make_store_map(&fp.z_map, z, true, L.ldz, rows, L.ldz * 4));
    FLCE_TRY(logged(FLCE_LAUNCH_FWD_LOGITS, st, [&] {
      return launch_fwd_gemm(bias != nullptr, softcap, pair_f, fm, sf, fp, status, dev.num_sms, st);
    }));
    MergeParams mp{};
    mp.n_tokens = rows;
    mp.vocab = V;
    mp.n_splits = splits * kEpilogueGroups;
    mp.reduction = p->reduction;
    mp.ignore_index = p->ignore_index;
    mp.part_m = fp.part_m;
    mp.part_s = fp.part_s;
    mp.part_a = fp.part_a;
    mp.part_best = fp.part_best;
    mp.part_idx = fp.part_idx;
    mp.z_target = fp.z_target;
    mp.targets = tgt;
    const int64_t o0 = pr.cmp ? 0 : r0;  // with a row map the merge writes token rows
    mp.lse = lse + o0;
    mp.entropy = entropy ? entropy + o0 : nullptr;
    mp.loss_tok = none ? loss + o0 : nullptr;
    mp.blocks = blocks + r0 / kMergeRows;  // r0 % kMergeRows == 0
    mp.row_map = rmap;
    mp.row_count = lim;
    mp.lse_compact = pr.cmp ? pr.c_lse + r0 : nullptr;
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_merge(mp, status, st); }));

    // (2) G and the dbias partials from the kept logits
    ZGradParams zp{};
    zp.rows = rows;
    zp.vocab = V;
    zp.z = z;
    zp.ldz = L.ldz;
    zp.g = g;
    zp.reduction = p->reduction;
    zp.scale = p->logit_scale;
    zp.softcap = fp.softcap;
    zp.inv_softcap = fp.inv_softcap;
    zp.ignore_index = p->ignore_index;
    zp.targets = tgt;
    zp.lse = pr.cmp ? pr.c_lse + r0 : lse + r0;
    zp.dloss = none ? (pr.c_dloss ? pr.c_dloss : dloss) + r0 : dloss;
    zp.row_limit = lim;
    zp.n_valid = n_valid;
    zp.num_items = static_cast<float>(p->num_items_in_batch);
    zp.dbias_part = dbias_part;
    FLCE_TRY(logged(FLCE_LAUNCH_BWD_LOGIT_GRAD, st, [&] { return launch_zgrad(zp, softcap, st); }));
    if (dbias) {  // the chunk's dbias partials, in row-tile order, into the fp32 accumulator (or dbias)
      FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
        return launch_dbias_reduce(dbias_part, L.ldz, static_cast<int>(cdiv(rows, kZGradRows)), kZGradRows, V,
                                   dbias, p->bias_dtype == FLCE_F32, lim, dbias_acc, c > 0 ? 1 : 0,
                                   last ? 1 : 0, st);
      }));
    }

    // (3) dh rows of the chunk = G W   (A = G K-major, B = W MN-major, K = V)
    TmaMaps mh;
    FLCE_TRY(make_map(&mh.a0, g, V, rows, L.ldz * 2, kBK, kBM));
    mh.a1 = mh.a2 = mh.a0;
    mh.b0 = wmn.b0;
    mh.b1 = wmn.b1;
    mh.b2 = wmn.b2;
    GemmSched s3 = base_sched(rows, D, V, dh_nseg, dh_segs, pair_dh);
    s3.b_mn = 1;
    s3.ksplit = ksplit;
    s3.kb_per_split = static_cast<int32_t>(cdiv(s3.k_blocks, ksplit));
    // K = V: the head and the chunk's G (each ~ V * D or rows * V bf16) stream
    // from HBM; groups of 8 m tiles run over one K slice at a time, so that
    // the units running together (8 m x ~9.5 n tiles on 76 pairs) share their
    // G and W slices in L2.  Measured DRAM reads of one 4096-token chunk's dh
    // at V = 37984, against 0.62 GB of G + W: 1.43 GB with groups of 8 m
    // tiles, 1.61 GB with 16, 2.02 GB with 4, 5.34 GB with the K split varying
    // fastest; the time was the same for 8 and 16.
    s3.group_m = 8;
    s3.ks_outer = 1;
    s3.m_limit = lim;
    finish_sched(s3);
    uint8_t* dh_out = static_cast<uint8_t*>(dhidden) + (pr.cmp ? 0 : size_t(r0) * D * out_elem);
    AccumParams ap{};
    ap.rows = rows;
    ap.cols = D;
    ap.part = dh_part;
    ap.part_stride = rows * D;
    ap.accumulate = 0;
    ap.write_final = ksplit == 1 ? 1 : 0;
    ap.out = dh_out;
    ap.out_f32 = h32 ? 1 : 0;
    ap.row_map = rmap;
    ap.row_count = lim;
    FLCE_TRY(logged(FLCE_LAUNCH_BWD_DHIDDEN, st,
                    [&] { return launch_accum_gemm(pair_dh, mh, s3, ap, status, dev.num_sms, st); }));
    if (ksplit > 1) {
      FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] {
        return launch_dh_finalize(dh_part, rows * D, ksplit, rows, D, dh_out, h32 ? 1 : 0, rmap, lim,
                                  dev.num_sms * 4, st);
      }));
    }

    // (4) dW (+)= G^T h[chunk]   (A = G MN-major, B = h MN-major, K = chunk rows); none with a frozen head
    if (!dweight) continue;
    TmaMaps mw;
    FLCE_TRY(make_map(&mw.a0, g, V, rows, L.ldz * 2, 64, kBK));
    mw.a1 = mw.a2 = mw.a0;
    FLCE_TRY(make_term_maps(&mw.b0, &mw.b1, &mw.b2, pr.h, pr.nh, h_off, D, rows, D * 2, 64, kBK));
    GemmSched s2 = base_sched(V, D, rows, dw_nseg, dw_segs, pair_dw);
    s2.a_mn = 1;
    s2.b_mn = 1;
    s2.group_m = std::max(1, dw_ctas / std::max(1, s2.n_tiles));
    s2.k_limit = lim;
    finish_sched(s2);
    if (L.n_tchunks == 1) {  // nothing to accumulate: dW goes out through TMA stores
      StoreParams sp{};
      sp.rows = V;
      sp.cols = D;
      sp.out_f32 = w_elem == 4 ? 1 : 0;
      FLCE_TRY(make_store_map(&sp.out_map, dweight, w_elem == 4, D, V, D * w_elem));
      FLCE_TRY(logged(FLCE_LAUNCH_BWD_DWEIGHT, st,
                      [&] { return launch_store_gemm(pair_dw, mw, s2, sp, status, dev.num_sms, st); }));
      continue;
    }
    AccumParams aw{};
    aw.rows = V;
    aw.cols = D;
    aw.part = dw_acc;
    aw.part_stride = V * D;
    aw.accumulate = c > 0 ? 1 : 0;
    aw.write_final = last ? 1 : 0;
    aw.out = dweight;
    aw.out_f32 = w_elem == 4 ? 1 : 0;
    FLCE_TRY(logged(FLCE_LAUNCH_BWD_DWEIGHT, st,
                    [&] { return launch_accum_gemm(pair_dw, mw, s2, aw, status, dev.num_sms, st); }));
  }
  const ReduceParams rp = reduce_params(p, L, ws, loss, correct, n_valid, entropy_sum);
  return logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_reduce(rp, st); });
}

int check_forward_args(const flce_problem* p, const void* hidden, const void* weight, const int64_t* targets,
                       const float* loss, const float* lse, const int64_t* correct, const int64_t* n_valid,
                       const float* entropy_sum, const void* workspace) {
  const int64_t N = p->n_tokens;
  if (!weight || !loss || !correct || !n_valid || !entropy_sum || !workspace) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!hidden || !targets || !lse)) return FLCE_ERR_INVALID_ARG;
  if (!aligned(weight, 16) || (N > 0 && !aligned(hidden, 16)) || !aligned(workspace, 256) ||
      (targets && !aligned(targets, 8)))
    return FLCE_ERR_MISALIGNED;
  return FLCE_OK;
}

int check_backward_args(const flce_problem* p, const void* hidden, const void* weight, const void* bias,
                        const int64_t* targets, const float* lse, const int64_t* n_valid, const float* dloss,
                        const void* dhidden, const void* dweight, const void* dbias, const void* workspace) {
  const int64_t N = p->n_tokens;
  if (!weight || !workspace || !n_valid || !dloss) return FLCE_ERR_INVALID_ARG;
  if (frozen(p)) {  // dhidden only: no weight or bias gradient is written
    if (dweight || dbias) return FLCE_ERR_INVALID_ARG;
  } else {
    if (!dweight || (bias == nullptr) != (dbias == nullptr)) return FLCE_ERR_INVALID_ARG;
  }
  if (N > 0 && (!hidden || !targets || !lse || !dhidden)) return FLCE_ERR_INVALID_ARG;
  if (!aligned(weight, 16) || !aligned(dweight, 16) || !aligned(workspace, 256) ||
      (N > 0 && (!aligned(hidden, 16) || !aligned(dhidden, 16))) || (targets && !aligned(targets, 8)))
    return FLCE_ERR_MISALIGNED;
  return FLCE_OK;
}

int zero_grads_for_empty(const flce_problem* p, void* dweight, void* dbias, cudaStream_t st) {
  const size_t bias_elem = p->bias_dtype == FLCE_F32 ? 4 : 2;
  if (dweight) FLCE_TRY(fail(cudaMemsetAsync(dweight, 0, size_t(p->vocab) * p->hidden * weight_elem(p), st)));
  if (dbias) FLCE_TRY(fail(cudaMemsetAsync(dbias, 0, size_t(p->vocab) * bias_elem, st)));
  return FLCE_OK;
}

// A one-word vocabulary: the softmax is exactly 1, so (softmax - onehot) and
// every gradient are exactly 0 (the kernels would leave rounding noise of
// e^(z - lse) - 1 instead).
int zero_grads_single_class(const flce_problem* p, void* dhidden, void* dweight, void* dbias, cudaStream_t st) {
  const size_t h_elem = p->hidden_dtype == FLCE_F32 ? 4 : 2;
  FLCE_TRY(fail(cudaMemsetAsync(dhidden, 0, size_t(p->n_tokens) * p->hidden * h_elem, st)));
  return zero_grads_for_empty(p, dweight, dbias, st);
}

}  // namespace
}  // namespace flce

extern "C" {

int flce_forward(const flce_problem* p, const void* hidden, const void* weight, const void* bias,
                 const int64_t* targets, float* loss, float* lse, float* entropy, int64_t* correct,
                 int64_t* n_valid, float* entropy_sum, void* workspace, size_t workspace_bytes,
                 flce_stream_t stream) {
  FLCE_TRY(validate(p));
  FLCE_TRY(check_bias_dtype(p, bias));
  FLCE_TRY(check_forward_args(p, hidden, weight, targets, loss, lse, correct, n_valid, entropy_sum, workspace));
  const Layout L = make_layout(p, kForward, true);
  if (workspace_bytes < L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  FLCE_TRY(get_device(&dev));
  FLCE_TRY(check_local(dev, hidden, weight, workspace));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  FLCE_TRY(fail(cudaMemsetAsync(status, 0, sizeof(int), st)));
  if (p->n_tokens == 0) {
    const ReduceParams rp = reduce_params(p, L, ws, loss, correct, n_valid, entropy_sum);
    return logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_reduce(rp, st); });
  }
  Prep pr;
  FLCE_TRY(prepare(p, L, dev, ws, status, st, hidden, weight, targets, nullptr, nullptr, lse, entropy,
                   p->reduction == FLCE_RED_NONE ? loss : nullptr, &pr));
  return run_forward(p, L, dev, ws, status, st, bias, pr, loss, lse, entropy, correct, n_valid, entropy_sum,
                     nullptr);
}

int flce_backward(const flce_problem* p, const void* hidden, const void* weight, const void* bias,
                  const int64_t* targets, const float* lse, const int64_t* n_valid, const float* dloss,
                  void* dhidden, void* dweight, void* dbias, void* workspace, size_t workspace_bytes,
                  flce_stream_t stream) {
  FLCE_TRY(validate(p));
  FLCE_TRY(check_bias_dtype(p, bias));
  FLCE_TRY(check_backward_args(p, hidden, weight, bias, targets, lse, n_valid, dloss, dhidden, dweight, dbias,
                               workspace));
  const Layout L = make_layout(p, kBackward, true);
  if (workspace_bytes < L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  FLCE_TRY(get_device(&dev));
  FLCE_TRY(check_local(dev, hidden, weight, dhidden, dweight, workspace));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  FLCE_TRY(fail(cudaMemsetAsync(status, 0, sizeof(int), st)));
  if (p->n_tokens == 0) return zero_grads_for_empty(p, dweight, dbias, st);
  if (p->vocab == 1) return zero_grads_single_class(p, dhidden, dweight, dbias, st);
  Prep pr;
  FLCE_TRY(prepare(p, L, dev, ws, status, st, hidden, weight, targets, lse, dloss, nullptr, nullptr, nullptr, &pr));
  const float* lse_use = pr.cmp ? pr.c_lse : lse;
  const float* dloss_use = pr.c_dloss ? pr.c_dloss : dloss;
  return run_backward(p, L, dev, ws, status, st, bias, pr, lse_use, n_valid, dloss_use, dhidden, dweight,
                      dbias);
}

int flce_forward_backward(const flce_problem* p, const void* hidden, const void* weight, const void* bias,
                          const int64_t* targets, const float* dloss, float* loss, float* lse, float* entropy,
                          int64_t* correct, int64_t* n_valid, float* entropy_sum, void* dhidden, void* dweight,
                          void* dbias, void* workspace, size_t workspace_bytes, flce_stream_t stream) {
  FLCE_TRY(validate(p));
  FLCE_TRY(check_bias_dtype(p, bias));
  FLCE_TRY(check_forward_args(p, hidden, weight, targets, loss, lse, correct, n_valid, entropy_sum, workspace));
  FLCE_TRY(check_backward_args(p, hidden, weight, bias, targets, lse, n_valid, dloss, dhidden, dweight, dbias,
                               workspace));
  const Layout L = make_layout(p, kFused, true);
  if (workspace_bytes < L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  FLCE_TRY(get_device(&dev));
  FLCE_TRY(check_local(dev, hidden, weight, dhidden, dweight, workspace));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  FLCE_TRY(fail(cudaMemsetAsync(status, 0, sizeof(int), st)));
  if (p->n_tokens == 0) {
    const ReduceParams rp = reduce_params(p, L, ws, loss, correct, n_valid, entropy_sum);
    FLCE_TRY(logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_fwd_reduce(rp, st); }));
    return zero_grads_for_empty(p, dweight, dbias, st);
  }
  Prep pr;
  FLCE_TRY(prepare(p, L, dev, ws, status, st, hidden, weight, targets, nullptr, dloss, lse, entropy,
                   p->reduction == FLCE_RED_NONE ? loss : nullptr, &pr));
  if (L.token) {
    FLCE_TRY(run_fused_tokens(p, L, dev, ws, status, st, bias, pr, dloss, loss, lse, entropy, correct, n_valid,
                              entropy_sum, dhidden, dweight, dbias));
    return p->vocab == 1 ? zero_grads_single_class(p, dhidden, dweight, dbias, st) : FLCE_OK;
  }
  FLCE_TRY(run_forward(p, L, dev, ws, status, st, bias, pr, loss, lse, entropy, correct, n_valid,
                       entropy_sum, pr.cmp ? pr.c_lse : nullptr));
  if (p->vocab == 1) return zero_grads_single_class(p, dhidden, dweight, dbias, st);
  const float* lse_use = pr.cmp ? pr.c_lse : lse;
  const float* dloss_use = pr.c_dloss ? pr.c_dloss : dloss;
  return run_backward(p, L, dev, ws, status, st, bias, pr, lse_use, n_valid, dloss_use, dhidden, dweight,
                      dbias);
}

int flce_scale_gradient(const float* scale, void* x, int64_t n, int32_t dtype, flce_stream_t stream) {
  if (!scale || n < 0 || (n > 0 && !x)) return FLCE_ERR_INVALID_ARG;
  if (dtype != FLCE_BF16 && dtype != FLCE_F32) return FLCE_ERR_UNSUPPORTED_DTYPE;
  if (n == 0) return FLCE_OK;
  DeviceInfo dev;
  FLCE_TRY(get_device(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return logged(FLCE_LAUNCH_OTHER, st, [&] {
    return launch_scale(scale, x, n, dtype == FLCE_F32 ? 1 : 0, dev.num_sms * 8, st);
  });
}

int flce_testing_set_tuning(int64_t chunk_cols, int dh_ksplit) {
  if (chunk_cols < 0 || dh_ksplit < 0 || dh_ksplit > kMaxKSplit) return FLCE_ERR_INVALID_ARG;
  g_force_chunk_cols.store(chunk_cols);
  g_force_dh_ksplit.store(dh_ksplit);
  return FLCE_OK;
}

int flce_testing_set_token_chunk(int64_t rows) {
  if (rows < 0) return FLCE_ERR_INVALID_ARG;
  g_force_token_rows.store(rows);
  return FLCE_OK;
}

int flce_testing_set_gemm_mode(int mode) {
  if (mode < 0 || mode > 2) return FLCE_ERR_INVALID_ARG;
  g_gemm_mode.store(mode);
  return FLCE_OK;
}

int flce_testing_plan(const flce_problem* problem, int for_backward, int num_sms, flce_testing_plan_info* out) {
  if (!out || num_sms < 2 || num_sms > 4096 || for_backward < 0 || for_backward > 2) return FLCE_ERR_INVALID_ARG;
  FLCE_TRY(validate(problem));
  const int64_t N = problem->n_tokens, D = problem->hidden, V = problem->vocab;
  flce_testing_plan_info info{};
  if (for_backward == 0) {
    const FwdPlan f = plan_forward(N, V, num_sms);
    info.fwd_pair = f.pair ? 1 : 0;
    info.fwd_splits = f.splits;
    info.fwd_tiles_per_split = f.per_unit;
    *out = info;
    return FLCE_OK;
  }
  const Layout L = make_layout(problem, for_backward == 2 ? kFused : kBackward, true);
  // The forward of the fused call with kept logits runs per token chunk.
  const FwdPlan f = plan_forward(L.token ? L.nc : N, V, num_sms);
  info.fwd_pair = f.pair ? 1 : 0;
  info.fwd_splits = f.splits;
  info.fwd_tiles_per_split = f.per_unit;
  DhPlan d;
  if (L.token) {
    info.keep_logits = 1;
    info.token_chunk_rows = L.nc;
    info.n_chunks = L.n_tchunks;
    d = plan_token_dh(L, D, num_sms);
  } else {
    info.vocab_chunk_cols = L.vc;
    info.run_chunk_cols = recompute_chunk_cols(L, N, D, V, num_sms);
    info.n_chunks = cdiv(V, info.run_chunk_cols);
    d = plan_recompute_dh(L, N, D, num_sms);
  }
  info.dh_ksplit_max = L.ksplit_max;
  info.dh_ksplit = d.ksplit;
  info.dh_pair = d.pair ? 1 : 0;
  *out = info;
  return FLCE_OK;
}

int flce_testing_set_launch_log(flce_launch_record* records, int32_t capacity, int32_t* count) {
  if (records && (capacity < 0 || !count)) return FLCE_ERR_INVALID_ARG;
  g_log = records;
  g_log_cap = records ? capacity : 0;
  g_log_count = records ? count : nullptr;
  return FLCE_OK;
}

int64_t flce_testing_launch_count(void) { return g_launches.load(); }

int flce_testing_gemm(int a_mn_major, int b_mn_major, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float* C, int64_t ldc, flce_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C) return FLCE_ERR_INVALID_ARG;
  if (lda % 8 || ldb % 8 || ldc % 4 || !aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16))
    return FLCE_ERR_MISALIGNED;
  DeviceInfo dev;
  FLCE_TRY(get_device(&dev));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool pair = use_pair(M, cdiv(N, kBN), dev.num_sms);
  GemmSched s = base_sched(M, N, K, 1, 0u, pair);
  s.a_mn = a_mn_major ? 1 : 0;
  s.b_mn = b_mn_major ? 1 : 0;
  finish_sched(s);
  // K-major B: each CTA of a pair loads a 128-row half.
  const uint32_t b_rows = pair ? kBN / 2 : kBN;
  TmaMaps m;
  if (!a_mn_major) FLCE_TRY(make_map(&m.a0, A, K, M, lda * 2, kBK, kBM));
  else FLCE_TRY(make_map(&m.a0, A, M, K, lda * 2, 64, kBK));
  if (!b_mn_major) FLCE_TRY(make_map(&m.b0, B, K, N, ldb * 2, kBK, b_rows));
  else FLCE_TRY(make_map(&m.b0, B, N, K, ldb * 2, 64, kBK));
  m.a1 = m.a2 = m.a0;
  m.b1 = m.b2 = m.b0;
  StoreParams sp{};
  sp.rows = M;
  sp.cols = N;
  sp.out_f32 = 1;
  FLCE_TRY(make_store_map(&sp.out_map, C, true, N, M, ldc * 4));
  return logged(FLCE_LAUNCH_OTHER, st, [&] { return launch_store_gemm(pair, m, s, sp, nullptr, dev.num_sms, st); });
}

}  // extern "C"
