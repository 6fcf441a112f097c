// flce_fwd.cu — forward kernels: the logit GEMM with the online-statistics
// epilogue (four variants: bias x soft cap), the split-partial merge, the final
// deterministic reduction, and the fp32-hidden hi/lo split.
#include <cuda_runtime.h>

#include "flce_gemm_launch.cuh"

namespace flce {

cudaError_t launch_fwd_gemm(bool bias, bool softcap, bool pair, const TmaMaps& maps, const GemmSched& sc,
                            const FwdParams& p, int* status, int num_sms, cudaStream_t stream) {
  if (bias && softcap) return launch_gemm<EpiFwd<true, true>>(pair, maps, sc, p, status, num_sms, stream);
  if (bias) return launch_gemm<EpiFwd<true, false>>(pair, maps, sc, p, status, num_sms, stream);
  if (softcap) return launch_gemm<EpiFwd<false, true>>(pair, maps, sc, p, status, num_sms, stream);
  return launch_gemm<EpiFwd<false, false>>(pair, maps, sc, p, status, num_sms, stream);
}

// ---------------------------------------------------------------------------
// fp32 hidden -> bf16 hi + bf16 lo, hi = rn(h), lo = rn(h - hi).  hi + lo
// carries about 16 bits of the 24-bit mantissa.
// ---------------------------------------------------------------------------
// x = t0 + t1 (+ t2) in bf16 terms: t0 = rn(x), t1 = rn(x - t0), t2 = rn(x - t0 - t1).
// Each difference is exact in fp32 (the term shares x's exponent range), so two
// terms carry about 16 significant bits of x and three all 24.
__device__ __forceinline__ void split_terms(float4 x, uint2& t0, uint2& t1, uint2& t2) {
  const float v[4] = {x.x, x.y, x.z, x.w};
  uint32_t a[2], b[2], c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t p0 = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    const float r0 = v[2 * i] - __uint_as_float(p0 << 16);
    const float r1 = v[2 * i + 1] - __uint_as_float(p0 & 0xFFFF0000u);
    const uint32_t p1 = pack_bf16x2(r0, r1);
    const float s0 = r0 - __uint_as_float(p1 << 16);
    const float s1 = r1 - __uint_as_float(p1 & 0xFFFF0000u);
    a[i] = p0;
    b[i] = p1;
    c[i] = pack_bf16x2(s0, s1);
  }
  t0 = make_uint2(a[0], a[1]);
  t1 = make_uint2(b[0], b[1]);
  t2 = make_uint2(c[0], c[1]);
}

__global__ void split_f32_kernel(const float4* __restrict__ x, uint2* __restrict__ t0, uint2* __restrict__ t1,
                                 uint2* __restrict__ t2, int64_t n4) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint2 a, b, c;
    split_terms(x[i], a, b, c);
    t0[i] = a;
    t1[i] = b;
    if (t2) t2[i] = c;
  }
}

cudaError_t launch_split_f32(const float* x, uint16_t* t0, uint16_t* t1, uint16_t* t2, int64_t n, int grid,
                             cudaStream_t stream) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  return launch_plain(split_f32_kernel, dim3(grid), dim3(256), 0, stream, reinterpret_cast<const float4*>(x),
                    reinterpret_cast<uint2*>(t0), reinterpret_cast<uint2*>(t1), reinterpret_cast<uint2*>(t2), n4);
}

// ---------------------------------------------------------------------------
// Merge of the split partials and block partial sums.  One warp per token at
// a time (kMergeRows / 8 tokens per warp); lane l takes the records l, l + 32,
// ..., and the lanes combine their results in a fixed butterfly order.
//   M = max_s m_s, S = sum_s s_s e^(m_s - M), A = sum_s a_s e^(m_s - M)
//   lse = M + ln S, sum p z = A / S, entropy = lse - A / S
//   argmax: the largest best_s, the lowest index on ties
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the warp in a fixed butterfly order; every lane gets the result.
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kMergeThreads) fwd_merge_kernel(MergeParams p, int* status) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  constexpr int kWarps = kMergeThreads / 32;
  constexpr int kPerWarp = kMergeRows / kWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = p.row_count ? static_cast<int64_t>(*p.row_count) : p.n_tokens;
  const int64_t N = p.n_tokens;
  double loss_d = 0.0, ent_d = 0.0;  // this warp's tokens (lane 0)
  long long corr = 0, val = 0;
  for (int i = 0; i < kPerWarp; ++i) {
    const int64_t row = blockIdx.x * static_cast<int64_t>(kMergeRows) + warp * kPerWarp + i;
    if (row >= rows) break;  // uniform over the warp
    float M = -INFINITY;
    for (int s = lane; s < p.n_splits; s += 32) M = fmaxf(M, p.part_m[s * N + row]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = 0.f, A = 0.f, best = -INFINITY;
    int32_t best_idx = INT32_MAX;
    for (int s = lane; s < p.n_splits; s += 32) {
      const float f = expf(p.part_m[s * N + row] - M);
      S = fmaf(p.part_s[s * N + row], f, S);
      A = fmaf(p.part_a[s * N + row], f, A);
      const float b = p.part_best[s * N + row];
      const int32_t bi = p.part_idx[s * N + row];
      if (b > best || (b == best && bi < best_idx)) {  // lowest index on ties
        best = b;
        best_idx = bi;
      }
    }
    S = warp_allsum(S);
    A = warp_allsum(A);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int32_t oi = __shfl_xor_sync(0xffffffffu, best_idx, o);
      if (ob > best || (ob == best && oi < best_idx)) {
        best = ob;
        best_idx = oi;
      }
    }
    if (lane == 0) {
      const int64_t orow = p.row_map ? static_cast<int64_t>(p.row_map[row]) : row;
      const float lse = M + logf(S);
      const float ent = lse - A / S;
      const int64_t t = p.targets[row];
      const bool in_range = t >= 0 && t < p.vocab;
      const bool valid = in_range && t != p.ignore_index;
      if (t != p.ignore_index && !in_range) atomicCAS(status, 0, kStatusTargetOutOfRange);
      const float loss = valid ? lse - p.z_target[row] : 0.f;
      p.lse[orow] = lse;
      if (p.lse_compact) p.lse_compact[row] = lse;
      if (p.entropy) p.entropy[orow] = ent;
      if (p.loss_tok) p.loss_tok[orow] = loss;
      loss_d += loss;
      ent_d += valid ? ent : 0.0;
      corr += (valid && best_idx == t) ? 1 : 0;
      val += valid ? 1 : 0;
    }
  }
  __shared__ double s_loss[kWarps], s_ent[kWarps];
  __shared__ long long s_corr[kWarps], s_val[kWarps];
  if (lane == 0) {
    s_loss[warp] = loss_d;
    s_ent[warp] = ent_d;
    s_corr[warp] = corr;
    s_val[warp] = val;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    BlockPartial bp{0.0, 0.0, 0, 0};
    for (int i = 0; i < kWarps; ++i) {
      bp.loss += s_loss[i];
      bp.entropy += s_ent[i];
      bp.correct += s_corr[i];
      bp.valid += s_val[i];
    }
    p.blocks[blockIdx.x] = bp;
  }
}

cudaError_t launch_fwd_merge(const MergeParams& p, int* status, cudaStream_t stream) {
  const int64_t blocks = (p.n_tokens + kMergeRows - 1) / kMergeRows;
  if (blocks == 0) return cudaSuccess;
  return launch_plain(fwd_merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kMergeThreads), 0, stream, p,
                    status);
}

// Valid-target count ahead of the forward (the token-chunked backward needs the
// mean's denominator before the last chunk's forward has run).
__global__ void __launch_bounds__(1024) count_valid_kernel(const int64_t* targets, int64_t n, int64_t vocab,
                                                           int64_t ignore_index, int64_t* n_valid) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  long long c = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t t = targets[i];
    c += (t != ignore_index && t >= 0 && t < vocab) ? 1 : 0;
  }
  __shared__ long long s_c[32];
  c = warp_sum(c);
  if ((threadIdx.x & 31) == 0) s_c[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long total = 0;
    for (int i = 0; i < 32; ++i) total += s_c[i];
    n_valid[0] = total;
  }
}

cudaError_t launch_count_valid(const int64_t* targets, int64_t n, int64_t vocab, int64_t ignore_index,
                               int64_t* n_valid, cudaStream_t stream) {
  return launch_plain(count_valid_kernel, dim3(1), dim3(1024), 0, stream, targets, n, vocab, ignore_index, n_valid);
}

// Rows of each token chunk under compaction: out[c] = clamp(count - c * rows_per_chunk, 0, rows_per_chunk).
__global__ void chunk_rows_kernel(const int32_t* count, int64_t rows_per_chunk, int n_chunks, int32_t* out) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) {
    const int64_t left = static_cast<int64_t>(*count) - c * rows_per_chunk;
    out[c] = static_cast<int32_t>(left <= 0 ? 0 : (left < rows_per_chunk ? left : rows_per_chunk));
  }
}

cudaError_t launch_chunk_rows(const int32_t* count, int64_t rows_per_chunk, int n_chunks, int32_t* out,
                              cudaStream_t stream) {
  return launch_plain(chunk_rows_kernel, dim3(1), dim3(256), 0, stream, count, rows_per_chunk, n_chunks, out);
}

// Final scalars from the block partials, in a fixed order (one block).
__global__ void __launch_bounds__(256) fwd_reduce_kernel(ReduceParams p) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  double loss_d = 0.0, ent_d = 0.0;
  long long corr = 0, val = 0;
  for (int i = threadIdx.x; i < p.n_blocks; i += blockDim.x) {
    const BlockPartial b = p.blocks[i];
    loss_d += b.loss;
    ent_d += b.entropy;
    corr += b.correct;
    val += b.valid;
  }
  __shared__ double s_loss[8], s_ent[8];
  __shared__ long long s_corr[8], s_val[8];
  loss_d = warp_sum(loss_d);
  ent_d = warp_sum(ent_d);
  corr = warp_sum(corr);
  val = warp_sum(val);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_loss[w] = loss_d;
    s_ent[w] = ent_d;
    s_corr[w] = corr;
    s_val[w] = val;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double L = 0.0, E = 0.0;
    long long C = 0, V = 0;
    for (int i = 0; i < 8; ++i) {
      L += s_loss[i];
      E += s_ent[i];
      C += s_corr[i];
      V += s_val[i];
    }
    const double den = p.num_items > 0.0 ? p.num_items : static_cast<double>(V);
    if (p.reduction == 2) p.loss[0] = den > 0.0 ? static_cast<float>(L / den) : 0.f;
    if (p.reduction == 1) p.loss[0] = static_cast<float>(L);
    p.correct[0] = C;
    p.n_valid[0] = V;
    p.entropy_sum[0] = static_cast<float>(E);
  }
}

cudaError_t launch_fwd_reduce(const ReduceParams& p, cudaStream_t stream) {
  return launch_plain(fwd_reduce_kernel, dim3(1), dim3(256), 0, stream, p);
}

// ---------------------------------------------------------------------------
// Valid-token compaction: the tokens whose target is valid, in their original
// order, are gathered into positions [0, count); positions [count, N) get a
// zero hidden row and the ignore index so that they contribute nothing.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool target_valid(const CompactParams& p, int64_t row, int64_t* t_out) {
  const int64_t t = p.targets[row];
  *t_out = t;
  return t != p.ignore_index && t >= 0 && t < p.vocab;
}

__global__ void __launch_bounds__(kCompactBlock) compact_count_kernel(CompactParams p, int* status) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  const int64_t row = blockIdx.x * static_cast<int64_t>(kCompactBlock) + threadIdx.x;
  int valid = 0;
  if (row < p.n_tokens) {
    int64_t t;
    valid = target_valid(p, row, &t) ? 1 : 0;
    if (!valid && t != p.ignore_index) atomicCAS(status, 0, kStatusTargetOutOfRange);
  }
  const int n = __syncthreads_count(valid);
  if (threadIdx.x == 0) p.block_counts[blockIdx.x] = n;
}

__global__ void compact_scan_kernel(CompactParams p, int n_blocks) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  if (threadIdx.x != 0) return;
  int acc = 0;
  for (int b = 0; b < n_blocks; ++b) {
    p.block_offsets[b] = acc;
    acc += p.block_counts[b];
  }
  *p.count = acc;
}

// Copies hidden row `src` to compacted row `dst` (bf16), or splits it into hi / lo (fp32).
__device__ __forceinline__ void copy_hidden_row(const CompactParams& p, int64_t src, int64_t dst, uint32_t lane) {
  const int64_t D = p.hidden;
  if (!p.hidden_f32) {
    const uint4* in = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.hidden_in) + src * D);
    uint4* out = reinterpret_cast<uint4*>(p.hc + dst * D);
    for (int64_t i = lane; i < D / 8; i += 32) out[i] = in[i];
  } else {
    const float4* in = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.hidden_in) + src * D);
    uint2* t0 = reinterpret_cast<uint2*>(p.hc + dst * D);
    uint2* t1 = reinterpret_cast<uint2*>(p.lo + dst * D);
    uint2* t2 = p.lo2 ? reinterpret_cast<uint2*>(p.lo2 + dst * D) : nullptr;
    for (int64_t i = lane; i < D / 4; i += 32) {
      uint2 a, b, c;
      split_terms(in[i], a, b, c);
      t0[i] = a;
      t1[i] = b;
      if (t2) t2[i] = c;
    }
  }
}

__device__ __forceinline__ void zero_hidden_row(const CompactParams& p, int64_t dst, uint32_t lane) {
  const int64_t D = p.hidden;
  uint4* out = reinterpret_cast<uint4*>(p.hc + dst * D);
  for (int64_t i = lane; i < D / 8; i += 32) out[i] = make_uint4(0, 0, 0, 0);
  if (p.hidden_f32) {
    uint4* out2 = reinterpret_cast<uint4*>(p.lo + dst * D);
    for (int64_t i = lane; i < D / 8; i += 32) out2[i] = make_uint4(0, 0, 0, 0);
    if (p.lo2) {
      uint4* out3 = reinterpret_cast<uint4*>(p.lo2 + dst * D);
      for (int64_t i = lane; i < D / 8; i += 32) out3[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

__global__ void __launch_bounds__(kCompactBlock) compact_gather_kernel(CompactParams p) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  __shared__ int s_warp[kCompactBlock / 32];
  const int64_t base = blockIdx.x * static_cast<int64_t>(kCompactBlock);
  const int64_t row = base + threadIdx.x;
  const uint32_t lane = threadIdx.x & 31u;
  const int warp = threadIdx.x >> 5;
  int64_t t = p.ignore_index;
  const bool valid = row < p.n_tokens && target_valid(p, row, &t);
  const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) s_warp[warp] = __popc(ballot);
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the per-warp counts
    const int c = s_warp[lane];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += y;
    }
    s_warp[lane] = incl - c;
  }
  __syncthreads();
  const int pos = valid ? p.block_offsets[blockIdx.x] + s_warp[warp] + __popc(ballot & ((1u << lane) - 1u)) : -1;
  if (valid) {
    p.row_map[pos] = static_cast<int32_t>(row);
    p.targets_out[pos] = t;
    if (p.lse_in) p.lse_out[pos] = p.lse_in[row];
    if (p.dloss_in) p.dloss_out[pos] = p.dloss_in[row];
  } else if (row < p.n_tokens) {  // ignored token: its per-token outputs are 0
    if (p.lse_default) p.lse_default[row] = 0.f;
    if (p.entropy_default) p.entropy_default[row] = 0.f;
    if (p.loss_default) p.loss_default[row] = 0.f;
  }
  const int64_t count = *p.count;
  const int64_t q = base + threadIdx.x;  // a compacted position in this block's window
  if (q >= count && q < p.n_tokens) {
    p.row_map[q] = 0;
    p.targets_out[q] = p.ignore_index;
    if (p.lse_out) p.lse_out[q] = 0.f;
    if (p.dloss_out) p.dloss_out[q] = 0.f;
  }
}

// Compacted row q <- hidden row row_map[q] (q < count), or a zero row; one warp
// per row, grid-stride, so that the copy runs on every SM.
__global__ void __launch_bounds__(256) compact_copy_kernel(CompactParams p) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t count = *p.count;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); q < p.n_tokens;
       q += warps) {
    if (q < count) {
      copy_hidden_row(p, p.row_map[q], q, lane);
    } else {
      zero_hidden_row(p, q, lane);
    }
  }
}

cudaError_t launch_compact(const CompactParams& p, int* status, int num_sms, cudaStream_t stream) {
  const int64_t blocks = (p.n_tokens + kCompactBlock - 1) / kCompactBlock;
  if (blocks == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e = launch_plain(compact_count_kernel, grid, dim3(kCompactBlock), 0, stream, p, status);
  if (e != cudaSuccess) return e;
  if ((e = launch_plain(compact_scan_kernel, dim3(1), dim3(32), 0, stream, p, static_cast<int>(blocks))) != cudaSuccess)
    return e;
  if ((e = launch_plain(compact_gather_kernel, grid, dim3(kCompactBlock), 0, stream, p)) != cudaSuccess) return e;
  return launch_plain(compact_copy_kernel, dim3(num_sms * 4), dim3(256), 0, stream, p);
}

}  // namespace flce
