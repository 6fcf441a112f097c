// flce_bwd.cu — backward kernels: the recompute GEMM with the logit-gradient
// epilogue (four variants: bias x soft cap), the dW store GEMM, the dh / dW
// accumulate GEMM, the logit gradient of the token-chunked backward (from kept
// logits), the ordered dbias reduction and the dh K-split finalize.
#include <cuda_runtime.h>

#include "flce_gemm_launch.cuh"

namespace flce {

cudaError_t launch_grad_gemm(bool bias, bool softcap, bool pair, const TmaMaps& maps, const GemmSched& sc,
                             const GradParams& p, int* status, int num_sms, cudaStream_t stream) {
  if (bias && softcap) return launch_gemm<EpiGrad<true, true>>(pair, maps, sc, p, status, num_sms, stream);
  if (bias) return launch_gemm<EpiGrad<true, false>>(pair, maps, sc, p, status, num_sms, stream);
  if (softcap) return launch_gemm<EpiGrad<false, true>>(pair, maps, sc, p, status, num_sms, stream);
  return launch_gemm<EpiGrad<false, false>>(pair, maps, sc, p, status, num_sms, stream);
}

cudaError_t launch_store_gemm(bool pair, const TmaMaps& maps, const GemmSched& sc, const StoreParams& p,
                              int* status, int num_sms, cudaStream_t stream) {
  return launch_gemm<EpiStore>(pair, maps, sc, p, status, num_sms, stream);
}

cudaError_t launch_accum_gemm(bool pair, const TmaMaps& maps, const GemmSched& sc, const AccumParams& p,
                              int* status, int num_sms, cudaStream_t stream) {
  return launch_gemm<EpiAccum>(pair, maps, sc, p, status, num_sms, stream);
}

// Token-chunked backward: G from the kept fp32 logits of one token chunk.
// Thread t of a block handles kZGradVec consecutive columns over one tile of
// kZGradRows rows at a time (row tiles grid-strided over blockIdx.y): per row
// one 32-byte load of z and one 16-byte store of G, both coalesced across the
// block (HBM-bound: 6 bytes per logit).  The column sums of G (fp32, before
// rounding) over a tile's rows are that tile's dbias partials, added in row
// order.  Short tiles (32 rows) keep the last wave of blocks small.
template <bool kSoftcap>
__global__ void __launch_bounds__(kZGradThreads) zgrad_kernel(ZGradParams p) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  __shared__ float s_lse2[kZGradRows];  // lse * log2(e)
  __shared__ float s_wd[kZGradRows];    // w_n * s (0 at ignored rows)
  __shared__ int64_t s_t[kZGradRows];   // target column
  int64_t lim = p.rows, lim_pad = p.rows;  // rows with a logit; rows the GEMMs read
  if (p.row_limit) {
    lim = *p.row_limit < p.rows ? *p.row_limit : p.rows;
    lim_pad = (lim + kTokenChunkAlign - 1) / kTokenChunkAlign * kTokenChunkAlign;
    if (lim_pad > p.rows) lim_pad = p.rows;
  }
  const int64_t row_tiles = (p.rows + kZGradRows - 1) / kZGradRows;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * kZGradThreads + threadIdx.x) * kZGradVec;
  const bool active = c0 < p.vocab;  // threads past the vocabulary still take the barriers
  const int valid_cols = !active ? 0 : (p.vocab - c0 < kZGradVec ? static_cast<int>(p.vocab - c0) : kZGradVec);
  for (int64_t rt = blockIdx.y; rt < row_tiles; rt += gridDim.y) {
    const int64_t r0 = rt * kZGradRows;
    if (r0 >= lim_pad) break;  // uniform over the block; later tiles are further out
    const int rows = lim - r0 < kZGradRows ? static_cast<int>(lim - r0 > 0 ? lim - r0 : 0) : kZGradRows;
    const int zero_rows = lim_pad - r0 < kZGradRows ? static_cast<int>(lim_pad - r0) : kZGradRows;
    __syncthreads();  // the previous tile's readers of the row data are done
    for (int i = threadIdx.x; i < kZGradRows; i += kZGradThreads) {
      float lse2 = 0.f, wd = 0.f;
      int64_t t = -1;
      if (i < rows) {
        const int64_t row = r0 + i;
        t = __ldg(p.targets + row);
        lse2 = __ldg(p.lse + row) * kLog2e;
        const bool valid = t != p.ignore_index && t >= 0 && t < p.vocab;
        if (valid) wd = token_weight(p.reduction, p.dloss, row, p.n_valid, p.num_items) * p.scale;
        if (!valid) t = -1;
      }
      s_lse2[i] = lse2;
      s_wd[i] = wd;
      s_t[i] = t;
    }
    __syncthreads();
    if (!active) continue;
    const float* __restrict__ zp = p.z + r0 * p.ldz + c0;  // 32-byte aligned: ldz % 32 == 0, c0 % 8 == 0
    uint16_t* __restrict__ gp = p.g + r0 * p.ldz + c0;
    float colsum[kZGradVec];
#pragma unroll
    for (int j = 0; j < kZGradVec; ++j) colsum[j] = 0.f;
#pragma unroll 4
    for (int r = 0; r < rows; ++r) {
      const float4 za = __ldcs(reinterpret_cast<const float4*>(zp + r * p.ldz));
      const float4 zb = __ldcs(reinterpret_cast<const float4*>(zp + r * p.ldz) + 1);
      const float z[kZGradVec] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
      const float lse2 = s_lse2[r], wd = s_wd[r];
      const int64_t tj = s_t[r] - c0;
      float g[kZGradVec];
#pragma unroll
      for (int j = 0; j < kZGradVec; ++j) {
        const float pr = ex2_approx(fmaf(z[j], kLog2e, -lse2));  // e^(z - lse)
        float d = wd;
        if (kSoftcap) {
          const float th = z[j] * p.inv_softcap;                   // z / c
          d = wd * fmaf(-th, th, 1.f);                             // w s (1 - (z/c)^2)
        }
        g[j] = d * (pr - (j == tj ? 1.f : 0.f));
        if (j >= valid_cols) g[j] = 0.f;
        colsum[j] += g[j];
      }
      uint4 pk;
      pk.x = pack_bf16x2(g[0], g[1]);
      pk.y = pack_bf16x2(g[2], g[3]);
      pk.z = pack_bf16x2(g[4], g[5]);
      pk.w = pack_bf16x2(g[6], g[7]);
      __stcs(reinterpret_cast<uint4*>(gp + r * p.ldz), pk);
    }
    for (int r = rows; r < zero_rows; ++r)  // past the valid rows of a compacted chunk: exact zeros
      __stcs(reinterpret_cast<uint4*>(gp + r * p.ldz), make_uint4(0u, 0u, 0u, 0u));
    if (p.dbias_part) {
      float* dst = p.dbias_part + rt * p.ldz + c0;
#pragma unroll
      for (int j = 0; j < kZGradVec; ++j)
        if (j < valid_cols) dst[j] = colsum[j];
    }
  }
}

cudaError_t launch_zgrad(const ZGradParams& p, bool softcap, cudaStream_t stream) {
  const int64_t gx = (p.vocab + kZGradCols - 1) / kZGradCols;
  const int64_t row_tiles = (p.rows + kZGradRows - 1) / kZGradRows;
  if (gx == 0 || row_tiles == 0) return cudaSuccess;
  if (gx > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(row_tiles < 65535 ? row_tiles : 65535));
  if (softcap) return launch_plain(zgrad_kernel<true>, grid, dim3(kZGradThreads), 0, stream, p);
  return launch_plain(zgrad_kernel<false>, grid, dim3(kZGradThreads), 0, stream, p);
}

// x[i] = rn(x[i] * s) in place (fp32 multiply, one rounding), s = *scale read
// on the device; nothing is read or written when s == 1.
__global__ void scale_kernel(const float* __restrict__ scale, void* x, int64_t n, int x_f32) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  const float s = __ldg(scale);
  if (s == 1.0f) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (x_f32) {
    float* v = static_cast<float*>(x);
    for (int64_t i = i0; i < n; i += stride) v[i] *= s;
  } else {
    uint16_t* v = static_cast<uint16_t*>(x);
    for (int64_t i = i0; i < n; i += stride)
      v[i] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(static_cast<uint32_t>(v[i]) << 16) * s, 0.f) & 0xFFFFu);
  }
}

cudaError_t launch_scale(const float* scale, void* x, int64_t n, int x_f32, int grid, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  return launch_plain(scale_kernel, dim3(grid), dim3(256), 0, stream, scale, x, n, x_f32);
}

// dbias[j] = sum over m tiles of the per-tile column sums, in m order; with an
// fp32 accumulator the sum is added to acc[j] (when `accumulate`) and kept
// there until the call that writes the result (`write_final`).
__global__ void dbias_reduce_kernel(const float* __restrict__ part, int64_t ldg, int m_tiles, int rows_per_tile,
                                    int64_t cols, void* dbias, int bias_f32, const int32_t* row_count, float* acc,
                                    int accumulate, int write_final) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (j >= cols) return;
  // Under compaction only the tiles that hold a valid token were computed.
  const int tiles = row_count ? min(m_tiles, (*row_count + rows_per_tile - 1) / rows_per_tile) : m_tiles;
  float s = 0.f;
  for (int m = 0; m < tiles; ++m) s += part[static_cast<int64_t>(m) * ldg + j];
  if (acc) {
    if (accumulate) s = acc[j] + s;
    if (!write_final) {
      acc[j] = s;
      return;
    }
  }
  if (bias_f32) {
    reinterpret_cast<float*>(dbias)[j] = s;
  } else {
    reinterpret_cast<uint16_t*>(dbias)[j] = static_cast<uint16_t>(pack_bf16x2(s, 0.f) & 0xFFFFu);
  }
}

cudaError_t launch_dbias_reduce(const float* part, int64_t ldg, int m_tiles, int rows_per_tile, int64_t cols,
                                void* dbias, int bias_f32, const int32_t* row_count, float* acc, int accumulate,
                                int write_final, cudaStream_t stream) {
  const int64_t blocks = (cols + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  return launch_plain(dbias_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, part, ldg,
                    m_tiles, rows_per_tile, cols, dbias, bias_f32, row_count, acc, accumulate, write_final);
}

// dh = sum over K-split slots, in slot order, cast to the output dtype; with a
// row map, compacted row k goes to output row row_map[k] (rows at or past
// *row_count are skipped).
__global__ void dh_finalize_kernel(const float4* __restrict__ part, int64_t stride4, int ksplit, int64_t rows,
                                   int64_t cols, void* out, int out_f32, const int32_t* row_map,
                                   const int32_t* row_count) {
  griddep_release();  // lets the next kernel (a GEMM) launch and set up
  const int64_t n4 = rows * cols / 4;
  const int64_t limit = row_count ? static_cast<int64_t>(*row_count) * cols / 4 : n4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4 && i < limit;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 s = part[i];
    for (int k = 1; k < ksplit; ++k) {
      const float4 o = part[k * stride4 + i];
      s.x += o.x;
      s.y += o.y;
      s.z += o.z;
      s.w += o.w;
    }
    int64_t o = i;
    if (row_map) {
      const int64_t r = (i * 4) / cols;
      o = (static_cast<int64_t>(row_map[r]) * cols + (i * 4 - r * cols)) / 4;
    }
    if (out_f32) {
      reinterpret_cast<float4*>(out)[o] = s;
    } else {
      reinterpret_cast<uint2*>(out)[o] = make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
    }
  }
}

cudaError_t launch_dh_finalize(const float* part, int64_t stride, int ksplit, int64_t rows, int64_t cols, void* out,
                               int out_f32, const int32_t* row_map, const int32_t* row_count, int grid,
                               cudaStream_t stream) {
  return launch_plain(dh_finalize_kernel, dim3(grid), dim3(256), 0, stream, reinterpret_cast<const float4*>(part),
                    stride / 4, ksplit, rows, cols, out, out_f32, row_map, row_count);
}

}  // namespace flce
