// flce_bwd.cu — backward kernels: the recompute GEMM with the logit-gradient
// epilogue (four variants: bias x soft cap), the dW store GEMM, the dh
// accumulate GEMM, the ordered dbias reduction and the dh K-split finalize.
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

// dbias[j] = sum over m tiles of the per-tile column sums, in m order.
__global__ void dbias_reduce_kernel(const float* __restrict__ part, int64_t ldg, int m_tiles, int64_t cols,
                                    void* dbias, int bias_f32, const int32_t* row_count) {
  const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (j >= cols) return;
  // Under compaction only the tiles that hold a valid token were computed.
  const int tiles = row_count ? min(m_tiles, (*row_count + kBM - 1) / kBM) : m_tiles;
  float s = 0.f;
  for (int m = 0; m < tiles; ++m) s += part[static_cast<int64_t>(m) * ldg + j];
  if (bias_f32) {
    reinterpret_cast<float*>(dbias)[j] = s;
  } else {
    reinterpret_cast<uint16_t*>(dbias)[j] = static_cast<uint16_t>(pack_bf16x2(s, 0.f) & 0xFFFFu);
  }
}

cudaError_t launch_dbias_reduce(const float* part, int64_t ldg, int m_tiles, int64_t cols, void* dbias,
                                int bias_f32, const int32_t* row_count, cudaStream_t stream) {
  const int64_t blocks = (cols + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  dbias_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(part, ldg, m_tiles, cols, dbias, bias_f32,
                                                                          row_count);
  return cudaGetLastError();
}

// dh = sum over K-split slots, in slot order, cast to the output dtype; with a
// row map, compacted row k goes to output row row_map[k] (rows at or past
// *row_count are skipped).
__global__ void dh_finalize_kernel(const float4* __restrict__ part, int64_t stride4, int ksplit, int64_t rows,
                                   int64_t cols, void* out, int out_f32, const int32_t* row_map,
                                   const int32_t* row_count) {
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
  dh_finalize_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(part), stride / 4, ksplit, rows, cols,
                                               out, out_f32, row_map, row_count);
  return cudaGetLastError();
}

}  // namespace flce
