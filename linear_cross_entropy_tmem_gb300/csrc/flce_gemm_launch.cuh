// flce_gemm_launch.cuh — launch helpers for the two GEMM kernels (single CTA
// and CTA pair), shared by flce_fwd.cu and flce_bwd.cu.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "flce_gemm.cuh"
#include "flce_launch.h"

namespace flce {

// kern<<<grid, block, smem, stream>>>(args...), returning the launch error;
// `dependent`: as a programmatic dependent of the previous kernel in the
// stream (it may start while that kernel finishes and waits for its results in
// griddep_wait before touching global memory).
template <class... Params, class... Args>
static cudaError_t launch_ex(bool dependent, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The light kernels: ordinary stream order.
template <class... Params, class... Args>
static cudaError_t launch_plain(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args... args) {
  return launch_ex(false, kern, grid, block, smem, stream, args...);
}

template <class Epi>
static cudaError_t launch_gemm_single(const TmaMaps& m, const GemmSched& sc, const typename Epi::Params& p,
                                      int* status, int num_sms, cudaStream_t stream) {
  auto kern = gemm_kernel<Epi>;
  constexpr int smem = kGemmSmemBase + Epi::kTailBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(sc.total_units, num_sms));
  return launch_ex(true, kern, dim3(grid), dim3(kThreads), smem, stream, m.a0, m.a1, m.a2, m.b0, m.b1, m.b2, sc,
                   p, status);
}

// Launch configuration of the pair kernel: clusters of two CTAs, and (when
// `dependent`) a programmatic dependent of the previous kernel in the stream.
template <class Epi>
static cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, cudaStream_t stream, bool dependent) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kGemmPairSmemBase + Epi::kTailBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
  return cfg;
}

// CTA pairs of the pair kernel that can be resident at once on the current
// device, one CTA per SM.  The kernel's shared-memory attribute is set on every
// call (it belongs to the current context); the occupancy query is cached per
// device, in atomics, so that host threads may call at once.
template <class Epi>
static cudaError_t resident_pairs(int num_sms, int* out) {
  auto kern = gemm_pair_kernel<Epi>;
  static std::atomic<int> resident[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kGemmPairSmemBase + Epi::kTailBytes)) != cudaSuccess)
    return e;
  int n = resident[dev].load(std::memory_order_relaxed);
  if (n == 0) {  // every thread that gets here computes the same value
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config<Epi>(attr, nullptr, false);
    cfg.gridDim = dim3(2 * std::max(1, num_sms / 2));
    if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
    n = std::max(1, n);
    resident[dev].store(n, std::memory_order_relaxed);
  }
  *out = std::min(n, std::max(1, num_sms / 2));
  return cudaSuccess;
}

template <class Epi>
static cudaError_t launch_gemm_pair(const TmaMaps& m, const GemmSched& sc, const typename Epi::Params& p,
                                    int* status, int num_sms, cudaStream_t stream) {
  auto kern = gemm_pair_kernel<Epi>;
  int resident = 0;
  cudaError_t e = resident_pairs<Epi>(num_sms, &resident);  // also sets the smem attribute
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config<Epi>(attr, stream, true);
  const int clusters = std::max(1, std::min(sc.total_units, resident));
  cfg.gridDim = dim3(2 * clusters);
  return cudaLaunchKernelEx(&cfg, kern, m.a0, m.a1, m.a2, m.b0, m.b1, m.b2, sc, p, status);
}

template <class Epi>
static cudaError_t launch_gemm(bool pair, const TmaMaps& m, const GemmSched& sc, const typename Epi::Params& p,
                               int* status, int num_sms, cudaStream_t stream) {
  return pair ? launch_gemm_pair<Epi>(m, sc, p, status, num_sms, stream)
              : launch_gemm_single<Epi>(m, sc, p, status, num_sms, stream);
}

}  // namespace flce
