// flce_noalloc.cu — flce_forward_noalloc: the forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin inside a host application that
// owns the whole device-memory budget and hands its plugins no allocator, or
// latency-critical code that must not pay for cudaMalloc's implicit device
// synchronisation.  For them this entry point runs the normal forward with its
// scratch (split partials, target logits, block sums, device status word) in a
// file-scope static device array of FLCE_NOALLOC_SCRATCH_BYTES, instead of a
// caller-provided workspace.  The caller still passes inputs and outputs.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits.  Every call uses the same array and it keeps the
// last call's contents; the forward clears the one word that must start at
// zero (the status word) and writes every other scratch byte before reading
// it.  Calls whose GPU work overlaps in time (different streams, threads or
// processes sharing the context) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "flce.h"

namespace {

constexpr size_t kScratchBytes = FLCE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return FLCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_noalloc(const flce_problem* problem, const void* hidden, const void* weight,
                                    const void* bias, const int64_t* targets, float* loss, float* lse,
                                    float* entropy, int64_t* correct, int64_t* n_valid, float* entropy_sum,
                                    flce_stream_t stream) {
  size_t need = 0;
  const int rc = flce_workspace_size(problem, 0, &need);
  if (rc != FLCE_OK) return rc;
  if (need > kScratchBytes) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rs = scratch_address(&scratch);
  if (rs != FLCE_OK) return rs;
  return flce_forward(problem, hidden, weight, bias, targets, loss, lse, entropy, correct, n_valid, entropy_sum,
                      scratch, kScratchBytes, stream);
}
