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
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "flce.h"

namespace {

constexpr size_t kScratchBytes = FLCE_NOALLOC_SCRATCH_BYTES;
constexpr int kCacheSlots = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
struct Slot {
  unsigned long long ctx_id;  // 0 = empty
  void* addr;
};
Slot g_slots[kCacheSlots] = {};
int g_next_slot = 0;

// Process-unique id of the current CUDA context (0 when none is current yet).
int current_context_id(unsigned long long* id) {
  if (!g_ctx_current || !g_ctx_id) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FLCE_ERR_CUDA;
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FLCE_ERR_CUDA;
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return FLCE_ERR_CUDA;
  *id = 0;
  if (ctx && g_ctx_id(ctx, id) != CUDA_SUCCESS) return FLCE_ERR_CUDA;
  return FLCE_OK;
}

// Device address of g_scratch in the current context.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress (with the caller's device current) the first time a
// context calls, and cached under the context's process-unique id: another
// context on the same device, or the new one after cudaDeviceReset, looks it
// up again instead of reusing an address that is not valid there.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long id = 0;
  if (current_context_id(&id) != FLCE_OK) return FLCE_ERR_CUDA;
  for (int i = 0; id != 0 && i < kCacheSlots; ++i) {
    if (g_slots[i].ctx_id == id) {
      *out = g_slots[i].addr;
      return FLCE_OK;
    }
  }
  void* p = nullptr;  // makes the device's primary context current when none was
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return FLCE_ERR_CUDA;
  if (id == 0 && current_context_id(&id) != FLCE_OK) return FLCE_ERR_CUDA;
  if (id != 0) {
    g_slots[g_next_slot] = Slot{id, p};
    g_next_slot = (g_next_slot + 1) % kCacheSlots;
  }
  *out = p;
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
