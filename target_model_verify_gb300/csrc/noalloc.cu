// specdec_verify_noalloc: the verify step with its scratch in a static
// device array, for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code that runs
// inside a host program that owns all device memory and offers its plug-ins
// no allocator, or a per-token decode loop whose memory was planned up front
// and where a cudaMalloc would synchronise the device (stalling every other
// stream) or fail because a caching allocator already reserved the memory.
// For them the scratch lives in a file-scope __device__ array of
// SPECDEC_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library
// holds until the process exits.
#include <cuda.h>

#include <mutex>

#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPECDEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's identity of the context current on this thread: 0 when it
// cannot be told (no context yet, or the driver lacks the calls). Context
// IDs are unique for the life of the process, so a context created after a
// reset never matches one from before it.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(b);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct ScratchEntry {
  unsigned long long ctx_id;   // context the address belongs to (0: unknown)
  void* addr;
};
std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the context current on this
// thread. The array's name in host code is only a host-side stand-in, so
// the address is looked up (cudaGetSymbolAddress) with the device current,
// once per device and context: a reset or another context loads the module
// anew, and the array may then sit elsewhere.
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPECDEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchEntry& e = g_scratch[dev];
  const unsigned long long id = current_context_id();
  if (e.addr == nullptr || id == 0 || e.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPECDEC_ERR_CUDA;
    e.addr = p;
    // The look-up creates the context if there was none yet: take its ID now.
    e.ctx_id = current_context_id();
  }
  *out = e.addr;
  return SPECDEC_OK;
}

}  // namespace

extern "C" int specdec_verify_noalloc(const void* hidden, const void* W_lm,
                                      const int32_t* draft_tokens, const void* draft_logits, int B,
                                      int gamma, int d, int V, int dtype, float temperature,
                                      uint64_t seed, int mode, int32_t* out_tokens,
                                      int32_t* n_accepted, void* stream) {
  const size_t need = specdec_verify_workspace_size(B, gamma, d, V, dtype, mode);
  if (need == 0) {
    // Invalid shape or enum: let the regular checks name the error.
    return specdec_verify(hidden, W_lm, draft_tokens, draft_logits, B, gamma, d, V, dtype,
                          temperature, seed, mode, out_tokens, n_accepted, nullptr, 0, stream);
  }
  if (need > (size_t)SPECDEC_NOALLOC_SCRATCH_BYTES) return SPECDEC_ERR_WORKSPACE;
  if (B == 0) return SPECDEC_OK;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SPECDEC_OK) return rc;
  // The step clears what must start at zero (status word, sampler tickets)
  // itself, so the previous call's leftovers in the array do no harm.
  return specdec_verify(hidden, W_lm, draft_tokens, draft_logits, B, gamma, d, V, dtype,
                        temperature, seed, mode, out_tokens, n_accepted, scratch,
                        (size_t)SPECDEC_NOALLOC_SCRATCH_BYTES, stream);
}
