// Forward entry point for callers that cannot allocate device memory.
//
// grpo_head_forward needs scratch space (per-split LSE partials and the
// gathered target logits) that the caller normally provides as `ws`.  Some
// callers cannot provide it: their device memory is entirely owned by another
// allocator (a framework's caching allocator that has reserved the pool, or a
// memory plan fixed before the step starts), or they must not call cudaMalloc
// in the middle of a step because cudaMalloc can synchronise the device.  For
// them grpo_head_forward_noalloc runs the same forward with its scratch in the
// fixed device array below, so the caller only passes inputs and outputs.
//
// The array is GH_NOALLOC_SCRATCH_BYTES (64 MiB); every GPU that loads this
// library holds it until the process exits.  Its device address is looked up
// on the first call made on each device (with that device current), so that
// first call should come before any stream capture.  The address belongs to
// the CUDA context it was looked up in: a later call from a different context
// (after cudaDeviceReset, say) looks it up again.  All calls share the array:
// calls whose GPU work overlaps (different streams or threads) race on it and
// must be serialised by the caller.  The array keeps the previous call's
// contents; nothing in it has to start at zero, because the forward writes
// every scratch slot it later reads within the same call.
#include <cuda.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "grpo_head.h"
#include "internal.h"

namespace gh {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GH_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
struct NoallocSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;  // unique id of the context the address belongs to (0: unknown)
};
NoallocSlot g_noalloc_slot[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}

// Unique id (for the life of the process) of the calling thread's current
// context, 0 when there is none or the driver cannot say.
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call there and again when the current context has changed since.
gh_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error_message(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return GH_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    set_error_message("device index out of range for the no-allocation scratch table");
    return GH_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoallocSlot& slot = g_noalloc_slot[dev];
  const unsigned long long cur = current_context_id();
  if (!slot.ptr || (cur != 0 && cur != slot.ctx_id)) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      set_error_message(std::string("cudaGetSymbolAddress(no-allocation scratch): ") + cudaGetErrorString(e));
      return GH_ERR_CUDA;
    }
    slot.ptr = p;
    slot.ctx_id = current_context_id();  // the lookup makes the device's primary context current
  }
  *out = slot.ptr;
  return GH_OK;
}

}  // namespace
}  // namespace gh

extern "C" gh_status grpo_head_forward_noalloc(const gh_head* head, const gh_grpo* grpo, float* logp, float* lse,
                                               float* coef, float* loss3, int32_t* status, void* stream) {
  const size_t need = grpo_head_forward_workspace_size(head);
  if (need == 0) {
    // invalid problem (the regular entry point reports why) or one needing no scratch
    return grpo_head_forward(head, grpo, logp, lse, coef, loss3, status, nullptr, 0, stream);
  }
  if (need > static_cast<size_t>(GH_NOALLOC_SCRATCH_BYTES)) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "problem needs %zu bytes of forward scratch, more than the %zu-byte no-allocation buffer "
             "(use grpo_head_forward with a caller workspace)",
             need, static_cast<size_t>(GH_NOALLOC_SCRATCH_BYTES));
    gh::set_error_message(buf);
    return GH_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const gh_status s = gh::noalloc_scratch(&scratch);
  if (s != GH_OK) return s;
  return grpo_head_forward(head, grpo, logp, lse, coef, loss3, status, scratch,
                           static_cast<size_t>(GH_NOALLOC_SCRATCH_BYTES), stream);
}
