// Fixed scratch for csa2_attend_static: the split partials of the sink-softmax attention live in
// a file-scope device array instead of a caller workspace, so that entry point never allocates.
//
// The array sits in its own translation unit (its own module): with lazy module loading the
// 19 MiB are claimed on a device only when the first csa2_attend_static call there resolves
// the symbol, and never by programs that use the other entry points alone.
#include <cuda.h>

#include <mutex>

#include "csa2_internal.h"

namespace csa2 {
namespace {

// Split partials: kStaticAttendRows rows of 64 heads x (512 unnormalised O values + m + l), fp32.
// attend_workspace_bytes() is the need of one launch; it stays within this on any device with at
// most kStaticAttendRows SMs, because a query batch is split only while queries x splits <= SMs.
constexpr size_t kStaticAttendFloats = kStaticAttendRows * kH * (kD + 2);
static __device__ __align__(256) float g_attend_scratch[kStaticAttendFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];
unsigned long long g_ctx[kMaxDevices];  // ID of the context each cached address belongs to

// The unique ID of the current context (driver entry points, found once), or false if there is
// none or the driver lacks the calls.  A device reset ends the primary context, and the one that
// replaces it has a new ID.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext c = nullptr;
  return get_current && get_id && get_current(&c) == CUDA_SUCCESS && c && get_id(c, id) == CUDA_SUCCESS;
}

}  // namespace

size_t attend_static_scratch_bytes() { return kStaticAttendFloats * sizeof(float); }

// Resolves the array's address on `device`, which must be the current device, under a lock:
// once per device and context (cudaGetSymbolAddress may load the module, which allocates the
// array).  Later calls in the same context only compare the context ID and read the cached
// pointer; a call in a new context (after a device reset) resolves the address again.
cudaError_t attend_static_scratch(int device, void** out) {
  *out = nullptr;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = 0;
  const bool known = current_context_id(&id);
  if (!g_addr[device] || !known || id != g_ctx[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attend_scratch);
    if (e != cudaSuccess) return e;
    g_addr[device] = p;
    g_ctx[device] = current_context_id(&id) ? id : 0;  // a context is current after that call
  }
  *out = g_addr[device];
  return cudaSuccess;
}

}  // namespace csa2
