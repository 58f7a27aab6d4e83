// Fixed scratch for csa2_attend_static: the split partials of the sink-softmax attention live in
// a file-scope device array instead of a caller workspace, so that entry point never allocates.
//
// The array sits in its own translation unit (its own module): with lazy module loading the
// 19 MiB are claimed on a device only when the first csa2_attend_static call there resolves
// the symbol, and never by programs that use the other entry points alone.
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

}  // namespace

size_t attend_static_scratch_bytes() { return kStaticAttendFloats * sizeof(float); }

// Resolves the array's address on `device`, which must be the current device.  Done once per
// device under a lock (cudaGetSymbolAddress may load the module, which allocates the array);
// later calls only read the cached pointer.
cudaError_t attend_static_scratch(int device, void** out) {
  *out = nullptr;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attend_scratch);
    if (e != cudaSuccess) return e;
    g_addr[device] = p;
  }
  *out = g_addr[device];
  return cudaSuccess;
}

}  // namespace csa2
