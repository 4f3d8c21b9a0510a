// int8_matmul_noalloc: the LLM.int8() matmul for callers that cannot allocate device
// memory when they call (an application whose device memory comes only from its own
// allocator, a latency-critical loop that must not call cudaMalloc, code running where
// allocation is not allowed). The pages have no counterpart to this call.
//
// Instead of a caller-provided workspace it uses one fixed scratch array in device memory,
// reserved by every GPU that loads this library until the process exits, and forwards to
// int8_matmul unchanged. Host code must not pass the array's name to a kernel: on the host
// it is only a stand-in symbol, so its device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current (the first call on a
// device does this; make it before any stream capture). int8_matmul clears the parts of
// the workspace that must start at zero on every call; the rest keeps the last call's
// contents. Calls that overlap on the GPU share the array and race.
#include <mutex>

#include "int8mm_internal.h"

#define I8_API extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[I8_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device (looked up once per device).
i8_status scratch_for_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return I8_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return I8_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return I8_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return I8_OK;
}

}  // namespace

I8_API i8_status int8_matmul_noalloc(const void* X, int T, int in, const int8_t* CB,
                                     const float* SCB, int out, float threshold,
                                     const void* bias, void* Y, void* stream) {
  // the smallest workspace int8_matmul accepts: a 64-column outlier capacity, unsplit
  // schedule (int8_matmul takes the split one when the scratch also holds its slots)
  if (int8_matmul_workspace_size(T, in, out, 64) == 0)
    // invalid sizes: the regular entry point reports them, launching nothing
    return int8_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, nullptr, 0, stream);
  const size_t need = i8mm::ws_layout(T, in, out, 64, false).total;
  if (need > I8_NOALLOC_SCRATCH_BYTES) return I8_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const i8_status st = scratch_for_current_device(&ws);
  if (st != I8_OK) return st;
  return int8_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, ws, I8_NOALLOC_SCRATCH_BYTES,
                     stream);
}
