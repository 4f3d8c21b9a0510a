// int8_matmul_noalloc: the LLM.int8() matmul for callers that cannot allocate device
// memory when they call (an application whose device memory comes only from its own
// allocator, a latency-critical loop that must not call cudaMalloc, code running where
// allocation is not allowed). The pages have no counterpart to this call.
//
// Instead of a caller-provided workspace it uses one fixed scratch array in device memory,
// reserved by every GPU that loads this library until the process exits, and forwards to
// int8_matmul unchanged. Host code must not pass the array's name to a kernel: on the host
// it is only a stand-in symbol, so its device address is looked up with
// cudaGetSymbolAddress, once per device and CUDA context, with that device current (the
// first call on a device does this; make it before any stream capture). A device whose
// context was destroyed (cudaDeviceReset) gets the address looked up again in its new
// context. int8_matmul clears the parts of the workspace that must start at zero on every
// call; the rest keeps the last call's contents. Calls that overlap on the GPU share the
// array and race. i8_noalloc_status reads the device status word the last call left at
// the start of the array.
#include <cudaTypedefs.h>

#include <mutex>

#include "int8mm_internal.h"

#define I8_API extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[I8_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchRef {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: unknown)
};
ScratchRef g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Unique id of the current CUDA context (never reused within the process), or 0 if the
// driver entry points are not available. Fetched through the runtime, so the library does
// not link libcuda.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q1, q2;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault,
                                         &q1) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    }
    cudaGetLastError();
    looked_up = true;
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device (looked up once per device and
// context).
i8_status scratch_for_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return I8_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return I8_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchRef& ref = g_scratch[dev];
  const unsigned long long ctx = current_context_id();
  if (!ref.addr || (ctx != 0 && ctx != ref.ctx_id)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no error pending for a later launch check
      return I8_ERR_CUDA;
    }
    ref.addr = p;
    ref.ctx_id = current_context_id();  // the lookup may have created the context
  }
  *addr = ref.addr;
  return I8_OK;
}

}  // namespace

I8_API i8_status int8_matmul_noalloc(const void* X, int T, int in, const int8_t* CB,
                                     const float* SCB, int out, float threshold,
                                     const void* bias, void* Y, void* stream) {
  // arguments, sizes and the device first: nothing here touches the scratch before they
  // pass
  i8_status st = i8mm::matmul_precheck(X, T, in, CB, SCB, out, threshold, bias, Y);
  if (st != I8_OK) return st;
  if (T == 0 || out == 0) return I8_OK;
  // the smallest workspace int8_matmul accepts: a 64-column outlier capacity, unsplit
  // schedule (int8_matmul takes the split one when the scratch also holds its slots)
  const size_t need = i8mm::ws_layout(T, in, out, 64, false).total;
  if (need > I8_NOALLOC_SCRATCH_BYTES) return I8_ERR_SCRATCH_LIMIT;
  if ((st = i8mm::current_device_check()) != I8_OK) return st;
  void* ws = nullptr;
  if ((st = scratch_for_current_device(&ws)) != I8_OK) return st;
  return int8_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, ws, I8_NOALLOC_SCRATCH_BYTES,
                     stream);
}

I8_API i8_status i8_noalloc_status(void* stream) {
  void* ws = nullptr;
  const i8_status st = scratch_for_current_device(&ws);
  if (st != I8_OK) return st;
  return i8_get_status(ws, stream);
}
