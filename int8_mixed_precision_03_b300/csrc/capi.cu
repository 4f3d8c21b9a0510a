// C-ABI entry points of libint8mm (declared in include/int8mm.h): host-side validation,
// workspace layout and the launch sequence. Nothing here computes on the host.
#include <cmath>
#include <cstring>

#include "int8mm_internal.h"

#define I8_API extern "C" __attribute__((visibility("default")))

namespace i8mm {
namespace {

thread_local int g_last_launches = 0;
thread_local cudaEvent_t g_prof[4] = {nullptr, nullptr, nullptr, nullptr};

void prof_mark(int i, cudaStream_t s) {
  if (g_prof[i]) cudaEventRecord(g_prof[i], s);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 1 = sm_103 device, 0 = other device, -1 = not checked yet (per device ordinal).
int g_dev_ok[64];
bool g_dev_init = false;

i8_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return I8_ERR_CUDA;
  if (dev < 0 || dev >= 64) return I8_ERR_UNSUPPORTED_DEVICE;
  if (!g_dev_init) {
    for (int& v : g_dev_ok) v = -1;
    g_dev_init = true;
  }
  if (g_dev_ok[dev] < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return I8_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
  }
  return g_dev_ok[dev] ? I8_OK : I8_ERR_UNSUPPORTED_DEVICE;
}

i8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? I8_OK : I8_ERR_CUDA; }

int ncap_limit(int in) { return (int)align_up((size_t)in, 64); }

// Largest outlier capacity (multiple of 64, at most ceil64(in)) whose layout fits.
int ncap_for_bytes(int T, int in, int out, size_t ws_bytes) {
  int hi = ncap_limit(in) / 64, lo = 0;
  while (lo < hi) {  // largest k in [0, hi] with layout(64k) fitting
    const int mid = (lo + hi + 1) / 2;
    if (ws_layout(T, in, out, 64 * mid).total <= ws_bytes) lo = mid; else hi = mid - 1;
  }
  return 64 * lo;
}

i8_status validate_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                          int out, float threshold, const void* bias, const void* Y,
                          const void* ws) {
  if (T < 0 || out < 0 || in <= 0 || in > I8_MAX_IN) return I8_ERR_INVALID_ARG;
  if (std::isnan(threshold) || threshold <= 0.0f) return I8_ERR_INVALID_ARG;
  if (!X || !CB || !SCB || !Y || !ws) return I8_ERR_INVALID_ARG;
  if (in % 16 != 0) return I8_ERR_ALIGNMENT;
  if (!aligned16(X) || !aligned16(CB) || !aligned16(SCB) || !aligned16(Y) || !aligned16(ws) ||
      (bias && !aligned16(bias)))
    return I8_ERR_ALIGNMENT;
  return I8_OK;
}

i8_status run_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB, int out,
                     float threshold, const void* bias, void* Y, void* workspace,
                     size_t ws_bytes, void* stream, int32_t* dbg_idx, int32_t* dbg_n,
                     int8_t* dbg_xq, float* dbg_rowabs, int32_t* dbg_acc,
                     uint64_t stall_ns = 0) {
  g_last_launches = 0;
  i8_status st = validate_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace);
  if (st != I8_OK) return st;
  if (stall_ns && gemv_fits(T, in)) return I8_ERR_INVALID_ARG;  // a tensor-core-path hook
  if ((dbg_idx && !aligned16(dbg_idx)) || (dbg_n && !aligned16(dbg_n)) ||
      (dbg_xq && !aligned16(dbg_xq)) || (dbg_rowabs && !aligned16(dbg_rowabs)) ||
      (dbg_acc && !aligned16(dbg_acc)))
    return I8_ERR_ALIGNMENT;
  if (T == 0 || out == 0) return I8_OK;
  const int ncap = ncap_for_bytes(T, in, out, ws_bytes);
  if (ncap < 64) return I8_ERR_WORKSPACE;
  if ((st = check_device()) != I8_OK) return st;
  const WsLayout L = ws_layout(T, in, out, ncap);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.header);
  uint32_t* mask = reinterpret_cast<uint32_t*>(ws + L.mask);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + L.idx);
  float* rowabs = reinterpret_cast<float*>(ws + L.rowabs);
  int32_t* l1 = reinterpret_cast<int32_t*>(ws + L.l1);

  if (cudaMemsetAsync(ws, 0, L.zero_bytes, s) != cudaSuccess) return I8_ERR_CUDA;
  ++g_last_launches;
  prof_mark(0, s);
  if ((st = from_cuda(launch_colstats(X, T, in, threshold_to_half_bits(threshold), hdr, mask,
                                      idx, ncap, s))) != I8_OK)
    return st;
  ++g_last_launches;
  prof_mark(1, s);
  if (gemv_fits(T, in)) {
    // decode sizes: int8 codes for the CUDA-core matmul, which reads the outlier weights
    // from CB itself (no W_out gather)
    int8_t* xq8 = reinterpret_cast<int8_t*>(ws + L.xq);
    if ((st = from_cuda(launch_quantize_gather(X, T, in, CB, SCB, out, hdr, mask, idx, ncap,
                                               nullptr, rowabs, ws + L.xout, nullptr, l1, xq8,
                                               s))) != I8_OK)
      return st;
    ++g_last_launches;
    prof_mark(2, s);
    GemvArgs g;
    g.CB = CB;
    g.SCB = SCB;
    g.T = T;
    g.in = in;
    g.out = out;
    g.xq8 = xq8;
    g.rowabs = rowabs;
    g.hdr = hdr;
    g.idx = idx;
    g.xout = ws + L.xout;
    g.ncap = ncap;
    g.bias = bias;
    g.Y = Y;
    g.acc_debug = dbg_acc;
    if ((st = from_cuda(launch_gemv_i8(g, s))) != I8_OK) return st;
    ++g_last_launches;
    prof_mark(3, s);
    if (dbg_xq && cudaMemcpyAsync(dbg_xq, xq8, (size_t)T * in, cudaMemcpyDeviceToDevice, s) !=
                      cudaSuccess)
      return I8_ERR_CUDA;
  } else {
    if ((st = from_cuda(launch_quantize_gather(X, T, in, CB, SCB, out, hdr, mask, idx, ncap,
                                               ws + L.xq, rowabs, ws + L.xout, ws + L.wout,
                                               l1, dbg_xq, s))) != I8_OK)
      return st;
    ++g_last_launches;
    prof_mark(2, s);
    GemmArgs g;
    g.a_int8 = CB;
    g.b_f16 = ws + L.xq;
    g.wout = ws + L.wout;
    g.xout = ws + L.xout;
    g.ncap = ncap;
    g.hdr = hdr;
    g.rowabs = rowabs;
    g.l1 = l1;
    g.acc_scratch = reinterpret_cast<int32_t*>(ws + L.acc);
    g.scb = SCB;
    g.bias = bias;
    g.Y = Y;
    g.acc_debug = dbg_acc;
    g.T = T;
    g.in = in;
    g.out = out;
    if (stall_ns) {  // test hook: nothing is loaded, so every pipeline wait runs out
      g.debug_skip_loads = 1;
      g.timeout_ns = stall_ns;
    }
    if ((st = from_cuda(launch_i8_gemm(g, s))) != I8_OK) return st;
    ++g_last_launches;
    prof_mark(3, s);
  }
  // debug copies of the intermediates (stream-ordered device copies)
  if (dbg_idx && cudaMemcpyAsync(dbg_idx, idx, sizeof(int32_t) * (size_t)in,
                                 cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  if (dbg_n && cudaMemcpyAsync(dbg_n, &hdr->n_out, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                               s) != cudaSuccess)
    return I8_ERR_CUDA;
  if (dbg_rowabs && cudaMemcpyAsync(dbg_rowabs, rowabs, sizeof(float) * (size_t)T,
                                    cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  return I8_OK;
}

}  // namespace
}  // namespace i8mm

using namespace i8mm;

I8_API i8_status int8_quantize_weight(const void* W, int out, int in, int8_t* CB, float* SCB,
                                      void* stream) {
  g_last_launches = 0;
  if (out < 0 || in < 0 || !W || !CB || !SCB) return I8_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(CB) || !aligned16(SCB)) return I8_ERR_ALIGNMENT;
  if (out == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  st = from_cuda(launch_absmax_rows(W, out, in, CB, SCB, static_cast<cudaStream_t>(stream)));
  if (st == I8_OK) g_last_launches = 1;
  return st;
}

I8_API size_t int8_matmul_workspace_size(int T, int in, int out, int max_outlier_cols) {
  if (T < 0 || out < 0 || in <= 0 || in > I8_MAX_IN) return 0;
  int cap = (max_outlier_cols <= 0 || max_outlier_cols > in) ? in : max_outlier_cols;
  cap = (int)align_up((size_t)cap, 64);
  return ws_layout(T, in, out, cap).total;
}

I8_API i8_status int8_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                             int out, float threshold, const void* bias, void* Y,
                             void* workspace, size_t ws_bytes, void* stream) {
  return run_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace, ws_bytes, stream,
                    nullptr, nullptr, nullptr, nullptr, nullptr);
}

I8_API i8_status int8_matmul_debug(const void* X, int T, int in, const int8_t* CB,
                                   const float* SCB, int out, float threshold, const void* bias,
                                   void* Y, void* workspace, size_t ws_bytes, void* stream,
                                   int32_t* outlier_idx, int32_t* n_out, int8_t* Xq,
                                   float* rowabs, int32_t* acc_s32) {
  return run_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace, ws_bytes, stream,
                    outlier_idx, n_out, Xq, rowabs, acc_s32);
}

I8_API i8_status i8_test_stalled_matmul(const void* X, int T, int in, const int8_t* CB,
                                        const float* SCB, int out, void* Y, void* workspace,
                                        size_t ws_bytes, uint64_t wait_limit_ns, void* stream) {
  if (wait_limit_ns == 0) return I8_ERR_INVALID_ARG;
  return run_matmul(X, T, in, CB, SCB, out, 6.0f, nullptr, Y, workspace, ws_bytes, stream,
                    nullptr, nullptr, nullptr, nullptr, nullptr, wait_limit_ns);
}

I8_API i8_status absmax_quantize_rows(const void* X, int rows, int cols, int8_t* Q,
                                      float* absmax, void* stream) {
  g_last_launches = 0;
  if (rows < 0 || cols < 0 || !X || !Q || !absmax) return I8_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || !aligned16(absmax)) return I8_ERR_ALIGNMENT;
  if (rows == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  st = from_cuda(launch_absmax_rows(X, rows, cols, Q, absmax, static_cast<cudaStream_t>(stream)));
  if (st == I8_OK) g_last_launches = 1;
  return st;
}

I8_API i8_status zeropoint_quantize_rows(const void* X, int rows, int cols, int8_t* Q, float* S,
                                         float* Z, void* stream) {
  g_last_launches = 0;
  if (rows < 0 || cols < 0 || !X || !Q || !S || !Z) return I8_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || !aligned16(S) || !aligned16(Z)) return I8_ERR_ALIGNMENT;
  if (rows == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  st = from_cuda(
      launch_zeropoint_rows(X, rows, cols, Q, S, Z, static_cast<cudaStream_t>(stream)));
  if (st == I8_OK) g_last_launches = 1;
  return st;
}

I8_API i8_status f16_matmul(const void* X, int T, int in, const void* W, int out,
                            const void* bias, void* Y, void* stream) {
  g_last_launches = 0;
  if (T < 0 || out < 0 || in <= 0 || !X || !W || !Y) return I8_ERR_INVALID_ARG;
  if (in % 16 != 0) return I8_ERR_ALIGNMENT;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (bias && !aligned16(bias)))
    return I8_ERR_ALIGNMENT;
  if (T == 0 || out == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  GemmArgs g;
  g.a_f16 = W;
  g.b_f16 = X;
  g.bias = bias;
  g.Y = Y;
  g.T = T;
  g.in = in;
  g.out = out;
  st = from_cuda(launch_f16_gemm(g, static_cast<cudaStream_t>(stream)));
  if (st == I8_OK) g_last_launches = 1;
  return st;
}

I8_API i8_status i8_get_status(const void* workspace, void* stream) {
  if (!workspace) return I8_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return I8_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return I8_ERR_CUDA;
  return static_cast<i8_status>(v);
}

I8_API const char* i8_status_string(i8_status s) {
  switch (s) {
    case I8_OK: return "ok";
    case I8_ERR_INVALID_ARG: return "invalid argument";
    case I8_ERR_ALIGNMENT: return "pointer not 16-byte aligned or in not a multiple of 16";
    case I8_ERR_WORKSPACE: return "workspace missing or too small";
    case I8_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (B300)";
    case I8_ERR_CUDA: return "CUDA runtime error";
    case I8_ERR_OUTLIER_CAP: return "more outlier columns than the workspace capacity";
    case I8_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case I8_ERR_SCRATCH_LIMIT: return "sizes exceed the built-in scratch of int8_matmul_noalloc";
  }
  return "unknown status";
}

I8_API int i8_last_launch_count(void) { return g_last_launches; }

I8_API void i8_set_profile_events(void** events) {
  for (int i = 0; i < 4; ++i)
    g_prof[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}
