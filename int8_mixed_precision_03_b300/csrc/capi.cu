// C-ABI entry points of libint8mm (declared in include/int8mm.h): host-side validation,
// workspace layout and the launch sequence. Nothing here computes on the host.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "int8mm_internal.h"

#define I8_API extern "C" __attribute__((visibility("default")))

namespace i8mm {

int sm_count() {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};  // 0: not looked up yet
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();  // no device here: leave no error pending for a later launch check
    return kSmFallback;
  }
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kSmFallback;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

thread_local int g_last_launches = 0;
constexpr int kProfSlots = 8;
thread_local cudaEvent_t g_prof[kProfSlots] = {};
thread_local int g_prof_n = 0;

void prof_mark(int i, cudaStream_t s) {
  if (i >= 0 && i < g_prof_n && g_prof[i]) cudaEventRecord(g_prof[i], s);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 1 = sm_103 device, 0 = other device, -1 = not checked yet (per device ordinal).
int g_dev_ok[64];
bool g_dev_init = false;

i8_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();  // leave no error pending for a later launch check
    return I8_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return I8_ERR_UNSUPPORTED_DEVICE;
  if (!g_dev_init) {
    for (int& v : g_dev_ok) v = -1;
    g_dev_init = true;
  }
  if (g_dev_ok[dev] < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return I8_ERR_CUDA;
    }
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
  }
  return g_dev_ok[dev] ? I8_OK : I8_ERR_UNSUPPORTED_DEVICE;
}

i8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? I8_OK : I8_ERR_CUDA; }

int ncap_limit(int in) { return (int)align_up((size_t)in, 64); }

// Largest outlier capacity (multiple of 64, at most ceil64(in)) whose layout fits.
int ncap_for_bytes(int T, int in, int out, size_t ws_bytes, bool split_ok) {
  int hi = ncap_limit(in) / 64, lo = 0;
  while (lo < hi) {  // largest k in [0, hi] with layout(64k) fitting
    const int mid = (lo + hi + 1) / 2;
    if (ws_layout(T, in, out, 64 * mid, split_ok).total <= ws_bytes) lo = mid; else hi = mid - 1;
  }
  return 64 * lo;
}

i8_status validate_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                          int out, float threshold, const void* bias, const void* Y,
                          const void* ws) {
  if (T < 0 || out < 0 || in <= 0 || in > I8_MAX_IN) return I8_ERR_INVALID_ARG;
  if (std::isnan(threshold) || threshold <= 0.0f) return I8_ERR_INVALID_ARG;
  if (!CB || !SCB || !ws) return I8_ERR_INVALID_ARG;
  if (T > 0 && (!X || !Y)) return I8_ERR_INVALID_ARG;  // an empty batch may pass nulls
  if (in % 16 != 0) return I8_ERR_ALIGNMENT;
  if (!aligned16(X) || !aligned16(CB) || !aligned16(SCB) || !aligned16(Y) || !aligned16(ws) ||
      (bias && !aligned16(bias)))
    return I8_ERR_ALIGNMENT;
  return I8_OK;
}

// One int8 matmul on its (already zeroed) workspace section: column statistics (or, when
// the previous matmul's epilogue has filled the mask, only its compaction), quantize +
// gather, then the tensor-core or decode matmul with the optional epilogue extras.
struct Layer {
  const void* X = nullptr;
  int T = 0, in = 0, out = 0;
  const int8_t* CB = nullptr;
  const float* SCB = nullptr;
  uint16_t thr_bits = 0x7C00u;
  const void* bias = nullptr;
  void* Y = nullptr;
  uint8_t* ws = nullptr;
  WsLayout L;
  NextLayer next;                  // FFN up projection: activation + next layer's mask
  bool stats_in_mask = false;      // the mask was filled by the previous matmul
  const WsHeader* prev = nullptr;  // its status word, carried into this one
  int8_t* dbg_xq = nullptr;
  int32_t* dbg_acc = nullptr;
  // zeropoint activation codes (tensor-core kernel at every T): the weight's code sums
  const int32_t* zp_cbsum = nullptr;
  float* dbg_S = nullptr;
  float* dbg_Z = nullptr;
  uint64_t stall_ns = 0;
  int prof_base = -1;              // profiling events prof_base .. +3, or -1: none
};

i8_status launch_layer(const Layer& ly, cudaStream_t s) {
  const WsLayout& L = ly.L;
  uint8_t* ws = ly.ws;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.header);
  uint32_t* mask = reinterpret_cast<uint32_t*>(ws + L.mask);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + L.idx);
  float* rowabs = reinterpret_cast<float*>(ws + L.rowabs);
  int32_t* l1 = reinterpret_cast<int32_t*>(ws + L.l1);
  const int ncap = L.ncap;
  i8_status st;
  if (ly.prof_base >= 0) prof_mark(ly.prof_base + 0, s);
  if (ly.stats_in_mask)
    st = from_cuda(launch_mask_index(ly.in, hdr, mask, idx, ncap, ly.prev, s));
  else
    st = from_cuda(launch_colstats(ly.X, ly.T, ly.in, ly.thr_bits, hdr, mask, idx, ncap, s));
  if (st != I8_OK) return st;
  ++g_last_launches;
  if (ly.prof_base >= 0) prof_mark(ly.prof_base + 1, s);
  const bool zp = ly.zp_cbsum != nullptr;
  if (!zp && gemv_fits(ly.T, ly.in)) {
    // decode sizes: int8 codes for the CUDA-core matmul, which reads the outlier weights
    // from CB itself (no W_out gather)
    int8_t* xq8 = reinterpret_cast<int8_t*>(ws + L.xq);
    if ((st = from_cuda(launch_quantize_gather(ly.X, ly.T, ly.in, ly.CB, ly.SCB, ly.out, hdr,
                                               mask, idx, ncap, nullptr, rowabs, ws + L.xout,
                                               nullptr, nullptr, l1, xq8, s))) != I8_OK)
      return st;
    ++g_last_launches;
    if (ly.prof_base >= 0) prof_mark(ly.prof_base + 2, s);
    GemvArgs g;
    g.CB = ly.CB;
    g.SCB = ly.SCB;
    g.T = ly.T;
    g.in = ly.in;
    g.out = ly.out;
    g.xq8 = xq8;
    g.rowabs = rowabs;
    g.hdr = hdr;
    g.idx = idx;
    g.xout = ws + L.xout;
    g.ncap = ncap;
    g.bias = ly.bias;
    g.Y = ly.Y;
    g.acc_debug = ly.dbg_acc;
    g.next = ly.next;
    if ((st = from_cuda(launch_gemv_i8(g, s))) != I8_OK) return st;
    ++g_last_launches;
    if (ly.prof_base >= 0) prof_mark(ly.prof_base + 3, s);
    if (ly.dbg_xq && cudaMemcpyAsync(ly.dbg_xq, xq8, (size_t)ly.T * ly.in,
                                     cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return I8_ERR_CUDA;
  } else {
    int32_t* zi = reinterpret_cast<int32_t*>(ws + L.zi);
    int32_t* cbout = reinterpret_cast<int32_t*>(ws + L.cbout);
    if (zp)
      st = from_cuda(launch_quantize_gather_zp(ly.X, ly.T, ly.in, ly.CB, ly.SCB, ly.out, hdr,
                                               mask, idx, ncap, ws + L.xq, rowabs, zi,
                                               ws + L.xout, ws + L.wout, ws + L.xoT, cbout, l1,
                                               ly.dbg_xq, ly.dbg_S, ly.dbg_Z, s));
    else
      st = from_cuda(launch_quantize_gather(ly.X, ly.T, ly.in, ly.CB, ly.SCB, ly.out, hdr,
                                            mask, idx, ncap, ws + L.xq, rowabs, ws + L.xout,
                                            ws + L.wout, ws + L.xoT, l1, ly.dbg_xq, s));
    if (st != I8_OK) return st;
    ++g_last_launches;
    if (ly.prof_base >= 0) prof_mark(ly.prof_base + 2, s);
    GemmArgs g;
    g.a_int8 = ly.CB;
    g.b_f16 = ws + L.xq;
    g.wout = ws + L.wout;
    g.xout = ws + L.xout;
    g.xoT = ws + L.xoT;
    g.ncap = ncap;
    g.hdr = hdr;
    g.rowabs = rowabs;
    g.l1 = l1;
    g.acc_scratch = reinterpret_cast<int32_t*>(ws + L.acc);
    g.scb = ly.SCB;
    g.bias = ly.bias;
    g.Y = ly.Y;
    g.acc_debug = ly.dbg_acc;
    g.T = ly.T;
    g.in = ly.in;
    g.out = ly.out;
    g.next = ly.next;
    if (L.split) {
      g.split = L.split;
      g.part = reinterpret_cast<int32_t*>(ws + L.part);
      g.part_f = reinterpret_cast<float*>(ws + L.part_f);
      g.tile_cnt = reinterpret_cast<int32_t*>(ws + L.tile_cnt);
    }
    if (zp) {
      g.zi = zi;
      g.cbsum = ly.zp_cbsum;
      g.cbout = cbout;
    }
    if (ly.stall_ns) {  // test hook: nothing is loaded, so every pipeline wait runs out
      g.debug_skip_loads = 1;
      g.timeout_ns = ly.stall_ns;
    }
    if ((st = from_cuda(launch_i8_gemm(g, s))) != I8_OK) return st;
    ++g_last_launches;
    if (ly.prof_base >= 0) prof_mark(ly.prof_base + 3, s);
  }
  return I8_OK;
}

i8_status run_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB, int out,
                     float threshold, const void* bias, void* Y, void* workspace,
                     size_t ws_bytes, void* stream, int32_t* dbg_idx, int32_t* dbg_n,
                     int8_t* dbg_xq, float* dbg_rowabs, int32_t* dbg_acc,
                     uint64_t stall_ns = 0, const int32_t* zp_cbsum = nullptr,
                     bool zp = false, float* dbg_S = nullptr, float* dbg_Z = nullptr) {
  g_last_launches = 0;
  i8_status st = validate_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace);
  if (st != I8_OK) return st;
  if (zp && !zp_cbsum) return I8_ERR_INVALID_ARG;
  if ((zp_cbsum && !aligned16(zp_cbsum)) || (dbg_S && !aligned16(dbg_S)) ||
      (dbg_Z && !aligned16(dbg_Z)))
    return I8_ERR_ALIGNMENT;
  if (stall_ns && gemv_fits(T, in)) return I8_ERR_INVALID_ARG;  // a tensor-core-path hook
  if ((dbg_idx && !aligned16(dbg_idx)) || (dbg_n && !aligned16(dbg_n)) ||
      (dbg_xq && !aligned16(dbg_xq)) || (dbg_rowabs && !aligned16(dbg_rowabs)) ||
      (dbg_acc && !aligned16(dbg_acc)))
    return I8_ERR_ALIGNMENT;
  if (T == 0 || out == 0) return I8_OK;
  // the split schedule's slots if the workspace holds them, else the unsplit schedule
  bool split_ok = true;
  int ncap = ncap_for_bytes(T, in, out, ws_bytes, true);
  if (ncap < 64) {
    split_ok = false;
    ncap = ncap_for_bytes(T, in, out, ws_bytes, false);
  }
  if (ncap < 64) return I8_ERR_WORKSPACE;
  if ((st = check_device()) != I8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Layer ly;
  ly.X = X;
  ly.T = T;
  ly.in = in;
  ly.out = out;
  ly.CB = CB;
  ly.SCB = SCB;
  ly.thr_bits = threshold_to_half_bits(threshold);
  ly.bias = bias;
  ly.Y = Y;
  ly.ws = static_cast<uint8_t*>(workspace);
  ly.L = ws_layout(T, in, out, ncap, split_ok);
  ly.dbg_xq = dbg_xq;
  ly.dbg_acc = dbg_acc;
  ly.stall_ns = stall_ns;
  ly.zp_cbsum = zp ? zp_cbsum : nullptr;
  ly.dbg_S = dbg_S;
  ly.dbg_Z = dbg_Z;
  ly.prof_base = 0;
  if (cudaMemsetAsync(ly.ws, 0, ly.L.zero_bytes, s) != cudaSuccess) return I8_ERR_CUDA;
  ++g_last_launches;
  if ((st = launch_layer(ly, s)) != I8_OK) return st;
  // debug copies of the intermediates (stream-ordered device copies)
  uint8_t* ws = ly.ws;
  if (dbg_idx && cudaMemcpyAsync(dbg_idx, ws + ly.L.idx, sizeof(int32_t) * (size_t)in,
                                 cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  if (dbg_n && cudaMemcpyAsync(dbg_n, &reinterpret_cast<WsHeader*>(ws + ly.L.header)->n_out,
                               sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  if (dbg_rowabs && cudaMemcpyAsync(dbg_rowabs, ws + ly.L.rowabs, sizeof(float) * (size_t)T,
                                    cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  return I8_OK;
}

// ---------------------------------------------------------------- FFN block
// Workspace: [second matmul's section | first matmul's section], both 256-byte aligned, so
// that the status word at offset 0 is the second matmul's, into which the first one's is
// carried (launch_mask_index) before the second matmul's own kernels run.
struct FfnPlan {
  WsLayout down, up;
  size_t up_off = 0, total = 0;
};

FfnPlan ffn_plan(int T, int d_model, int d_ff, int cap, bool split_ok = true) {
  FfnPlan P;
  const int cap_up = std::min(cap, ncap_limit(d_model));
  const int cap_down = std::min(cap, ncap_limit(d_ff));
  P.down = ws_layout(T, d_ff, d_model, cap_down, split_ok);
  P.up = ws_layout(T, d_model, d_ff, cap_up, split_ok);
  P.up_off = align_up(P.down.total, 256);
  P.total = P.up_off + P.up.total;
  return P;
}

// Largest capacity (multiple of 64, at most the wider input's limit) whose plan fits.
int ffn_cap_for_bytes(int T, int d_model, int d_ff, size_t ws_bytes, bool split_ok) {
  int hi = std::max(ncap_limit(d_model), ncap_limit(d_ff)) / 64, lo = 0;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (ffn_plan(T, d_model, d_ff, 64 * mid, split_ok).total <= ws_bytes) lo = mid;
    else hi = mid - 1;
  }
  return 64 * lo;
}

i8_status run_ffn(const void* X, int T, int d_model, int d_ff, const int8_t* CB_up,
                  const float* SCB_up, const void* bias_up, const int8_t* CB_down,
                  const float* SCB_down, const void* bias_down, float threshold, int act,
                  void* H, void* Y, void* workspace, size_t ws_bytes, void* stream,
                  int32_t* dbg_idx, int32_t* dbg_n) {
  g_last_launches = 0;
  if (act != I8_ACT_NONE && act != I8_ACT_RELU) return I8_ERR_INVALID_ARG;
  if (d_ff <= 0 || d_ff > I8_MAX_IN || !CB_down || !SCB_down) return I8_ERR_INVALID_ARG;
  i8_status st = validate_matmul(X, T, d_model, CB_up, SCB_up, d_ff, threshold, bias_up, H,
                                 workspace);
  if (st != I8_OK) return st;
  if (T > 0 && !Y) return I8_ERR_INVALID_ARG;
  if (d_ff % 16 != 0) return I8_ERR_ALIGNMENT;
  if (!aligned16(CB_down) || !aligned16(SCB_down) || !aligned16(Y) ||
      (bias_down && !aligned16(bias_down)) || (dbg_idx && !aligned16(dbg_idx)) ||
      (dbg_n && !aligned16(dbg_n)))
    return I8_ERR_ALIGNMENT;
  if (T == 0) return I8_OK;
  bool split_ok = true;
  int cap = ffn_cap_for_bytes(T, d_model, d_ff, ws_bytes, true);
  if (cap < 64) {
    split_ok = false;
    cap = ffn_cap_for_bytes(T, d_model, d_ff, ws_bytes, false);
  }
  if (cap < 64) return I8_ERR_WORKSPACE;
  if ((st = check_device()) != I8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const FfnPlan P = ffn_plan(T, d_model, d_ff, cap, split_ok);
  uint8_t* ws_down = static_cast<uint8_t*>(workspace);
  uint8_t* ws_up = ws_down + P.up_off;
  const uint16_t thr_bits = threshold_to_half_bits(threshold);

  Layer up;
  up.X = X;
  up.T = T;
  up.in = d_model;
  up.out = d_ff;
  up.CB = CB_up;
  up.SCB = SCB_up;
  up.thr_bits = thr_bits;
  up.bias = bias_up;
  up.Y = H;
  up.ws = ws_up;
  up.L = P.up;
  up.next.relu = act == I8_ACT_RELU ? 1 : 0;
  up.next.mask = reinterpret_cast<uint32_t*>(ws_down + P.down.mask);
  up.next.thr_bits = thr_bits;

  Layer down;
  down.X = H;
  down.T = T;
  down.in = d_ff;
  down.out = d_model;
  down.CB = CB_down;
  down.SCB = SCB_down;
  down.thr_bits = thr_bits;
  down.bias = bias_down;
  down.Y = Y;
  down.ws = ws_down;
  down.L = P.down;
  down.stats_in_mask = true;
  down.prev = reinterpret_cast<const WsHeader*>(ws_up + P.up.header);
  up.prof_base = 0;
  down.prof_base = 4;

  // both masks start empty: the first matmul's epilogue writes the second one's
  if (cudaMemsetAsync(ws_down, 0, P.down.zero_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(ws_up, 0, P.up.zero_bytes, s) != cudaSuccess)
    return I8_ERR_CUDA;
  g_last_launches += 2;
  if ((st = launch_layer(up, s)) != I8_OK) return st;
  if ((st = launch_layer(down, s)) != I8_OK) return st;
  if (dbg_idx && cudaMemcpyAsync(dbg_idx, ws_down + P.down.idx, sizeof(int32_t) * (size_t)d_ff,
                                 cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  if (dbg_n &&
      cudaMemcpyAsync(dbg_n, &reinterpret_cast<WsHeader*>(ws_down + P.down.header)->n_out,
                      sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return I8_ERR_CUDA;
  return I8_OK;
}

}  // namespace

i8_status matmul_precheck(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                          int out, float threshold, const void* bias, const void* Y) {
  // validate_matmul with a stand-in workspace pointer (aligned, never dereferenced)
  const void* ws_stand_in = reinterpret_cast<const void*>(uintptr_t{256});
  return validate_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, ws_stand_in);
}

i8_status current_device_check() { return check_device(); }

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

I8_API i8_status int8_weight_code_sums(const int8_t* CB, int out, int in, int32_t* CBsum,
                                       void* stream) {
  g_last_launches = 0;
  if (out < 0 || in < 0 || !CB || !CBsum) return I8_ERR_INVALID_ARG;
  if (!aligned16(CB) || !aligned16(CBsum)) return I8_ERR_ALIGNMENT;
  if (out == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  st = from_cuda(launch_code_sums(CB, out, in, CBsum, static_cast<cudaStream_t>(stream)));
  if (st == I8_OK) g_last_launches = 1;
  return st;
}

I8_API i8_status int8_matmul_zeropoint(const void* X, int T, int in, const int8_t* CB,
                                       const float* SCB, const int32_t* CBsum, int out,
                                       float threshold, const void* bias, void* Y,
                                       void* workspace, size_t ws_bytes, void* stream) {
  return run_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace, ws_bytes, stream,
                    nullptr, nullptr, nullptr, nullptr, nullptr, 0, CBsum, true);
}

I8_API i8_status int8_matmul_zeropoint_debug(const void* X, int T, int in, const int8_t* CB,
                                             const float* SCB, const int32_t* CBsum, int out,
                                             float threshold, const void* bias, void* Y,
                                             void* workspace, size_t ws_bytes, void* stream,
                                             int32_t* outlier_idx, int32_t* n_out, int8_t* Xq,
                                             float* S, float* Z, int32_t* acc_s32) {
  return run_matmul(X, T, in, CB, SCB, out, threshold, bias, Y, workspace, ws_bytes, stream,
                    outlier_idx, n_out, Xq, nullptr, acc_s32, 0, CBsum, true, S, Z);
}

I8_API size_t int8_ffn_workspace_size(int T, int d_model, int d_ff, int max_outlier_cols) {
  if (T < 0 || d_model <= 0 || d_ff <= 0 || d_model > I8_MAX_IN || d_ff > I8_MAX_IN) return 0;
  const int wide = std::max(d_model, d_ff);
  int cap = (max_outlier_cols <= 0 || max_outlier_cols > wide) ? wide : max_outlier_cols;
  return ffn_plan(T, d_model, d_ff, (int)align_up((size_t)cap, 64)).total;
}

I8_API i8_status int8_ffn(const void* X, int T, int d_model, int d_ff, const int8_t* CB_up,
                          const float* SCB_up, const void* bias_up, const int8_t* CB_down,
                          const float* SCB_down, const void* bias_down, float threshold,
                          int act, void* H, void* Y, void* workspace, size_t ws_bytes,
                          void* stream) {
  return run_ffn(X, T, d_model, d_ff, CB_up, SCB_up, bias_up, CB_down, SCB_down, bias_down,
                 threshold, act, H, Y, workspace, ws_bytes, stream, nullptr, nullptr);
}

I8_API i8_status int8_ffn_debug(const void* X, int T, int d_model, int d_ff,
                                const int8_t* CB_up, const float* SCB_up, const void* bias_up,
                                const int8_t* CB_down, const float* SCB_down,
                                const void* bias_down, float threshold, int act, void* H,
                                void* Y, void* workspace, size_t ws_bytes, void* stream,
                                int32_t* down_outlier_idx, int32_t* down_n_out) {
  return run_ffn(X, T, d_model, d_ff, CB_up, SCB_up, bias_up, CB_down, SCB_down, bias_down,
                 threshold, act, H, Y, workspace, ws_bytes, stream, down_outlier_idx,
                 down_n_out);
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

I8_API i8_status absmax_quantize_blocks(const void* X, int rows, int cols, int block, int8_t* Q,
                                        float* absmax, void* stream) {
  g_last_launches = 0;
  if (rows < 0 || cols < 0 || block <= 0 || !X || !Q || !absmax) return I8_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || !aligned16(absmax)) return I8_ERR_ALIGNMENT;
  if (rows == 0 || cols == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  st = from_cuda(launch_absmax_blocks(X, rows, cols, block, Q, absmax,
                                      static_cast<cudaStream_t>(stream)));
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

I8_API i8_status f16_ffn(const void* X, int T, int d_model, int d_ff, const void* W_up,
                         const void* bias_up, const void* W_down, const void* bias_down,
                         int act, void* H, void* Y, void* stream) {
  g_last_launches = 0;
  if (act != I8_ACT_NONE && act != I8_ACT_RELU) return I8_ERR_INVALID_ARG;
  if (T < 0 || d_model <= 0 || d_ff <= 0 || !W_up || !W_down) return I8_ERR_INVALID_ARG;
  if (T > 0 && (!X || !H || !Y)) return I8_ERR_INVALID_ARG;
  if (d_model % 16 != 0 || d_ff % 16 != 0) return I8_ERR_ALIGNMENT;
  if (!aligned16(X) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(H) ||
      !aligned16(Y) || (bias_up && !aligned16(bias_up)) || (bias_down && !aligned16(bias_down)))
    return I8_ERR_ALIGNMENT;
  if (T == 0) return I8_OK;
  i8_status st = check_device();
  if (st != I8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmArgs g;
  g.a_f16 = W_up;
  g.b_f16 = X;
  g.bias = bias_up;
  g.Y = H;
  g.T = T;
  g.in = d_model;
  g.out = d_ff;
  g.relu = act == I8_ACT_RELU ? 1 : 0;
  if ((st = from_cuda(launch_f16_gemm(g, s))) != I8_OK) return st;
  GemmArgs g2;
  g2.a_f16 = W_down;
  g2.b_f16 = H;
  g2.bias = bias_down;
  g2.Y = Y;
  g2.T = T;
  g2.in = d_ff;
  g2.out = d_model;
  if ((st = from_cuda(launch_f16_gemm(g2, s))) != I8_OK) return st;
  g_last_launches = 2;
  return I8_OK;
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

I8_API void i8_set_profile_events_n(void** events, int n) {
  g_prof_n = (events && n > 0) ? std::min(n, kProfSlots) : 0;
  for (int i = 0; i < kProfSlots; ++i)
    g_prof[i] = i < g_prof_n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

I8_API void i8_set_profile_events(void** events) { i8_set_profile_events_n(events, 4); }
