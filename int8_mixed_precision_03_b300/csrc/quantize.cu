// Row quantizers: vector-wise absmax (activations and weights), the fused activation
// quantize + outlier gather of the matmul, and zeropoint rows.
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq):
//   section "core idea", step 2: the non-outlier part is quantized to int8 vector-wise
//     (activations per row, weights per output feature) and the outlier part stays fp16;
//   section "zeropoint vs absmax": absmax scaling, divide by absmax and multiply by 127;
//   section "transformers integration": CB in [-127,127], W ~ (CB * SCB) / 127.
// "LLM.int8() summary" (zenn), section "Zeropoint Quantization":
//   X8 = INT8(X16*S - Z), X16 = (X8 + Z)/S, S = 254/(max - min).
//
// Every rounding step uses an explicit IEEE intrinsic (__fdiv_rn, __fmul_rn, __fsub_rn,
// __float2int_rn), so the codes do not depend on contraction flags:
//   s = 127/absmax (0 if absmax is 0), code = clamp(rint(x*s), -127, 127).
// One CTA of 256 threads quantizes one row; rows are read with 16-byte loads when the
// row length is a multiple of 8 elements, element by element otherwise.
#include "int8mm_internal.h"
#include "sm103_ptx.cuh"

namespace i8mm {

constexpr int kRowThreads = 256;

__device__ __forceinline__ int absmax_code(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  return max(-127, min(127, q));
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Block-wide max of non-negative values held as unsigned bit patterns.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* s_red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) r = max(r, s_red[w]);
  __syncthreads();
  return r;
}

// Masked-column test: bit j of the mask words flags column j as an outlier.
__device__ __forceinline__ bool is_masked(const uint32_t* smask, int j) {
  return (smask[j >> 5] >> (j & 31)) & 1u;
}

// Mask bits of the 8 columns of 16-byte chunk c (bit e <-> column 8c + e).
__device__ __forceinline__ uint32_t chunk_mask(const uint32_t* smask, int c) {
  return (smask[c >> 2] >> ((c & 3) * 8)) & 0xffu;
}

// Max |x| bit pattern of the 8 fp16 values of a chunk (masked columns excluded).
template <bool kMasked>
__device__ __forceinline__ uint32_t chunk_absmax(const uint4& v, uint32_t mb) {
  uint32_t w[4] = {v.x & 0x7fff7fffu, v.y & 0x7fff7fffu, v.z & 0x7fff7fffu, v.w & 0x7fff7fffu};
  if (kMasked) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t keep = ((mb >> (2 * k)) & 1u ? 0u : 0x0000ffffu) |
                            ((mb >> (2 * k + 1)) & 1u ? 0u : 0xffff0000u);
      w[k] &= keep;
    }
  }
  uint32_t mx = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0xffffu, w[k] >> 16));
  return mx;
}

// Codes of the 8 values of chunk c with scale s; writes them to q8 / q16 (either may be
// null) and returns sum |code|.
template <bool kMasked>
__device__ __forceinline__ int chunk_codes(const uint4& v, uint32_t mb, float s, int c,
                                           int8_t* __restrict__ q8, uint16_t* __restrict__ q16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  int q[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    q[2 * k] = absmax_code(h2f(w[k] & 0xffffu), s);
    q[2 * k + 1] = absmax_code(h2f(w[k] >> 16), s);
  }
  if (kMasked) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if ((mb >> e) & 1u) q[e] = 0;
  }
  int a1 = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) a1 += abs(q[e]);
  if (q8) {
    uint2 o;
    o.x = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) |
          ((uint32_t)(q[3] & 0xff) << 24);
    o.y = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) |
          ((uint32_t)(q[7] & 0xff) << 24);
    reinterpret_cast<uint2*>(q8)[c] = o;
  }
  if (q16) {
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      ow[k] = (uint32_t)__half_as_ushort(__int2half_rn(q[2 * k])) |
              ((uint32_t)__half_as_ushort(__int2half_rn(q[2 * k + 1])) << 16);
    reinterpret_cast<uint4*>(q16)[c] = o;
  }
  return a1;
}

// Quantizes one row of `cols` fp16 values.
//   kMasked: columns flagged in smask are excluded from the absmax and coded 0.
//   q8 (nullable): int8 codes; q16 (nullable): the same codes as exact fp16 values.
//   s_l1 (nullable, shared, zeroed): += sum of |code| per 1024-column chunk.
// Returns the row absmax (over unmasked columns).
//
// kNV > 0: the row is read from memory once and held in registers, thread t owning 16-byte
// chunks t, t + 256, ..., t + 256 (kNV - 1) (needs cols % 8 == 0, cols <= 2048 kNV).
// kNV == 0: two passes over the row (any length).
template <bool kMasked, int kNV>
__device__ float quantize_row(const uint16_t* __restrict__ x, int cols,
                              const uint32_t* smask, int8_t* __restrict__ q8,
                              uint16_t* __restrict__ q16, uint32_t* s_red,
                              int* s_l1 = nullptr) {
  const int tid = threadIdx.x;
  if constexpr (kNV > 0) {
    const int nch = cols >> 3;
    uint4 v[kNV];
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      v[i] = c < nch ? __ldg(reinterpret_cast<const uint4*>(x) + c) : make_uint4(0, 0, 0, 0);
      mx = max(mx, chunk_absmax<kMasked>(v[i], kMasked && c < nch ? chunk_mask(smask, c) : 0u));
    }
    const float a = h2f((uint16_t)block_max_u32(mx, s_red));
    const float s = a > 0.0f ? __fdiv_rn(127.0f, a) : 0.0f;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      int a1 = 0;
      if (c < nch) a1 = chunk_codes<kMasked>(v[i], kMasked ? chunk_mask(smask, c) : 0u, s, c, q8, q16);
      if (s_l1) {
        // the warp's 32 chunks (256 columns) lie in one 1024-column chunk
        a1 = __reduce_add_sync(0xffffffffu, a1);
        if ((tid & 31) == 0 && a1 > 0) atomicAdd(&s_l1[(c * 8) / kChunkK], a1);
      }
    }
    return a;
  } else {
    const bool vec = (cols & 7) == 0;
    uint32_t mx = 0;  // running max of |x| bit patterns
    if (vec) {
      const int nch = cols >> 3;
      for (int c = tid; c < nch; c += kRowThreads)
        mx = max(mx, chunk_absmax<kMasked>(__ldg(reinterpret_cast<const uint4*>(x) + c),
                                           kMasked ? chunk_mask(smask, c) : 0u));
    } else {
      for (int j = tid; j < cols; j += kRowThreads) {
        if (kMasked && is_masked(smask, j)) continue;
        mx = max(mx, (uint32_t)(x[j] & 0x7fffu));
      }
    }
    const float a = h2f((uint16_t)block_max_u32(mx, s_red));
    const float s = a > 0.0f ? __fdiv_rn(127.0f, a) : 0.0f;
    if (vec) {
      const int nch = cols >> 3;
      for (int c = tid; c < nch; c += kRowThreads) {
        const int a1 = chunk_codes<kMasked>(__ldg(reinterpret_cast<const uint4*>(x) + c),
                                            kMasked ? chunk_mask(smask, c) : 0u, s, c, q8, q16);
        if (s_l1) atomicAdd(&s_l1[(c * 8) / kChunkK], a1);
      }
    } else {
      for (int j = tid; j < cols; j += kRowThreads) {
        int q = absmax_code(h2f(x[j]), s);
        if (kMasked && is_masked(smask, j)) q = 0;
        if (q8) q8[j] = (int8_t)q;
        if (q16) q16[j] = __half_as_ushort(__int2half_rn(q));
      }
    }
    return a;
  }
}

// Register chunks per thread for a row of `cols` values: 1, 2, 4 or 8, or 0 when the row
// is longer than 16384 or not a multiple of 8 (two-pass path; deeper register rows would
// cost more in occupancy than the second read of the row costs).
inline int row_nv(int cols) {
  if (cols % 8 != 0) return 0;
  const int nch = cols / 8;
  for (int nv = 1; nv <= 8; nv *= 2)
    if (nch <= nv * kRowThreads) return nv;
  return 0;
}

// Standalone absmax rows; also the weight quantizer (rows = output features).
template <int kNV>
__global__ void __launch_bounds__(kRowThreads) absmax_rows_kernel(
    const uint16_t* __restrict__ X, int cols, int8_t* __restrict__ Q, float* __restrict__ amax) {
  __shared__ uint32_t s_red[kRowThreads / 32];
  const size_t row = blockIdx.x;
  const float a = quantize_row<false, kNV>(X + row * cols, cols, nullptr, Q + row * cols,
                                           nullptr, s_red);
  if (threadIdx.x == 0) amax[row] = a;
}

// Row i's outlier values into the transposed slice of the matmul's CUDA-core outlier
// product: xoT[k * xo_stride(T) + i] = X[i, idx[k]] for k < n, 0 for n <= k < kCcOutlierCols.
__device__ __forceinline__ void gather_transposed(const uint16_t* __restrict__ x,
                                                  const int32_t* __restrict__ idx, int n,
                                                  uint16_t* __restrict__ xoT, int T, size_t i) {
  if (!xoT) return;
  const size_t stride = xo_stride(T);
  for (int k = threadIdx.x; k < kCcOutlierCols; k += kRowThreads)
    xoT[(size_t)k * stride + i] = k < n ? x[__ldg(&idx[k])] : (uint16_t)0;
}

// Blocks [T, ..) of the quantize passes: 32 output features per block, 8 threads per
// feature o: W_out[o, k] = fp16((CB[o,idx[k]]*SCB[o])/127) for k < n, zeros up to npad.
// Returns, in the feature's first thread, sum_k CB[o, idx[k]] (the other threads: partial).
__device__ int gather_outlier_weights(const int8_t* __restrict__ CB,
                                      const float* __restrict__ SCB, int in, int out,
                                      const int32_t* __restrict__ idx, int n, int npad,
                                      int ncap, int T, uint16_t* __restrict__ wout) {
  const int o = (blockIdx.x - T) * 32 + (threadIdx.x >> 3);
  int csum = 0;
  if (o < out) {
    const float scb = __ldg(&SCB[o]);
    for (int k = threadIdx.x & 7; k < npad; k += 8) {
      uint16_t v = 0;
      if (k < n) {
        const int cb = __ldg(&CB[(size_t)o * in + __ldg(&idx[k])]);
        csum += cb;
        v = __half_as_ushort(__float2half_rn(__fdiv_rn(__fmul_rn((float)cb, scb), 127.0f)));
      }
      wout[(size_t)o * ncap + k] = v;
    }
  }
  // the 8 threads of a feature are 8 consecutive lanes
  csum += __shfl_xor_sync(0xffffffffu, csum, 1);
  csum += __shfl_xor_sync(0xffffffffu, csum, 2);
  csum += __shfl_xor_sync(0xffffffffu, csum, 4);
  return csum;
}

// Fused activation quantize + outlier gather of the matmul.
//   blocks [0, T): row i -> fp16 codes (outlier columns 0), rowabs[i], and
//                  X_out[i, k] = X[i, idx[k]] for k < n, zeros up to a multiple of 64;
//   blocks [T, ..): 32 output features each -> W_out[o, k] = fp16((CB[o,idx[k]]*SCB[o])/127).
template <int kNV>
__global__ void __launch_bounds__(kRowThreads) quantize_gather_kernel(
    const uint16_t* __restrict__ X, int T, int in, const int8_t* __restrict__ CB,
    const float* __restrict__ SCB, int out, const WsHeader* __restrict__ hdr,
    const uint32_t* __restrict__ mask, const int32_t* __restrict__ idx, int ncap,
    uint16_t* __restrict__ xq16, float* __restrict__ rowabs, uint16_t* __restrict__ xout,
    uint16_t* __restrict__ wout, uint16_t* __restrict__ xoT, int32_t* __restrict__ l1, int bn,
    int8_t* __restrict__ xq8) {
  extern __shared__ uint32_t s_mask[];  // (in + 31) / 32 words
  __shared__ uint32_t s_red[kRowThreads / 32];
  __shared__ int s_l1[I8_MAX_IN / kChunkK];
  const int n = hdr->n_out_used;
  const int npad = (n + 63) / 64 * 64;
  if (blockIdx.x < (unsigned)T) {
    const int words = (in + 31) / 32;
    const int nch = (in + kChunkK - 1) / kChunkK;
    for (int w = threadIdx.x; w < words; w += kRowThreads) s_mask[w] = __ldg(&mask[w]);
    for (int c = threadIdx.x; c < nch; c += kRowThreads) s_l1[c] = 0;
    __syncthreads();
    const size_t i = blockIdx.x;
    const uint16_t* x = X + i * in;
    const float a = quantize_row<true, kNV>(x, in, s_mask, xq8 ? xq8 + i * in : nullptr,
                                            xq16 ? xq16 + i * in : nullptr, s_red, s_l1);
    if (threadIdx.x == 0) rowabs[i] = a;
    __syncthreads();
    // bound of the matmul's fp32 chunk sums: max over the token tile of sum |code|
    for (int c = threadIdx.x; c < nch; c += kRowThreads)
      if (s_l1[c] > 0) atomicMax(&l1[(size_t)(i / bn) * nch + c], s_l1[c]);
    for (int k = threadIdx.x; k < npad; k += kRowThreads)
      xout[i * ncap + k] = k < n ? x[__ldg(&idx[k])] : (uint16_t)0;
    gather_transposed(x, idx, n, xoT, T, i);
  } else {
    if (npad == 0) return;
    gather_outlier_weights(CB, SCB, in, out, idx, n, npad, ncap, T, wout);
  }
}

__device__ __forceinline__ int zp_code(float x, float sc, float z) {
  return max(-127, min(127, __float2int_rn(__fsub_rn(__fmul_rn(x, sc), z))));
}

// Zeropoint rows: S = 254/(max-min), Z = rint(S*min) + 127, code = clamp(rint(x*S - Z)).
// kNV > 0: the row is read once and held in registers (as in quantize_row); kNV == 0:
// element by element, two passes.
template <int kNV>
__global__ void __launch_bounds__(kRowThreads) zeropoint_rows_kernel(
    const uint16_t* __restrict__ X, int cols, int8_t* __restrict__ Q, float* __restrict__ S,
    float* __restrict__ Z) {
  __shared__ float s_mn[kRowThreads / 32], s_mx[kRowThreads / 32];
  const size_t row = blockIdx.x;
  const uint16_t* x = X + row * cols;
  int8_t* q = Q + row * cols;
  const int tid = threadIdx.x;
  float mn = INFINITY, mx = -INFINITY;
  [[maybe_unused]] uint4 v[kNV > 0 ? kNV : 1];
  if constexpr (kNV > 0) {
    const int nch = cols >> 3;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      if (c < nch) {
        v[i] = __ldg(reinterpret_cast<const uint4*>(x) + c);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = h2f(w[k] & 0xffffu), hi = h2f(w[k] >> 16);
          mn = fminf(mn, fminf(lo, hi));
          mx = fmaxf(mx, fmaxf(lo, hi));
        }
      }
    }
  } else {
    for (int j = tid; j < cols; j += kRowThreads) {
      const float xv = h2f(x[j]);
      mn = fminf(mn, xv);
      mx = fmaxf(mx, xv);
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) { s_mn[warp] = mn; s_mx[warp] = mx; }
  __syncthreads();
  mn = s_mn[0];
  mx = s_mx[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) { mn = fminf(mn, s_mn[w]); mx = fmaxf(mx, s_mx[w]); }
  if (cols == 0) { mn = 0.0f; mx = 0.0f; }
  const bool spread = mx > mn;
  const float sc = spread ? __fdiv_rn(254.0f, __fsub_rn(mx, mn)) : 0.0f;
  const float z = spread ? __fadd_rn(rintf(__fmul_rn(sc, mn)), 127.0f) : mn;
  if (tid == 0) { S[row] = sc; Z[row] = z; }
  if constexpr (kNV > 0) {
    const int nch = cols >> 3;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      if (c < nch) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        int cq[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          cq[2 * k] = spread ? zp_code(h2f(w[k] & 0xffffu), sc, z) : 0;
          cq[2 * k + 1] = spread ? zp_code(h2f(w[k] >> 16), sc, z) : 0;
        }
        uint2 o;
        o.x = (cq[0] & 0xff) | ((cq[1] & 0xff) << 8) | ((cq[2] & 0xff) << 16) |
              ((uint32_t)(cq[3] & 0xff) << 24);
        o.y = (cq[4] & 0xff) | ((cq[5] & 0xff) << 8) | ((cq[6] & 0xff) << 16) |
              ((uint32_t)(cq[7] & 0xff) << 24);
        reinterpret_cast<uint2*>(q)[c] = o;
      }
    }
  } else {
    for (int j = tid; j < cols; j += kRowThreads)
      q[j] = spread ? (int8_t)zp_code(h2f(x[j]), sc, z) : (int8_t)0;
  }
}

// ---------------------------------------------------------------- zeropoint variant
// Zeropoint codes of the 8 values of chunk c (masked columns 0; all 0 when the row has no
// spread); writes q8 / q16 (either may be null) and returns sum |code|.
__device__ __forceinline__ int chunk_zp_codes(const uint4& v, uint32_t mb, bool spread,
                                              float sc, float z, int c,
                                              int8_t* __restrict__ q8,
                                              uint16_t* __restrict__ q16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  int q[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    q[2 * k] = zp_code(h2f(w[k] & 0xffffu), sc, z);
    q[2 * k + 1] = zp_code(h2f(w[k] >> 16), sc, z);
  }
  int a1 = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (!spread || ((mb >> e) & 1u)) q[e] = 0;
    a1 += abs(q[e]);
  }
  if (q8) {
    uint2 o;
    o.x = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) |
          ((uint32_t)(q[3] & 0xff) << 24);
    o.y = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) |
          ((uint32_t)(q[7] & 0xff) << 24);
    reinterpret_cast<uint2*>(q8)[c] = o;
  }
  if (q16) {
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      ow[k] = (uint32_t)__half_as_ushort(__int2half_rn(q[2 * k])) |
              ((uint32_t)__half_as_ushort(__int2half_rn(q[2 * k + 1])) << 16);
    reinterpret_cast<uint4*>(q16)[c] = o;
  }
  return a1;
}

// Min and max of the unmasked values of a chunk, folded into mn / mx.
__device__ __forceinline__ void chunk_minmax(const uint4& v, uint32_t mb, float& mn,
                                             float& mx) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if ((mb >> e) & 1u) continue;
    const float x = h2f(e & 1 ? w[e >> 1] >> 16 : w[e >> 1] & 0xffffu);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
}

// Block-wide min and max (kRowThreads threads).
__device__ __forceinline__ void block_minmax(float& mn, float& mx, float* s_mn, float* s_mx) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { s_mn[warp] = mn; s_mx[warp] = mx; }
  __syncthreads();
  mn = s_mn[0];
  mx = s_mx[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) { mn = fminf(mn, s_mn[w]); mx = fmaxf(mx, s_mx[w]); }
  __syncthreads();
}

// Zeropoint quantization of one row over its unmasked columns, the analogue of
// quantize_row (same kNV register staging, same per-chunk code statistics in s_l1):
// S = 254/(max - min), Z = rint(S*min) + 127, code = clamp(rint(x*S - Z)); no unmasked
// column gives min = max = 0; no spread gives S = 0, Z = min and codes 0.
template <int kNV>
__device__ void quantize_row_zp(const uint16_t* __restrict__ x, int cols, const uint32_t* smask,
                                int8_t* __restrict__ q8, uint16_t* __restrict__ q16,
                                float* s_mn, float* s_mx, int* s_l1, float& S, float& Z) {
  const int tid = threadIdx.x;
  const bool vec = (cols & 7) == 0;
  const int nch = cols >> 3;
  float mn = INFINITY, mx = -INFINITY;
  [[maybe_unused]] uint4 v[kNV > 0 ? kNV : 1];
  if constexpr (kNV > 0) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      v[i] = c < nch ? __ldg(reinterpret_cast<const uint4*>(x) + c) : make_uint4(0, 0, 0, 0);
      if (c < nch) chunk_minmax(v[i], chunk_mask(smask, c), mn, mx);
    }
  } else if (vec) {
    for (int c = tid; c < nch; c += kRowThreads)
      chunk_minmax(__ldg(reinterpret_cast<const uint4*>(x) + c), chunk_mask(smask, c), mn, mx);
  } else {
    for (int j = tid; j < cols; j += kRowThreads) {
      if (is_masked(smask, j)) continue;
      const float xv = h2f(x[j]);
      mn = fminf(mn, xv);
      mx = fmaxf(mx, xv);
    }
  }
  block_minmax(mn, mx, s_mn, s_mx);
  if (!(mn <= mx)) { mn = 0.0f; mx = 0.0f; }  // no unmasked column
  const bool spread = mx > mn;
  const float sc = spread ? __fdiv_rn(254.0f, __fsub_rn(mx, mn)) : 0.0f;
  const float z = spread ? __fadd_rn(rintf(__fmul_rn(sc, mn)), 127.0f) : mn;
  S = sc;
  Z = z;
  if constexpr (kNV > 0) {
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c = tid + i * kRowThreads;
      int a1 = c < nch ? chunk_zp_codes(v[i], chunk_mask(smask, c), spread, sc, z, c, q8, q16)
                       : 0;
      // the warp's 32 chunks (256 columns) lie in one 1024-column chunk
      a1 = __reduce_add_sync(0xffffffffu, a1);
      if ((tid & 31) == 0 && a1 > 0) atomicAdd(&s_l1[(c * 8) / kChunkK], a1);
    }
  } else if (vec) {
    for (int c = tid; c < nch; c += kRowThreads) {
      const int a1 = chunk_zp_codes(__ldg(reinterpret_cast<const uint4*>(x) + c),
                                    chunk_mask(smask, c), spread, sc, z, c, q8, q16);
      if (a1 > 0) atomicAdd(&s_l1[(c * 8) / kChunkK], a1);
    }
  } else {
    for (int j = tid; j < cols; j += kRowThreads) {
      int q = spread ? zp_code(h2f(x[j]), sc, z) : 0;
      if (is_masked(smask, j)) q = 0;
      if (q8) q8[j] = (int8_t)q;
      if (q16) q16[j] = __half_as_ushort(__int2half_rn(q));
      if (q) atomicAdd(&s_l1[j / kChunkK], abs(q));
    }
  }
}

// The zeropoint variant of quantize_gather_kernel (see launch_quantize_gather_zp).
template <int kNV>
__global__ void __launch_bounds__(kRowThreads) quantize_gather_zp_kernel(
    const uint16_t* __restrict__ X, int T, int in, const int8_t* __restrict__ CB,
    const float* __restrict__ SCB, int out, const WsHeader* __restrict__ hdr,
    const uint32_t* __restrict__ mask, const int32_t* __restrict__ idx, int ncap,
    uint16_t* __restrict__ xq16, float* __restrict__ rowabs, int32_t* __restrict__ zi,
    uint16_t* __restrict__ xout, uint16_t* __restrict__ wout, uint16_t* __restrict__ xoT,
    int32_t* __restrict__ cbout, int32_t* __restrict__ l1, int bn, int8_t* __restrict__ xq8,
    float* __restrict__ dbg_S, float* __restrict__ dbg_Z) {
  extern __shared__ uint32_t s_mask[];  // (in + 31) / 32 words
  __shared__ float s_mn[kRowThreads / 32], s_mx[kRowThreads / 32];
  __shared__ int s_l1[I8_MAX_IN / kChunkK];
  const int n = hdr->n_out_used;
  const int npad = (n + 63) / 64 * 64;
  if (blockIdx.x < (unsigned)T) {
    const int words = (in + 31) / 32;
    const int nch = (in + kChunkK - 1) / kChunkK;
    for (int w = threadIdx.x; w < words; w += kRowThreads) s_mask[w] = __ldg(&mask[w]);
    for (int c = threadIdx.x; c < nch; c += kRowThreads) s_l1[c] = 0;
    __syncthreads();
    const size_t i = blockIdx.x;
    const uint16_t* x = X + i * in;
    float S, Z;
    quantize_row_zp<kNV>(x, in, s_mask, xq8 ? xq8 + i * in : nullptr,
                         xq16 ? xq16 + i * in : nullptr, s_mn, s_mx, s_l1, S, Z);
    if (threadIdx.x == 0) {
      // epilogue factors: y = (acc + zi * sum of inlier codes) * rowabs * SCB / 127^2
      const bool spread = S > 0.0f;
      rowabs[i] = spread ? __fdiv_rn(127.0f, S) : __fmul_rn(127.0f, Z);
      zi[i] = spread ? (int32_t)Z : 1;
      if (dbg_S) dbg_S[i] = S;
      if (dbg_Z) dbg_Z[i] = Z;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < nch; c += kRowThreads)
      if (s_l1[c] > 0) atomicMax(&l1[(size_t)(i / bn) * nch + c], s_l1[c]);
    for (int k = threadIdx.x; k < npad; k += kRowThreads)
      xout[i * ncap + k] = k < n ? x[__ldg(&idx[k])] : (uint16_t)0;
    gather_transposed(x, idx, n, xoT, T, i);
  } else {
    const int csum = gather_outlier_weights(CB, SCB, in, out, idx, n, npad, ncap, T, wout);
    const int o = (blockIdx.x - T) * 32 + (threadIdx.x >> 3);
    if ((threadIdx.x & 7) == 0 && o < out) cbout[o] = csum;
  }
}

// Row sums of int8 codes: one warp per row, 16-byte loads where the row allows.
__global__ void __launch_bounds__(256) code_sums_kernel(const int8_t* __restrict__ CB, int out,
                                                        int in, int32_t* __restrict__ sums) {
  const int o = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (o >= out) return;
  const int8_t* row = CB + (size_t)o * in;
  int acc = 0;
  if (in % 16 == 0) {
    for (int c = lane; c < in / 16; c += 32) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + c);
      acc = __dp4a((int)v.x, 0x01010101, acc);
      acc = __dp4a((int)v.y, 0x01010101, acc);
      acc = __dp4a((int)v.z, 0x01010101, acc);
      acc = __dp4a((int)v.w, 0x01010101, acc);
    }
  } else {
    for (int j = lane; j < in; j += 32) acc += row[j];
  }
  acc = __reduce_add_sync(0xffffffffu, acc);
  if (lane == 0) sums[o] = acc;
}

// Instantiates F<kNV> for the register depth that fits `cols` (0: two-pass path).
#define I8_DISPATCH_NV(cols, F)                      \
  switch (row_nv(cols)) {                            \
    case 1: F(1); break;                             \
    case 2: F(2); break;                             \
    case 4: F(4); break;                             \
    case 8: F(8); break;                             \
    default: F(0); break;                            \
  }

cudaError_t launch_absmax_rows(const void* X, int rows, int cols, int8_t* Q, float* absmax,
                               cudaStream_t s) {
#define I8_LAUNCH(NV)                                                                    \
  absmax_rows_kernel<NV><<<rows, kRowThreads, 0, s>>>(static_cast<const uint16_t*>(X), cols, \
                                                       Q, absmax)
  I8_DISPATCH_NV(cols, I8_LAUNCH)
#undef I8_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_zeropoint_rows(const void* X, int rows, int cols, int8_t* Q, float* S,
                                  float* Z, cudaStream_t s) {
#define I8_LAUNCH(NV)                                                                    \
  zeropoint_rows_kernel<NV><<<rows, kRowThreads, 0, s>>>(static_cast<const uint16_t*>(X), \
                                                          cols, Q, S, Z)
  I8_DISPATCH_NV(cols, I8_LAUNCH)
#undef I8_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_quantize_gather(const void* X, int T, int in, const int8_t* CB,
                                   const float* SCB, int out, const WsHeader* hdr,
                                   const uint32_t* mask, const int32_t* idx, int ncap,
                                   void* xq16, float* rowabs, void* xout, void* wout,
                                   void* xoT, int32_t* l1, int8_t* xq8_debug, cudaStream_t s) {
  // without a W_out buffer (the decode path reads the outlier weights from CB itself) only
  // the T row blocks run
  const int wblocks = wout ? (out + 31) / 32 : 0;
  const size_t smem = sizeof(uint32_t) * (size_t)((in + 31) / 32);
#define I8_LAUNCH(NV)                                                                       \
  quantize_gather_kernel<NV><<<T + wblocks, kRowThreads, smem, s>>>(                         \
      static_cast<const uint16_t*>(X), T, in, CB, SCB, out, hdr, mask, idx, ncap,           \
      static_cast<uint16_t*>(xq16), rowabs, static_cast<uint16_t*>(xout),                   \
      static_cast<uint16_t*>(wout), static_cast<uint16_t*>(xoT), l1, i8_bn(T), xq8_debug)
  I8_DISPATCH_NV(in, I8_LAUNCH)
#undef I8_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_quantize_gather_zp(const void* X, int T, int in, const int8_t* CB,
                                      const float* SCB, int out, const WsHeader* hdr,
                                      const uint32_t* mask, const int32_t* idx, int ncap,
                                      void* xq16, float* rowabs, int32_t* zi, void* xout,
                                      void* wout, void* xoT, int32_t* cbout, int32_t* l1,
                                      int8_t* xq8_debug, float* dbg_S, float* dbg_Z,
                                      cudaStream_t s) {
  const int wblocks = (out + 31) / 32;
  const size_t smem = sizeof(uint32_t) * (size_t)((in + 31) / 32);
#define I8_LAUNCH(NV)                                                                       \
  quantize_gather_zp_kernel<NV><<<T + wblocks, kRowThreads, smem, s>>>(                      \
      static_cast<const uint16_t*>(X), T, in, CB, SCB, out, hdr, mask, idx, ncap,           \
      static_cast<uint16_t*>(xq16), rowabs, zi, static_cast<uint16_t*>(xout),               \
      static_cast<uint16_t*>(wout), static_cast<uint16_t*>(xoT), cbout, l1, i8_bn(T),        \
      xq8_debug, dbg_S, dbg_Z)
  I8_DISPATCH_NV(in, I8_LAUNCH)
#undef I8_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_code_sums(const int8_t* CB, int out, int in, int32_t* CBsum,
                             cudaStream_t s) {
  code_sums_kernel<<<(out + 7) / 8, 256, 0, s>>>(CB, out, in, CBsum);
  return cudaGetLastError();
}

}  // namespace i8mm
