// Block-wise absmax quantization.
//
// "[論文レビュー] The case for 4-bit precision: k-bit Inference Scaling Laws" (nubint review),
// sections "提案手法" and "主な発見": the block size is a parameter of the quantizer, and small
// blocks (64-128 values), each normalized by its own absmax, quantize better than large
// ones. Here each row of X [rows, cols] is cut into blocks of `block` consecutive columns
// (the last block of a row shorter when block does not divide cols); block k of row i gets
// absmax[i, k] = max |x| over the block and the codes clamp(rint(x * (127/absmax))), with the
// rounding of the row-wise quantizer (s = 127/absmax in IEEE fp32, one fp32 multiply, round
// half to even; absmax 0 gives codes 0).
//
// Vector path (cols % 8 == 0 and block = 8 * g with g a power of two, 2 <= g <= 32): a
// thread owns one 16-byte chunk (8 values) of a block of g chunks held by g consecutive
// lanes; the block's absmax is a max over those lanes by shuffles, so no shared memory and
// no block-wide barrier. A warp walks a row kSlots x 32 chunks at a time, issuing all their
// loads before using any (HBM latency is paid once per kSlots chunks), then writes 8 codes
// (8 bytes) per chunk and, from the group's first lane, the block's absmax.
// Other shapes: one thread per block, element by element.
#include <cuda_fp16.h>

#include <algorithm>

#include "int8mm_internal.h"

namespace i8mm {
namespace {

constexpr int kBlkThreads = 256;
constexpr int kSlots = 8;  // 16-byte chunks in flight per thread

__device__ __forceinline__ float bh2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ int blk_code(float x, float s) {
  const int q = __float2int_rn(__fmul_rn(x, s));
  return max(-127, min(127, q));
}

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// G = lanes per block (block = 8 G values). The work units are segments of 32 x kSlots
// chunks of a row (a whole number of blocks); warp w of the grid takes units w, w + W, ...
// In a segment, lane l takes chunks l, l + 32, ..., all loaded before any is used, so the G
// lanes of a group always hold one block (G divides 32 and a pass starts at a multiple of
// 32). Chunks past the row end load nothing.
template <int G>
__global__ void __launch_bounds__(kBlkThreads) blocks_vec_kernel(
    const uint16_t* __restrict__ X, int rows, int cols, int nblocks, int8_t* __restrict__ Q,
    float* __restrict__ absmax) {
  constexpr int kSeg = 32 * kSlots;  // chunks per unit
  const int cpr = cols >> 3;          // chunks per row
  const int spr = (cpr + kSeg - 1) / kSeg;
  const long long units = (long long)rows * spr;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (kBlkThreads / 32);
  for (long long un = (long long)blockIdx.x * (kBlkThreads / 32) + (threadIdx.x >> 5);
       un < units; un += nwarps) {
    const int row = (int)(un / spr), cb = (int)(un - (long long)row * spr) * kSeg;
    const uint4* x4 = reinterpret_cast<const uint4*>(X + (size_t)row * cols);
    uint2* q2 = reinterpret_cast<uint2*>(Q + (size_t)row * cols);
    float* am = absmax + (size_t)row * nblocks;
    {
      uint4 v[kSlots];
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {  // all loads first
        const int c = cb + 32 * u + lane;
        v[u] = c < cpr ? ld_stream16(x4 + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        if (cb + 32 * u >= cpr) break;  // uniform: no chunk of this pass is in the row
        const int c = cb + 32 * u + lane;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
#pragma unroll
        for (int d = 1; d < G; d <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
        const float a = bh2f((uint16_t)m);
        const float s = a > 0.0f ? __fdiv_rn(127.0f, a) : 0.0f;
        if (c < cpr) {
          int q[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            q[2 * k] = blk_code(bh2f((uint16_t)(w[k] & 0xffffu)), s);
            q[2 * k + 1] = blk_code(bh2f((uint16_t)(w[k] >> 16)), s);
          }
          uint2 o;
          o.x = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) |
                ((uint32_t)(q[3] & 0xff) << 24);
          o.y = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) |
                ((uint32_t)(q[7] & 0xff) << 24);
          q2[c] = o;
          if (c % G == 0) am[c / G] = a;
        }
      }
    }
  }
}

// Any shape: one thread per block of one row.
__global__ void __launch_bounds__(kBlkThreads) blocks_scalar_kernel(
    const uint16_t* __restrict__ X, int rows, int cols, int block, int nblocks,
    int8_t* __restrict__ Q, float* __restrict__ absmax) {
  const long long nb = (long long)rows * nblocks;
  for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nb;
       b += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(b / nblocks), k = (int)(b % nblocks);
    const int j0 = k * block, j1 = min(cols, j0 + block);
    const uint16_t* x = X + (size_t)i * cols;
    uint32_t m = 0;
    for (int j = j0; j < j1; ++j) m = max(m, (uint32_t)(x[j] & 0x7fffu));
    const float a = bh2f((uint16_t)m);
    const float s = a > 0.0f ? __fdiv_rn(127.0f, a) : 0.0f;
    for (int j = j0; j < j1; ++j) Q[(size_t)i * cols + j] = (int8_t)blk_code(bh2f(x[j]), s);
    absmax[b] = a;
  }
}

template <int G>
cudaError_t launch_vec(const uint16_t* X, int rows, int cols, int8_t* Q, float* absmax,
                       cudaStream_t s) {
  const int nblocks = (cols + 8 * G - 1) / (8 * G);
  // a warp per unit while units last, at most 8 CTAs of 8 warps per SM
  const long long units = (long long)rows * ((cols / 8 + 32 * kSlots - 1) / (32 * kSlots));
  const long long want = (units + kBlkThreads / 32 - 1) / (kBlkThreads / 32);
  const int grid = (int)std::max(1LL, std::min(want, (long long)sm_count() * 8));
  blocks_vec_kernel<G><<<grid, kBlkThreads, 0, s>>>(X, rows, cols, nblocks, Q, absmax);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absmax_blocks(const void* X, int rows, int cols, int block, int8_t* Q,
                                 float* absmax, cudaStream_t s) {
  const uint16_t* x = static_cast<const uint16_t*>(X);
  if (cols % 8 == 0) {
    switch (block) {
      case 16: return launch_vec<2>(x, rows, cols, Q, absmax, s);
      case 32: return launch_vec<4>(x, rows, cols, Q, absmax, s);
      case 64: return launch_vec<8>(x, rows, cols, Q, absmax, s);
      case 128: return launch_vec<16>(x, rows, cols, Q, absmax, s);
      case 256: return launch_vec<32>(x, rows, cols, Q, absmax, s);
      default: break;
    }
  }
  const int nblocks = (cols + block - 1) / block;
  const long long nb = (long long)rows * nblocks;
  const int grid = (int)std::max(1LL, std::min((nb + kBlkThreads - 1) / kBlkThreads,
                                               (long long)sm_count() * 8));
  blocks_scalar_kernel<<<grid, kBlkThreads, 0, s>>>(x, rows, cols, block, nblocks, Q, absmax);
  return cudaGetLastError();
}

}  // namespace i8mm
