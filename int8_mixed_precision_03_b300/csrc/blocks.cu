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
// no block-wide barrier. Rows are padded to whole blocks of chunk slots (a slot past the row
// end loads nothing), so groups never straddle rows or warps. Each thread takes kSlots slots
// spaced one grid apart and issues all their loads before using any (HBM latency is paid
// once per kSlots chunks), then writes 8 codes (8 bytes) per chunk and, from the group's
// first lane, the block's absmax. The grid covers the slots in one pass when it can.
// Other shapes: one thread per block, element by element.
#include <cuda_fp16.h>

#include <algorithm>

#include "int8mm_internal.h"

namespace i8mm {
namespace {

constexpr int kBlkThreads = 256;
constexpr int kSlots = 4;  // 16-byte chunks in flight per thread

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

// G = lanes per block (block = 8 G values).
template <int G>
__global__ void __launch_bounds__(kBlkThreads) blocks_vec_kernel(
    const uint16_t* __restrict__ X, int rows, int cols, long long nslots, int slots_per_row,
    int nblocks, int8_t* __restrict__ Q, float* __restrict__ absmax) {
  const int cpr = cols >> 3;  // chunks per row
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x + threadIdx.x; base < nslots;
       base += stride * kSlots) {
    uint4 v[kSlots];
    int row[kSlots], c[kSlots];
#pragma unroll
    for (int u = 0; u < kSlots; ++u) {  // all loads first
      const long long slot = base + stride * u;
      row[u] = (int)(slot / slots_per_row);
      c[u] = (int)(slot - (long long)row[u] * slots_per_row);
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (slot < nslots && row[u] < rows && c[u] < cpr)
        v[u] = ld_stream16(X + (size_t)row[u] * cols + (size_t)c[u] * 8);
    }
#pragma unroll
    for (int u = 0; u < kSlots; ++u) {
      const long long slot = base + stride * u;
      // slot < nslots is the same for the whole warp (nslots is a multiple of 32 slots)
      if (slot >= nslots) break;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
#pragma unroll
      for (int d = 1; d < G; d <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
      const float a = bh2f((uint16_t)m);
      const float s = a > 0.0f ? __fdiv_rn(127.0f, a) : 0.0f;
      if (row[u] < rows && c[u] < cpr) {
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
        *reinterpret_cast<uint2*>(Q + (size_t)row[u] * cols + (size_t)c[u] * 8) = o;
        if (c[u] % G == 0) absmax[(size_t)row[u] * nblocks + c[u] / G] = a;
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
  const int cpr = cols / 8;
  const int slots_per_row = (cpr + G - 1) / G * G;
  long long nslots = (long long)rows * slots_per_row;
  nslots = (nslots + 31) / 32 * 32;  // whole warps (the padding slots load and store nothing)
  const int nblocks = (cols + 8 * G - 1) / (8 * G);
  // enough threads for every slot in one pass of kSlots, at most 8 CTAs per SM
  const long long want = (nslots + (long long)kBlkThreads * kSlots - 1) / (kBlkThreads * kSlots);
  const int grid = (int)std::max(1LL, std::min(want, (long long)sm_count() * 8));
  blocks_vec_kernel<G><<<grid, kBlkThreads, 0, s>>>(X, rows, cols, nslots, slots_per_row,
                                                    nblocks, Q, absmax);
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
