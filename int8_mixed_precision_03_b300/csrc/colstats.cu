// Outlier column statistics (step 1 of the method).
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
// idea", step 1: outliers are found per column of the hidden-state matrix by a magnitude
// threshold (about 6). "LLM.int8() summary" (zenn), section "method": the decomposition
// splits the matmul by input dimension.
//
// Column j is an outlier iff some row i has |X[i,j]| >= threshold. For fp16 inputs this is
// the same as comparing the magnitude bit pattern with the smallest fp16 pattern >= the
// threshold, so the pass keeps a running unsigned max of |x| bits per column (two columns
// per 32-bit lane word, __vmaxu2) and compares once at the end.
//
// Layout: X fp16 [T, in] row-major. Grid (ceil(in/256), row splits); each CTA covers 256
// columns (one 16-byte load per lane per row) and a contiguous range of rows. A CTA ORs
// its flags into the 32-column mask words with one atomicOr per non-zero word; the last
// CTA to arrive turns the mask into the ascending index list (block scan of per-word
// popcounts), so the order never depends on scheduling.
//
// When the matmul that produced X already ORed its columns' flags into the mask (its
// epilogue sees every output value once), mask_index_kernel does only the compaction.
#include "int8mm_internal.h"
#include "sm103_ptx.cuh"

namespace i8mm {

constexpr int kColsPerCta = 256;
constexpr int kColThreads = 256;

__device__ __forceinline__ uint4 ld_nc_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void fold_absmax(uint32_t (&m)[4], const uint4& v) {
  m[0] = __vmaxu2(m[0], v.x & 0x7fff7fffu);
  m[1] = __vmaxu2(m[1], v.y & 0x7fff7fffu);
  m[2] = __vmaxu2(m[2], v.z & 0x7fff7fffu);
  m[3] = __vmaxu2(m[3], v.w & 0x7fff7fffu);
}

// Block-wide compaction (kColThreads threads): the set bits of mask[0, words) become the
// ascending column list idx[0, n); hdr gets n, min(n, ncap) and, past the capacity,
// I8_ERR_OUTLIER_CAP. Each thread takes a contiguous run of words; a block scan of their
// popcounts gives every run its output position, so the order never depends on timing.
__device__ void compact_mask(const uint32_t* mask, int words, int32_t* idx, WsHeader* hdr,
                             int ncap, int* s_warp_sum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (words + kColThreads - 1) / kColThreads;
  const int w0 = min(words, threadIdx.x * per), w1 = min(words, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(__ldcg(&mask[w]));
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kColThreads / 32; ++w) {
    before += (w < warp) ? s_warp_sum[w] : 0;
    total += s_warp_sum[w];
  }
  int pos = before + incl - cnt;
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = __ldcg(&mask[w]);
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      idx[pos++] = w * 32 + b;
    }
  }
  if (threadIdx.x == 0) {
    hdr->n_out = total;
    hdr->n_out_used = min(total, ncap);
    if (total > ncap) atomicCAS(&hdr->status, 0, (int)I8_ERR_OUTLIER_CAP);
  }
}

__global__ void __launch_bounds__(kColThreads) colstats_kernel(
    const uint16_t* __restrict__ X, int T, int in, int rows_per_split, uint32_t thr_bits,
    WsHeader* hdr, uint32_t* mask, int32_t* idx, int words, int ncap) {
  __shared__ uint32_t s_flags[kColThreads / 32][32];
  __shared__ int s_warp_sum[kColThreads / 32];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int col0 = blockIdx.x * kColsPerCta + lane * 8;
  const int r0 = blockIdx.y * rows_per_split;
  const int r1 = min(T, r0 + rows_per_split);

  uint32_t m[4] = {0u, 0u, 0u, 0u};
  if (col0 < in) {  // in % 16 == 0, so the whole 8-column group is in range
    const uint16_t* base = X + col0;
    int r = r0 + warp;
    for (; r + 24 < r1; r += 32) {  // four independent 16-byte loads in flight per lane
      const uint4 v0 = ld_nc_stream(base + (size_t)r * in);
      const uint4 v1 = ld_nc_stream(base + (size_t)(r + 8) * in);
      const uint4 v2 = ld_nc_stream(base + (size_t)(r + 16) * in);
      const uint4 v3 = ld_nc_stream(base + (size_t)(r + 24) * in);
      fold_absmax(m, v0);
      fold_absmax(m, v1);
      fold_absmax(m, v2);
      fold_absmax(m, v3);
    }
    for (; r < r1; r += 8) fold_absmax(m, ld_nc_stream(base + (size_t)r * in));
  }
  // one flag bit per column: bit c of the lane byte <-> column col0 + c
  uint32_t byte = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    byte |= ((m[q] & 0xffffu) >= thr_bits ? 1u : 0u) << (2 * q);
    byte |= ((m[q] >> 16) >= thr_bits ? 1u : 0u) << (2 * q + 1);
  }
  s_flags[warp][lane] = byte;
  __syncthreads();
  if (warp == 0) {
    uint32_t b = 0;
#pragma unroll
    for (int w = 0; w < kColThreads / 32; ++w) b |= s_flags[w][lane];
    // 32-column word k of this CTA = bytes of lanes 4k..4k+3
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 1);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 2);
    const uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 3);
    if ((lane & 3) == 0) {
      const uint32_t word = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
      const int gw = blockIdx.x * (kColsPerCta / 32) + (lane >> 2);
      if (word != 0u && gw < words) atomicOr(&mask[gw], word);
    }
  }

  // The last CTA to arrive compacts the mask into the ordered index list.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    s_last = (atomicAdd(&hdr->arrive, 1u) == total - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  compact_mask(mask, words, idx, hdr, ncap, s_warp_sum);
}

// One CTA of kColThreads: mask words -> ascending column list, count, capacity check.
__global__ void __launch_bounds__(kColThreads) mask_index_kernel(
    WsHeader* hdr, const uint32_t* mask, int32_t* idx, int words, int ncap,
    const WsHeader* prev) {
  __shared__ int s_warp_sum[kColThreads / 32];
  if (prev && threadIdx.x == 0) {
    const int ps = *reinterpret_cast<volatile const int*>(&prev->status);
    if (ps != 0) atomicCAS(&hdr->status, 0, ps);
  }
  compact_mask(mask, words, idx, hdr, ncap, s_warp_sum);
}

uint16_t threshold_to_half_bits(float threshold) {
  if (!(threshold <= 65504.0f)) return 0x7C00u;  // above the largest finite fp16 (or inf)
  // the fp16 nearest to threshold, then step up while it is below threshold
  uint16_t b = __half_as_ushort(__float2half_rn(threshold));
  while (b < 0x7C00u && __half2float(__ushort_as_half(b)) < threshold) ++b;
  return b;
}

cudaError_t launch_colstats(const void* X, int T, int in, uint16_t thr_bits, WsHeader* hdr,
                            uint32_t* mask, int32_t* idx, int ncap, cudaStream_t s) {
  const int colblocks = (in + kColsPerCta - 1) / kColsPerCta;
  // about four CTAs per SM in total, at least 8 rows per split
  int splits = (4 * sm_count() + colblocks - 1) / colblocks;
  splits = max(1, min(splits, (T + 7) / 8));
  const int rows_per_split = (T + splits - 1) / splits;
  splits = (T + rows_per_split - 1) / rows_per_split;
  dim3 grid(colblocks, splits);
  colstats_kernel<<<grid, kColThreads, 0, s>>>(static_cast<const uint16_t*>(X), T, in,
                                                rows_per_split, thr_bits, hdr, mask, idx,
                                                (in + 31) / 32, ncap);
  return cudaGetLastError();
}

cudaError_t launch_mask_index(int in, WsHeader* hdr, uint32_t* mask, int32_t* idx, int ncap,
                              const WsHeader* prev, cudaStream_t s) {
  mask_index_kernel<<<1, kColThreads, 0, s>>>(hdr, mask, idx, (in + 31) / 32, ncap, prev);
  return cudaGetLastError();
}

}  // namespace i8mm
