// Decode-size LLM.int8() matmul for 9 <= T <= 16 tokens on the legacy fp16 tensor path
// (mma.sync m16n8k16, fp32 accumulation), streaming CB at HBM rate.
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
// idea" steps 2-3: with a handful of tokens the int8 matmul is a pass over the weights.
// Compared with dp4a on the CUDA cores, one m16n8k16 instruction does 2048 products, so
// the per-byte instruction count drops to the int8 -> fp16 conversion of the weights and
// stays flat up to 16 tokens. (At T = 8 the dp4a kernel, whose warps read 512 contiguous
// bytes of each row per load, measured faster on B300; this kernel takes T = 9 .. 16.)
//
// Exactness: int8 codes are exact fp16 values and the fp32 fragment sums stay integers
// below 2^24 over 1024 K (1024 * 127 * 127 < 2^24); every 16 steps of 64 K the fragments are
// drained into int32 registers, so the int32 result is exact.
//
// Layout: x codes int8 [T, in] staged in shared memory (row stride = 64 mod 128 bytes,
// which keeps the 16-byte reads of a quarter warp on distinct banks). Warp w of the grid
// owns the rows [w*out/W, (w+1)*out/W) and walks them 16 at a time. Lane (g, c) = (l / 4,
// l % 4) loads, per 64-byte K step, bytes [16c, 16c + 16) of rows g and g + 8 and of token g
// (and g + 8). Within a step, sub-step s takes bytes 16c + 4s .. +3 of each: the first two
// are the MMA's k = 2c, 2c+1 and the last two its k = 2c+8, 2c+9, the same permutation of K
// for the weights and the codes, so the dot products are unchanged. Four steps of weight
// loads are in flight per warp. Lane (g, c) ends with the sums of rows {g, g + 8} x tokens
// {2c, 2c + 1} (+8 for the second token tile) and finishes them as the CUDA-core decode
// kernel does (outlier bytes of the CTA's rows gathered once into a shared-memory table).
#include <cuda_fp16.h>

#include "int8mm_internal.h"

namespace i8mm {
namespace {

constexpr int kMvThreads = 512;
constexpr int kMvWarps = kMvThreads / 32;
constexpr int kMvRows = 16;   // rows of CB per warp group (the MMA's M)
constexpr int kMvBuf = 4;     // 64-byte K steps of weight loads in flight per warp
constexpr int kMvTab = 64;    // outlier columns held in the shared-memory table

__host__ __device__ constexpr size_t mv_align16(size_t x) { return (x + 15) / 16 * 16; }
// x row stride in shared memory: >= in and = 64 (mod 128)
__host__ __device__ constexpr int mv_xstride(int in) { return (in + 127) / 128 * 128 + 64; }

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// int8 x 4 (one word) -> two half2 words (b0, b1) and (b2, b3), exactly: fp16 0x6400|u is
// 1024 + u, and u = b ^ 0x80 is b + 128.
__device__ __forceinline__ void cvt_s8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t p0 = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t p1 = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
  const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
  const __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
  lo = *reinterpret_cast<const uint32_t*>(&h0);
  hi = *reinterpret_cast<const uint32_t*>(&h1);
}

// d += A (16 x 16, row) * B (16 x 8, col), fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int s) {
  return s == 0 ? v.x : s == 1 ? v.y : s == 2 ? v.z : v.w;
}

template <int NT>  // token tiles of 8
__global__ void __launch_bounds__(kMvThreads, 1) gemv_mma_kernel(
    const int8_t* __restrict__ CB, const float* __restrict__ SCB, int T, int in, int out,
    const int8_t* __restrict__ xq, const float* __restrict__ rowabs,
    const WsHeader* __restrict__ hdr, const int32_t* __restrict__ idx,
    const uint16_t* __restrict__ xout, int ncap, const uint16_t* __restrict__ bias,
    uint16_t* __restrict__ Y, int32_t* __restrict__ acc_debug, int use_tab,
    const NextLayer next) {
  // shared memory: x codes [T][xs] | outlier bytes [rows of this CTA][kMvTab] |
  //                X_out [T][kMvTab] fp32
  extern __shared__ uint4 smv[];
  const int xs = mv_xstride(in);
  uint8_t* sx = reinterpret_cast<uint8_t*>(smv);
  const long long W = (long long)gridDim.x * kMvWarps;
  const int cta_r0 = (int)((long long)blockIdx.x * kMvWarps * out / W);
  const int cta_r1 = (int)((long long)(blockIdx.x + 1) * kMvWarps * out / W);
  int8_t* otab = reinterpret_cast<int8_t*>(sx + mv_align16((size_t)T * xs));
  float* xo = reinterpret_cast<float*>(otab + mv_align16((size_t)(cta_r1 - cta_r0) * kMvTab));
  const int n_out = *reinterpret_cast<volatile const int*>(&hdr->n_out_used);
  const int n_tab = min(n_out, use_tab ? kMvTab : 0);

  const int nvec = in / 16;  // in % 16 == 0
  for (int i = threadIdx.x; i < T * nvec; i += kMvThreads) {
    const int t = i / nvec, j = i - t * nvec;
    *reinterpret_cast<uint4*>(sx + (size_t)t * xs + 16 * j) =
        __ldg(reinterpret_cast<const uint4*>(xq) + i);
  }
  for (int i = threadIdx.x; i < (cta_r1 - cta_r0) * n_tab; i += kMvThreads) {
    const int rr = i / n_tab, k = i - rr * n_tab;
    otab[rr * kMvTab + k] = __ldg(&CB[(size_t)(cta_r0 + rr) * in + __ldg(&idx[k])]);
  }
  for (int i = threadIdx.x; i < T * n_tab; i += kMvThreads) {
    const int t = i / n_tab, k = i - t * n_tab;
    xo[t * kMvTab + k] = __half2float(__ushort_as_half(__ldg(&xout[(size_t)t * ncap + k])));
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const long long gw = (long long)blockIdx.x * kMvWarps + warp;
  const int r_begin = (int)(gw * out / W), r_end = (int)((gw + 1) * out / W);
  const int nsteps = (in + 63) / 64;

  for (int r0 = r_begin; r0 < r_end; r0 += kMvRows) {
    // rows past the warp's range re-read its last row; their results are not stored
    const int8_t* pa = CB + (size_t)min(r0 + g, r_end - 1) * in + 16 * c;
    const int8_t* pb = CB + (size_t)min(r0 + g + 8, r_end - 1) * in + 16 * c;
    float d[NT][4];
    int acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) { d[n][i] = 0.0f; acc[n][i] = 0; }
    uint4 wa[kMvBuf], wb[kMvBuf];
#pragma unroll
    for (int b = 0; b < kMvBuf; ++b) {
      const bool in_k = b < nsteps && 64 * b + 16 * c < in;
      wa[b] = in_k ? ld_stream16(pa + 64 * b) : make_uint4(0, 0, 0, 0);
      wb[b] = in_k ? ld_stream16(pb + 64 * b) : make_uint4(0, 0, 0, 0);
    }
    for (int s0 = 0; s0 < nsteps; s0 += kMvBuf) {
#pragma unroll
      for (int b = 0; b < kMvBuf; ++b) {
        const int step = s0 + b;
        if (step >= nsteps) break;
        const int kofs = 64 * step + 16 * c;
        uint4 xv[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int t = g + 8 * n;
          xv[n] = (t < T && kofs < in)
                      ? *reinterpret_cast<const uint4*>(sx + (size_t)t * xs + kofs)
                      : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int ss = 0; ss < 4; ++ss) {
          uint32_t a0, a2, a1, a3;
          cvt_s8x4(word(wa[b], ss), a0, a2);  // row g:     k 2c, 2c+1 | k 2c+8, 2c+9
          cvt_s8x4(word(wb[b], ss), a1, a3);  // row g + 8: the same k
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            uint32_t b0, b1;
            cvt_s8x4(word(xv[n], ss), b0, b1);
            mma16816(d[n], a0, a1, a2, a3, b0, b1);
          }
        }
        const int nstep = step + kMvBuf;
        if (nstep < nsteps) {
          const bool in_k = 64 * nstep + 16 * c < in;
          wa[b] = in_k ? ld_stream16(pa + 64 * nstep) : make_uint4(0, 0, 0, 0);
          wb[b] = in_k ? ld_stream16(pb + 64 * nstep) : make_uint4(0, 0, 0, 0);
        }
        if ((step & 15) == 15 || step == nsteps - 1) {  // drain the exact fp32 sums
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[n][i] += __float2int_rn(d[n][i]);
              d[n][i] = 0.0f;
            }
        }
      }
    }
    // finish this lane's outputs: rows g, g+8 x tokens 2c, 2c+1 (+ 8n)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int o = r0 + g + (i >= 2 ? 8 : 0);
        const int t = 8 * n + 2 * c + (i & 1);
        if (o >= r_end || t >= T) continue;
        const float scb = __ldg(&SCB[o]);
        float fo = 0.0f;
        const int8_t* orow = otab + (size_t)(o - cta_r0) * kMvTab;
        for (int k = 0; k < n_tab; ++k) {
          const float wk =
              __half2float(__float2half_rn(__fdiv_rn(__fmul_rn((float)orow[k], scb), 127.0f)));
          fo = fmaf(xo[t * kMvTab + k], wk, fo);
        }
        for (int k = n_tab; k < n_out; ++k) {  // columns beyond the table
          const float cw = (float)__ldg(&CB[(size_t)o * in + __ldg(&idx[k])]);
          const float wk = __half2float(__float2half_rn(__fdiv_rn(__fmul_rn(cw, scb), 127.0f)));
          fo = fmaf(__half2float(__ushort_as_half(__ldg(&xout[(size_t)t * ncap + k]))), wk, fo);
        }
        const float so = scb * (1.0f / 16129.0f);
        const float bo = bias ? __half2float(__ushort_as_half(__ldg(&bias[o]))) : 0.0f;
        const float ra = __ldg(&rowabs[t]);
        float y = (float)acc[n][i] * (ra * so) + fo + bo;
        if (next.relu) y = fmaxf(y, 0.0f);
        const uint32_t h = __half_as_ushort(__float2half_rn(y));
        Y[(size_t)t * out + o] = (uint16_t)h;
        // FFN up projection: flag column o of Y for the next matmul (at most T atomics
        // per flagged column)
        if (next.mask && (h & 0x7fffu) >= next.thr_bits)
          atomicOr(&next.mask[o >> 5], 1u << (o & 31));
        if (acc_debug) acc_debug[(size_t)t * out + o] = acc[n][i];
      }
  }
}

size_t mv_smem(int T, int in, int out, bool use_tab) {
  const int G = sm_count();  // the grid of launch_nt
  const int rows_cta = (out + G - 1) / G;
  size_t b = mv_align16((size_t)T * mv_xstride(in));
  if (use_tab) b += mv_align16((size_t)rows_cta * kMvTab) + (size_t)T * kMvTab * 4;
  return b;
}

template <int NT>
cudaError_t launch_nt(const GemvArgs& a, cudaStream_t s) {
  const bool use_tab = mv_smem(a.T, a.in, a.out, true) <= kGemvMaxSmem;
  const size_t smem = mv_smem(a.T, a.in, a.out, use_tab);
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gemv_mma_kernel<NT><<<sm_count(), kMvThreads, smem, s>>>(
      a.CB, a.SCB, a.T, a.in, a.out, a.xq8, a.rowabs, a.hdr, a.idx,
      static_cast<const uint16_t*>(a.xout), a.ncap, static_cast<const uint16_t*>(a.bias),
      static_cast<uint16_t*>(a.Y), a.acc_debug, use_tab ? 1 : 0, a.next);
  return cudaGetLastError();
}

}  // namespace

bool gemv_mma_fits(int T, int in) {
  return T >= kGemvMmaMinT && T <= kGemvMaxT &&
         mv_align16((size_t)T * mv_xstride(in)) <= kGemvMaxSmem;
}

cudaError_t launch_gemv_mma(const GemvArgs& a, cudaStream_t s) {
  return a.T <= 8 ? launch_nt<1>(a, s) : launch_nt<2>(a, s);
}

}  // namespace i8mm
