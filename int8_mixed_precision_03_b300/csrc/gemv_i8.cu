// Decode-size LLM.int8() matmul (T <= 8 tokens) on the CUDA cores.
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
// idea" steps 2-3, and section "speed" (per-token generation latency): with a handful of
// tokens the int8 matmul is a pass over the weights, so its speed is the rate at which CB
// streams from HBM. The tensor cores would idle here; instead every warp streams whole
// rows of CB with 16-byte loads and accumulates exact int32 dot products with dp4a
// (4 x int8 products per instruction), so there is no fp32 exactness bound to manage.
//
// Layout: x codes int8 [T, in] (outlier columns 0) are staged in shared memory for the
// whole call. Warp w of the grid owns the rows [w*out/W, (w+1)*out/W) and walks them four
// at a time; per step lane l reads bytes [16*(32*v + l), +16) of each of the four rows and
// the same bytes of every token's codes, so a step covers 512 bytes of K per row. A
// rolling register pipeline keeps four steps of weight loads in flight per warp, and the
// next group's first loads go out before a group's sums are reduced. The reduction gives
// lane (r, t) = (l / 8, l % 8) the warp sum of row r, token t (a reduce-scatter for T = 8,
// a butterfly otherwise), and that lane finishes output feature o = row r of the group for
// token t:
//   Y[t, o] = fp16( acc * rowabs[t] * SCB[o]/127^2 + sum_k X_out[t,k] * W_out[o,k] + bias[o] )
// with W_out[o,k] = fp16(CB[o, idx_k] * SCB[o] / 127), in the same fp32 expressions as
// the tensor-core path. The outlier bytes CB[o, idx_k] of the CTA's rows (for the first
// kOutTab outlier columns) are gathered into a shared-memory table at the start, with
// independent loads, and X_out is staged there as fp32; outlier columns past kOutTab are
// read from global memory in the epilogue.
#include <cuda_fp16.h>

#include "int8mm_internal.h"

namespace i8mm {
namespace {

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) / 16 * 16; }

// Threads per CTA and weight-load steps in flight per warp: 512 threads with 4 steps for
// T <= 2; 384 threads with 4 steps (the registers of 8 tokens' sums) from T = 3 (timed on
// B300: 2-4 % faster at T = 8 than 512 threads with 2 steps).
template <int T> struct GvShape {
  static constexpr int kThreads = T <= 2 ? 512 : 384;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kBuf = 4;
};
constexpr int kGvRows = 4;     // rows of CB per warp step
constexpr int kOutTab = 64;    // outlier columns held in the shared-memory table

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int T>
__device__ __forceinline__ void dot_step(int (&acc)[kGvRows][T], const uint4 (&w)[kGvRows],
                                         const uint4* sx, int nvec, int v) {
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const uint4 x = sx[t * nvec + v];
#pragma unroll
    for (int r = 0; r < kGvRows; ++r) {
      acc[r][t] = __dp4a((int)w[r].x, (int)x.x, acc[r][t]);
      acc[r][t] = __dp4a((int)w[r].y, (int)x.y, acc[r][t]);
      acc[r][t] = __dp4a((int)w[r].z, (int)x.z, acc[r][t]);
      acc[r][t] = __dp4a((int)w[r].w, (int)x.w, acc[r][t]);
    }
  }
}

template <int T>
__global__ void __launch_bounds__(GvShape<T>::kThreads, 1) gemv_i8_kernel(
    const int8_t* __restrict__ CB, const float* __restrict__ SCB, int in, int out,
    const int8_t* __restrict__ xq, const float* __restrict__ rowabs,
    const WsHeader* __restrict__ hdr, const int32_t* __restrict__ idx,
    const uint16_t* __restrict__ xout, int ncap, const uint16_t* __restrict__ bias,
    uint16_t* __restrict__ Y, int32_t* __restrict__ acc_debug, int use_tab,
    const NextLayer next) {
  // shared memory: x codes [T][in] | outlier bytes [rows of this CTA][kOutTab] |
  //                X_out [T][kOutTab] fp32
  constexpr int kGvThreads = GvShape<T>::kThreads, kGvWarps = GvShape<T>::kWarps;
  constexpr int kBuf = GvShape<T>::kBuf;
  extern __shared__ uint4 sx[];
  const int nvec = in / 16;  // in % 16 == 0
  const long long W = (long long)gridDim.x * kGvWarps;
  const int cta_r0 = (int)((long long)blockIdx.x * kGvWarps * out / W);
  const int cta_r1 = (int)((long long)(blockIdx.x + 1) * kGvWarps * out / W);
  int8_t* otab = reinterpret_cast<int8_t*>(sx + (size_t)T * nvec);
  float* xo = reinterpret_cast<float*>(otab + align16((size_t)(cta_r1 - cta_r0) * kOutTab));
  const int n_out = *reinterpret_cast<volatile const int*>(&hdr->n_out_used);
  const int n_tab = min(n_out, use_tab ? kOutTab : 0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kGvWarps + warp;
  const int r_begin = (int)(gw * out / W), r_end = (int)((gw + 1) * out / W);
  const int lr = lane / 8, lt = lane % 8;  // the (row, token) this lane finishes
  const float ra_l = lt < T ? __ldg(&rowabs[lt]) : 0.0f;

  // weight rows of group r0 (rows past the warp's range re-read its last row)
  auto group_rows = [&](int r0, const uint4* (&wrow)[kGvRows]) {
    const int nr = min(kGvRows, r_end - r0);
#pragma unroll
    for (int r = 0; r < kGvRows; ++r)
      wrow[r] = reinterpret_cast<const uint4*>(CB + (size_t)(r0 + min(r, nr - 1)) * in);
  };
  // rolling pipeline of kBuf steps: a buffer is reloaded right after it is consumed; the
  // next group's first steps are issued before this group's sums are reduced and finished
  uint4 w[kBuf][kGvRows];
  auto load_first = [&](const uint4* (&wrow)[kGvRows]) {
#pragma unroll
    for (int bi = 0; bi < kBuf; ++bi) {
      const int vb = lane + 32 * bi;
      if (vb < nvec) {
#pragma unroll
        for (int r = 0; r < kGvRows; ++r) w[bi][r] = ld_stream16(wrow[r] + vb);
      }
    }
  };
  const uint4* wrow[kGvRows];
  if (r_begin < r_end) {
    group_rows(r_begin, wrow);
    load_first(wrow);
  }
  // shared-memory staging overlaps the first weight loads
  for (int i = threadIdx.x; i < T * nvec; i += kGvThreads)
    sx[i] = __ldg(reinterpret_cast<const uint4*>(xq) + i);
  for (int i = threadIdx.x; i < (cta_r1 - cta_r0) * n_tab; i += kGvThreads) {
    const int rr = i / n_tab, k = i - rr * n_tab;
    otab[rr * kOutTab + k] = __ldg(&CB[(size_t)(cta_r0 + rr) * in + __ldg(&idx[k])]);
  }
  for (int i = threadIdx.x; i < T * n_tab; i += kGvThreads) {
    const int t = i / n_tab, k = i - t * n_tab;
    xo[t * kOutTab + k] = __half2float(__ushort_as_half(__ldg(&xout[(size_t)t * ncap + k])));
  }
  __syncthreads();

  for (int r0 = r_begin; r0 < r_end; r0 += kGvRows) {
    const int nr = min(kGvRows, r_end - r0);
    int acc[kGvRows][T];
#pragma unroll
    for (int r = 0; r < kGvRows; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) acc[r][t] = 0;
    for (int v = lane; v < nvec; v += 32 * kBuf) {
#pragma unroll
      for (int bi = 0; bi < kBuf; ++bi) {
        const int vb = v + 32 * bi;
        if (vb < nvec) dot_step<T>(acc, w[bi], sx, nvec, vb);
        const int vn = vb + 32 * kBuf;
        if (vn < nvec) {
#pragma unroll
          for (int r = 0; r < kGvRows; ++r) w[bi][r] = ld_stream16(wrow[r] + vn);
        }
      }
    }
    if (r0 + kGvRows < r_end) {  // the next group's loads go out now
      group_rows(r0 + kGvRows, wrow);
      load_first(wrow);
    }
    int a = 0;  // this lane's total: (row, token) = (lane / 8, lane % 8)
    if constexpr (kGvRows * T == 32) {
      // reduce-scatter: each round halves the values a lane holds, exchanging the other
      // half with the partner lane, until lane l holds the warp sum of value l
      int v[32];
#pragma unroll
      for (int r = 0; r < kGvRows; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t) v[r * T + t] = acc[r][t];
#pragma unroll
      for (int wd = 16; wd >= 1; wd >>= 1) {
        const bool upper = (lane & wd) != 0;
#pragma unroll
        for (int i = 0; i < wd; ++i) {
          const int send = upper ? v[i] : v[i + wd];
          const int keep = upper ? v[i + wd] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, wd);
        }
      }
      a = v[0];
    } else {
      // every lane gets every total
#pragma unroll
      for (int r = 0; r < kGvRows; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t)
#pragma unroll
          for (int d = 16; d >= 1; d >>= 1)
            acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], d);
      // select without dynamic register indexing
#pragma unroll
      for (int r = 0; r < kGvRows; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t)
          if (r == lr && t == lt) a = acc[r][t];
    }
    if (lt < T && lr < nr) {
      const int o = r0 + lr;
      const float scb = __ldg(&SCB[o]);
      float fo = 0.0f;
      const int8_t* orow = otab + (size_t)(o - cta_r0) * kOutTab;
      for (int k = 0; k < n_tab; ++k) {
        const float wk =
            __half2float(__float2half_rn(__fdiv_rn(__fmul_rn((float)orow[k], scb), 127.0f)));
        fo = fmaf(xo[lt * kOutTab + k], wk, fo);
      }
      for (int k = n_tab; k < n_out; ++k) {  // columns beyond the table
        const float c = (float)__ldg(&CB[(size_t)o * in + __ldg(&idx[k])]);
        const float wk = __half2float(__float2half_rn(__fdiv_rn(__fmul_rn(c, scb), 127.0f)));
        fo = fmaf(__half2float(__ushort_as_half(__ldg(&xout[(size_t)lt * ncap + k]))), wk, fo);
      }
      const float so = scb * (1.0f / 16129.0f);
      const float bo = bias ? __half2float(__ushort_as_half(__ldg(&bias[o]))) : 0.0f;
      float y = (float)a * (ra_l * so) + fo + bo;
      if (next.relu) y = fmaxf(y, 0.0f);
      const uint32_t h = __half_as_ushort(__float2half_rn(y));
      Y[(size_t)lt * out + o] = (uint16_t)h;
      // FFN up projection: flag column o of Y for the next matmul (at most T atomics
      // per flagged column)
      if (next.mask && (h & 0x7fffu) >= next.thr_bits)
        atomicOr(&next.mask[o >> 5], 1u << (o & 31));
      if (acc_debug) acc_debug[(size_t)lt * out + o] = a;
    }
  }
}

// Shared memory of the kernel: x codes, the outlier-byte table (if use_tab) and X_out.
size_t gemv_smem(int T, int in, int out, bool use_tab) {
  // with G = sm_count() CTAs, a CTA owns floor((b+1)*out/G) - floor(b*out/G) <= ceil(out/G)
  // rows
  const int G = sm_count();
  const int rows_cta = (out + G - 1) / G;
  size_t b = (size_t)T * in;
  if (use_tab) b += align16((size_t)rows_cta * kOutTab) + (size_t)T * kOutTab * 4;
  return b;
}

template <int T>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t s) {
  const bool use_tab = gemv_smem(T, a.in, a.out, true) <= kGemvMaxSmem;
  const size_t smem = gemv_smem(T, a.in, a.out, use_tab);
  cudaError_t e = cudaFuncSetAttribute(gemv_i8_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gemv_i8_kernel<T><<<sm_count(), GvShape<T>::kThreads, smem, s>>>(
      a.CB, a.SCB, a.in, a.out, a.xq8, a.rowabs, a.hdr, a.idx,
      static_cast<const uint16_t*>(a.xout), a.ncap, static_cast<const uint16_t*>(a.bias),
      static_cast<uint16_t*>(a.Y), a.acc_debug, use_tab ? 1 : 0, a.next);
  return cudaGetLastError();
}

}  // namespace

bool gemv_fits(int T, int in) {
  if (T >= kGemvMmaMinT) return gemv_mma_fits(T, in);
  return T >= 1 && (size_t)T * in <= kGemvMaxSmem;
}

cudaError_t launch_gemv_i8(const GemvArgs& a, cudaStream_t s) {
  if (a.T >= kGemvMmaMinT) return launch_gemv_mma(a, s);
  switch (a.T) {
    case 1: return launch_t<1>(a, s);
    case 2: return launch_t<2>(a, s);
    case 3: return launch_t<3>(a, s);
    case 4: return launch_t<4>(a, s);
    case 5: return launch_t<5>(a, s);
    case 6: return launch_t<6>(a, s);
    case 7: return launch_t<7>(a, s);
    case 8: return launch_t<8>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace i8mm
