// Pieces shared by the two tensor-core matmul kernels (the LLM.int8() matmul in gemm_i8.cu
// and the fp16 comparator in gemm_f16.cu): tile constants, the bounded pipeline wait,
// shared-memory and TMEM access wrappers, the exact int8 -> fp16 conversion, the staged
// TMA-store epilogue helpers and the host-side tensor-map encoder.
#pragma once
#include <cudaTypedefs.h>

#include "int8mm_internal.h"
#include "sm103_ptx.cuh"

namespace i8mm {
namespace gemm {

constexpr int BM = 128;          // output features per tile (TMEM lanes)
constexpr int BK = kKBlock;      // 64 K elements per pipeline stage
constexpr int kA16Bytes = BM * BK * 2;  // one fp16 A stage (16 KB)
constexpr int kA8Bytes = BM * BK;       // one int8 A stage (8 KB)
constexpr int kMaxSmem = 232448;        // dynamic shared memory limit per CTA (227 KB)

// Abort flag and status word of one CTA's pipeline.
struct Abort {
  volatile int* flag;  // CTA-local: set when any role gives up
  WsHeader* hdr;       // device status word (may be null)
  uint64_t timeout_ns;
};

// Bounded wait: false if the pipeline was aborted or this wait ran past the time limit
// (then the status word records I8_ERR_TIMEOUT and every role unwinds).
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, const Abort& ab) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    // sleep in the barrier (woken when the phase completes) rather than spin
    if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
    if (*ab.flag) return false;
    if (globaltimer_ns() - t0 > ab.timeout_ns) {
      *ab.flag = 1;
      if (ab.hdr) atomicCAS(&ab.hdr->status, 0, (int)I8_ERR_TIMEOUT);
      return false;
    }
  }
}

// int8 x16 (one 16-byte chunk, K order) -> fp16 x16 as 8 words of (even K, odd K) pairs,
// exactly. fp16 with bits 0x6400|u is 1024+u for a byte u; u = b ^ 0x80 maps int8 b to
// b+128, so (0x6400|(b^0x80)) - 1152 == b.
__device__ __forceinline__ void cvt_s8x16_to_f16x16(const uint4& in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u, in.z ^ 0x80808080u,
                         in.w ^ 0x80808080u};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t p0 = __byte_perm(w[k], 0x64646464u, 0x5140);  // bytes b0,b1 -> 2 halves
    const uint32_t p1 = __byte_perm(w[k], 0x64646464u, 0x7362);  // bytes b2,b3
    __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
    __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
    o[2 * k] = *reinterpret_cast<uint32_t*>(&h0);
    o[2 * k + 1] = *reinterpret_cast<uint32_t*>(&h1);
  }
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  st_shared_u32(addr, __float_as_uint(v));
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
template <int W> __device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[W]);
template <> __device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld_32x32b_x32(taddr, r);
}
template <> __device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld_32x32b_x16(taddr, r);
}
template <int W> __device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[W]);
template <> __device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) {
  tmem_st_32x32b_x32(taddr, r);
}
template <> __device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t (&r)[16]) {
  tmem_st_32x32b_x16(taddr, r);
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Epilogue output boxes: each epilogue warp stages kW tokens x 32 features of Y (fp16) in
// shared memory and writes them with one TMA store. Two boxes per warp alternate, so the
// store of one slice overlaps the next slice's arithmetic. Before a box is written again,
// the store issued from it two slices ago must have finished reading it; at most the one
// newer store (from the other box) may still be reading.
__device__ __forceinline__ void box_reuse_wait(int lane) {
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  __syncwarp();
}

// Writes this lane's kW outputs (one feature, kW tokens; fp16 pairs in yh) into its box
// column and stores the box to Y[tok0 .. +kW, feat0 .. +32]. With a Y tensor map (Y's row
// pitch a multiple of 16 bytes) that is one TMA store, clipped by the map at the edges of
// Y, whose lines are marked first to leave L2 (`policy`: Y is not read again here, and the
// operands the matmul re-reads across waves should stay); without one the lanes copy the
// box out element by element.
template <int kW>
__device__ __forceinline__ void box_store(uint8_t* box, const uint32_t (&yh)[kW / 2],
                                          const CUtensorMap* mapY, uint16_t* Y, int T, int out,
                                          int feat0, int tok0, int lane, uint64_t policy) {
  const uint32_t b = smem_u32(box);
#pragma unroll
  for (int j = 0; j < kW; ++j) {
    const uint16_t h = (j & 1) ? (uint16_t)(yh[j / 2] >> 16) : (uint16_t)(yh[j / 2] & 0xffffu);
    st_shared_u16(b + (j * 32 + lane) * 2, h);
  }
  if (mapY) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d_hint(mapY, box, feat0, tok0, policy);
      bulk_commit_group();
    }
  } else {
    __syncwarp();
    const int o = feat0 + lane;
#pragma unroll 1
    for (int j = 0; j < kW; ++j) {
      const int tok = tok0 + j;
      if (o < out && tok < T)
        Y[(size_t)tok * out + o] = reinterpret_cast<const uint16_t*>(box)[j * 32 + lane];
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D row-major map: rows x cols elements, box box_rows x box_cols.
inline bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
                     uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                     CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm
}  // namespace i8mm
