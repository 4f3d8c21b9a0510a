// Tensor-core matmul of the LLM.int8() method (steps 2 and 3) on tcgen05, plus the fp16
// comparator GEMM on the same pipeline.
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
// idea": the int8 part is multiplied with int8 vector-wise scales, the outlier part in
// fp16, and the int8 result is dequantized and added to the fp16 result.
// "LLM.int8() summary" (zenn), section "method": outlier input dimensions and the matching
// weight dimensions are split off and kept in 16 bit.
//
// sm_103a has no int8 tcgen05 MMA (ptxas rejects .kind::i8 for this target), so the int8
// product runs on .kind::f16: int8 codes are exact fp16 values and fp32 sums of integers
// are exact while every partial sum stays within 2^24 in magnitude. The K loop is cut into
// 1024-element chunks; for each (token tile, chunk) the quantize pass records
// L1 = max over the tile's rows of sum |code|, and since |CB| <= 127 every partial sum of
// a run of chunks is bounded by 127 * (sum of their L1). Consecutive chunks share one fp32
// accumulation ("segment") while that bound stays <= 2^24; a single chunk always fits
// (127 * 127 * 1024 < 2^24). At a segment boundary the epilogue warps convert the fp32
// tile to int32 and add it to an int32 running sum kept in a second TMEM region. The
// int32 result is therefore exact for any input; for activation-like data most tiles
// need a single segment.
//
// Tile: M = 128 output features (TMEM lanes) x N = BN tokens (TMEM columns), K stage 64.
//   A (M side) = CB int8 [out, in]  -> TMA (64-byte swizzle) -> converter warps -> fp16
//                tile in the 128-byte-swizzled K-major UMMA layout;
//   B (N side) = activation codes as fp16 [T, in] (written by the quantize pass) -> TMA.
//   Outlier segment: W_out fp16 [out, ncap] and X_out fp16 [T, ncap] by TMA, fp32 result.
// Epilogue: Y[t, o] = fp16(acc * rowabs[t] * SCB[o] / 127^2 + outlier + bias[o]), staged
// per warp in shared memory as a token x 32-feature box and written by a TMA store.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 4-7 int8->fp16 converters, warps 8-11 epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31). Persistent CTAs, one per SM, walk tiles token-block fastest so that
// concurrently running CTAs share the same weight strip in L2.
#include <cudaTypedefs.h>

#include "int8mm_internal.h"
#include "sm103_ptx.cuh"

namespace i8mm {

#ifdef I8MM_TRACE
// Trace build only: CTA 0 timestamps pipeline events (SM clock) into a host-provided
// buffer, one region of 2^16 entries per role: tag (high 16 bits) | clock (low 48 bits).
// The buffer pointer is read once per thread, so a record costs a clock read and a store.
__device__ uint64_t* g_i8_trace = nullptr;
#define I8_TRACE_INIT uint64_t* const i8_trace_buf = (blockIdx.x == 0) ? g_i8_trace : nullptr
#define I8_TRACE(role, n, tag)                                                         \
  do {                                                                                 \
    if (i8_trace_buf && (n) < 65536)                                                   \
      i8_trace_buf[((role) << 16) + (n)] =                                             \
          ((uint64_t)(tag) << 48) | ((uint64_t)clock64() & 0xFFFFFFFFFFFFull);         \
    ++(n);                                                                             \
  } while (0)
#else
#define I8_TRACE_INIT do { } while (0)
#define I8_TRACE(role, n, tag) do { } while (0)
#endif

namespace {

constexpr int BM = 128;
constexpr int BK = kKBlock;  // 64
constexpr int kStages = 4;   // fp16 A + B ring
constexpr int kStages8 = 3;  // int8 A staging ring
constexpr int kThreads = 384;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpConv0 = 4, kWarpEpi0 = 8;
constexpr int kA16Bytes = BM * BK * 2;  // 16 KB
constexpr int kA8Bytes = BM * BK;       // 8 KB
constexpr uint32_t kExactLimit = 1u << 24;                      // integers exact in fp32
constexpr uint32_t kWorstChunkBound = 127u * 127u * kChunkK;    // < kExactLimit

template <int BN>
struct Smem {
  static constexpr int kW = BN < 32 ? BN : 32;           // tokens per epilogue slice
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = 32 * kW * 2;        // one warp's output box (fp16)
  static constexpr int a16 = 0;
  static constexpr int b = a16 + kStages * kA16Bytes;
  static constexpr int a8 = b + kStages * kBBytes;
  static constexpr int stage = a8 + kStages8 * kA8Bytes;
  static constexpr int bars = stage + 4 * kStageBytes;
  // full_a[S], full_b[S], empty[S], a8_full[S8], a8_empty[S8], tmem_full, tmem_empty, done
  static constexpr int kNumBars = 3 * kStages + 2 * kStages8 + 3;
  static constexpr int misc = bars + kNumBars * 8;
  static constexpr int total = misc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                        : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
};

struct Params {
  int T, in, out;
  int m_tiles, n_tiles, nkb;  // nkb = ceil(in / 64)
  int nchunks;                // ceil(in / 1024)
  int int8_path;              // 1: LLM.int8 matmul, 0: fp16 comparator
  int y_tma;                  // 1: epilogue writes Y with TMA stores (out % 8 == 0)
  WsHeader* hdr;
  const float* rowabs;
  const int32_t* l1;
  const float* scb;
  const uint16_t* bias;
  uint16_t* Y;
  int32_t* acc_debug;
  uint64_t timeout_ns;
  int debug_skip_loads;
};

struct Pipe {
  uint64_t* full_a;
  uint64_t* full_b;
  uint64_t* empty;
  uint64_t* a8_full;
  uint64_t* a8_empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* done;
  volatile int* abort;
};

// Bounded wait: false if the pipeline was aborted or this wait ran past the time limit
// (then the status word records I8_ERR_TIMEOUT and every role unwinds).
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, const Params& p,
                                          const Pipe& pp) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    // sleep in the barrier (woken when the phase completes) rather than spin
    if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
    if (*pp.abort) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      *pp.abort = 1;
      if (p.hdr) atomicCAS(&p.hdr->status, 0, (int)I8_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ int outlier_kblocks(const Params& p) {
  if (!p.int8_path) return 0;
  const int n = *reinterpret_cast<volatile const int*>(&p.hdr->n_out_used);
  return (n + 63) / 64;
}

// ---------------------------------------------------------------- segment plan
// Chunks of the K loop: 1024 K each on the int8 path, one chunk over all of K for fp16.
__device__ __forceinline__ int plan_nchunks(const Params& p) {
  return p.int8_path ? p.nchunks : 1;
}
__device__ __forceinline__ void chunk_kblocks(const Params& p, int c, int& kb0, int& kb1) {
  if (!p.int8_path) { kb0 = 0; kb1 = p.nkb; return; }
  kb0 = c * kChunkKBlocks;
  kb1 = min(p.nkb, kb0 + kChunkKBlocks);
}
// Bound on |partial sums| of chunk c for token tile n_blk (see the file comment).
__device__ __forceinline__ uint32_t chunk_bound(const Params& p, int n_blk, int c) {
  if (!p.int8_path) return 0;
  if (!p.l1) return kWorstChunkBound;
  return 127u * (uint32_t)__ldg(&p.l1[(size_t)n_blk * p.nchunks + c]);
}
// Greedy rule shared by the MMA issuer and the epilogue: chunk c opens a new segment when
// it is the first chunk or adding its bound would exceed 2^24.
struct SegWalker {
  uint32_t run = 0;
  __device__ __forceinline__ bool opens(uint32_t b, int c) {
    if (c == 0 || run + b > kExactLimit) { run = b; return true; }
    run += b;
    return false;
  }
};
__device__ __forceinline__ int count_int_segments(const Params& p, int n_blk) {
  SegWalker w;
  int n = 0;
  const int nc = plan_nchunks(p);
  for (int c = 0; c < nc; ++c) n += w.opens(chunk_bound(p, n_blk, c), c) ? 1 : 0;
  return n;
}

// int8 x16 (one 16-byte chunk) -> fp16 x16 (two 16-byte chunks), exactly.
// fp16 with bits 0x6400|u is 1024+u for a byte u; u = b ^ 0x80 maps int8 b to b+128,
// so (0x6400|(b^0x80)) - 1152 == b.
__device__ __forceinline__ void cvt_s8x16_to_f16x16(const uint4& in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u, in.z ^ 0x80808080u,
                         in.w ^ 0x80808080u};
  uint32_t o[8];
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
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
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

// kMode: 0 = fp16 comparator, 1 = LLM.int8 matmul, 2 = LLM.int8 matmul that also exports
// the exact int32 products (test path). Each mode is its own instantiation so that the
// hot loops carry no code for the other paths.
template <int BN, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA8, const __grid_constant__ CUtensorMap tmA16,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmWo,
                const __grid_constant__ CUtensorMap tmXo, const __grid_constant__ CUtensorMap tmY,
                const Params p) {
  using L = Smem<BN>;
  constexpr int kW = L::kW;
  constexpr bool kInt8 = kMode != 0;
  constexpr bool kDebug = kMode == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  Pipe pp;
  pp.full_a = bars;
  pp.full_b = bars + kStages;
  pp.empty = bars + 2 * kStages;
  pp.a8_full = bars + 3 * kStages;
  pp.a8_empty = bars + 3 * kStages + kStages8;
  pp.tmem_full = bars + 3 * kStages + 2 * kStages8;
  pp.tmem_empty = pp.tmem_full + 1;
  pp.done = pp.tmem_full + 2;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + L::misc);
  pp.abort = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  I8_TRACE_INIT;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&pp.full_a[s], 4);  // 4 converter warps, or the producer with count 4
      mbar_init(&pp.full_b[s], 1);
      mbar_init(&pp.empty[s], 1);
    }
    for (int s = 0; s < kStages8; ++s) {
      mbar_init(&pp.a8_full[s], 1);
      mbar_init(&pp.a8_empty[s], 4);  // one arrival per converter warp
    }
    mbar_init(pp.tmem_full, 1);
    mbar_init(pp.tmem_empty, 4);      // one arrival per epilogue warp
    mbar_init(pp.done, 1);
    *pp.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmA8);
    tma_prefetch_desc(&tmA16);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmWo);
    tma_prefetch_desc(&tmXo);
    tma_prefetch_desc(&tmY);
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_base_smem, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;

  const int tiles = p.m_tiles * p.n_tiles;
  const int nkb_out = outlier_kblocks(p);
  const uint32_t sbase = smem_u32(smem);

  if (warp == kWarpTma) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && !p.debug_skip_loads) {
      uint32_t it = 0, it8 = 0;
      [[maybe_unused]] uint32_t tn = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t / p.n_tiles) * BM, n0 = (t % p.n_tiles) * BN;
        const int nkb_total = p.nkb + nkb_out;
        for (int kb = 0; kb < nkb_total && ok; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          I8_TRACE(0, tn, 1);
          if (!(ok = pipe_wait(&pp.empty[s], ph ^ 1u, p, pp))) break;
          I8_TRACE(0, tn, 2);
          uint8_t* a16 = smem + L::a16 + s * kA16Bytes;
          uint8_t* bb = smem + L::b + s * L::kBBytes;
          if (kb < p.nkb) {
            if (kInt8) {
              const uint32_t s8 = it8 % kStages8, ph8 = (it8 / kStages8) & 1u;
              if (!(ok = pipe_wait(&pp.a8_empty[s8], ph8 ^ 1u, p, pp))) break;
              mbar_arrive_expect_tx(&pp.a8_full[s8], kA8Bytes);
              tma_load_2d(smem + L::a8 + s8 * kA8Bytes, &tmA8, &pp.a8_full[s8], kb * BK, m0);
              ++it8;
              mbar_arrive_expect_tx(&pp.full_b[s], L::kBBytes);
              tma_load_2d(bb, &tmB, &pp.full_b[s], kb * BK, n0);
            } else {
              mbar_arrive_expect_tx(&pp.full_b[s], kA16Bytes + L::kBBytes);
              tma_load_2d(a16, &tmA16, &pp.full_b[s], kb * BK, m0);
              tma_load_2d(bb, &tmB, &pp.full_b[s], kb * BK, n0);
              mbar_arrive_cnt(&pp.full_a[s], 4);
            }
          } else {
            const int ko = kb - p.nkb;
            mbar_arrive_expect_tx(&pp.full_b[s], kA16Bytes + L::kBBytes);
            tma_load_2d(a16, &tmWo, &pp.full_b[s], ko * BK, m0);
            tma_load_2d(bb, &tmXo, &pp.full_b[s], ko * BK, n0);
            mbar_arrive_cnt(&pp.full_a[s], 4);
          }
        }
      }
      // Do not leave the CTA with copies in flight: wait for the last issued stages.
      for (uint32_t k = 0; k < kStages && k < it; ++k) {
        const uint32_t j = it - 1 - k;
        mbar_wait_bounded(&pp.full_b[j % kStages], (j / kStages) & 1u, p.timeout_ns);
      }
      for (uint32_t k = 0; k < kStages8 && k < it8; ++k) {
        const uint32_t j = it8 - 1 - k;
        mbar_wait_bounded(&pp.a8_full[j % kStages8], (j / kStages8) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32acc(BM, BN);
      uint32_t it = 0, nseg = 0;
      [[maybe_unused]] uint32_t tn = 0;
      bool ok = true;
      const int nc = plan_nchunks(p);
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int n_blk = t % p.n_tiles;
        SegWalker walker;
        bool seg_first_kb = true;
        // int (or fp16) chunks, grouped into exact segments
        for (int c = 0; c < nc && ok; ++c) {
          if (walker.opens(chunk_bound(p, n_blk, c), c)) {
            if (c > 0) { mma_commit(pp.tmem_full); ++nseg; }
            I8_TRACE(1, tn, 10);
            if (!(ok = pipe_wait(pp.tmem_empty, (nseg & 1u) ^ 1u, p, pp))) break;
            I8_TRACE(1, tn, 11);
            tc_fence_after();
            seg_first_kb = true;
          }
          int kb0, kb1;
          chunk_kblocks(p, c, kb0, kb1);
          for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
            I8_TRACE(1, tn, 12);
            if (!(ok = pipe_wait(&pp.full_a[s], ph, p, pp))) break;
            I8_TRACE(1, tn, 13);
            if (!(ok = pipe_wait(&pp.full_b[s], ph, p, pp))) break;
            I8_TRACE(1, tn, 14);
            tc_fence_after();
            const uint64_t ad = sdesc_kmajor_sw128(sbase + L::a16 + s * kA16Bytes);
            const uint64_t bd = sdesc_kmajor_sw128(sbase + L::b + s * L::kBBytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_f16_ss(tmem_base, ad + 2 * k, bd + 2 * k, idesc,
                         (seg_first_kb && k == 0) ? 0u : 1u);
            seg_first_kb = false;
            mma_commit(&pp.empty[s]);
          }
        }
        if (!ok) break;
        mma_commit(pp.tmem_full);
        ++nseg;
        // outlier segment (fp16 x fp16, fp32 result)
        if (nkb_out > 0) {
          if (!(ok = pipe_wait(pp.tmem_empty, (nseg & 1u) ^ 1u, p, pp))) break;
          tc_fence_after();
          for (int kb = p.nkb; kb < p.nkb + nkb_out; ++kb, ++it) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
            if (!(ok = pipe_wait(&pp.full_a[s], ph, p, pp))) break;
            if (!(ok = pipe_wait(&pp.full_b[s], ph, p, pp))) break;
            tc_fence_after();
            const uint64_t ad = sdesc_kmajor_sw128(sbase + L::a16 + s * kA16Bytes);
            const uint64_t bd = sdesc_kmajor_sw128(sbase + L::b + s * L::kBBytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_f16_ss(tmem_base, ad + 2 * k, bd + 2 * k, idesc,
                         (kb == p.nkb && k == 0) ? 0u : 1u);
            mma_commit(&pp.empty[s]);
          }
          if (!ok) break;
          mma_commit(pp.tmem_full);
          ++nseg;
        }
      }
      // all issued MMAs have completed before TMEM is released
      mma_commit(pp.done);
      mbar_wait_bounded(pp.done, 0, p.timeout_ns);
    }
  } else if (warp >= kWarpConv0 && warp < kWarpConv0 + 4) {
    // ------------------------------------------------------------------ int8 -> fp16
    if (kInt8 && !p.debug_skip_loads) {
      const int cw = warp - kWarpConv0;
      const int c = lane >> 3;           // 16-byte int8 chunk of the 64-byte row (0..3)
      uint32_t it = 0, it8 = 0;
      [[maybe_unused]] uint32_t tn = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int nkb_total = p.nkb + nkb_out;
        for (int kb = 0; kb < nkb_total && ok; ++kb, ++it) {
          if (kb >= p.nkb) continue;  // outlier K blocks arrive as fp16 by TMA
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          const uint32_t s8 = it8 % kStages8, ph8 = (it8 / kStages8) & 1u;
          if (cw == 0 && lane == 0) I8_TRACE(2, tn, 20);
          if (!(ok = pipe_wait(&pp.a8_full[s8], ph8, p, pp))) break;
          if (cw == 0 && lane == 0) I8_TRACE(2, tn, 21);
          if (!(ok = pipe_wait(&pp.empty[s], ph ^ 1u, p, pp))) break;
          if (cw == 0 && lane == 0) I8_TRACE(2, tn, 22);
          const uint32_t src = sbase + L::a8 + s8 * kA8Bytes;
          const uint32_t dst = sbase + L::a16 + s * kA16Bytes;
          uint4 v[4];
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 32 + cw * 8 + (lane & 7);
            v[pass] = ld_shared_v4(src + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
          }
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 32 + cw * 8 + (lane & 7);
            uint4 lo, hi;
            cvt_s8x16_to_f16x16(v[pass], lo, hi);
            st_shared_v4(dst + r * 128 + (((2 * c) ^ (r & 7)) << 4), lo);
            st_shared_v4(dst + r * 128 + (((2 * c + 1) ^ (r & 7)) << 4), hi);
          }
          // each thread orders its shared stores before the async proxy reads them; the
          // warp then signals once (both barriers count one arrival per converter warp)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&pp.a8_empty[s8]);
            mbar_arrive(&pp.full_a[s]);
          }
          if (cw == 0 && lane == 0) I8_TRACE(2, tn, 23);
          ++it8;
        }
      }
    }
  } else if (warp >= kWarpEpi0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant
    const uint32_t tF = tmem_base + ((uint32_t)(q * 32) << 16);
    const uint32_t tI = tF + BN;
    uint8_t* stage = smem + L::stage + q * L::kStageBytes;  // [kW tokens][32 features]
    const uint32_t stg = smem_u32(stage);
    uint32_t nseg = 0;
    [[maybe_unused]] uint32_t tn = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const int m_blk = t / p.n_tiles, n_blk = t % p.n_tiles;
      const int m0 = m_blk * BM, n0 = n_blk * BN;
      const int o = m0 + q * 32 + lane;
      const bool o_ok = o < p.out;
      const float bo = (o_ok && p.bias) ? __half2float(__ushort_as_half(p.bias[o])) : 0.0f;
      const float so = (kInt8 && o_ok) ? __ldg(&p.scb[o]) * (1.0f / 16129.0f) : 0.0f;
      const int nseg_int = count_int_segments(p, n_blk);
      const int nseg_tile = nseg_int + (nkb_out > 0 ? 1 : 0);
      for (int si = 0; si < nseg_tile && ok; ++si, ++nseg) {
        const bool is_out = si >= nseg_int;
        const bool first = si == 0;
        const bool last = si == nseg_tile - 1;
        if (q == 0 && lane == 0) I8_TRACE(3, tn, 30);
        if (!(ok = pipe_wait(pp.tmem_full, nseg & 1u, p, pp))) break;
        if (q == 0 && lane == 0) I8_TRACE(3, tn, 31);
        tc_fence_after();
        if (kInt8 && !last) {
          // int segment: I (+)= int(F)
#pragma unroll 1
          for (int j0 = 0; j0 < BN; j0 += kW) {
            uint32_t f[kW], r[kW];
            tmem_ld<kW>(tF + j0, f);
            if (!first) tmem_ld<kW>(tI + j0, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < kW; ++j) {
              const int v = __float2int_rn(__uint_as_float(f[j]));
              r[j] = first ? (uint32_t)v : (uint32_t)((int)r[j] + v);
            }
            tmem_st<kW>(tI + j0, r);
          }
          tmem_st_wait();
        } else {
#pragma unroll 1
          for (int j0 = 0; j0 < BN; j0 += kW) {
            uint32_t f[kW], r[kW];
            if (q == 0 && lane == 0) I8_TRACE(3, tn, 40);
            tmem_ld<kW>(tF + j0, f);
            if (kInt8 && !first) tmem_ld<kW>(tI + j0, r);
            tmem_ld_wait();
            if (q == 0 && lane == 0) I8_TRACE(3, tn, 41);
            // row scales of this slice's tokens: one coalesced load, broadcast by shuffles
            float ra_lane = 0.0f;
            if (kInt8) {
              const int tk = n0 + j0 + lane;
              if (lane < kW && tk < p.T) ra_lane = __ldg(&p.rowabs[tk]);
            }
            if (lane == 0) bulk_wait_group_read0();  // the staging box is free again
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kW; ++j) {
              float y;
              if constexpr (kInt8) {
                int acc;
                float fo = 0.0f;
                if (is_out) {
                  acc = (int)r[j];
                  fo = __uint_as_float(f[j]);
                } else {
                  acc = __float2int_rn(__uint_as_float(f[j])) + (first ? 0 : (int)r[j]);
                }
                const float ra = __shfl_sync(0xffffffffu, ra_lane, j);
                y = (float)acc * (ra * so) + fo + bo;
                if constexpr (kDebug) r[j] = (uint32_t)acc;
              } else {
                y = __uint_as_float(f[j]) + bo;
              }
              st_shared_u16(stg + (j * 32 + lane) * 2, __half_as_ushort(__float2half_rn(y)));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (q == 0 && lane == 0) I8_TRACE(3, tn, 42);
            if (p.y_tma) {
              // one TMA store of the [kW tokens][32 features] box per warp
              if (lane == 0) {
                tma_store_2d(&tmY, stage, m0 + q * 32, n0 + j0);
                bulk_commit_group();
              }
            } else {
              // Y's row pitch is not a multiple of 16 bytes: copy the box out lane by lane
#pragma unroll 1
              for (int j = 0; j < kW; ++j) {
                const int tok = n0 + j0 + j;
                if (o_ok && tok < p.T)
                  p.Y[(size_t)tok * p.out + o] =
                      reinterpret_cast<const uint16_t*>(stage)[j * 32 + lane];
              }
              __syncwarp();
            }
            if constexpr (kDebug) {
#pragma unroll
              for (int j = 0; j < kW; ++j) {
                const int tok = n0 + j0 + j;
                if (o_ok && tok < p.T) p.acc_debug[(size_t)tok * p.out + o] = (int)r[j];
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pp.tmem_empty);
        if (q == 0 && lane == 0) I8_TRACE(3, tn, last ? 33 : 32);
      }
    }
    if (lane == 0) bulk_wait_group0();  // output stores complete before the CTA exits
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem_base, L::kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
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

template <int BN, int kMode>
cudaError_t launch_mode(cudaStream_t s, const CUtensorMap& mA8, const CUtensorMap& mA16,
                        const CUtensorMap& mB, const CUtensorMap& mWo, const CUtensorMap& mXo,
                        const CUtensorMap& mY, const Params& p, int grid) {
  using L = Smem<BN>;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
  if (e != cudaSuccess) return e;
  gemm_kernel<BN, kMode><<<grid, kThreads, L::total, s>>>(mA8, mA16, mB, mWo, mXo, mY, p);
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_bn(const GemmArgs& a, cudaStream_t s) {
  using L = Smem<BN>;
  CUtensorMap mA8, mA16, mB, mWo, mXo, mY;
  const bool i8 = a.a_int8 != nullptr;
  bool ok = true;
  // Maps that a path does not read still need to be valid descriptors: reuse B.
  ok &= make_map(&mB, a.b_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.in, BN, BK,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (i8) {
    ok &= make_map(&mA8, a.a_int8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.out, a.in, BM, BK,
                   CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= make_map(&mWo, a.wout, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.out, a.ncap, BM, BK,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= make_map(&mXo, a.xout, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.ncap, BN, BK,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    mA16 = mWo;
  } else {
    ok &= make_map(&mA16, a.a_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.out, a.in, BM, BK,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    mA8 = mB;
    mWo = mB;
    mXo = mB;
  }
  // Y [T, out] fp16 through TMA stores when its row pitch is a multiple of 16 bytes.
  const bool y_tma = (a.out % 8) == 0;
  if (y_tma)
    ok &= make_map(&mY, a.Y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.out, L::kW, 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mY = mB;
  if (!ok) return cudaErrorInvalidValue;
  Params p{};
  p.T = a.T;
  p.in = a.in;
  p.out = a.out;
  p.m_tiles = (a.out + BM - 1) / BM;
  p.n_tiles = (a.T + BN - 1) / BN;
  p.nkb = (a.in + BK - 1) / BK;
  p.nchunks = num_chunks(a.in);
  p.int8_path = i8 ? 1 : 0;
  p.y_tma = y_tma ? 1 : 0;
  p.hdr = a.hdr;
  p.rowabs = a.rowabs;
  p.l1 = a.l1;
  p.scb = a.scb;
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.Y = static_cast<uint16_t*>(a.Y);
  p.acc_debug = a.acc_debug;
  p.timeout_ns = a.timeout_ns;
  p.debug_skip_loads = a.debug_skip_loads;
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < kSmCount ? tiles : kSmCount;
  if (!i8) return launch_mode<BN, 0>(s, mA8, mA16, mB, mWo, mXo, mY, p, grid);
  if (a.acc_debug) return launch_mode<BN, 2>(s, mA8, mA16, mB, mWo, mXo, mY, p, grid);
  return launch_mode<BN, 1>(s, mA8, mA16, mB, mWo, mXo, mY, p, grid);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  switch (gemm_bn(a.T)) {
    case 16: return launch_bn<16>(a, s);
    case 32: return launch_bn<32>(a, s);
    case 64: return launch_bn<64>(a, s);
    case 128: return launch_bn<128>(a, s);
    default: return launch_bn<256>(a, s);
  }
}

}  // namespace i8mm

#ifdef I8MM_TRACE
// Trace build only: points CTA 0's timestamp records at a device buffer of 4 x 2^16 u64.
extern "C" __attribute__((visibility("default"))) int i8_trace_set(void* buf) {
  return cudaMemcpyToSymbol(i8mm::g_i8_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
#endif
