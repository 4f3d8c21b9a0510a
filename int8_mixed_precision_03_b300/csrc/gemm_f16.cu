// Our own fp16 GEMM on tcgen05: Y = X . W^T + bias with fp32 accumulation. It is the
// 16-bit comparator for the speed trade-off of the int8 matmul that the pages discuss
// ("Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section
// "speed"; "LLM.int8() summary" (zenn), section "INT8 speed").
//
// Tile: M = 128 output features (TMEM lanes) x N = BN tokens (TMEM columns), K stage 64.
// A = W fp16 [out, in] and B = X fp16 [T, in], both by TMA with the 128-byte swizzle,
// K-major, read by the MMA from shared memory. Two accumulators (2 x BN TMEM columns)
// alternate between tiles, so the epilogue of one tile overlaps the MMAs of the next.
// Epilogue: fp16(acc + bias[o]), optionally through ReLU (the fp16 FFN block), staged per
// warp in shared memory, written by TMA stores.
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 4-7 epilogue. Persistent CTAs, one per SM, tiles token-block fastest.
#include "gemm_common.cuh"

namespace i8mm {
namespace gemm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpEpi0 = 4;
constexpr int kStages = 4;

template <int BN>
struct CfgF {
  static constexpr int kW = BN < 32 ? BN : 32;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kBoxBytes = kW * 32 * 2;
  static constexpr uint32_t kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN;  // power of two >= 32
  static constexpr int a = 0;
  static constexpr int b = a + kStages * kA16Bytes;
  static constexpr int box = b + kStages * kBBytes;
  static constexpr int bars = box + 4 * 2 * kBoxBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * 2 + 1;  // full, empty; tmem full/empty; done
  static constexpr int misc = bars + kNumBars * 8;
  static constexpr int total = misc + 16 + 1024;
  static_assert(b % 1024 == 0 && kBBytes % 1024 == 0, "alignment");
  static_assert(total <= kMaxSmem, "shared memory per CTA");
};

struct ParamsF {
  int T, in, out;
  int m_tiles, n_tiles, nkb;
  int y_tma;
  const uint16_t* bias;
  uint16_t* Y;
  int relu;  // ReLU on Y (the fp16 FFN's up projection)
  uint64_t timeout_ns;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    f16_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmY, const ParamsF p) {
  using C = CfgF<BN>;
  constexpr int kW = C::kW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* done = tmem_empty + 2;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::misc);
  const Abort ab{reinterpret_cast<volatile int*>(smem + C::misc + 4), nullptr, p.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 4);
    }
    mbar_init(done, 1);
    *ab.flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmY);
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_base_smem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;
  const int tiles = p.m_tiles * p.n_tiles;
  const uint32_t sbase = smem_u32(smem);

  if (warp == kWarpTma) {
    if (lane == 0) {
      // X (the B operand) is re-read by every weight strip: keep it in L2 across waves
      const uint64_t keep = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t / p.n_tiles) * BM, n0 = (t % p.n_tiles) * BN;
        for (int kb = 0; kb < p.nkb && ok; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!(ok = pipe_wait(&empty[s], ph ^ 1u, ab))) break;
          mbar_arrive_expect_tx(&full[s], kA16Bytes + C::kBBytes);
          tma_load_2d(smem + C::a + s * kA16Bytes, &tmA, &full[s], kb * BK, m0);
          tma_load_2d_hint(smem + C::b + s * C::kBBytes, &tmB, &full[s], kb * BK, n0, keep);
        }
      }
      for (uint32_t k = 0; k < (uint32_t)kStages && k < it; ++k) {
        const uint32_t j = it - 1 - k;
        mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32acc(BM, BN);
      uint32_t it = 0, nt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++nt) {
        const uint32_t b = nt & 1u;
        if (!(ok = pipe_wait(&tmem_empty[b], ((nt >> 1) & 1u) ^ 1u, ab))) break;
        tc_fence_after();
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!(ok = pipe_wait(&full[s], ph, ab))) break;
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(sbase + C::a + s * kA16Bytes);
          const uint64_t bd = sdesc_kmajor_sw128(sbase + C::b + s * C::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss(tmem_base + b * BN, ad + 2 * k, bd + 2 * k, idesc,
                       (kb == 0 && k == 0) ? 0u : 1u);
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&tmem_full[b]);
      }
      mma_commit(done);
      mbar_wait_bounded(done, 0, p.timeout_ns);
    }
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;
    const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
    uint8_t* boxes = smem + C::box + q * 2 * C::kBoxBytes;
    const CUtensorMap* mapY = p.y_tma ? &tmY : nullptr;
    const uint64_t y_policy = l2_policy_evict_first();
    uint32_t nt = 0, slot = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++nt) {
      const int m0 = (t / p.n_tiles) * BM, n0 = (t % p.n_tiles) * BN;
      const int o = m0 + q * 32 + lane;
      const float bo = (o < p.out && p.bias) ? __half2float(__ushort_as_half(p.bias[o])) : 0.0f;
      const uint32_t b = nt & 1u;
      if (!(ok = pipe_wait(&tmem_full[b], (nt >> 1) & 1u, ab))) break;
      tc_fence_after();
#pragma unroll 1
      for (int j0 = 0; j0 < BN; j0 += kW) {
        uint32_t f[kW];
        tmem_ld<kW>(tq + b * BN + j0, f);
        tmem_ld_wait();
        uint32_t yh[kW / 2];
#pragma unroll
        for (int j = 0; j < kW; ++j) {
          float v = __uint_as_float(f[j]) + bo;
          if (p.relu) v = fmaxf(v, 0.0f);
          const uint32_t h = __half_as_ushort(__float2half_rn(v));
          yh[j / 2] = (j & 1) ? (yh[j / 2] | (h << 16)) : h;
        }
        box_reuse_wait(lane);
        box_store<kW>(boxes + slot * C::kBoxBytes, yh, mapY, p.Y, p.T, p.out, m0 + 32 * q,
                      n0 + j0, lane, y_policy);
        slot ^= 1u;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[b]);
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int BN>
cudaError_t launch_f16_bn(const GemmArgs& a, cudaStream_t s) {
  using C = CfgF<BN>;
  CUtensorMap mA, mB, mY;
  bool ok = true;
  ok &= make_map(&mA, a.a_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.out, a.in, BM, BK,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= make_map(&mB, a.b_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.in, BN, BK,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  const bool y_tma = (a.out % 8) == 0;
  if (y_tma)
    ok &= make_map(&mY, a.Y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.out, C::kW, 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mY = mB;  // a valid descriptor that is never used
  if (!ok) return cudaErrorInvalidValue;
  ParamsF p{};
  p.T = a.T;
  p.in = a.in;
  p.out = a.out;
  p.m_tiles = (a.out + BM - 1) / BM;
  p.n_tiles = (a.T + BN - 1) / BN;
  p.nkb = (a.in + BK - 1) / BK;
  p.y_tma = y_tma ? 1 : 0;
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.Y = static_cast<uint16_t*>(a.Y);
  p.relu = a.relu;
  p.timeout_ns = a.timeout_ns;
  const int tiles = p.m_tiles * p.n_tiles;
  const int sms = sm_count();
  const int grid = tiles < sms ? tiles : sms;
  cudaError_t e = cudaFuncSetAttribute(f16_gemm_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::total);
  if (e != cudaSuccess) return e;
  f16_gemm_kernel<BN><<<grid, kThreads, C::total, s>>>(mA, mB, mY, p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace gemm

cudaError_t launch_f16_gemm(const GemmArgs& a, cudaStream_t s) {
  const int T = a.T;
  if (T <= 16) return gemm::launch_f16_bn<16>(a, s);
  if (T <= 32) return gemm::launch_f16_bn<32>(a, s);
  if (T <= 64) return gemm::launch_f16_bn<64>(a, s);
  if (T <= 128) return gemm::launch_f16_bn<128>(a, s);
  return gemm::launch_f16_bn<256>(a, s);
}

}  // namespace i8mm
