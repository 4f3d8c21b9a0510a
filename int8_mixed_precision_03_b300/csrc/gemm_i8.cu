// Tensor-core matmul of the LLM.int8() method (steps 2 and 3) on tcgen05.
//
// "Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
// idea": the int8 part is multiplied with int8 vector-wise scales, the outlier part in
// fp16, and the int8 result is dequantized and added to the fp16 result.
// "LLM.int8() summary" (zenn), section "method": outlier input dimensions and the matching
// weight dimensions are split off and kept in 16 bit.
//
// Exact int8 products on the fp16 tensor path. sm_103a has no int8 tcgen05 MMA (ptxas
// rejects .kind::i8 for this target), so the int8 product runs on .kind::f16: int8 codes
// are exact fp16 values and fp32 sums of integers are exact while every partial sum stays
// within 2^24 in magnitude. The K loop is cut into 1024-element chunks; for each (token
// tile, chunk) the quantize pass records L1 = max over the tile's rows of sum |code|, and
// since |CB| <= 127 every partial sum of a run of chunks is bounded by 127 * (sum of their
// L1). Consecutive chunks share one fp32 accumulation ("segment") while that bound stays
// <= 2^24; a single chunk always fits (127 * 127 * 1024 < 2^24). At a segment boundary the
// epilogue converts the fp32 tile to int32 and adds it to a running int32 sum.
//
// Tile: M = 128 output features (TMEM lanes) x N = BN tokens (TMEM columns); a pipeline
// stage is one 64-K block, or four for token tiles of at most 64 (below).
//   A = CB int8 [out, in]: streamed by TMA into a weight ring of its own (64-byte-wide boxes
//       with the 64-byte swizzle; 128-byte-wide boxes with the 128-byte swizzle when a stage
//       holds several K blocks); two sets of four converter warps (alternate stages) turn
//       each 128 x 64 block into fp16, stored in the 128-byte-swizzled K-major layout in
//       shared memory, or, for token tiles of at most 64, into TMEM (tcgen05.st; the MMAs
//       then read A from TMEM). The outlier weight slice W_out fp16 [out, ncap] takes the
//       same route as two boxes per stage, copied without conversion.
//   B = activation codes as fp16 [T, in] (written by the quantize pass), or the outlier
//       slice X_out fp16 [T, ncap]: TMA, 128-byte swizzle, K-major, one box per K block.
//   A and B stages form one ring, released by one MMA commit per stage. The MMA issuer
//   waits on one barrier per stage (full_a): a converter warp completes its share of it
//   only once the stage's B has landed (full_b).
// For small token tiles an MMA takes about 56 cycles while each barrier query and each
// step of the issuing thread's own loop takes tens of cycles, so stages hold four K blocks
// (16 MMAs) there, and the issuer's loop over a chunk's stages does nothing but wait, issue,
// commit and advance the stage.
// TMEM: two accumulators F0 [0, BN) and F1 [BN, 2BN) take the segments in turn (the int
// segments of a tile, then its outlier segment if it has one, then the next tile's), so the
// epilogue of one segment overlaps the MMAs of the next. The epilogue's running int32 sum of
// a tile lives in a per-CTA slot of the workspace (L2 resident): a segment that is not the
// last of its tile is folded into it, and the tile's last segment reads it back.
// Outlier product: with at most kCcOut outlier columns (the usual case: about 0.1% of the
// hidden dimensions) the epilogue computes it on the CUDA cores, sum_k X_out[t,k] W_out[o,k]
// in fp32 from a token-contiguous transposed copy of X_out and this feature's W_out row
// held in registers. On the whole-tile schedule the four epilogue warps copy the tile's rows
// of that copy into shared memory once per tile and each 16-token slice reads them with
// broadcast loads; on the split schedule lane k loads row k of a slice and shuffles pass it
// on (shuffles compete with the mainloop's shared-memory traffic). A tile then has no short
// outlier segment after its long int segment, so the next tile's MMAs never wait for the
// epilogue to drain the int accumulator. With more outlier columns they run as the tile's
// last MMA segment (fp16 operands, fp32 accumulation in TMEM) of ceil(n/64) K blocks.
// Epilogue: Y[t, o] = fp16(acc * rowabs[t] * SCB[o] / 127^2 + outlier + bias[o]), staged
// per warp in shared memory (two boxes of tokens x 32 features) and written by TMA stores.
// The tokens' row scales come from a per-tile copy in shared memory on the whole-tile
// schedule (broadcast loads, four per 16-token slice), from shuffles otherwise.
// L2 policy: the activation codes, re-read by every weight strip, are loaded evict-last,
// and Y, written once, is stored evict-first, so that the codes stay in L2 across waves.
// With zeropoint activation codes (x ~ (q + Z)/S per token, "LLM.int8() summary" (zenn),
// "Zeropoint Quantization") the epilogue adds Z_t times the feature's code sum over the
// inlier columns to the exact int32 product before scaling by rowabs = 127/S: in int32
// when |Z| is small enough for every token of a 32-token group, in 64 bits otherwise.
// When Y is the input of a following int8 matmul (an FFN's up projection), the epilogue
// also applies the activation (ReLU or none) and computes that matmul's outlier flags:
// each lane owns one column of Y, keeps the largest fp16 magnitude over the tile's valid
// tokens, and the warp ORs one 32-column mask word per tile (step 1 of the next matmul
// without reading Y again).
//
// Warp roles (512 threads): warp 0 TMA for B, warp 1 MMA issuer and TMEM owner, warp 2 TMA
// for the weight stream, warps 4-7 and 12-15 converters, warps 8-11 epilogue (warp w
// reaches TMEM lanes 32*(w%4) .. +31). Persistent CTAs, one per SM, walk tiles
// token-block fastest so that concurrently running CTAs share the same weight strip in L2.
//
// CTA pairs: 256-token tiles on the whole-tile schedule run on clusters of two CTAs (two
// SMs) that share one tile of 256 output features x 256 tokens through tcgen05 cta_group::2
// MMAs with M = 256: CTA r (its rank in the pair) converts and holds A rows 128r .. 128r + 127
// and holds B rows (tokens) 128r .. 128r + 127, and its TMEM receives its 128 feature rows of
// the accumulator for all 256 tokens. The even CTA issues the MMAs; both CTAs' B halves
// complete on its barrier (TMA with .cta_group::2), the odd CTA's converter and epilogue
// warps arrive on its barriers remotely, and its commits reach both CTAs (multicast). Per
// SM the tensor core reads half of B per K block instead of all of it, which halves the
// operand traffic of the shared-memory port and lets B stages be half as large. The
// epilogue is unchanged: each CTA writes its own 128 features.
//
// Schedules: whole tiles per CTA (t = b, b + G, ...), or, where that leaves the last wave
// unbalanced (i8_split_ctas), the split schedule (kSplit): the (tile, 1024-K chunk) units
// are cut into one contiguous range per CTA, and a tile cut into pieces is finished by the
// last of its pieces to arrive, from the exact int32 sums (and the tile-ending piece's fp32
// outlier sums) the pieces leave in their CTAs' slots. No CTA ever waits for another.
#include "gemm_common.cuh"

namespace i8mm {
namespace gemm {
namespace {

constexpr int kThreads = 512;
constexpr int kWarpB = 0, kWarpMma = 1, kWarpA8 = 2;
constexpr int kWarpConv0 = 4, kWarpEpi0 = 8, kWarpConv1 = 12;
constexpr uint32_t kExactLimit = 1u << 24;                    // integers exact in fp32
// Up to this many outlier columns the epilogue adds the outlier product on the CUDA cores;
// beyond it the outlier product runs as the tile's last MMA segment (see the file comment).
constexpr int kCcOut = kCcOutlierCols;
static_assert(kCcOut == 32, "one transposed X_out row per lane");
// Largest outlier count sent to the CUDA-core path (<= kCcOut): above it the outlier
// product is cheaper as an MMA segment than as per-element work in the epilogue.
constexpr int kCcMaxDefault = 32;
// 256-token tiles run on CTA pairs (cta_group::2) unless this is set.
constexpr bool kDisablePairs = false;
constexpr uint32_t kWorstChunkBound = 127u * 127u * kChunkK;  // < kExactLimit
static_assert(kWorstChunkBound <= kExactLimit, "one chunk must always be exact");

// Token tiles up to this size keep the converted weights (A) in TMEM instead of shared
// memory: the two accumulators of a small tile leave room for the A stages.
constexpr int kATmemMaxBN = 64;
// K blocks per stage of those tiles (2 or 4; with 4, three stages fill TMEM). Measured on
// the 176B decode shape (64 tokens x 14336 -> 57344): one K block 264 us, two 209 us, four
// 191 us.
constexpr int kATKBlocks = 4;
// a 128-row x 128-byte weight box in shared memory
constexpr int kBox8Bytes = 128 * 128;

// Selects the zeropoint epilogue's 64-bit form (true) or its int32 form (false) at compile
// time, so that a slice's loop carries only one of them.
template <bool B>
struct Wide {
  static constexpr bool value = B;
};

template <int BN, bool kPair = false>
struct Cfg {
  static constexpr int kW = 16;  // tokens per epilogue slice
  // A stages in TMEM (small token tiles): the converters write them with tcgen05.st and the
  // MMA reads A from TMEM, so shared memory holds only B and the int8 weight ring.
  static constexpr bool kAT = !kPair && BN <= kATmemMaxBN;
  // K blocks (64 K each) per pipeline stage: kATKBlocks for the A-in-TMEM tiles, whose
  // weight boxes are then 128 bytes wide (whole 128-byte lines) and whose roles wait, arrive
  // and commit once per 16 or 32 KB of weights; one otherwise.
  // Ring depths (kStages, kStages8): A (fp16, in TMEM or shared memory) + B in one ring of
  // stages, the int8 weight stream in its own ring of slots; with A in TMEM both hold 12 K
  // blocks. A CTA of a pair holds half of the tile's B rows, so its stages are half as large
  // and it affords one more of them.
  static constexpr int kKB = kAT ? kATKBlocks : 1;
  static constexpr int kA8Slot = kKB * kA8Bytes;       // one weight-ring slot
  static constexpr int kBoxKB = kKB >= 2 ? 2 : 1;      // K blocks per weight box
  static constexpr int kSub = kKB / kBoxKB;            // weight boxes per slot
  static constexpr int kStages = kAT ? 12 / kKB : kPair ? 4 : BN == 256 ? 3 : 4;
  static constexpr int kStages8 = kAT ? 12 / kKB : BN == 256 ? 8 : BN == 128 ? 6 : BN == 64 ? 10 : 12;
  static constexpr int kBRows = kPair ? BN / 2 : BN;  // B rows (tokens) in this CTA's stages
  static constexpr int kBBytes = kBRows * BK * 2;     // B of one K block
  static constexpr int kBStage = kKB * kBBytes;
  static constexpr int kBoxBytes = kW * 32 * 2;
  // TMEM: F0 + F1 (2 BN columns), then with kAT the A stages, 32 columns per K block (128
  // lanes x 64 fp16 K values, two per column)
  static constexpr uint32_t kAcol0 = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr uint32_t kTmemCols = kAT ? 512 : 2 * BN <= 32 ? 32 : 2 * BN;
  static_assert(!kAT || kAcol0 + 32 * kKB * kStages <= 512, "TMEM columns");
  // shared memory (stage bases 1024-byte aligned for the swizzled layouts)
  static constexpr int a16 = 0;
  static constexpr int b = a16 + (kAT ? 0 : kStages * kA16Bytes);
  static constexpr int a8 = b + kStages * kBStage;
  static constexpr int box = a8 + kStages8 * kA8Slot;
  // the tile's transposed X_out rows (CUDA-core outlier product, whole-tile schedule), where
  // they fit: [kCcOut rows][BN tokens] fp16
  static constexpr int xo = box + 4 * 2 * kBoxBytes;
  static constexpr int kXoWant = kCcOut * BN * 2 + BN * 4;  // + the tile's row scales
  static constexpr int kXoBytes =
      xo + kXoWant + (3 * kStages + 2 * kStages8 + 6) * 8 + 16 + 1024 <= kMaxSmem ? kXoWant : 0;
  static constexpr int bars = xo + kXoBytes;
  // full_a, full_b, empty [kStages]; a8_full, a8_empty [kStages8]; tmem_full,
  // tmem_empty [2]; done; epi (the four epilogue warps' rendezvous of split tiles)
  static constexpr int kNumBars = 3 * kStages + 2 * kStages8 + 2 * 2 + 2;
  static constexpr int misc = bars + kNumBars * 8;
  static constexpr int total = misc + 16 + 1024;  // + alignment slack
  static_assert(b % 1024 == 0 && kBBytes % 1024 == 0 && a8 % 1024 == 0, "alignment");
  static_assert(total <= kMaxSmem, "shared memory per CTA");
};

struct Params {
  int T, in, out;
  int m_tiles, n_tiles, nkb;  // nkb = ceil(in / 64)
  int nchunks;                // ceil(in / 1024)
  int y_tma;                  // 1: Y written by TMA stores (out % 8 == 0)
  WsHeader* hdr;
  const float* rowabs;
  const int32_t* l1;
  int32_t* acc_scratch;       // [gridDim.x][BN][128] int32
  const float* scb;
  const uint16_t* bias;
  uint16_t* Y;
  int32_t* acc_debug;
  uint32_t* next_mask;        // FFN up projection: the next matmul's outlier mask
  uint32_t next_thr;          // its threshold as fp16 magnitude bits
  int next_relu;              // ReLU on Y before the statistics
  int z_safe;                 // zeropoint: |Z| up to which acc + Z * cbin fits in int32
  const int32_t* zi;          // zeropoint variant: per-token zero points [T]
  const int32_t* cbsum;       // and per-feature code sums over all / outlier columns
  const int32_t* cbout;
  // split schedule (split != 0): units are (tile, 1024-K chunk) in tile-major order and
  // CTA b takes units [units*b/G, units*(b+1)/G); tiles cut between CTAs finish through
  // the part slots and a per-tile arrival counter (the last piece to arrive writes Y)
  int split;
  long long units;
  int32_t* part;              // [G][2][BN][128] int32: a CTA's first / last piece's sums
  float* part_f;              // [G][BN][128] fp32: outlier sums of a tile-ending piece
  int32_t* tile_cnt;          // [tiles] arrivals, zeroed per call
  // outlier product on the CUDA cores (0 < n_out <= kCcOut): W_out [out, ncap] and X_out
  // transposed, xoT [kCcOut][xo_stride] (token-contiguous rows, zeros past n_out)
  const uint16_t* wout;
  int ncap;
  const uint16_t* xoT;
  int xo_stride;
  int cc_max;                 // outlier counts 1 .. cc_max take the CUDA-core path
  uint64_t timeout_ns;
  int debug_skip_loads;
};

// The pieces of work of one CTA: whole tiles t = b, b + G, ... (unsplit), or the runs of
// its unit range that fall in one tile (split). A piece is (tile t, chunks [c0, c1)); its K
// blocks are [16 c0, min(16 c1, nkb)) plus the outlier K blocks when c1 == nchunks.
// First tile and tile stride of this CTA's whole-tile schedule: CTA b of a single-CTA grid,
// or the pair (cluster) b / 2 of a grid of CTA pairs, whose two CTAs work on the same tiles.
template <bool kPair>
__device__ __forceinline__ int tile_first() { return kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x; }
template <bool kPair>
__device__ __forceinline__ int tile_stride() { return kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x; }

template <bool kSplit, bool kPair = false>
struct Sched {
  long long u = 0, ue = 0;
  int t = 0;
  __device__ explicit Sched(const Params& p) {
    if constexpr (kSplit) {
      u = p.units * blockIdx.x / gridDim.x;
      ue = p.units * (blockIdx.x + 1) / gridDim.x;
    } else {
      t = tile_first<kPair>();
    }
  }
  __device__ bool next(const Params& p, int& tt, int& c0, int& c1) {
    if constexpr (!kSplit) {
      if (t >= p.m_tiles * p.n_tiles) return false;
      tt = t;
      c0 = 0;
      c1 = p.nchunks;
      t += tile_stride<kPair>();
      return true;
    }
    if (u >= ue) return false;
    tt = (int)(u / p.nchunks);
    c0 = (int)(u % p.nchunks);
    const long long e = min(ue, (long long)(tt + 1) * p.nchunks);
    c1 = c0 + (int)(e - u);
    u = e;
    return true;
  }
};
// First unit of CTA b, and the CTA that owns unit u, under the split schedule.
__device__ __forceinline__ long long unit_start(const Params& p, int b) {
  return p.units * b / gridDim.x;
}
__device__ __forceinline__ int unit_owner(const Params& p, long long u) {
  return (int)(((u + 1) * gridDim.x + p.units - 1) / p.units - 1);
}

// Epilogue variants: plain, plain + int32 export, activation + next matmul's column flags,
// zeropoint codes (acc + zi[t] * inlier code sum of feature o), the same + int32 export.
enum EpiMode { kEpiPlain = 0, kEpiDebug = 1, kEpiNext = 2, kEpiZp = 3, kEpiZpDebug = 4 };

__device__ __forceinline__ int outlier_count(const Params& p) {
  return *reinterpret_cast<volatile const int*>(&p.hdr->n_out_used);
}
// The outlier columns are multiplied on the CUDA cores in the epilogue when there are at
// most kCcOut of them (and the transposed slice was written); otherwise, and in every role
// alike, they form the tile's last MMA segment of ceil(n/64) K blocks.
__device__ __forceinline__ bool cc_outliers(const Params& p, int n) {
  return p.xoT != nullptr && n > 0 && n <= p.cc_max;
}

// This lane's outlier weights W_out[o, 0 .. kCcOut) as fp16 pairs (W_out is zero past the
// outlier count; a feature beyond `out` gets zeros).
__device__ __forceinline__ void load_cc_weights(const Params& p, int o, bool o_ok, int n,
                                                uint32_t (&wh)[kCcOut / 2]) {
#pragma unroll
  for (int c = 0; c < kCcOut / 8; ++c) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (o_ok && 8 * c < n) v = __ldg(reinterpret_cast<const uint4*>(p.wout + (size_t)o * p.ncap) + c);
    wh[4 * c + 0] = v.x;
    wh[4 * c + 1] = v.y;
    wh[4 * c + 2] = v.z;
    wh[4 * c + 3] = v.w;
  }
}

// lo += x.lo * w, hi += x.hi * w for the two fp16 values of x (low and high half) and the
// fp16 weight in half `wsel` of w2: fp16 products are exact in fp32 and each sum is rounded
// once, as fmaf on the converted values would.
__device__ __forceinline__ void fma2_f16_f32(float& lo, float& hi, uint32_t x, uint32_t w2,
                                             int wsel) {
  if (wsel)
    asm("{\n.reg .f16 xl, xh, wl, wh;\n"
        "mov.b32 {xl, xh}, %2;\n"
        "mov.b32 {wl, wh}, %3;\n"
        "fma.rn.f32.f16 %0, xl, wh, %0;\n"
        "fma.rn.f32.f16 %1, xh, wh, %1;\n}"
        : "+f"(lo), "+f"(hi)
        : "r"(x), "r"(w2));
  else
    asm("{\n.reg .f16 xl, xh, wl, wh;\n"
        "mov.b32 {xl, xh}, %2;\n"
        "mov.b32 {wl, wh}, %3;\n"
        "fma.rn.f32.f16 %0, xl, wl, %0;\n"
        "fma.rn.f32.f16 %1, xh, wl, %1;\n}"
        : "+f"(lo), "+f"(hi)
        : "r"(x), "r"(w2));
}

// The transposed X_out rows of a slice of 16 tokens tok0 .. tok0 + 15: lane k loads row k
// (outlier column k, 32 bytes), so one coalesced load per lane brings the whole slice; rows
// k >= n and slices past the last token are zero.
__device__ __forceinline__ void cc_load_rows(const Params& p, int tok0, int n, int lane,
                                             uint4& a, uint4& b) {
  a = make_uint4(0u, 0u, 0u, 0u);
  b = a;
  if (lane < n && tok0 < p.T) {
    const uint4* src = reinterpret_cast<const uint4*>(p.xoT + (size_t)lane * p.xo_stride + tok0);
    a = __ldg(src);
    b = __ldg(src + 1);
  }
}

// The same product with the slice's rows read from the tile's staged copy in shared memory
// (row k of the tile at xo + k * pitch bytes, tokens from the slice's first): every lane
// reads the same 32 bytes per row (broadcast loads), so no shuffles are needed.
__device__ __forceinline__ void cc_outlier_slice_smem(int n, const uint32_t (&wh)[kCcOut / 2],
                                                      uint32_t xo, uint32_t pitch,
                                                      float (&fo)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) fo[j] = 0.0f;
#pragma unroll
  for (int k0 = 0; k0 < kCcOut; k0 += 4) {
    if (k0 >= n) break;
    uint4 xa[4], xb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t a = xo + (uint32_t)(k0 + u) * pitch;
      xa[u] = ld_shared_v4(a);
      xb[u] = ld_shared_v4(a + 16);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u;
      const uint32_t w2 = wh[k >> 1];
      const uint32_t xw[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w,
                              xb[u].x, xb[u].y, xb[u].z, xb[u].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) fma2_f16_f32(fo[2 * e], fo[2 * e + 1], xw[e], w2, k & 1);
    }
  }
}

// Outlier product of the 16 tokens of a slice for this lane's feature:
// fo[j] = sum_{k < n} X_out[tok0 + j, k] * W_out[o, k], fp32 fused multiply-adds in
// ascending k, so every schedule gives the same bits. Row k of the slice (loaded by lane k
// with cc_load_rows) reaches every lane by shuffles; rows n .. are zero, so steps of four
// columns need no mask (n is the same for the whole warp).
__device__ __forceinline__ void cc_outlier_slice(int n, const uint32_t (&wh)[kCcOut / 2],
                                                 const uint4& a, const uint4& b,
                                                 float (&fo)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) fo[j] = 0.0f;
#pragma unroll
  for (int k0 = 0; k0 < kCcOut; k0 += 4) {
    if (k0 >= n) break;
#pragma unroll
    for (int k = k0; k < k0 + 4; ++k) {
      const uint32_t w2 = wh[k >> 1];
      const uint32_t xw[8] = {__shfl_sync(0xffffffffu, a.x, k), __shfl_sync(0xffffffffu, a.y, k),
                              __shfl_sync(0xffffffffu, a.z, k), __shfl_sync(0xffffffffu, a.w, k),
                              __shfl_sync(0xffffffffu, b.x, k), __shfl_sync(0xffffffffu, b.y, k),
                              __shfl_sync(0xffffffffu, b.z, k), __shfl_sync(0xffffffffu, b.w, k)};
#pragma unroll
      for (int e = 0; e < 8; ++e) fma2_f16_f32(fo[2 * e], fo[2 * e + 1], xw[e], w2, k & 1);
    }
  }
}

// Bound on |partial sums| of chunk c for token tile n_blk (see the file comment).
__device__ __forceinline__ uint32_t chunk_bound(const Params& p, int n_blk, int c) {
  if (!p.l1) return kWorstChunkBound;
  return 127u * (uint32_t)__ldg(&p.l1[(size_t)n_blk * p.nchunks + c]);
}
// Greedy rule shared by the MMA issuer and the epilogue: chunk c opens a new segment when
// it is the first chunk of a piece or adding its bound would exceed 2^24.
struct SegWalker {
  uint32_t run = 0;
  __device__ __forceinline__ bool opens(uint32_t b, bool first) {
    if (first || run + b > kExactLimit) { run = b; return true; }
    run += b;
    return false;
  }
};
__device__ __forceinline__ int count_int_segments(const Params& p, int n_blk, int c0, int c1) {
  SegWalker w;
  int n = 0;
  for (int c = c0; c < c1; ++c) n += w.opens(chunk_bound(p, n_blk, c), c == c0) ? 1 : 0;
  return n;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Pipeline waits (the same in a CTA pair: see mbar_arrive_cluster for the arrivals).
template <bool kPair>
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, const Abort& ab) {
  return pipe_wait(bar, parity, ab);
}
template <bool kPair>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t ns) {
  return mbar_wait_bounded(bar, parity, ns);
}
// Arrival on a barrier of the pair's even CTA (the MMA issuer's), or a local arrival.
template <bool kPair>
__device__ __forceinline__ void arrive_leader(uint64_t* bar) {
  if constexpr (kPair) {
    if (cluster_ctarank() == 0) mbar_arrive(bar);
    else mbar_arrive_cluster(mapa_rank(bar, 0));
  } else {
    mbar_arrive(bar);
  }
}

template <int BN, int kMode, bool kSplit, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    i8_gemm_kernel(const __grid_constant__ CUtensorMap tmA8, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmWo, const __grid_constant__ CUtensorMap tmXo,
                   const __grid_constant__ CUtensorMap tmY, const Params p) {
  static_assert(!kPair || (BN == 256 && !kSplit), "CTA pairs run 256-token whole tiles");
  using C = Cfg<BN, kPair>;
  constexpr int kS = C::kStages, kS8 = C::kStages8, kW = C::kW;
  // rank in the CTA pair (0 = the MMA issuer) and this CTA's share of a tile: feature rows
  // [128 rank, 128 rank + 128) of the 256 (pair) or 128 rows, B rows (tokens) likewise
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  constexpr int kFeatTile = kPair ? 2 * BM : BM;
  constexpr bool kDebug = kMode == kEpiDebug || kMode == kEpiZpDebug;
  constexpr bool kNext = kMode == kEpiNext;
  constexpr bool kZp = kMode == kEpiZp || kMode == kEpiZpDebug;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* full_b = full_a + kS;
  uint64_t* empty = full_b + kS;
  uint64_t* a8_full = empty + kS;
  uint64_t* a8_empty = a8_full + kS8;
  uint64_t* tmem_full = a8_empty + kS8;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* done = tmem_empty + 2;
  uint64_t* epi_bar = done + 1;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::misc);
  const Abort ab{reinterpret_cast<volatile int*>(smem + C::misc + 4), p.hdr, p.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(&full_a[s], kPair ? 8 : 4);  // the four warps of the converter set (each CTA's)
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kS8; ++s) {
      mbar_init(&a8_full[s], 1);
      mbar_init(&a8_empty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], kPair ? 8 : 4);  // one arrival per epilogue warp (each CTA's)
    }
    mbar_init(done, 1);
    mbar_init(epi_bar, 4);
    *ab.flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpB && lane == 0) {
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmXo);
    tma_prefetch_desc(&tmY);
  }
  if (warp == kWarpA8 && lane == 0) {
    tma_prefetch_desc(&tmA8);
    tma_prefetch_desc(&tmWo);
  }
  if (warp == kWarpMma) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_base_smem, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_base_smem, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers exist before any arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;

  const int tiles = p.m_tiles * p.n_tiles;
  // outlier columns: on the CUDA cores in the epilogue (n_cc of them), or as the tile's last
  // MMA segment (nkb_out K blocks); every role takes the same decision
  const int n_out_all = outlier_count(p);
  const bool cc = cc_outliers(p, n_out_all);
  const int n_cc = cc ? n_out_all : 0;
  const int nkb_out = cc ? 0 : (n_out_all + 63) / 64;
  // stages of kKB K blocks: a tile's int stages (the last one padded with zeros past K),
  // then its outlier stages; kChunkSt stages per 1024-K chunk
  constexpr int kKB = C::kKB;
  constexpr int kChunkSt = kChunkKBlocks / kKB;
  const int nst_int = (p.nkb + kKB - 1) / kKB;
  const int nst_all = nst_int + (nkb_out + kKB - 1) / kKB;
  const uint32_t sbase = smem_u32(smem);

  if (warp == kWarpB) {
    // -------------------------------------------------------- TMA: B operand
    if (lane == 0 && !p.debug_skip_loads) {
      // the activation codes are re-read by every weight strip: keep them in L2 across waves
      const uint64_t keep = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      Sched<kSplit, kPair> sc(p);
      int t, c0, c1;
      while (ok && sc.next(p, t, c0, c1)) {
        const int n0 = (t % p.n_tiles) * BN + (int)rank * C::kBRows;  // this CTA's B rows
        const int st_end = c1 == p.nchunks ? nst_all : c1 * kChunkSt;
        for (int st = c0 * kChunkSt; st < st_end && ok; ++st, ++it) {
          const uint32_t s = it % kS, ph = (it / kS) & 1u;
          if (!(ok = pwait<kPair>(&empty[s], ph ^ 1u, ab))) break;
          const bool is_int = st < nst_int;
          // first K (in elements) of the stage in B (activation codes) or X_out
          const int x0 = (is_int ? st : st - nst_int) * kKB * BK;
          if constexpr (kPair) {
            // both halves complete on the MMA issuer's barrier, which expects both
            if (rank == 0) mbar_arrive_expect_tx(&full_b[s], 2 * C::kBStage);
            const uint32_t bar = mapa_rank(&full_b[s], 0);
            for (int k = 0; k < kKB; ++k) {
              uint8_t* dst = smem + C::b + s * C::kBStage + k * C::kBBytes;
              tma_load_2d_pair(dst, is_int ? &tmB : &tmXo, bar, x0 + k * BK, n0, keep);
            }
          } else {
            mbar_arrive_expect_tx(&full_b[s], C::kBStage);
            for (int k = 0; k < kKB; ++k) {
              uint8_t* dst = smem + C::b + s * C::kBStage + k * C::kBBytes;
              if (is_int)
                tma_load_2d_hint(dst, &tmB, &full_b[s], x0 + k * BK, n0, keep);
              else
                tma_load_2d(dst, &tmXo, &full_b[s], x0 + k * BK, n0);
            }
          }
        }
      }
      // Do not leave the CTA with copies in flight: wait for the last issued stages (in a
      // pair the issuer's barrier counts both CTAs' copies, and the peer leaves only after
      // the issuer, at the final cluster barrier).
      if (rank == 0) {
        for (uint32_t k = 0; k < (uint32_t)kS && k < it; ++k) {
          const uint32_t j = it - 1 - k;
          wait_bounded<kPair>(&full_b[j % kS], (j / kS) & 1u, p.timeout_ns);
        }
      }
    }
  } else if (warp == kWarpA8) {
    // -------------------------------------------------------- TMA: weight stream
    // One 128 x 64 kKB int8 box per int stage; two 128 x 32 kKB fp16 boxes per outlier stage.
    if (lane == 0 && !p.debug_skip_loads) {
      uint32_t i8 = 0;
      bool ok = true;
      Sched<kSplit, kPair> sc(p);
      int t, c0, c1;
      while (ok && sc.next(p, t, c0, c1)) {
        const int m0 = (t / p.n_tiles) * kFeatTile + (int)rank * BM;
        const int st_end = c1 == p.nchunks ? nst_all : c1 * kChunkSt;
        for (int st = c0 * kChunkSt; st < st_end && ok; ++st) {
          const bool is_int = st < nst_int;
          const int nbox = is_int ? 1 : 2;
          for (int h = 0; h < nbox && ok; ++h, ++i8) {
            const uint32_t s8 = i8 % kS8, ph8 = (i8 / kS8) & 1u;
            if (!(ok = pipe_wait(&a8_empty[s8], ph8 ^ 1u, ab))) break;
            mbar_arrive_expect_tx(&a8_full[s8], C::kA8Slot);
#pragma unroll
            for (int b = 0; b < C::kSub; ++b) {  // boxes of 64 kBoxKB bytes side by side in K
              uint8_t* dst = smem + C::a8 + s8 * C::kA8Slot + b * (C::kA8Slot / C::kSub);
              if (is_int)
                tma_load_2d(dst, &tmA8, &a8_full[s8], (st * kKB + b * C::kBoxKB) * BK, m0);
              else
                tma_load_2d(dst, &tmWo, &a8_full[s8],
                            (st - nst_int) * kKB * BK + 32 * kKB * h + 32 * C::kBoxKB * b, m0);
            }
          }
        }
      }
      for (uint32_t k = 0; k < (uint32_t)kS8 && k < i8; ++k) {
        const uint32_t j = i8 - 1 - k;
        mbar_wait_bounded(&a8_full[j % kS8], (j / kS8) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == kWarpMma) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_f16_f32acc(kPair ? 2 * BM : BM, BN);
      uint32_t s = 0, ph = 0, nseg = 0;  // ring stage and its phase; segments issued
      bool ok = true;
      Sched<kSplit, kPair> sc(p);
      int t, c0, c1;
      while (ok && sc.next(p, t, c0, c1)) {
        const int n_blk = t % p.n_tiles;
        SegWalker walker;
        bool seg_first = true;
        uint32_t dcol = 0;
        int c = c0 - 1;  // current int chunk
        const int st_lo = c0 * kChunkSt;
        const int st_end = c1 == p.nchunks ? nst_all : c1 * kChunkSt;
        for (int st = st_lo; st < st_end && ok;) {
          // Segment boundaries, checked once per run of stages (the rest of an int chunk,
          // or the outlier segment): int chunks grouped by the exactness bound, then the
          // outlier segment; each segment takes the next accumulator (F0/F1).
          bool opens;
          int st_stop;
          if (st < nst_int) {  // st starts an int chunk
            ++c;
            opens = walker.opens(chunk_bound(p, n_blk, c), c == c0);
            st_stop = st + kChunkSt < nst_int ? st + kChunkSt : nst_int;
          } else {  // st == nst_int: the outlier segment
            opens = true;
            st_stop = st_end;
          }
          if (st_stop > st_end) st_stop = st_end;
          if (opens) {
            if (st > st_lo) {
              if constexpr (kPair) mma_commit_pair(&tmem_full[nseg & 1u], 3);
              else mma_commit(&tmem_full[nseg & 1u]);
              ++nseg;
            }
            if (!(ok = pwait<kPair>(&tmem_empty[nseg & 1u], ((nseg >> 1) & 1u) ^ 1u, ab))) break;
            tc_fence_after();
            dcol = (nseg & 1u) * BN;
            seg_first = true;
          }
          // The run itself does as little as possible per K block: this thread's
          // instruction stream, not the tensor core, bounds small token tiles. One wait per
          // stage: a converter arrives on full_a only once the stage's B has landed.
          for (; st < st_stop; ++st) {
            if (!(ok = pwait<kPair>(&full_a[s], ph, ab))) break;
            tc_fence_after();
            const uint64_t bd = sdesc_kmajor_sw128(sbase + C::b + s * C::kBStage);
            if constexpr (C::kAT) {  // A from TMEM: 16 K values = 8 columns per step
              const uint32_t ta = tmem_base + C::kAcol0 + 32 * kKB * s;
              // K blocks of the stage that hold data: past K the int boxes read zeros (outside
              // the tensors), but the outlier slices are zero-padded only to a multiple of 64
              // columns, so an outlier stage stops at its last K block
              const int nvalid = st < nst_int ? kKB : nkb_out - (st - nst_int) * kKB;
              // the MMAs of K block j of the stage
              auto kblock = [&](int j) {
                const uint64_t bdj = bd + (uint64_t)((j * C::kBBytes) >> 4);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                  mma_f16_ts(tmem_base + dcol, ta + 32 * j + 8 * k, bdj + 2 * k, idesc,
                             (seg_first && j == 0 && k == 0) ? 0u : 1u);
              };
              if (nvalid >= kKB) {
                // a whole stage (every int stage): one straight run of MMAs, no test
                // between them (a test inside the unrolled run cost 6-10 % at 16-64 tokens)
#pragma unroll
                for (int j = 0; j < kKB; ++j) kblock(j);
              } else {
                for (int j = 0; j < nvalid; ++j) kblock(j);
              }
            } else {
              const uint64_t ad = sdesc_kmajor_sw128(sbase + C::a16 + s * kA16Bytes);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                if constexpr (kPair)
                  mma_f16_ss_pair(tmem_base + dcol, ad + 2 * k, bd + 2 * k, idesc,
                                  (seg_first && k == 0) ? 0u : 1u);
                else
                  mma_f16_ss(tmem_base + dcol, ad + 2 * k, bd + 2 * k, idesc,
                             (seg_first && k == 0) ? 0u : 1u);
              }
            }
            seg_first = false;
            if constexpr (kPair) mma_commit_pair(&empty[s], 3);
            else mma_commit(&empty[s]);
            if (++s == (uint32_t)kS) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        if (!ok) break;
        if constexpr (kPair) mma_commit_pair(&tmem_full[nseg & 1u], 3);
        else mma_commit(&tmem_full[nseg & 1u]);
        ++nseg;
      }
      // all issued MMAs have completed before TMEM is released (in both CTAs of a pair)
      if constexpr (kPair) mma_commit_pair(done, 3);
      else mma_commit(done);
      wait_bounded<kPair>(done, 0, p.timeout_ns);
    } else if (kPair && lane == 0) {
      wait_bounded<kPair>(done, 0, p.timeout_ns);  // the issuer's MMAs, before TMEM is freed
    }
  } else if ((warp >= kWarpConv0 && warp < kWarpConv0 + 4) || warp >= kWarpConv1) {
    // -------------------------------------------------------- weights into fp16 A
    // Thread `lane` of warp q of a set handles row r = 32q + lane of each stage's 128 x 64 kKB
    // A block: 16-byte loads from the weight ring (TMA swizzle of the slot's row width: 64
    // bytes, chunk c of row r at chunk c ^ ((r >> 1) & 3); 128 bytes, at c ^ (r & 7)), int8
    // -> fp16 in registers (fp16 outlier weights are copied as they are), then either TMEM
    // stores (kAT) or eight 16-byte stores into the 128-byte-swizzled A stage in shared
    // memory (chunk c of row r at chunk c ^ (r & 7)).
    if (!p.debug_skip_loads) {
      const int set = warp >= kWarpConv1 ? 1 : 0;
      const int r = 32 * (warp & 3) + lane;
      const uint32_t swz8 = (uint32_t)(r >> 1) & 3u;  // 64-byte-wide boxes (kKB = 1)
      const uint32_t swz16 = (uint32_t)r & 7u;
      uint32_t it = 0, i8 = 0;
      bool ok = true;
      Sched<kSplit, kPair> sc(p);
      int t, c0, c1;
      while (ok && sc.next(p, t, c0, c1)) {
        const int st_end = c1 == p.nchunks ? nst_all : c1 * kChunkSt;
        for (int st = c0 * kChunkSt; st < st_end && ok; ++st, ++it) {
          const bool is_int = st < nst_int;
          const uint32_t i8_0 = i8;
          i8 += is_int ? 1u : 2u;
          if ((int)(it & 1u) != set) continue;  // stage `it` belongs to set it & 1
          const uint32_t s = it % kS, ph = (it / kS) & 1u;
          // the MMAs that last read A stage s have completed
          if (!(ok = pwait<kPair>(&empty[s], ph ^ 1u, ab))) break;
          if constexpr (C::kAT) tc_fence_after();
          if constexpr (C::kAT) {
            // One K block at a time from the slot's 128-byte-wide boxes (128 rows x 128
            // bytes, 128-byte swizzle: chunk c of row r at c ^ (r & 7)): an int box holds two
            // K blocks, an fp16 outlier box one. Converted (int) or copied (fp16), then
            // stored to TMEM lane r: 32 columns of (even K, odd K) per K block.
            const uint32_t ta =
                tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + C::kAcol0 + 32 * kKB * s;
            uint32_t held = ~0u;  // the slot whose barrier this thread has waited on
#pragma unroll
            for (int j = 0; j < kKB; ++j) {
              const uint32_t h = is_int ? 0u : (uint32_t)(2 * j / kKB);  // slot of the stage
              const uint32_t j8 = i8_0 + h, s8 = j8 % kS8;
              if (j8 != held) {
                if (!(ok = pwait<kPair>(&a8_full[s8], (j8 / kS8) & 1u, ab))) break;
                held = j8;
              }
              const uint32_t box = is_int ? (uint32_t)j / 2 : (uint32_t)(j - (int)h * kKB / 2);
              const uint32_t row = sbase + C::a8 + s8 * C::kA8Slot + box * kBox8Bytes + r * 128;
              uint32_t a[32];
              if (is_int) {
                const uint32_t cb = 4u * (uint32_t)(j % 2);
                uint4 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  v[c] = ld_shared_v4(row + ((((uint32_t)c + cb) ^ swz16) << 4));
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  uint32_t o[8];
                  cvt_s8x16_to_f16x16(v[c], o);
#pragma unroll
                  for (int k = 0; k < 8; ++k) a[8 * c + k] = o[k];
                }
              } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const uint4 v = ld_shared_v4(row + (((uint32_t)c ^ swz16) << 4));
                  a[4 * c + 0] = v.x;
                  a[4 * c + 1] = v.y;
                  a[4 * c + 2] = v.z;
                  a[4 * c + 3] = v.w;
                }
              }
              tmem_st<32>(ta + 32 * j, a);
            }
            if (!ok) break;
            tmem_st_wait();
            tc_fence_before();
          } else {
            static_assert(C::kKB == 1, "shared-memory A stages hold one K block");
            uint32_t a[32];
            if (is_int) {
              const uint32_t s8 = i8_0 % kS8;
              if (!(ok = pwait<kPair>(&a8_full[s8], (i8_0 / kS8) & 1u, ab))) break;
              const uint32_t src = sbase + C::a8 + s8 * C::kA8Slot + r * 64;
              uint4 v[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) v[c] = ld_shared_v4(src + (((uint32_t)c ^ swz8) << 4));
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t o[8];
                cvt_s8x16_to_f16x16(v[c], o);
#pragma unroll
                for (int k = 0; k < 8; ++k) a[8 * c + k] = o[k];
              }
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {  // slot h: fp16 columns [32 h, 32 h + 32)
                const uint32_t j8 = i8_0 + h, s8 = j8 % kS8;
                if (!(ok = pwait<kPair>(&a8_full[s8], (j8 / kS8) & 1u, ab))) break;
                const uint32_t src = sbase + C::a8 + s8 * C::kA8Slot + r * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const uint4 v = ld_shared_v4(src + (((uint32_t)c ^ swz8) << 4));
                  a[16 * h + 4 * c + 0] = v.x;
                  a[16 * h + 4 * c + 1] = v.y;
                  a[16 * h + 4 * c + 2] = v.z;
                  a[16 * h + 4 * c + 3] = v.w;
                }
              }
              if (!ok) break;
            }
            const uint32_t dst = sbase + C::a16 + s * kA16Bytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(dst + (((uint32_t)c ^ swz16) << 4), a[4 * c], a[4 * c + 1],
                           a[4 * c + 2], a[4 * c + 3]);
            // each thread orders its shared stores before the tensor core reads them
            fence_proxy_async_smem();
          }
          // The stage's B must have landed before the MMA issuer sees full_a complete: warp
          // 0 of the set waits for it (in a pair, the issuer's full_b counts both halves).
          if ((warp & 3) == 0 && rank == 0) {
            if (!(ok = pwait<kPair>(&full_b[s], ph, ab))) break;
          }
          // the warp then signals once
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&a8_empty[i8_0 % kS8]);
            if (!is_int) mbar_arrive(&a8_empty[(i8_0 + 1) % kS8]);
            arrive_leader<kPair>(&full_a[s]);
          }
        }
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    // -------------------------------------------------------- epilogue
    if constexpr (!kSplit) {
      // whole tiles, t = b, b + G, ...
      constexpr int kNR = (BN + 31) / 32;  // prefetched row scales per lane
      const int q = warp & 3;
      const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
      uint8_t* boxes = smem + C::box + q * 2 * C::kBoxBytes;
      const CUtensorMap* mapY = p.y_tma ? &tmY : nullptr;
      const uint64_t y_policy = l2_policy_evict_first();
      // this CTA's running-sum slot, [BN tokens][128 features]; lane = feature 32q + lane
      int32_t* accs = p.acc_scratch + (size_t)blockIdx.x * BN * 128 + 32 * q + lane;
      uint32_t nseg = 0, slot = 0, ephase = 0;
      bool ok = true;
      // CUDA-core outlier product: the tile's transposed X_out rows are staged once in shared
      // memory by the four epilogue warps (where they fit), so that each slice reads them
      // with broadcast loads instead of shuffles
      constexpr bool kXoSmem = C::kXoBytes > 0;
      // the tile's row scales likewise (their per-token shuffles go too); the zeropoint
      // epilogue keeps its shuffles, as its zero points would cost registers it lacks
      constexpr bool kRsSmem = kXoSmem && !kZp;
      [[maybe_unused]] const uint32_t xo_s = sbase + C::xo;
      // rendezvous of the four epilogue warps (bounded: an aborted pipeline unwinds)
      [[maybe_unused]] auto epi_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_bar);
        const bool r = pipe_wait(epi_bar, ephase & 1u, ab);
        ++ephase;
        return r;
      };
      for (int t = tile_first<kPair>(); t < tiles && ok; t += tile_stride<kPair>()) {
        const int m_blk = t / p.n_tiles, n_blk = t % p.n_tiles;
        const int m0 = m_blk * kFeatTile + (int)rank * BM, n0 = n_blk * BN;
        const int o = m0 + q * 32 + lane;
        const bool o_ok = o < p.out;
        const float bo = (o_ok && p.bias) ? __half2float(__ushort_as_half(p.bias[o])) : 0.0f;
        const float so = o_ok ? __ldg(&p.scb[o]) * (1.0f / 16129.0f) : 0.0f;
        float ra[kNR];  // row scales of the tile's tokens, 32 per register, one per lane
        [[maybe_unused]] int za[kZp ? kNR : 1] = {};  // zeropoint: the tokens' zero points
  #pragma unroll
        for (int i = 0; i < kNR; ++i) {
          const int tk = n0 + 32 * i + lane;
          ra[i] = tk < p.T ? __ldg(&p.rowabs[tk]) : 0.0f;
          if constexpr (kZp) za[i] = tk < p.T ? __ldg(&p.zi[tk]) : 0;
        }
        // zeropoint: sum of this feature's codes over the inlier columns
        [[maybe_unused]] const int cbin =
            (kZp && o_ok) ? __ldg(&p.cbsum[o]) - __ldg(&p.cbout[o]) : 0;
        uint32_t wh[kCcOut / 2];  // this feature's outlier weights (CUDA-core outlier product)
        load_cc_weights(p, o, o_ok, n_cc, wh);
        if constexpr (kXoSmem) {
          // the previous tile's rows and scales are no longer read once all four warps arrive;
          // then the tile's row scales and (n_cc > 0) its transposed outlier rows
          if (kRsSmem || n_cc > 0) {
            if (!(ok = epi_sync())) break;
          }
          if constexpr (kRsSmem) {
            for (int j = 32 * q + lane; j < BN; j += 128) {
              const int tk = n0 + j;
              st_shared_f32(xo_s + kCcOut * BN * 2 + 4 * j, tk < p.T ? __ldg(&p.rowabs[tk]) : 0.0f);
            }
          }
          if (n_cc > 0) {
            // rows 0 .. n_cc rounded up to 4 (zeros past n_cc), the tile's tokens present in
            // the transposed copy (its rows hold T rounded up to 16), in 16-byte chunks
            const int rows = (n_cc + 3) & ~3;
            const int cpr = min(BN, p.xo_stride - n0) / 8;
            const int et = 32 * q + lane;
            for (int c = et; c < rows * cpr; c += 128) {
              const int k = c / cpr, ch = c - k * cpr;
              const uint4 v =
                  __ldg(reinterpret_cast<const uint4*>(p.xoT + (size_t)k * p.xo_stride + n0) + ch);
              st_shared_v4(xo_s + (uint32_t)(k * BN + ch * 8) * 2u, v.x, v.y, v.z, v.w);
            }
          }
          if (kRsSmem || n_cc > 0) {
            if (!(ok = epi_sync())) break;
          }
        }
        const int nseg_int = count_int_segments(p, n_blk, 0, p.nchunks);
        const int nseg_tile = nseg_int + (nkb_out > 0 ? 1 : 0);
        uint32_t ymax = 0;  // kNext: largest fp16 magnitude bits of this lane's column
        for (int si = 0; si < nseg_tile && ok; ++si, ++nseg) {
          const bool is_out = si >= nseg_int;
          const bool first = si == 0;
          const bool last = si == nseg_tile - 1;
          const uint32_t b = nseg & 1u;
          if (!(ok = pwait<kPair>(&tmem_full[b], (nseg >> 1) & 1u, ab))) break;
          tc_fence_after();
          const uint32_t tF = tq + b * BN;
          // Running sums of the tile (not for its first segment): slice j0's are in pc while
          // the next slice's load into pn, so the L2 latency is paid once per segment.
          int pn[kW];
  #pragma unroll
          for (int j = 0; j < kW; ++j) pn[j] = first ? 0 : accs[(size_t)j * 128];
          static_assert(kW == 16, "CUDA-core outlier slices are 16 tokens");
          uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;  // the slice's transposed X_out
          if (!kXoSmem && last) cc_load_rows(p, n0, n_cc, lane, xa, xb);  // rows (shuffled)
          if (!last) {
            // an int segment that is not the last one of the tile: fold it into the
            // running sum (first segment: store it)
  #pragma unroll 1
            for (int j0 = 0; j0 < BN; j0 += kW) {
              int pc[kW];
  #pragma unroll
              for (int j = 0; j < kW; ++j) pc[j] = pn[j];
              if (!first && j0 + kW < BN) {
  #pragma unroll
                for (int j = 0; j < kW; ++j) pn[j] = accs[(size_t)(j0 + kW + j) * 128];
              }
              uint32_t f[kW];
              tmem_ld<kW>(tF + j0, f);
              tmem_ld_wait();
  #pragma unroll
              for (int j = 0; j < kW; ++j)
                accs[(size_t)(j0 + j) * 128] = pc[j] + __float2int_rn(__uint_as_float(f[j]));
            }
            // the accumulator is free as soon as it has been read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_leader<kPair>(&tmem_empty[b]);
          } else {
  #pragma unroll 1
            for (int j0 = 0; j0 < BN; j0 += kW) {
              int pc[kW];
  #pragma unroll
              for (int j = 0; j < kW; ++j) pc[j] = pn[j];
              if (!first && j0 + kW < BN) {
  #pragma unroll
                for (int j = 0; j < kW; ++j) pn[j] = accs[(size_t)(j0 + kW + j) * 128];
              }
              float fcc[kW];  // outlier product of this slice (zeros unless cc)
              if constexpr (kXoSmem) {
                cc_outlier_slice_smem(n_cc, wh, xo_s + (uint32_t)j0 * 2u, (uint32_t)BN * 2u, fcc);
              } else {
                uint4 na, nb;  // the next slice's rows, loaded while this one is computed
                cc_load_rows(p, n0 + j0 + kW < n0 + BN ? n0 + j0 + kW : p.T, n_cc, lane, na, nb);
                cc_outlier_slice(n_cc, wh, xa, xb, fcc);
                xa = na;
                xb = nb;
              }
              uint32_t f[kW];
              tmem_ld<kW>(tF + j0, f);
              tmem_ld_wait();
              if (j0 + kW >= BN) {  // all of F has been read: release it to the MMA
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader<kPair>(&tmem_empty[b]);
              }
              const float ra_s = ra[0];  // this slice's tokens, one per lane
              [[maybe_unused]] const int za_s = kZp ? za[0] : 0;
              // zeropoint: the int32 form is exact for all 32 tokens of the group (uniform)
              [[maybe_unused]] const bool z32 =
                  kZp && __all_sync(0xffffffffu, abs(za_s) <= p.z_safe);
              uint32_t yh[kW / 2];
              [[maybe_unused]] uint32_t rsv[kW];  // the slice's row scales (kRsSmem)
              if constexpr (kRsSmem) {
  #pragma unroll
                for (int c = 0; c < kW / 4; ++c) {
                  const uint4 r4 = ld_shared_v4(xo_s + kCcOut * BN * 2 + 4 * (j0 + 4 * c));
                  rsv[4 * c] = r4.x;
                  rsv[4 * c + 1] = r4.y;
                  rsv[4 * c + 2] = r4.z;
                  rsv[4 * c + 3] = r4.w;
                }
              }
              auto slice_y = [&](auto wide) {
  #pragma unroll
                for (int j = 0; j < kW; ++j) {
                  int acc;
                  float fo = fcc[j];
                  if (is_out) {
                    acc = pc[j];
                    fo = __uint_as_float(f[j]);
                  } else {
                    acc = __float2int_rn(__uint_as_float(f[j])) + pc[j];
                  }
                  float rj;
                  if constexpr (kRsSmem) rj = __uint_as_float(rsv[j]);
                  else rj = __shfl_sync(0xffffffffu, ra_s, (j0 % 32) + j);
                  float y;
                  if constexpr (kZp) {
                    // x ~ (q + Z)/S: sum_j (q_j + Z) CB_j = acc + Z * cbin, exact: in int32
                    // when |Z| <= z_safe bounds it below 2^31, in 64 bits otherwise
                    const int zj = __shfl_sync(0xffffffffu, za_s, (j0 % 32) + j);
                    if constexpr (decltype(wide)::value) {
                      const long long az = (long long)acc + (long long)zj * (long long)cbin;
                      y = __fmaf_rn(__ll2float_rn(az), rj * so, fo) + bo;
                    } else {
                      y = __fmaf_rn((float)(acc + zj * cbin), rj * so, fo) + bo;
                    }
                  } else {
                    y = __fmaf_rn((float)acc, rj * so, fo) + bo;
                  }
                  if constexpr (kNext) {
                    if (p.next_relu) y = fmaxf(y, 0.0f);
                  }
                  const uint32_t h = __half_as_ushort(__float2half_rn(y));
                  if constexpr (kNext) {
                    if (n0 + j0 + j < p.T) ymax = max(ymax, h & 0x7fffu);
                  }
                  yh[j / 2] = (j & 1) ? (yh[j / 2] | (h << 16)) : h;
                  if constexpr (kDebug) pc[j] = acc;
                }
              };
              // the whole group's test picks one form for the slice (a uniform branch)
              if (kZp && !z32) slice_y(Wide<true>{});
              else slice_y(Wide<false>{});
              box_reuse_wait(lane);
              box_store<kW>(boxes + slot * C::kBoxBytes, yh, mapY, p.Y, p.T, p.out, m0 + 32 * q,
                            n0 + j0, lane, y_policy);
              slot ^= 1u;
              if constexpr (kDebug) {
  #pragma unroll 1
                for (int j = 0; j < kW; ++j) {
                  const int tok = n0 + j0 + j;
                  if (o_ok && tok < p.T) p.acc_debug[(size_t)tok * p.out + o] = pc[j];
                }
              }
              if ((j0 + kW) % 32 == 0) {  // next 32 tokens: rotate the prefetched row scales
  #pragma unroll
                for (int i = 0; i + 1 < kNR; ++i) ra[i] = ra[i + 1];
                if constexpr (kZp) {
  #pragma unroll
                  for (int i = 0; i + 1 < kNR; ++i) za[i] = za[i + 1];
                }
              }
            }
            if constexpr (kNext) {  // the tile's flags of columns m0 + 32q .. + 31
              const uint32_t word = __ballot_sync(0xffffffffu, o_ok && ymax >= p.next_thr);
              if (lane == 0 && word != 0u) atomicOr(&p.next_mask[(m0 + 32 * q) >> 5], word);
            }
          }
        }
      }
      if (lane == 0) bulk_wait_group0();  // output stores complete before the CTA exits
    } else {
      // pieces of the split schedule
      constexpr int kNR = (BN + 31) / 32;  // prefetched row scales per lane
      const int q = warp & 3;
      const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
      uint8_t* boxes = smem + C::box + q * 2 * C::kBoxBytes;
      const CUtensorMap* mapY = p.y_tma ? &tmY : nullptr;
      const uint64_t y_policy = l2_policy_evict_first();
      volatile int* s_fin = reinterpret_cast<volatile int*>(smem + C::misc + 8);
      // this CTA's running-sum slot, [BN tokens][128 features]; lane = feature 32q + lane
      int32_t* accs = p.acc_scratch + (size_t)blockIdx.x * BN * 128 + 32 * q + lane;
      uint32_t nseg = 0, slot = 0, ephase = 0;
      bool ok = true;
      // rendezvous of the four epilogue warps (bounded: an aborted pipeline unwinds)
      auto epi_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_bar);
        const bool r = pipe_wait(epi_bar, ephase & 1u, ab);
        ++ephase;
        return r;
      };
      Sched<kSplit> sc(p);
      int t, c0, c1;
      while (ok && sc.next(p, t, c0, c1)) {
        const int m_blk = t / p.n_tiles, n_blk = t % p.n_tiles;
        const int m0 = m_blk * BM, n0 = n_blk * BN;
        const int o = m0 + q * 32 + lane;
        const bool o_ok = o < p.out;
        const float bo = (o_ok && p.bias) ? __half2float(__ushort_as_half(p.bias[o])) : 0.0f;
        const float so = o_ok ? __ldg(&p.scb[o]) * (1.0f / 16129.0f) : 0.0f;
        float ra[kNR];  // row scales of the tile's tokens, 32 per register, one per lane
        [[maybe_unused]] int za[kZp ? kNR : 1] = {};  // zeropoint: the tokens' zero points
  #pragma unroll
        for (int i = 0; i < kNR; ++i) {
          const int tk = n0 + 32 * i + lane;
          ra[i] = tk < p.T ? __ldg(&p.rowabs[tk]) : 0.0f;
          if constexpr (kZp) za[i] = tk < p.T ? __ldg(&p.zi[tk]) : 0;
        }
        // zeropoint: sum of this feature's codes over the inlier columns
        [[maybe_unused]] const int cbin =
            (kZp && o_ok) ? __ldg(&p.cbsum[o]) - __ldg(&p.cbout[o]) : 0;
        uint32_t wh[kCcOut / 2];  // this feature's outlier weights (CUDA-core outlier product)
        load_cc_weights(p, o, o_ok, n_cc, wh);
        const bool has_out = c1 == p.nchunks && nkb_out > 0;
        const int nseg_int = count_int_segments(p, n_blk, c0, c1);
        const int nseg_tile = nseg_int + (has_out ? 1 : 0);
        // a piece that is not the whole tile publishes its sums; the tile's last piece to
        // arrive adds all pieces and writes Y
        const bool whole = c0 == 0 && c1 == p.nchunks;
        int32_t* my_part = nullptr;
        float* my_part_f = nullptr;
        if (!whole) {
          const int pslot = unit_start(p, blockIdx.x) >= (long long)t * p.nchunks ? 0 : 1;
          my_part = p.part + ((size_t)blockIdx.x * 2 + pslot) * BN * 128 + 32 * q + lane;
          my_part_f = p.part_f + (size_t)blockIdx.x * BN * 128 + 32 * q + lane;
        }
        uint32_t ymax = 0;  // kNext: largest fp16 magnitude bits of this lane's column

        // Y of token slice j0 from its int sums and fp32 outlier sums (one per lane = feature)
        auto emit = [&](int j0, const int (&accv)[kW], const float (&fov)[kW]) {
          const float ra_s = ra[0];  // this slice's tokens, one per lane
          [[maybe_unused]] const int za_s = kZp ? za[0] : 0;
          // zeropoint: the int32 form is exact for all 32 tokens of the group (uniform)
          [[maybe_unused]] const bool z32 = kZp && __all_sync(0xffffffffu, abs(za_s) <= p.z_safe);
          uint4 xa, xb;
          cc_load_rows(p, n0 + j0, n_cc, lane, xa, xb);
          float fcc[kW];  // outlier product of this slice (zeros unless cc)
          cc_outlier_slice(n_cc, wh, xa, xb, fcc);
          uint32_t yh[kW / 2];
          auto slice_y = [&](auto wide) {
  #pragma unroll
            for (int j = 0; j < kW; ++j) {
              const int acc = accv[j];
              const float fo = fov[j] + fcc[j];
              const float rj = __shfl_sync(0xffffffffu, ra_s, (j0 % 32) + j);
              float y;
              if constexpr (kZp) {
                // x ~ (q + Z)/S: sum_j (q_j + Z) CB_j = acc + Z * cbin, exact: in int32 when
                // |Z| <= z_safe bounds it below 2^31, in 64 bits otherwise
                const int zj = __shfl_sync(0xffffffffu, za_s, (j0 % 32) + j);
                if constexpr (decltype(wide)::value) {
                  const long long az = (long long)acc + (long long)zj * (long long)cbin;
                  y = __fmaf_rn(__ll2float_rn(az), rj * so, fo) + bo;
                } else {
                  y = __fmaf_rn((float)(acc + zj * cbin), rj * so, fo) + bo;
                }
              } else {
                y = __fmaf_rn((float)acc, rj * so, fo) + bo;
              }
              if constexpr (kNext) {
                if (p.next_relu) y = fmaxf(y, 0.0f);
              }
              const uint32_t h = __half_as_ushort(__float2half_rn(y));
              if constexpr (kNext) {
                if (n0 + j0 + j < p.T) ymax = max(ymax, h & 0x7fffu);
              }
              yh[j / 2] = (j & 1) ? (yh[j / 2] | (h << 16)) : h;
            }
          };
          // the whole group's test picks one form for the slice (a uniform branch)
          if (kZp && !z32) slice_y(Wide<true>{});
          else slice_y(Wide<false>{});
          box_reuse_wait(lane);
          box_store<kW>(boxes + slot * C::kBoxBytes, yh, mapY, p.Y, p.T, p.out, m0 + 32 * q,
                        n0 + j0, lane, y_policy);
          slot ^= 1u;
          if constexpr (kDebug) {
  #pragma unroll 1
            for (int j = 0; j < kW; ++j) {
              const int tok = n0 + j0 + j;
              if (o_ok && tok < p.T) p.acc_debug[(size_t)tok * p.out + o] = accv[j];
            }
          }
          if ((j0 + kW) % 32 == 0) {  // next 32 tokens: rotate the prefetched row scales
  #pragma unroll
            for (int i = 0; i + 1 < kNR; ++i) ra[i] = ra[i + 1];
            if constexpr (kZp) {
  #pragma unroll
              for (int i = 0; i + 1 < kNR; ++i) za[i] = za[i + 1];
            }
          }
        };

        for (int si = 0; si < nseg_tile && ok; ++si, ++nseg) {
          const bool is_out = si >= nseg_int;
          const bool first = si == 0;
          const bool last = si == nseg_tile - 1;
          const uint32_t b = nseg & 1u;
          if (!(ok = pipe_wait(&tmem_full[b], (nseg >> 1) & 1u, ab))) break;
          tc_fence_after();
          const uint32_t tF = tq + b * BN;
          // Running sums of the piece (not for its first segment): slice j0's are in pc
          // while the next slice's load into pn, so the L2 latency is paid once per segment.
          int pn[kW];
  #pragma unroll
          for (int j = 0; j < kW; ++j) pn[j] = first ? 0 : accs[(size_t)j * 128];
  #pragma unroll 1
          for (int j0 = 0; j0 < BN; j0 += kW) {
            int pc[kW];
  #pragma unroll
            for (int j = 0; j < kW; ++j) pc[j] = pn[j];
            if (!first && j0 + kW < BN) {
  #pragma unroll
              for (int j = 0; j < kW; ++j) pn[j] = accs[(size_t)(j0 + kW + j) * 128];
            }
            uint32_t f[kW];
            tmem_ld<kW>(tF + j0, f);
            tmem_ld_wait();
            if (j0 + kW >= BN) {  // all of F has been read: release it to the MMA
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tmem_empty[b]);
            }
            if (!last) {
              // an int segment that is not the last one of the piece: fold it into the
              // running sum (first segment: store it)
  #pragma unroll
              for (int j = 0; j < kW; ++j)
                accs[(size_t)(j0 + j) * 128] = pc[j] + __float2int_rn(__uint_as_float(f[j]));
              continue;
            }
            int accv[kW];
            float fov[kW];
  #pragma unroll
            for (int j = 0; j < kW; ++j) {
              accv[j] = is_out ? pc[j] : pc[j] + __float2int_rn(__uint_as_float(f[j]));
              fov[j] = is_out ? __uint_as_float(f[j]) : 0.0f;
            }
            if (whole) {
              emit(j0, accv, fov);
            } else {
  #pragma unroll
              for (int j = 0; j < kW; ++j) {
                my_part[(size_t)(j0 + j) * 128] = accv[j];
                if (has_out) my_part_f[(size_t)(j0 + j) * 128] = fov[j];
              }
            }
          }
        }
        if (!ok) break;
        if (!whole) {
          // arrive on the tile; the last of its pieces (b_first .. b_last) finishes it
          const long long ut0 = (long long)t * p.nchunks;
          const int b_first = unit_owner(p, ut0);
          const int b_last = unit_owner(p, ut0 + p.nchunks - 1);
          __threadfence();  // this thread's part stores before the arrival (all four warps)
          if (!(ok = epi_sync())) break;
          if (q == 0 && lane == 0) {
            __threadfence();
            *s_fin = atomicAdd(&p.tile_cnt[t], 1) == b_last - b_first ? 1 : 0;
          }
          if (!(ok = epi_sync())) break;
          if (*s_fin) {
            __threadfence();
            const bool t_out = nkb_out > 0;
            const float* pf = p.part_f + (size_t)b_last * BN * 128 + 32 * q + lane;
  #pragma unroll 1
            for (int j0 = 0; j0 < BN; j0 += kW) {
              int accv[kW];
              float fov[kW];
  #pragma unroll
              for (int j = 0; j < kW; ++j) {
                accv[j] = 0;
                fov[j] = t_out ? __ldcg(pf + (size_t)(j0 + j) * 128) : 0.0f;
              }
  #pragma unroll 1
              for (int bb = b_first; bb <= b_last; ++bb) {
                const int ps = unit_start(p, bb) >= ut0 ? 0 : 1;
                const int32_t* src =
                    p.part + ((size_t)bb * 2 + ps) * BN * 128 + 32 * q + lane + (size_t)j0 * 128;
  #pragma unroll
                for (int j = 0; j < kW; ++j) accv[j] += __ldcg(src + (size_t)j * 128);
              }
              emit(j0, accv, fov);
            }
          }
        }
        if constexpr (kNext) {  // the tile's flags of columns m0 + 32q .. + 31
          const uint32_t word = __ballot_sync(0xffffffffu, o_ok && ymax >= p.next_thr);
          if (lane == 0 && word != 0u) atomicOr(&p.next_mask[(m0 + 32 * q) >> 5], word);
        }
      }
      if (lane == 0) bulk_wait_group0();  // output stores complete before the CTA exits
    }
  }

  // -------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  // a pair's CTAs leave together: neither exits while the other may still arrive on its
  // barriers or read its shared memory through the MMAs
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == kWarpMma) {
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, int kMode, bool kSplit, bool kPair>
cudaError_t launch_variant(cudaStream_t s, const CUtensorMap& mA8, const CUtensorMap& mB,
                           const CUtensorMap& mWo, const CUtensorMap& mXo,
                           const CUtensorMap& mY, const Params& p, int grid) {
  using C = Cfg<BN, kPair>;
  auto kernel = i8_gemm_kernel<BN, kMode, kSplit, kPair>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::total);
  if (e != cudaSuccess) return e;
  if constexpr (!kPair) {
    kernel<<<grid, kThreads, C::total, s>>>(mA8, mB, mWo, mXo, mY, p);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, mA8, mB, mWo, mXo, mY, p);
  }
}

// Pairs of CTAs (2-SM clusters) that can be resident at once for this kernel, looked up once
// per device; 0 if the device cannot run it.
template <int kMode>
int max_pairs() {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};  // 0: not looked up yet, -1: none
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 0;
  }
  if (cache[dev] == 0) {
    using C = Cfg<256, true>;
    auto kernel = i8_gemm_kernel<256, kMode, false, true>;
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::total) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * sm_count(), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = C::total;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[dev] = n > 0 ? n : -1;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

template <int BN, int kMode>
cudaError_t launch_kernel(cudaStream_t s, const CUtensorMap& mA8, const CUtensorMap& mB,
                          const CUtensorMap& mWo, const CUtensorMap& mXo, const CUtensorMap& mY,
                          const Params& p, int grid, bool pair) {
  if constexpr (BN == 256) {
    if (pair) return launch_variant<BN, kMode, false, true>(s, mA8, mB, mWo, mXo, mY, p, grid);
  }
  if (p.split) return launch_variant<BN, kMode, true, false>(s, mA8, mB, mWo, mXo, mY, p, grid);
  return launch_variant<BN, kMode, false, false>(s, mA8, mB, mWo, mXo, mY, p, grid);
}

// Kernel mode of a call (the epilogue variant).
inline int epi_mode(const GemmArgs& a) {
  if (a.zi) return a.acc_debug ? kEpiZpDebug : kEpiZp;
  if (a.next.mask) return kEpiNext;
  return a.acc_debug ? kEpiDebug : kEpiPlain;
}

template <int BN>
cudaError_t launch_bn(const GemmArgs& a, cudaStream_t s) {
  // 256-token tiles on the whole-tile schedule run on CTA pairs (M = 256 per MMA, each CTA
  // holding half of the tile's B rows) when the device can hold at least one pair
  int pairs = 0;
  if constexpr (BN == 256) {
    if (!a.split && !kDisablePairs) {
      switch (epi_mode(a)) {
        case kEpiPlain: pairs = max_pairs<kEpiPlain>(); break;
        case kEpiDebug: pairs = max_pairs<kEpiDebug>(); break;
        case kEpiNext: pairs = max_pairs<kEpiNext>(); break;
        case kEpiZp: pairs = max_pairs<kEpiZp>(); break;
        default: pairs = max_pairs<kEpiZpDebug>(); break;
      }
    }
  }
  const bool pair = pairs > 0;
  const int b_rows = pair ? BN / 2 : BN;  // B rows per CTA and stage
  using C = Cfg<BN>;
  CUtensorMap mA8, mB, mWo, mXo, mY;
  bool ok = true;
  // weight boxes: 128 rows x one stage of K (64 or 128 bytes), swizzled across the row
  const CUtensorMapSwizzle sw8 =
      C::kBoxKB == 2 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  ok &= make_map(&mA8, a.a_int8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.out, a.in, BM,
                 BK * C::kBoxKB, sw8);
  ok &= make_map(&mB, a.b_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.in, b_rows, BK,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  // outlier weights: 128 rows x 32 kKB fp16 (the same bytes as a weight box), two boxes per
  // stage
  ok &= make_map(&mWo, a.wout, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.out, a.ncap, BM,
                 BK / 2 * C::kBoxKB, sw8);
  ok &= make_map(&mXo, a.xout, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.ncap, b_rows, BK,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  // Y [T, out] fp16 through TMA stores when its row pitch is a multiple of 16 bytes
  const bool y_tma = (a.out % 8) == 0;
  if (y_tma)
    ok &= make_map(&mY, a.Y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.T, a.out, C::kW, 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mY = mB;  // a valid descriptor that is never used
  if (!ok) return cudaErrorInvalidValue;
  Params p{};
  p.T = a.T;
  p.in = a.in;
  p.out = a.out;
  p.m_tiles = (a.out + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM);
  p.n_tiles = (a.T + BN - 1) / BN;
  p.nkb = (a.in + BK - 1) / BK;
  p.nchunks = num_chunks(a.in);
  p.y_tma = y_tma ? 1 : 0;
  p.hdr = a.hdr;
  p.rowabs = a.rowabs;
  p.l1 = a.l1;
  p.acc_scratch = a.acc_scratch;
  p.scb = a.scb;
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.Y = static_cast<uint16_t*>(a.Y);
  p.acc_debug = a.acc_debug;
  p.next_mask = a.next.mask;
  p.next_thr = a.next.thr_bits;
  p.next_relu = a.next.relu;
  // |acc| <= 127^2 in and |cbin| <= 127 in, so |acc + Z cbin| < 2^31 while
  // |Z| <= (2^31 - 1 - 127^2 in) / (127 in)
  p.z_safe = (int)((2147483647LL - 16129LL * a.in) / (127LL * a.in));
  p.zi = a.zi;
  p.cbsum = a.cbsum;
  p.cbout = a.cbout;
  p.wout = static_cast<const uint16_t*>(a.wout);
  p.ncap = a.ncap;
  p.xoT = static_cast<const uint16_t*>(a.xoT);
  p.xo_stride = xo_stride(a.T);
  p.cc_max = kCcMaxDefault;
  p.timeout_ns = a.timeout_ns;
  p.debug_skip_loads = a.debug_skip_loads;
  const int tiles = p.m_tiles * p.n_tiles;
  const int sms = sm_count();
  int grid = tiles < sms ? tiles : sms;
  if (pair) grid = 2 * (tiles < pairs ? tiles : pairs);  // whole clusters, one per tile at most
  p.split = 0;
  if (a.split) {  // cut tiles between CTAs by 1024-K chunks (see i8_split_ctas)
    if (!a.part || !a.part_f || !a.tile_cnt) return cudaErrorInvalidValue;
    p.split = 1;
    p.units = (long long)tiles * p.nchunks;
    p.part = a.part;
    p.part_f = a.part_f;
    p.tile_cnt = a.tile_cnt;
    grid = a.split;
  }
  // ReLU comes only with the statistics epilogue (an FFN's up projection)
  if ((a.next.relu && !a.next.mask) || (a.next.mask && (a.acc_debug || a.zi)))
    return cudaErrorInvalidValue;
  if (a.zi && (!a.cbsum || !a.cbout)) return cudaErrorInvalidValue;
  switch (epi_mode(a)) {
    case kEpiZpDebug:
      return launch_kernel<BN, kEpiZpDebug>(s, mA8, mB, mWo, mXo, mY, p, grid, pair);
    case kEpiZp: return launch_kernel<BN, kEpiZp>(s, mA8, mB, mWo, mXo, mY, p, grid, pair);
    case kEpiNext: return launch_kernel<BN, kEpiNext>(s, mA8, mB, mWo, mXo, mY, p, grid, pair);
    case kEpiDebug: return launch_kernel<BN, kEpiDebug>(s, mA8, mB, mWo, mXo, mY, p, grid, pair);
    default: return launch_kernel<BN, kEpiPlain>(s, mA8, mB, mWo, mXo, mY, p, grid, pair);
  }
}

}  // namespace
}  // namespace gemm

cudaError_t launch_i8_gemm(const GemmArgs& a, cudaStream_t s) {
  switch (i8_bn(a.T)) {
    case 16: return gemm::launch_bn<16>(a, s);
    case 32: return gemm::launch_bn<32>(a, s);
    case 64: return gemm::launch_bn<64>(a, s);
    case 128: return gemm::launch_bn<128>(a, s);
    default: return gemm::launch_bn<256>(a, s);
  }
}

}  // namespace i8mm
