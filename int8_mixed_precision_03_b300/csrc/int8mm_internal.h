// Internal declarations shared by the kernel translation units and the C-ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/int8mm.h"

namespace i8mm {

// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount, looked
// up once per device). The persistent grids, the split plan and the per-SM workspace slots
// are sized from it. Without a usable device (workspace sizing on a host with no GPU) it
// returns kSmFallback, B300's count (2 dies x 74 SMs).
constexpr int kSmFallback = 148;
int sm_count();
constexpr int kKBlock = 64;         // K elements per pipeline stage (128 bytes of fp16)
constexpr int kChunkKBlocks = 16;   // K blocks per exact fp32 accumulation chunk (1024 K)
constexpr int kChunkK = kKBlock * kChunkKBlocks;
// Outlier columns up to this count are multiplied on the CUDA cores in the tensor-core
// matmul's epilogue, from a transposed copy of X_out (kCcOutlierCols rows of tokens).
constexpr int kCcOutlierCols = 32;
// Token stride of that copy: T rounded up to 16 (16-token slices, 32-byte aligned rows).
__host__ __device__ inline int xo_stride(int T) { return (T + 15) / 16 * 16; }

// Token tile (MMA N) of the int8 tensor-core matmul for T tokens: the smallest supported
// size that covers T, 256 for large T. The quantize pass uses it to group its per-chunk
// code statistics by token tile.
inline int i8_bn(int T) {
  return T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256;
}
inline int num_chunks(int in) { return (in + kChunkK - 1) / kChunkK; }

// Work split of the tensor-core matmul. Unsplit, CTA b of G = min(tiles, 148) takes the
// whole tiles b, b + G, ...; the slowest CTA does ceil(tiles / G) tiles of `chunks`
// 1024-K chunks each. Split, the (tile, chunk) units are cut into G = min(units, 148)
// contiguous ranges (ceil(units / G) units at most). A tile cut into pieces costs its
// epilogue warps a second pass (the pieces' sums are published and the last piece to
// arrive adds them up), which the epilogue of a 128- or 256-token tile cannot hide:
// measured on B300, splitting the 13B up and down projections (critical path -3% and
// -13%) made them 20% and 15% slower, while the 64-token decode tile gained 11%. Returns
// the split's CTA count when it shortens the slowest CTA's work by more than 3% (token
// tiles up to 64) or 25% (larger tiles), else 0 (unsplit).
inline int i8_split_ctas(int T, int in, int out) {
  const int bn = i8_bn(T);
  const long long tiles = (long long)((out + 127) / 128) * ((T + bn - 1) / bn);
  const long long chunks = num_chunks(in);
  if (tiles <= 0 || chunks <= 1) return 0;
  const long long sms = sm_count();
  const long long g0 = tiles < sms ? tiles : sms;
  const long long whole = (tiles + g0 - 1) / g0 * chunks;
  const long long units = tiles * chunks;
  const long long g1 = units < sms ? units : sms;
  const long long cut = (units + g1 - 1) / g1;
  return cut * 100 < whole * (bn <= 64 ? 97 : 75) ? (int)g1 : 0;
}

// Device status header at the start of every int8_matmul workspace (zeroed per call).
struct WsHeader {
  int32_t status;         // first device-side error (i8_status), 0 if none
  uint32_t arrive;        // CTA arrival counter of the column-statistics pass
  int32_t n_out;          // number of outlier columns found
  int32_t n_out_used;     // min(n_out, capacity): columns actually gathered
  int32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte block");

// Byte offsets of the int8_matmul workspace sections. Computed identically by
// int8_matmul_workspace_size() and int8_matmul().
struct WsLayout {
  size_t header = 0, mask = 0, l1 = 0, idx = 0, xq = 0, rowabs = 0, xout = 0, wout = 0;
  size_t xoT = 0;         // X_out transposed [kCcOutlierCols][xo_stride(T)] fp16
  size_t zi = 0;          // zeropoint variant: int32 per-row zero points [T]
  size_t cbout = 0;       // zeropoint variant: int32 sums of the outlier columns' codes [out]
  size_t acc = 0;         // int32 running sums of the matmul's epilogue, one tile per SM
  // split work (i8_split_ctas > 0): per-tile arrival counters (zeroed with the header),
  // the pieces' int32 sums [G][2][BN][128] and outlier sums [G][BN][128]
  size_t tile_cnt = 0, part = 0, part_f = 0;
  int split = 0;          // the split's CTA count, 0 if unsplit
  size_t total = 0;
  size_t zero_bytes = 0;  // header + mask + l1: memset at the start of every call
  int words = 0;          // 32-column words of the outlier mask
  int ncap = 0;           // outlier column capacity (multiple of 64)
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// split_ok = false: the layout of the unsplit schedule (no split sections).
inline WsLayout ws_layout(int T, int in, int out, int ncap, bool split_ok = true) {
  WsLayout L;
  size_t off = 0;
  L.words = (in + 31) / 32;
  L.ncap = ncap;
  L.header = off; off += sizeof(WsHeader);
  L.mask = off; off = align_up(off + sizeof(uint32_t) * L.words, 256);
  // per (token tile, 1024-K chunk): max over the tile's rows of sum |code| in the chunk
  L.l1 = off;
  off = align_up(off + sizeof(int32_t) * (size_t)((T + i8_bn(T) - 1) / i8_bn(T)) *
                           num_chunks(in), 256);
  L.split = split_ok ? i8_split_ctas(T, in, out) : 0;
  L.tile_cnt = off;
  if (L.split)
    off = align_up(off + sizeof(int32_t) * (size_t)((out + 127) / 128) *
                             ((T + i8_bn(T) - 1) / i8_bn(T)), 256);
  L.zero_bytes = off;
  L.idx = off; off = align_up(off + sizeof(int32_t) * (size_t)in, 256);
  L.xq = off; off = align_up(off + 2 * (size_t)T * in, 256);
  L.rowabs = off; off = align_up(off + 4 * (size_t)T, 256);
  L.xout = off; off = align_up(off + 2 * (size_t)T * ncap, 256);
  L.wout = off; off = align_up(off + 2 * (size_t)out * ncap, 256);
  L.xoT = off; off = align_up(off + 2 * (size_t)kCcOutlierCols * xo_stride(T), 256);
  L.zi = off; off = align_up(off + 4 * (size_t)T, 256);
  L.cbout = off; off = align_up(off + 4 * (size_t)out, 256);
  L.acc = off; off = align_up(off + 4 * (size_t)sm_count() * 128 * i8_bn(T), 256);
  L.part = off;
  if (L.split) off = align_up(off + 4 * (size_t)L.split * 2 * 128 * i8_bn(T), 256);
  L.part_f = off;
  if (L.split) off = align_up(off + 4 * (size_t)L.split * 128 * i8_bn(T), 256);
  L.total = off;
  return L;
}

// Host checks of int8_matmul's arguments (sizes, threshold, pointers, alignment) without a
// workspace: I8_OK, or the status int8_matmul would return before launching anything.
i8_status matmul_precheck(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                          int out, float threshold, const void* bias, const void* Y);
// I8_OK if the current device is an sm_103 GPU (I8_ERR_UNSUPPORTED_DEVICE, I8_ERR_CUDA).
i8_status current_device_check();

// Smallest fp16 bit pattern whose value is >= threshold (0x7C00 = +inf if none is finite).
uint16_t threshold_to_half_bits(float threshold);

// ---- kernel launchers (each returns cudaGetLastError() of its launch)
cudaError_t launch_colstats(const void* X, int T, int in, uint16_t thr_bits, WsHeader* hdr,
                            uint32_t* mask, int32_t* idx, int ncap, cudaStream_t s);
// Column statistics already in the mask (ORed by the previous matmul's epilogue): one CTA
// turns the mask into the ordered index list and the count. A non-null `prev` status
// word is carried into hdr->status first, so a chain reports its first error in one word.
cudaError_t launch_mask_index(int in, WsHeader* hdr, uint32_t* mask, int32_t* idx, int ncap,
                              const WsHeader* prev, cudaStream_t s);

// Optional epilogue work of a matmul whose output feeds another int8 matmul: ReLU on Y,
// and the next matmul's outlier mask (one bit per column of Y) ORed with the columns where
// some valid token has |fp16 y| >= the next threshold (compared as fp16 magnitude bits).
struct NextLayer {
  int relu = 0;
  uint32_t* mask = nullptr;      // null: no statistics
  uint32_t thr_bits = 0x7C00u;
};
// xoT (nullable): X_out transposed, rows k < kCcOutlierCols (zeros past the outlier count).
cudaError_t launch_quantize_gather(const void* X, int T, int in, const int8_t* CB,
                                   const float* SCB, int out, const WsHeader* hdr,
                                   const uint32_t* mask, const int32_t* idx, int ncap,
                                   void* xq16, float* rowabs, void* xout, void* wout,
                                   void* xoT, int32_t* l1, int8_t* xq8_debug, cudaStream_t s);
// Zeropoint variant of quantize + gather: per row S, Z over the inlier columns, codes
// clamp(rint(x*S - Z)) (outlier columns 0) as fp16, the epilogue's row factor
// rowabs[i] = 127/S (127*min for a constant row) and zero point zi[i] = Z (1 for a constant
// row), X_out; per output feature W_out and cbout[o] = sum of CB over the outlier columns.
// dbg_S, dbg_Z, xq8_debug are optional exports.
cudaError_t launch_quantize_gather_zp(const void* X, int T, int in, const int8_t* CB,
                                      const float* SCB, int out, const WsHeader* hdr,
                                      const uint32_t* mask, const int32_t* idx, int ncap,
                                      void* xq16, float* rowabs, int32_t* zi, void* xout,
                                      void* wout, void* xoT, int32_t* cbout, int32_t* l1,
                                      int8_t* xq8_debug, float* dbg_S, float* dbg_Z,
                                      cudaStream_t s);
// Sum of each row's int8 codes: CBsum[o] = sum_j CB[o, j] (int32).
cudaError_t launch_code_sums(const int8_t* CB, int out, int in, int32_t* CBsum, cudaStream_t s);
cudaError_t launch_absmax_rows(const void* X, int rows, int cols, int8_t* Q, float* absmax,
                               cudaStream_t s);
// Block-wise absmax: blocks of `block` columns per row, absmax [rows, ceil(cols / block)].
cudaError_t launch_absmax_blocks(const void* X, int rows, int cols, int block, int8_t* Q,
                                 float* absmax, cudaStream_t s);
cudaError_t launch_zeropoint_rows(const void* X, int rows, int cols, int8_t* Q, float* S,
                                  float* Z, cudaStream_t s);

struct GemmArgs {
  // A operand (M side = output features): int8 CB [out, in] converted in-kernel, or an
  // fp16 weight [out, in] loaded directly (the fp16 comparator).
  const void* a_int8 = nullptr;
  const void* a_f16 = nullptr;
  // B operand (N side = tokens): fp16 [T, in] (activation codes, or raw X for fp16)
  const void* b_f16 = nullptr;
  // Outlier slices (fp16): W_out [out, ncap] and X_out [T, ncap]; n_out read on device
  const void* wout = nullptr;
  const void* xout = nullptr;
  int ncap = 0;
  // X_out transposed [kCcOutlierCols][xo_stride(T)] for the CUDA-core outlier product (null:
  // the outlier product always runs on the tensor cores)
  const void* xoT = nullptr;
  WsHeader* hdr = nullptr;      // status word + n_out (int8 path), may be null for fp16
  const float* rowabs = nullptr;
  const int32_t* l1 = nullptr;  // per (token tile, chunk) code-magnitude bounds, or null
  int32_t* acc_scratch = nullptr;  // [sm_count()][BN][128] int32 epilogue running sums
  const float* scb = nullptr;
  const void* bias = nullptr;
  void* Y = nullptr;
  int32_t* acc_debug = nullptr; // optional [T, out] int32 export
  int T = 0, in = 0, out = 0;
  NextLayer next;               // int8 path: ReLU + next layer's column statistics
  // zeropoint variant (int8 path): per-row zero points, per-feature code sums of all
  // columns and of the outlier columns; the epilogue adds zi * (cbsum - cbout) to acc
  const int32_t* zi = nullptr;
  const int32_t* cbsum = nullptr;
  const int32_t* cbout = nullptr;
  // split work (split = CTA count, 0: whole tiles per CTA); see WsLayout
  int split = 0;
  int32_t* part = nullptr;
  float* part_f = nullptr;
  int32_t* tile_cnt = nullptr;
  int relu = 0;                 // fp16 comparator: ReLU on Y
  uint64_t timeout_ns = 2000000000ull;
  int debug_skip_loads = 0;     // test hook: the producer issues nothing (waits time out)
};
// Decode-size int8 matmuls (T <= kGemvMaxT tokens whose int8 codes fit in shared memory),
// streaming CB at HBM rate: exact int32 dp4a sums on the CUDA cores for T < kGemvMmaMinT,
// mma.sync m16n8k16 (fp16, exact fp32 fragments drained to int32) from kGemvMmaMinT on.
constexpr int kGemvMaxT = 16;
constexpr int kGemvMmaMinT = 9;  // below: dp4a (measured faster at T = 8 on B300)
constexpr size_t kGemvMaxSmem = 200 * 1024;
struct GemvArgs {
  const int8_t* CB = nullptr;
  const float* SCB = nullptr;
  int T = 0, in = 0, out = 0;
  const int8_t* xq8 = nullptr;    // int8 codes [T, in], outlier columns 0
  const float* rowabs = nullptr;  // [T]
  const WsHeader* hdr = nullptr;  // n_out_used
  const int32_t* idx = nullptr;   // outlier columns
  const void* xout = nullptr;     // fp16 [T, ncap]
  int ncap = 0;
  const void* bias = nullptr;
  void* Y = nullptr;
  int32_t* acc_debug = nullptr;
  NextLayer next;
};
bool gemv_fits(int T, int in);                            // either decode kernel applies
cudaError_t launch_gemv_i8(const GemvArgs& a, cudaStream_t s);  // dispatches on T
bool gemv_mma_fits(int T, int in);
cudaError_t launch_gemv_mma(const GemvArgs& a, cudaStream_t s);

// The int8 path (a_int8 set) and the fp16 comparator (a_f16 set).
cudaError_t launch_i8_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_f16_gemm(const GemmArgs& a, cudaStream_t s);

}  // namespace i8mm
