/*
 * int8mm -- LLM.int8() mixed-precision matrix multiply for NVIDIA B300 (sm_103a).
 *
 *   Y = dequant( int8(X_inlier) . int8(W)^T ) + X_outlier . W_outlier^T (fp16) + bias
 *
 * The method, as the source pages state it:
 *   "Hugging Face, LLM.int8() 8-bit matrix multiplication integrated into Transformers
 *    and Accelerate" (agentlenshq summary), section "core idea": (1) find hidden-state
 *    columns holding a value of magnitude above a threshold (about 6); (2) multiply those
 *    outlier columns in fp16 and quantize the rest to int8 vector-wise (activations per
 *    row, weights per output feature); (3) dequantize the int8 product to fp16 and add the
 *    fp16 outlier product. Section "zeropoint vs absmax": absmax scaling by 127/absmax.
 *    Section "transformers integration": weights kept as int8 CB in [-127,127] with
 *    W ~ (CB * SCB) / 127, quantized on the GPU when moved to it.
 *   "LLM.int8() summary" (zenn, bilzard), section "method": the decomposition splits the
 *    input dimensions and the matching weight dimensions; section "Zeropoint
 *    Quantization": X8 = INT8(X16*S - Z), X16 = (X8 + Z)/S, S = 254/(max - min).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers to caller-owned memory; the library never
 *     allocates or frees memory on these calls. Matrices are dense and row-major.
 *   - fp16 tensors are passed as `void*` holding IEEE binary16 values.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call is
 *     asynchronous on it and does not synchronize the host.
 *   - Errors found on the host (arguments, alignment, device) are returned at once and
 *     nothing is launched. Errors found on the device (outlier capacity exceeded, a wait
 *     that timed out) are recorded in the workspace status word; read it with
 *     i8_get_status(). No C++ exception crosses this interface.
 *   - Every device pointer must be 16-byte aligned, else I8_ERR_ALIGNMENT.
 *   - The device must be compute capability 10.3 (B300); there is no fallback.
 *
 * Rounding (fixed so that codes are reproducible bit for bit): absmax and absmax scale
 * s = 127/absmax in IEEE fp32, code = rint(x*s) with one fp32 multiply (no fused
 * multiply-add), round half to even, clamped to [-127,127]. An absmax of 0 gives scale 0
 * and codes 0. Codes, outlier column sets and int32 accumulators are exact; Y is fp16.
 */
#ifndef INT8MM_H_
#define INT8MM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  I8_OK = 0,
  I8_ERR_INVALID_ARG = 1,        /* null pointer, bad size, bad threshold */
  I8_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned, or `in` not a multiple of 16 */
  I8_ERR_WORKSPACE = 3,          /* workspace null or smaller than required */
  I8_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103 */
  I8_ERR_CUDA = 5,               /* a CUDA runtime call failed (launch, tensor map, ...) */
  I8_ERR_OUTLIER_CAP = 6,        /* device: more outlier columns than the workspace holds */
  I8_ERR_TIMEOUT = 7,            /* device: a pipeline wait gave up (kernel unwound safely) */
  I8_ERR_SCRATCH_LIMIT = 8       /* int8_matmul_noalloc: sizes exceed its built-in scratch */
} i8_status;

/* Largest supported `in`: keeps |acc| <= 127*127*in below 2^31. */
#define I8_MAX_IN 131072

/*
 * Vector-wise weight quantization ("core idea" step 2; "transformers integration":
 * CB in [-127,127], W ~ CB*SCB/127, done once when the weight moves to the GPU).
 *   W   : fp16 [out, in]            input
 *   CB  : int8 [out, in]            output codes, CB[o,j] = rint(W[o,j] * 127/SCB[o])
 *   SCB : fp32 [out]                output, SCB[o] = max_j |W[o,j]| (the absmax itself)
 * out >= 0, in >= 0 (0 is a no-op). One kernel launch.
 */
i8_status int8_quantize_weight(const void* W, int out, int in, int8_t* CB, float* SCB,
                               void* stream);

/*
 * Bytes of device workspace int8_matmul needs for these sizes. max_outlier_cols is the
 * largest number of outlier columns the call must handle (<= 0 means `in`, the worst
 * case); it is rounded up to a multiple of 64. Returns 0 for invalid sizes. The size
 * includes the slots of the split schedule, used when whole tiles per CTA would leave
 * the last wave of the tensor-core matmul unbalanced (tiles are then cut between CTAs
 * by 1024-K chunks); a workspace too small for them runs the unsplit schedule, which
 * needs less.
 */
size_t int8_matmul_workspace_size(int T, int in, int out, int max_outlier_cols);

/*
 * The LLM.int8() matmul (all three steps of "core idea").
 *   X         : fp16 [T, in]       activations (hidden states), row-major
 *   CB, SCB   : from int8_quantize_weight for W [out, in]
 *   threshold : a column j is an outlier iff some |X[i,j]| >= threshold. +INF disables the
 *               decomposition (plain vector-wise int8). NaN or <= 0: I8_ERR_INVALID_ARG.
 *   bias      : fp16 [out] or NULL
 *   Y         : fp16 [T, out]      output, Y = acc*rowabs_i*SCB_o/127^2 + outlier + bias
 *   workspace : device buffer of ws_bytes >= int8_matmul_workspace_size(T,in,out,cap).
 *               The outlier capacity used is the largest multiple of 64 columns that fits
 *               in ws_bytes. Contents on entry are ignored. Two calls that run at the same
 *               time must not share a workspace.
 * `in` must be a multiple of 16 and <= I8_MAX_IN; T == 0 or out == 0 is a no-op (with
 * T == 0, X and Y may be NULL).
 * Launches: one memset of the workspace header and three kernels (column statistics,
 * row quantize + outlier gather, matmul). The matmul is the tensor-core kernel, or, for
 * decode sizes, a kernel that streams CB at HBM rate: T <= 8 with T*in <= 200 KB on the
 * CUDA cores (exact int32 dp4a sums), 9 <= T <= 16 with the padded codes in 200 KB on
 * mma.sync (exact fp32 fragments drained to int32). The outlier count stays on the device;
 * no host synchronization.
 */
i8_status int8_matmul(const void* X, int T, int in, const int8_t* CB, const float* SCB, int out,
                      float threshold, const void* bias, void* Y, void* workspace,
                      size_t ws_bytes, void* stream);

/*
 * int8_matmul plus copies of its intermediates, for tests. Each extra pointer may be NULL.
 *   outlier_idx : int32 [in]       ascending outlier columns (first *n_out entries valid)
 *   n_out       : int32 [1]        number of outlier columns
 *   Xq          : int8 [T, in]     activation codes (outlier columns are 0)
 *   rowabs      : fp32 [T]         per-row absmax over inlier columns
 *   acc_s32     : int32 [T, out]   exact int8 product sum_j Xq[i,j]*CB[o,j]
 */
i8_status int8_matmul_debug(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                            int out, float threshold, const void* bias, void* Y,
                            void* workspace, size_t ws_bytes, void* stream,
                            int32_t* outlier_idx, int32_t* n_out, int8_t* Xq, float* rowabs,
                            int32_t* acc_s32);

/*
 * Row-wise absmax quantization ("zeropoint vs absmax", absmax paragraph).
 *   X      : fp16 [rows, cols]  input
 *   Q      : int8 [rows, cols]  codes rint(x * 127/absmax)
 *   absmax : fp32 [rows]        per-row max |x|
 * One kernel launch.
 */
i8_status absmax_quantize_rows(const void* X, int rows, int cols, int8_t* Q, float* absmax,
                               void* stream);

/*
 * Block-wise absmax quantization ("[論文レビュー] The case for 4-bit precision: k-bit Inference
 * Scaling Laws" (nubint review), sections "提案手法" and "主な発見": small blocks of 64-128
 * values, each with its own absmax scale). Each row is cut into blocks of `block`
 * consecutive columns (the last block of a row is shorter when block does not divide
 * cols); each block is quantized as absmax_quantize_rows quantizes a row.
 *   X      : fp16 [rows, cols]                    input
 *   block  : values per block (> 0); block >= cols gives absmax_quantize_rows' result
 *   Q      : int8 [rows, cols]                    codes rint(x * 127/absmax of the block)
 *   absmax : fp32 [rows, ceil(cols / block)]     per-block max |x| (0: codes 0)
 * rows == 0 or cols == 0 is a no-op. One kernel launch; it streams X at HBM rate when
 * cols % 8 == 0 and block is 16, 32, 64, 128 or 256, element by element otherwise.
 */
i8_status absmax_quantize_blocks(const void* X, int rows, int cols, int block, int8_t* Q,
                                 float* absmax, void* stream);

/*
 * Row-wise zeropoint quantization ("Zeropoint Quantization": X8 = INT8(X*S - Z),
 * S = 254/(max - min)). Z = rint(S*min) + 127 is an integer so that 0 maps to an exact
 * code; dequantize with X ~ (Q + Z)/S. A constant row stores S = 0, Z = min, codes 0.
 *   X : fp16 [rows, cols]; Q : int8 [rows, cols]; S, Z : fp32 [rows]. One kernel launch.
 */
i8_status zeropoint_quantize_rows(const void* X, int rows, int cols, int8_t* Q, float* S,
                                  float* Z, void* stream);

/*
 * Our own fp16 GEMM on the same tensor-core pipeline (no int8 step): the 16-bit
 * comparator for the speed trade-off the pages discuss ("speed trade-off"; "INT8 speed").
 *   X : fp16 [T, in]; W : fp16 [out, in]; bias : fp16 [out] or NULL; Y : fp16 [T, out]
 *   Y = X . W^T + bias with fp32 accumulation. `in` a multiple of 16.
 */
i8_status f16_matmul(const void* X, int T, int in, const void* W, int out, const void* bias,
                     void* Y, void* stream);

/*
 * Sums of each weight row's int8 codes, CBsum[o] = sum_j CB[o, j] (int32 [out]): the
 * per-weight input of int8_matmul_zeropoint, computed once with the codes. One launch.
 */
i8_status int8_weight_code_sums(const int8_t* CB, int out, int in, int32_t* CBsum,
                                void* stream);

/*
 * The matmul with zeropoint activation codes ("LLM.int8() summary" (zenn), section
 * "Zeropoint Quantization": X8 = INT8(X16*S - Z), X16 = (X8 + Z)/S, S = 254/(max - min),
 * which uses the whole code range on one-sided rows such as ReLU outputs; "Hugging Face,
 * LLM.int8() ..." (agentlenshq), section "zeropoint vs absmax").
 * Outlier columns are found and multiplied in fp16 exactly as in int8_matmul. Each row's
 * inlier columns are quantized with S = 254/(max - min), Z = rint(S*min) + 127 (min, max
 * over the inlier columns; none: 0, 0), code = clamp(rint(x*S - Z), -127, 127); a row
 * without spread has S = 0, Z = min and codes 0. The weights stay CB/SCB (absmax), so
 *   Y = (acc + Z * sum_{inlier j} CB[o,j]) * SCB[o] / (127 S) + outlier product + bias,
 * acc the exact int32 code product, the correction exact in 64-bit integers; a row without
 * spread contributes Z * sum_{inlier j} CB[o,j] * SCB[o] / 127.
 *   CBsum : int32 [out] from int8_weight_code_sums(CB)
 * Other arguments, the workspace (int8_matmul_workspace_size) and the errors are those of
 * int8_matmul. Every T runs on the tensor-core kernel (no decode-kernel variant).
 * Launches: one memset and three kernels.
 */
i8_status int8_matmul_zeropoint(const void* X, int T, int in, const int8_t* CB,
                                const float* SCB, const int32_t* CBsum, int out,
                                float threshold, const void* bias, void* Y, void* workspace,
                                size_t ws_bytes, void* stream);

/*
 * int8_matmul_zeropoint plus its intermediates, for tests (each extra pointer may be NULL):
 * outlier_idx int32 [in], n_out int32 [1], Xq int8 [T, in] (outlier columns 0),
 * S and Z fp32 [T], acc_s32 int32 [T, out] = sum_j Xq[i,j]*CB[o,j] (without the Z term).
 */
i8_status int8_matmul_zeropoint_debug(const void* X, int T, int in, const int8_t* CB,
                                      const float* SCB, const int32_t* CBsum, int out,
                                      float threshold, const void* bias, void* Y,
                                      void* workspace, size_t ws_bytes, void* stream,
                                      int32_t* outlier_idx, int32_t* n_out, int8_t* Xq,
                                      float* S, float* Z, int32_t* acc_s32);

/* Activation between the two matmuls of int8_ffn / f16_ffn. */
#define I8_ACT_NONE 0
#define I8_ACT_RELU 1

/*
 * Bytes of device workspace int8_ffn needs: the workspaces of its two matmuls (each with
 * an outlier capacity of max_outlier_cols rounded up to 64, at most its own input width;
 * <= 0 means the input width). Returns 0 for invalid sizes.
 */
size_t int8_ffn_workspace_size(int T, int d_model, int d_ff, int max_outlier_cols);

/*
 * An FFN block of two LLM.int8() matmuls, H = act(X . W_up^T + b_up) and
 * Y = H . W_down^T + b_down, each with the decomposition of int8_matmul ("LLM.int8()
 * summary" (zenn), section "INT8 speed": the benchmarked matmul is an FFN layer whose
 * intermediate size is four times the model size).
 *   X                  : fp16 [T, d_model]
 *   CB_up, SCB_up      : int8_quantize_weight of W_up [d_ff, d_model]
 *   CB_down, SCB_down  : int8_quantize_weight of W_down [d_model, d_ff]
 *   bias_up, bias_down : fp16 [d_ff], [d_model] or NULL
 *   threshold          : outlier threshold of both matmuls (as in int8_matmul)
 *   act                : I8_ACT_NONE or I8_ACT_RELU (H = max(y, 0)); else I8_ERR_INVALID_ARG
 *   H                  : fp16 [T, d_ff]    output: the intermediate activations
 *   Y                  : fp16 [T, d_model] output
 *   workspace          : ws_bytes >= int8_ffn_workspace_size(...); the capacity used is the
 *                        largest multiple of 64 columns that fits for both matmuls
 * H and Y are exactly what int8_matmul(X, up) -> act -> int8_matmul(H, down) gives; the
 * difference is where step 1 of the second matmul happens: the first matmul's epilogue
 * applies `act` and ORs each column of H whose fp16 magnitude reaches the threshold into
 * the second matmul's outlier mask, so H is not read an extra time for its column
 * statistics. d_model and d_ff must be multiples of 16 (<= I8_MAX_IN); T == 0 is a no-op
 * (X, H and Y may then be NULL).
 * Launches: two memsets and six kernels. Device errors of either matmul (outlier capacity,
 * timeout) end up in the one status word i8_get_status(workspace) reads, the first one
 * in stream order. With act == I8_ACT_NONE the second matmul's statistics are taken the
 * same way.
 */
i8_status int8_ffn(const void* X, int T, int d_model, int d_ff, const int8_t* CB_up,
                   const float* SCB_up, const void* bias_up, const int8_t* CB_down,
                   const float* SCB_down, const void* bias_down, float threshold, int act,
                   void* H, void* Y, void* workspace, size_t ws_bytes, void* stream);

/*
 * int8_ffn plus the second matmul's outlier columns, for tests (either pointer may be
 * NULL): down_outlier_idx int32 [d_ff] (first *down_n_out valid, ascending),
 * down_n_out int32 [1].
 */
i8_status int8_ffn_debug(const void* X, int T, int d_model, int d_ff, const int8_t* CB_up,
                         const float* SCB_up, const void* bias_up, const int8_t* CB_down,
                         const float* SCB_down, const void* bias_down, float threshold,
                         int act, void* H, void* Y, void* workspace, size_t ws_bytes,
                         void* stream, int32_t* down_outlier_idx, int32_t* down_n_out);

/*
 * The fp16 comparator of int8_ffn: f16_matmul(X, W_up) with `act` in its epilogue, then
 * f16_matmul(H, W_down). W_up fp16 [d_ff, d_model], W_down fp16 [d_model, d_ff]; H, Y as
 * in int8_ffn. Two kernel launches.
 */
i8_status f16_ffn(const void* X, int T, int d_model, int d_ff, const void* W_up,
                  const void* bias_up, const void* W_down, const void* bias_down, int act,
                  void* H, void* Y, void* stream);

/*
 * Synchronizes `stream` and returns the device status word of the last int8_matmul that
 * used this workspace (I8_OK, I8_ERR_OUTLIER_CAP or I8_ERR_TIMEOUT).
 */
i8_status i8_get_status(const void* workspace, void* stream);

/*
 * Test hook for the failure path of the tensor-core matmul (T > 16 tokens, or codes too
 * large for the decode kernels): runs int8_matmul (threshold 6, no bias) but the matmul's
 * loaders load nothing, so every pipeline wait gives up after wait_limit_ns; the kernel then
 * records I8_ERR_TIMEOUT in the workspace status word, frees its tensor memory and returns,
 * and the context stays usable. Read the status with i8_get_status. Y is left undefined.
 * Returns I8_ERR_INVALID_ARG for decode sizes or wait_limit_ns == 0. No counterpart in the
 * pages.
 */
i8_status i8_test_stalled_matmul(const void* X, int T, int in, const int8_t* CB,
                                 const float* SCB, int out, void* Y, void* workspace,
                                 size_t ws_bytes, uint64_t wait_limit_ns, void* stream);

/* Static description of a status code. */
const char* i8_status_string(i8_status s);

/* Number of kernels (and memsets) the last successful call on this host thread launched. */
int i8_last_launch_count(void);

/* Size of the built-in device scratch used by int8_matmul_noalloc (32 MiB per GPU). */
#define I8_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * int8_matmul without a caller-provided workspace, for callers that cannot allocate device
 * memory when they call: applications whose device memory is handed out only by their own
 * allocator (plug-ins, embedded inference runtimes), latency-critical loops that must not
 * call cudaMalloc (it can synchronize the device and takes a driver-wide lock), and code
 * that runs where allocation is not allowed at all. The pages have no counterpart to this
 * call; it is a deployment convenience.
 *
 * Arguments, layouts, results and errors are those of int8_matmul minus the workspace;
 * arguments and the device are checked before the scratch is touched.
 * The scratch is a fixed array of I8_NOALLOC_SCRATCH_BYTES in device memory that every GPU
 * which loads this library reserves until the process exits. Sizes whose workspace (with a
 * 64-column outlier capacity) does not fit return I8_ERR_SCRATCH_LIMIT before any launch;
 * within the limit the outlier capacity is the largest multiple of 64 columns that fits.
 * Roughly: 2*T*in + 132*(T + out) + 4*in + 512*BN*SMs bytes plus a few KB must fit in
 * 32 MiB, with BN the matmul's token tile (16, 32, 64, 128 or, above 128 tokens, 256) and
 * SMs the device's multiprocessor count.
 * - The first call on a device looks up the scratch's device address (once per device and
 *   CUDA context, with that device current); make that first call before any stream
 *   capture. After cudaDeviceReset the next call looks the address up again.
 * - All calls share the one scratch and it keeps the last call's contents; the parts that
 *   must start at zero are cleared by every call. Calls that overlap on the GPU (other
 *   streams, other host threads) race on the scratch: serialize them.
 * - Device-side errors (more outlier columns than the capacity, a wait that timed out) are
 *   recorded in the scratch's status word: read them with i8_noalloc_status.
 * Calls no allocating routine.
 */
i8_status int8_matmul_noalloc(const void* X, int T, int in, const int8_t* CB, const float* SCB,
                              int out, float threshold, const void* bias, void* Y,
                              void* stream);

/*
 * The device status word of the last int8_matmul_noalloc that launched work on the current
 * device (I8_OK, I8_ERR_OUTLIER_CAP or I8_ERR_TIMEOUT; I8_OK before any such call), the
 * counterpart of i8_get_status for the built-in scratch. Synchronizes `stream` first, so
 * that the calls queued on it have finished. No counterpart in the pages.
 */
i8_status i8_noalloc_status(void* stream);

/*
 * Profiling aid. `events` is NULL (off) or an array of 4 cudaEvent_t handles owned by the
 * caller. While set, every int8_matmul / int8_matmul_debug on this host thread records
 * events[0] before the column statistics, events[1] before the quantize pass, events[2]
 * before the matmul kernel and events[3] after it, on the call's stream, so that the
 * caller can time each kernel with cudaEventElapsedTime. Changes nothing else.
 */
void i8_set_profile_events(void** events);

/*
 * The same with n events (at most 8; NULL or n <= 0: off). int8_matmul records events
 * 0..3 as above; int8_ffn / int8_ffn_debug record 0..3 around its first matmul and 4..7
 * around its second (events[4] before the mask compaction that replaces its column
 * statistics). Slots beyond n are not recorded.
 */
void i8_set_profile_events_n(void** events, int n);

#ifdef __cplusplus
}
#endif
#endif /* INT8MM_H_ */
