/*
 * CPU oracle for the LLM.int8() mixed-precision matmul -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark may load this
 * library. The product path (the CUDA library) never calls it and shares no code with it.
 *
 * It follows the method step by step, in the order the pages state it, with no blocking,
 * fusion or reordering:
 *   "Hugging Face, LLM.int8() ... integrated into Transformers and Accelerate"
 *     (agentlenshq summary) -- section "core idea": (1) outlier extraction by column with a
 *     magnitude threshold of about 6, (2) outliers multiplied in 16 bit while the rest is
 *     quantized to int8 vector-wise (rows of the activations, columns of the weight), (3) the
 *     int8 result dequantized and added to the fp16 outlier result.
 *     Section "zeropoint vs absmax": absmax scaling by 127/absmax and rounding
 *     (worked example: absmax 5.4 gives scale 127/5.4 ~ 23.5).
 *     Section "transformers integration": weights stored as int8 CB in [-127,127] with
 *     W ~ (CB * SCB) / 127.
 *   "LLM.int8() summary" (zenn, bilzard) -- section "method": decomposition by input
 *     dimension, the matching weight dimensions split too, outliers kept in 16 bit;
 *     section "Zeropoint Quantization": X8 = INT8(X16*S - Z), X16 = (X8 + Z)/S,
 *     S = 254/(max - min).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - a column is an outlier iff some |x| >= threshold (threshold compared in fp32);
 *   - scale s = 127.0f / absmax as one IEEE fp32 division, code = rint(x * s) as one fp32
 *     multiply (no contraction) rounded half-to-even, clamped to [-127, 127];
 *   - absmax 0 (all-zero or all-outlier row, all-zero weight row) gives scale 0 and codes 0;
 *   - outlier weights are the dequantized codes rounded to fp16: fp16((CB * SCB) / 127);
 *   - Z = rint(S * min) + 127 (an integer), codes = clamp(rint(x*S - Z)); max == min gives
 *     S = 0, Z = min, codes 0.
 *
 * Floating point: fp32 where the method fixes it (the quantizers), fp64 for the output.
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared -pthread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* fp16 <-> fp32 conversion through the compiler's IEEE binary16 type. */
static float h2f(uint16_t bits) {
  _Float16 h;
  memcpy(&h, &bits, sizeof h);
  return (float)h;
}
static uint16_t f2h(float f) {
  _Float16 h = (_Float16)f; /* round to nearest even */
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

static int8_t clamp_code(float r) {
  if (r > 127.0f) return 127;
  if (r < -127.0f) return -127;
  return (int8_t)r;
}

/* absmax code: rint(x * s) with s = 127/absmax (fp32), clamped. */
static int8_t absmax_code(float x, float s) {
  float p = x * s;           /* one IEEE fp32 multiply */
  return clamp_code(rintf(p)); /* round half to even (default rounding mode) */
}

static float absmax_scale(float absmax) {
  return absmax > 0.0f ? 127.0f / absmax : 0.0f;
}

void orc_half_to_float(const uint16_t* h, int64_t n, float* f) {
  for (int64_t i = 0; i < n; ++i) f[i] = h2f(h[i]);
}
void orc_float_to_half(const float* f, int64_t n, uint16_t* h) {
  for (int64_t i = 0; i < n; ++i) h[i] = f2h(f[i]);
}

/* Step 1, outlier extraction: column j of X [T, in] is an outlier iff some row has
 * |X[i,j]| >= threshold. Writes the ascending column list to idx (capacity in) and
 * returns the count. */
int32_t orc_outlier_columns(const uint16_t* X, int64_t T, int64_t in, float threshold,
                            int32_t* idx) {
  int32_t n = 0;
  for (int64_t j = 0; j < in; ++j) {
    int hit = 0;
    for (int64_t i = 0; i < T && !hit; ++i)
      if (fabsf(h2f(X[i * in + j])) >= threshold) hit = 1;
    if (hit) idx[n++] = (int32_t)j;
  }
  return n;
}

/* Vector-wise weight quantization: for each output row o of W [out, in],
 * SCB[o] = max_j |W[o,j]|, CB[o,j] = clamp(rint(W[o,j] * (127/SCB[o]))). */
void orc_quantize_weight(const uint16_t* W, int64_t out, int64_t in, int8_t* CB, float* SCB) {
  for (int64_t o = 0; o < out; ++o) {
    const uint16_t* w = W + o * in;
    float a = 0.0f;
    for (int64_t j = 0; j < in; ++j) {
      float v = fabsf(h2f(w[j]));
      if (v > a) a = v;
    }
    SCB[o] = a;
    float s = absmax_scale(a);
    for (int64_t j = 0; j < in; ++j) CB[o * in + j] = absmax_code(h2f(w[j]), s);
  }
}

/* Row-wise absmax quantization of X [rows, cols]. Columns flagged in `outlier`
 * (nullable, one byte per column) are excluded from the absmax and get code 0. */
void orc_quantize_rows_absmax(const uint16_t* X, int64_t rows, int64_t cols,
                              const uint8_t* outlier, int8_t* Q, float* absmax) {
  for (int64_t i = 0; i < rows; ++i) {
    const uint16_t* x = X + i * cols;
    float a = 0.0f;
    for (int64_t j = 0; j < cols; ++j) {
      if (outlier && outlier[j]) continue;
      float v = fabsf(h2f(x[j]));
      if (v > a) a = v;
    }
    absmax[i] = a;
    float s = absmax_scale(a);
    for (int64_t j = 0; j < cols; ++j)
      Q[i * cols + j] = (outlier && outlier[j]) ? 0 : absmax_code(h2f(x[j]), s);
  }
}

/* Block-wise absmax quantization ("[論文レビュー] The case for 4-bit precision: k-bit
 * Inference Scaling Laws" (nubint review), sections "提案手法" and "主な発見": the block size
 * is a parameter of the quantizer, small blocks of 64-128 values each with their own
 * normalization). Reading: each row of X [rows, cols] is cut into blocks of `block`
 * consecutive columns, the last block of a row shorter when block does not divide cols;
 * block k of row i holds absmax[i * nblocks + k] = max |x| over its columns and the codes
 * clamp(rint(x * (127/absmax))) as in the row-wise quantizer (absmax 0: codes 0). */
void orc_quantize_blocks_absmax(const uint16_t* X, int64_t rows, int64_t cols, int64_t block,
                                int8_t* Q, float* absmax) {
  const int64_t nblocks = (cols + block - 1) / block;
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t k = 0; k < nblocks; ++k) {
      const int64_t j0 = k * block;
      const int64_t j1 = (j0 + block < cols) ? j0 + block : cols;
      float a = 0.0f;
      for (int64_t j = j0; j < j1; ++j) {
        float v = fabsf(h2f(X[i * cols + j]));
        if (v > a) a = v;
      }
      absmax[i * nblocks + k] = a;
      float s = absmax_scale(a);
      for (int64_t j = j0; j < j1; ++j) Q[i * cols + j] = absmax_code(h2f(X[i * cols + j]), s);
    }
  }
}

/* Zeropoint (asymmetric) quantization of one row, X8 = INT8(X*S - Z) with
 * S = 254/(max-min) and Z = rint(S*min) + 127, so that min maps to -127, max to +127 and 0
 * to the integer -Z. min and max are taken over the columns not flagged in `outlier`
 * (nullable); flagged columns get code 0. No such column: min = max = 0. A constant row
 * stores S = 0, Z = min and codes 0. */
static void zeropoint_row(const uint16_t* x, int64_t cols, const uint8_t* outlier, int8_t* q,
                          float* S, float* Z) {
  float mn = INFINITY, mx = -INFINITY;
  int any = 0;
  for (int64_t j = 0; j < cols; ++j) {
    if (outlier && outlier[j]) continue;
    float v = h2f(x[j]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
    any = 1;
  }
  if (!any) { mn = 0.0f; mx = 0.0f; }
  if (mx > mn) {
    float range = mx - mn;         /* fp32 subtraction */
    float s = 254.0f / range;      /* fp32 division */
    float z = rintf(s * mn) + 127.0f;
    *S = s;
    *Z = z;
    for (int64_t j = 0; j < cols; ++j) {
      if (outlier && outlier[j]) { q[j] = 0; continue; }
      float p = h2f(x[j]) * s;     /* fp32 multiply */
      float t = p - z;             /* fp32 subtract, not fused */
      q[j] = clamp_code(rintf(t));
    }
  } else {
    *S = 0.0f;
    *Z = mn;
    for (int64_t j = 0; j < cols; ++j) q[j] = 0;
  }
}

void orc_zeropoint_rows(const uint16_t* X, int64_t rows, int64_t cols, int8_t* Q, float* S,
                        float* Z) {
  for (int64_t i = 0; i < rows; ++i)
    zeropoint_row(X + i * cols, cols, NULL, Q + i * cols, &S[i], &Z[i]);
}

/* FFN block intermediate: H = fp16(act(y)) for the fp64 output y of the first matmul,
 * act = identity (relu == 0) or ReLU (max(y, 0); y <= 0 gives +0). One rounding from
 * fp64 to fp16, to nearest even. */
void orc_activation_to_half(const double* y, int64_t n, int relu, uint16_t* h) {
  for (int64_t i = 0; i < n; ++i) {
    double v = y[i];
    if (relu && !(v > 0.0)) v = 0.0;
    _Float16 t = (_Float16)v;
    memcpy(&h[i], &t, sizeof t);
  }
}

/* ---------------------------------------------------------------- full matmul */

typedef struct {
  /* shared inputs */
  const uint16_t* X;
  int64_t T, in, out;
  const int8_t* CB;
  const float* SCB;
  const uint16_t* bias;
  const int64_t* rows;
  int64_t nrows;
  const int32_t* idx;
  int32_t n_out;
  const int8_t* Q;       /* [nrows, in] codes of the selected rows */
  const float* rowabs;   /* [nrows] */
  const uint16_t* Wout;  /* [out, n_out] fp16 dequantized outlier weights */
  /* zeropoint variant (zp != 0): per selected row S and Z, per output the sum of the
   * weight codes over the inlier columns */
  int zp;
  const float* rowS;
  const float* rowZ;
  const int64_t* cbin;
  /* outputs */
  double* Y;             /* [nrows, out] */
  int64_t* acc;          /* [nrows, out] nullable */
  /* work split: output features [o0, o1) */
  int64_t o0, o1;
} mm_job;

static void* mm_worker(void* p) {
  mm_job* jb = (mm_job*)p;
  for (int64_t r = 0; r < jb->nrows; ++r) {
    const int8_t* q = jb->Q + r * jb->in;
    const uint16_t* x = jb->X + jb->rows[r] * jb->in;
    for (int64_t o = jb->o0; o < jb->o1; ++o) {
      const int8_t* c = jb->CB + o * jb->in;
      /* int8 x int8 products summed exactly in 64-bit integers */
      int64_t a = 0;
      for (int64_t j = 0; j < jb->in; ++j) a += (int64_t)q[j] * (int64_t)c[j];
      /* 16-bit outlier product: fp16 activations times fp16 dequantized weights */
      double f = 0.0;
      for (int32_t k = 0; k < jb->n_out; ++k)
        f += (double)h2f(x[jb->idx[k]]) * (double)h2f(jb->Wout[o * jb->n_out + k]);
      double y;
      if (!jb->zp) {
        /* dequantize: x ~ q*absmax/127 and w ~ CB*SCB/127 */
        y = (double)a * (double)jb->rowabs[r] * (double)jb->SCB[o] / (127.0 * 127.0);
      } else if (jb->rowS[r] != 0.0f) {
        /* x ~ (q + Z)/S over the inlier columns: sum_j (q_j + Z) CB_j = a + Z * cbin */
        double az = (double)a + (double)jb->rowZ[r] * (double)jb->cbin[o];
        y = az * (double)jb->SCB[o] / (127.0 * (double)jb->rowS[r]);
      } else {
        /* constant inlier row: every inlier x is Z (= min) */
        y = (double)jb->rowZ[r] * (double)jb->cbin[o] * (double)jb->SCB[o] / 127.0;
      }
      y += f;
      if (jb->bias) y += (double)h2f(jb->bias[o]);
      jb->Y[r * jb->out + o] = y;
      if (jb->acc) jb->acc[r * jb->out + o] = a;
    }
  }
  return NULL;
}

/* Outlier weight slice: Wout[o,k] = fp16((CB[o, idx[k]] * SCB[o]) / 127), the 16-bit
 * weights of the outlier input dimensions recovered from the int8 weights. */
void orc_outlier_weights(const int8_t* CB, const float* SCB, int64_t out, int64_t in,
                         const int32_t* idx, int32_t n_out, uint16_t* Wout) {
  for (int64_t o = 0; o < out; ++o)
    for (int32_t k = 0; k < n_out; ++k) {
      float w = ((float)CB[o * in + idx[k]] * SCB[o]) / 127.0f;
      Wout[o * n_out + k] = f2h(w);
    }
}

/* The LLM.int8() matmul for selected rows of X:
 *   1. outlier columns of X (over all T rows);
 *   2. row codes of the selected rows over inlier columns (outliers -> 0): absmax, or in
 *      the zeropoint variant (zp != 0) zeropoint with S and Z per row;
 *   3. acc = codes . CB^T exactly; outlier product in fp64 from fp16 operands;
 *   4. Y = acc * rowabs * SCB / 127^2 + outlier product + bias   (fp64), or with zeropoint
 *      codes Y = (acc + Z * sum of the inlier weight codes) * SCB / (127 S) + ... .
 * Outputs (all caller-allocated): Y [nrows,out]; acc [nrows,out] (nullable);
 * Q [nrows,in]; rowabs [nrows] (absmax) or S, Z [nrows] (zeropoint; rowabs unused);
 * idx [in]; returns n_out. nthreads <= 0 means 1. */
static int32_t int8_matmul_any(const uint16_t* X, int64_t T, int64_t in, const int8_t* CB,
                               const float* SCB, int64_t out, float threshold,
                               const uint16_t* bias, const int64_t* rows, int64_t nrows,
                               double* Y, int64_t* acc, int8_t* Q, float* rowabs, int zp,
                               float* S, float* Z, int32_t* idx, int nthreads) {
  int32_t n_out = orc_outlier_columns(X, T, in, threshold, idx);
  uint8_t* mask = (uint8_t*)calloc((size_t)(in > 0 ? in : 1), 1);
  for (int32_t k = 0; k < n_out; ++k) mask[idx[k]] = 1;
  int64_t* cbin = NULL;
  for (int64_t r = 0; r < nrows; ++r) {
    if (zp)
      zeropoint_row(X + rows[r] * in, in, mask, Q + r * in, &S[r], &Z[r]);
    else
      orc_quantize_rows_absmax(X + rows[r] * in, 1, in, mask, Q + r * in, rowabs + r);
  }
  if (zp) {
    cbin = (int64_t*)calloc((size_t)(out > 0 ? out : 1), sizeof(int64_t));
    for (int64_t o = 0; o < out; ++o)
      for (int64_t j = 0; j < in; ++j)
        if (!mask[j]) cbin[o] += CB[o * in + j];
  }
  uint16_t* Wout = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(out * (n_out > 0 ? n_out : 1)));
  orc_outlier_weights(CB, SCB, out, in, idx, n_out, Wout);

  if (nthreads < 1) nthreads = 1;
  if (nthreads > out && out > 0) nthreads = (int)out;
  if (nthreads < 1) nthreads = 1;
  mm_job* jobs = (mm_job*)calloc((size_t)nthreads, sizeof(mm_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    mm_job j = {X, T, in, out, CB, SCB, bias, rows, nrows, idx, n_out, Q, rowabs, Wout,
                zp, S, Z, cbin, Y, acc, out * t / nthreads, out * (t + 1) / nthreads};
    jobs[t] = j;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, mm_worker, &jobs[t]);
  mm_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  free(Wout);
  free(cbin);
  free(mask);
  return n_out;
}

int32_t orc_int8_matmul(const uint16_t* X, int64_t T, int64_t in, const int8_t* CB,
                        const float* SCB, int64_t out, float threshold, const uint16_t* bias,
                        const int64_t* rows, int64_t nrows, double* Y, int64_t* acc, int8_t* Q,
                        float* rowabs, int32_t* idx, int nthreads) {
  return int8_matmul_any(X, T, in, CB, SCB, out, threshold, bias, rows, nrows, Y, acc, Q,
                         rowabs, 0, NULL, NULL, idx, nthreads);
}

/* Zeropoint variant ("LLM.int8() summary" (zenn), section "Zeropoint Quantization", applied
 * to the activations of the decomposed matmul; the weights stay CB/SCB): S and Z [nrows]. */
int32_t orc_int8_matmul_zp(const uint16_t* X, int64_t T, int64_t in, const int8_t* CB,
                           const float* SCB, int64_t out, float threshold, const uint16_t* bias,
                           const int64_t* rows, int64_t nrows, double* Y, int64_t* acc,
                           int8_t* Q, float* S, float* Z, int32_t* idx, int nthreads) {
  return int8_matmul_any(X, T, in, CB, SCB, out, threshold, bias, rows, nrows, Y, acc, Q,
                         NULL, 1, S, Z, idx, nthreads);
}
