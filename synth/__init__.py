"""Seeded synthetic inputs shaped like the LLM.int8() FFN workloads.

This module only draws random numbers; it holds none of the method's arithmetic, so the
CPU oracle (``oracle/``) and the CUDA path can both be fed from it without sharing code.

Recipe (every tensor comes from ``numpy.random.default_rng((base_seed, sub_seed))``):

* X: N(0, x_std) drawn in float32, cast to float16 (round to nearest).
* outlier columns: ``choice(d_in, k, replace=False)``, sorted ascending.
* outlier values: for each (row, outlier column) an independent Bernoulli(row_frac)
  decides whether the entry is replaced; the replacement is sign * U[lo, hi] with a fair
  random sign, again drawn in float32 and cast to float16.
* W: N(0, w_std) in float32 -> float16, generated in blocks of rows from one generator.
* bias: N(0, 0.01) float32 -> float16.
* zeropoint input: |N(0, 1)| (a ReLU-like, one-sided distribution).

FFN blocks (``FfnWorkload``, X -> up projection -> ReLU -> down projection), with random
weights in place of trained ones:

* X as above (outlier columns of the up projection's input);
* W_up: N(0, s) with s chosen so that the up projection's output has standard deviation
  pre_std: s = pre_std / sqrt(E[sum_j x_j^2]), the expectation taken over the recipe of X
  (inlier columns N(0, 1), outlier columns replaced with probability row_frac);
* outlier features of H: choice(d_ff, k_h) columns (sorted) whose up-projection bias is
  U[lo, hi] (positive, so they pass the ReLU and every row of them exceeds the threshold);
  the other biases N(0, 0.01);
* W_down: N(0, w_down_std); b_down: N(0, 0.01).

The shapes and outlier statistics follow the pages' description of the workload:
about 0.1% of hidden dimensions carry outliers of magnitude well above the threshold of 6
("LLM.int8(): 8-bit Matrix Multiplication for Transformers at Scale" summary, sections on
outliers and decomposition), and the benchmarked matmul is the first FFN layer, whose
intermediate size is four times the model size (same summary, INT8 speed section).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
import math

import numpy as np

SUB_X, SUB_W, SUB_BIAS, SUB_COLS, SUB_OUTLIER, SUB_ZP = 0, 1, 2, 3, 4, 5
SUB_W_UP, SUB_B_UP, SUB_W_DOWN, SUB_B_DOWN, SUB_H_COLS, SUB_H_MAG = 6, 7, 8, 9, 10, 11


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens (rows of X)
    d_in: int         # input features (columns of X, K of the matmul)
    d_out: int        # output features (rows of W)
    x_std: float = 1.0
    w_std: float = 0.02
    n_outlier_cols: int = 0
    outlier_lo: float = 8.0
    outlier_hi: float = 60.0
    row_frac: float = 0.9
    threshold: float = 6.0
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _k(frac: float, d: int) -> int:
    """Number of outlier columns for a fraction of d, rounded to nearest."""
    return int(math.floor(frac * d + 0.5))


WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("tiny", 16, 256, 1024, n_outlier_cols=2, outlier_lo=8, outlier_hi=40, row_frac=1.0))
_add(Workload("ffn_6.7b_up", 2048, 4096, 16384, n_outlier_cols=_k(0.001, 4096)))
_add(Workload("ffn_13b_up", 4096, 5120, 20480, n_outlier_cols=_k(0.002, 5120)))
_add(Workload("ffn_13b_down", 4096, 20480, 5120, x_std=0.5, w_std=0.01,
              n_outlier_cols=_k(0.001, 20480)))
for _t in (1, 8, 64):
    _add(Workload(f"decode_176b_t{_t}", _t, 14336, 57344, n_outlier_cols=_k(0.001, 14336),
                  row_frac=1.0))
for _f, _tag in ((0.0, "0"), (0.001, "0.1"), (0.005, "0.5"), (0.02, "2")):
    for _thr, _ttag in ((6.0, "6"), (math.inf, "inf")):
        _add(Workload(f"sweep_f{_tag}_thr{_ttag}", 1024, 8192, 32768,
                      n_outlier_cols=_k(_f, 8192), outlier_lo=8, outlier_hi=100,
                      threshold=_thr))


@dataclass(frozen=True)
class FfnWorkload:
    name: str
    T: int
    d_model: int
    d_ff: int
    x_outlier_frac: float = 0.002   # outlier columns of X (13B: 10 of 5120)
    h_outlier_frac: float = 0.001   # outlier features of H (13B: 20 of 20480)
    min_outlier_cols: int = 1
    outlier_lo: float = 8.0
    outlier_hi: float = 60.0
    row_frac: float = 0.9
    pre_std: float = 0.5            # std of the up projection's output (13B down: X ~ N(0, 0.5))
    w_down_std: float = 0.01
    threshold: float = 6.0
    seed: int = 0

    def with_(self, **kw) -> "FfnWorkload":
        return replace(self, **kw)

    def x_workload(self) -> Workload:
        k = max(self.min_outlier_cols, _k(self.x_outlier_frac, self.d_model))
        return Workload(self.name + "/x", self.T, self.d_model, self.d_ff,
                        n_outlier_cols=min(k, self.d_model), outlier_lo=self.outlier_lo,
                        outlier_hi=self.outlier_hi, row_frac=self.row_frac,
                        threshold=self.threshold, seed=self.seed)

    def n_h_outliers(self) -> int:
        return min(self.d_ff, max(self.min_outlier_cols, _k(self.h_outlier_frac, self.d_ff)))


FFN_WORKLOADS: dict[str, FfnWorkload] = {}
for _f in (FfnWorkload("ffn_13b_block", 4096, 5120, 20480),
           FfnWorkload("ffn_small", 200, 256, 1024, min_outlier_cols=2),
           FfnWorkload("ffn_decode_t8", 8, 1024, 4096, min_outlier_cols=2),
           FfnWorkload("ffn_decode_t13", 13, 512, 2048, min_outlier_cols=2)):
    FFN_WORKLOADS[_f.name] = _f


def rng(w: Workload, sub: int) -> np.random.Generator:
    return np.random.default_rng((w.seed, sub))


def outlier_columns(w: Workload) -> np.ndarray:
    """The columns the generator plants outliers in (sorted, int64)."""
    if w.n_outlier_cols == 0:
        return np.zeros(0, dtype=np.int64)
    cols = rng(w, SUB_COLS).choice(w.d_in, w.n_outlier_cols, replace=False)
    return np.sort(cols).astype(np.int64)


def make_x(w: Workload) -> np.ndarray:
    """X float16 [T, d_in] with planted outlier columns."""
    x = rng(w, SUB_X).standard_normal((w.T, w.d_in), dtype=np.float32) * np.float32(w.x_std)
    cols = outlier_columns(w)
    if cols.size:
        g = rng(w, SUB_OUTLIER)
        hit = g.random((w.T, cols.size)) < w.row_frac
        sign = np.where(g.random((w.T, cols.size)) < 0.5, -1.0, 1.0).astype(np.float32)
        mag = g.uniform(w.outlier_lo, w.outlier_hi, (w.T, cols.size)).astype(np.float32)
        x[:, cols] = np.where(hit, sign * mag, x[:, cols])
    return x.astype(np.float16)


def make_w(w: Workload, block_rows: int = 4096) -> np.ndarray:
    """W float16 [d_out, d_in], drawn block of rows by block of rows from one generator."""
    g = rng(w, SUB_W)
    out = np.empty((w.d_out, w.d_in), dtype=np.float16)
    for r0 in range(0, w.d_out, block_rows):
        r1 = min(w.d_out, r0 + block_rows)
        blk = g.standard_normal((r1 - r0, w.d_in), dtype=np.float32) * np.float32(w.w_std)
        out[r0:r1] = blk.astype(np.float16)
    return out


def make_bias(w: Workload) -> np.ndarray:
    b = rng(w, SUB_BIAS).standard_normal(w.d_out, dtype=np.float32) * np.float32(0.01)
    return b.astype(np.float16)


def make_relu_like(w: Workload) -> np.ndarray:
    """|N(0,1)| float16 [T, d_in]: one-sided input for the zeropoint row quantizer."""
    x = np.abs(rng(w, SUB_ZP).standard_normal((w.T, w.d_in), dtype=np.float32))
    return x.astype(np.float16)


def make_random_f16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """Generic seeded N(0, std) float16 tensor for ragged/edge-case tests."""
    g = np.random.default_rng((seed, 99))
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float16)


def make_random_int(seed: int, shape, lo: int, hi: int) -> np.ndarray:
    """Seeded integers in [lo, hi] (int64)."""
    g = np.random.default_rng((seed, 98))
    return g.integers(lo, hi + 1, size=shape, dtype=np.int64)


def _frng(f: FfnWorkload, sub: int) -> np.random.Generator:
    return np.random.default_rng((f.seed, sub))


def make_ffn(f: FfnWorkload, block_rows: int = 4096) -> dict:
    """X, W_up, b_up, W_down, b_down (float16) and h_cols (planted outlier features of H)."""
    xw = f.x_workload()
    X = make_x(xw)
    k = xw.n_outlier_cols
    u2 = (xw.outlier_lo ** 2 + xw.outlier_lo * xw.outlier_hi + xw.outlier_hi ** 2) / 3.0
    energy = (f.d_model - k) + k * (f.row_frac * u2 + (1.0 - f.row_frac))
    s_up = f.pre_std / math.sqrt(energy)

    def normal_rows(sub, rows, cols, std):
        g = _frng(f, sub)
        out = np.empty((rows, cols), dtype=np.float16)
        for r0 in range(0, rows, block_rows):
            r1 = min(rows, r0 + block_rows)
            out[r0:r1] = (g.standard_normal((r1 - r0, cols), dtype=np.float32)
                          * np.float32(std)).astype(np.float16)
        return out

    W_up = normal_rows(SUB_W_UP, f.d_ff, f.d_model, s_up)
    W_down = normal_rows(SUB_W_DOWN, f.d_model, f.d_ff, f.w_down_std)
    b_up = (_frng(f, SUB_B_UP).standard_normal(f.d_ff, dtype=np.float32)
            * np.float32(0.01))
    h_cols = np.sort(_frng(f, SUB_H_COLS).choice(f.d_ff, f.n_h_outliers(), replace=False))
    b_up[h_cols] = _frng(f, SUB_H_MAG).uniform(f.outlier_lo, f.outlier_hi,
                                              h_cols.size).astype(np.float32)
    b_down = (_frng(f, SUB_B_DOWN).standard_normal(f.d_model, dtype=np.float32)
              * np.float32(0.01))
    return {"X": X, "W_up": W_up, "b_up": b_up.astype(np.float16), "W_down": W_down,
            "b_down": b_down.astype(np.float16), "h_cols": h_cols.astype(np.int64)}


def make_integer_ffn(seed: int, T: int, d_model: int, d_ff: int, outliers: bool,
                     n_big: int = 3) -> dict:
    """Integer-valued FFN inputs whose LLM.int8() evaluation is exact (float16 arrays).

    Every weight row holds values in {-1, 0, 1} with at least one nonzero, so its absmax is
    1 and its codes are 127 * w. X holds {-1, 0, 1}, except column 0, which is 8 when
    `outliers` (an outlier column at threshold 6) and 1 otherwise. The up projection has
    `n_big` "big" features (only with `outliers`): weight 1 on column 0 plus at most two
    more nonzeros, so their output lies in [6, 10] for every token (outlier features of H
    at threshold 6). Every other feature has a single nonzero weight off column 0, so its
    output is in {-1, 0, 1}. b_down holds integers in [-2, 2]; there is no up bias.
    Returns X, W_up, W_down, b_down and big (the big features, sorted)."""
    g = np.random.default_rng((seed, 97))
    X = g.integers(-1, 2, size=(T, d_model)).astype(np.float16)
    X[:, 0] = 8 if outliers else 1
    W_up = np.zeros((d_ff, d_model), np.float16)
    big = np.sort(g.choice(d_ff, n_big, replace=False)) if outliers else np.zeros(0, np.int64)
    for o in range(d_ff):
        if o in big:
            W_up[o, 0] = 1
            extra = g.choice(np.arange(1, d_model), 2, replace=False)
            W_up[o, extra] = g.integers(-1, 2, size=2)
        else:
            W_up[o, g.integers(1, d_model)] = 1 if g.random() < 0.5 else -1
    W_down = g.integers(-1, 2, size=(d_model, d_ff)).astype(np.float16)
    W_down[np.arange(d_model), g.integers(0, d_ff, size=d_model)] = 1
    b_down = g.integers(-2, 3, size=d_model).astype(np.float16)
    return {"X": X, "W_up": W_up, "W_down": W_down, "b_down": b_down,
            "big": big.astype(np.int64)}
