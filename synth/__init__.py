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
