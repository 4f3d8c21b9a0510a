"""CPU oracle for the LLM.int8() mixed-precision matmul -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The CUDA library never calls it, and it imports nothing from the
CUDA package: the two sides only share the seeded input generators in ``synth``.

The arithmetic lives in ``int8mm_oracle.c`` (plain C, IEEE fp32 for the quantizers, exact
integers for the int8 products, fp64 for the output). This module is numpy marshalling.

The zeropoint variant (``int8_matmul_zeropoint``) quantizes the activations' inlier columns
per row with S and Z (the zenn summary's "Zeropoint Quantization") instead of absmax and
adds the correction Z * (sum of the inlier weight codes) to the exact integer product.

Block-wise absmax (``quantize_blocks_absmax``) gives every block of ``block`` consecutive
columns of a row its own absmax scale (the k-bit scaling review's small blocks of 64-128).

The FFN block (``ffn``) chains two of these matmuls with ReLU (or nothing) between them,
the intermediate rounded once from fp64 to fp16 as the second matmul's input.

Pins (checked by ``tests/test_oracle.py`` without a GPU): the pages' worked absmax example,
an integer-valued case where the method reduces to an exact integer matmul, the
quantization error bounds, threshold = inf reducing to plain vector-wise int8, zeroing the
outlier columns reproducing the inlier product, the zeropoint range and round-trip
bounds, brute-force outlier sets on tiny inputs, and integer-valued FFN blocks (with and
without outlier columns in either matmul) that reduce to exact integer matmuls with ReLU. The quality of the method against
the unquantized product is reported, not pinned (the pages print no per-matmul error).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def load(path: str) -> C.CDLL:
    """Loads an oracle build and declares its C signatures."""
    L = C.CDLL(path)
    p = C.c_void_p
    i64 = C.c_int64
    L.orc_outlier_columns.argtypes = [p, i64, i64, C.c_float, p]
    L.orc_outlier_columns.restype = C.c_int32
    L.orc_quantize_weight.argtypes = [p, i64, i64, p, p]
    L.orc_quantize_rows_absmax.argtypes = [p, i64, i64, p, p, p]
    L.orc_zeropoint_rows.argtypes = [p, i64, i64, p, p, p]
    L.orc_quantize_blocks_absmax.argtypes = [p, i64, i64, i64, p, p]
    L.orc_outlier_weights.argtypes = [p, p, i64, i64, p, C.c_int32, p]
    L.orc_int8_matmul.argtypes = [p, i64, i64, p, p, i64, C.c_float, p, p, i64, p, p, p,
                                  p, p, C.c_int]
    L.orc_int8_matmul.restype = C.c_int32
    L.orc_int8_matmul_zp.argtypes = [p, i64, i64, p, p, i64, C.c_float, p, p, i64, p, p, p,
                                     p, p, p, C.c_int]
    L.orc_int8_matmul_zp.restype = C.c_int32
    L.orc_half_to_float.argtypes = [p, i64, p]
    L.orc_float_to_half.argtypes = [p, i64, p]
    L.orc_activation_to_half.argtypes = [p, i64, C.c_int, p]
    return L


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16, a.dtype
    return a


def default_threads() -> int:
    return os.cpu_count() or 1


def half_to_float(h: np.ndarray) -> np.ndarray:
    h = _f16(h)
    f = np.empty(h.shape, np.float32)
    lib().orc_half_to_float(_ptr(h.view(np.uint16)), h.size, _ptr(f))
    return f


def float_to_half(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    h = np.empty(f.shape, np.uint16)
    lib().orc_float_to_half(_ptr(f), f.size, _ptr(h))
    return h.view(np.float16)


def outlier_columns(X: np.ndarray, threshold: float) -> np.ndarray:
    """Ascending int32 list of columns j with some |X[i,j]| >= threshold."""
    X = _f16(X)
    T, d = X.shape
    idx = np.empty(max(d, 1), np.int32)
    n = lib().orc_outlier_columns(_ptr(X), T, d, float(threshold), _ptr(idx))
    return idx[:n].copy()


def quantize_weight(W: np.ndarray):
    """(CB int8 [out,in], SCB float32 [out]) with W ~ CB * SCB / 127."""
    W = _f16(W)
    out, d = W.shape
    CB = np.empty((out, d), np.int8)
    SCB = np.empty(out, np.float32)
    lib().orc_quantize_weight(_ptr(W), out, d, _ptr(CB), _ptr(SCB))
    return CB, SCB


def quantize_rows_absmax(X: np.ndarray, outlier_mask: np.ndarray | None = None):
    """(Q int8 [rows,cols], absmax float32 [rows]); masked columns excluded and coded 0."""
    X = _f16(X)
    rows, cols = X.shape
    m = None if outlier_mask is None else np.ascontiguousarray(outlier_mask, dtype=np.uint8)
    Q = np.empty((rows, cols), np.int8)
    a = np.empty(rows, np.float32)
    lib().orc_quantize_rows_absmax(_ptr(X), rows, cols, _ptr(m), _ptr(Q), _ptr(a))
    return Q, a


def quantize_blocks_absmax(X: np.ndarray, block: int):
    """(Q int8 [rows,cols], absmax float32 [rows, ceil(cols/block)]): each row cut into
    blocks of `block` columns (the last one shorter if block does not divide cols), each
    block quantized with its own absmax."""
    X = _f16(X)
    rows, cols = X.shape
    if block <= 0:
        raise ValueError("block must be positive")
    nb = (cols + block - 1) // block
    Q = np.empty((rows, cols), np.int8)
    a = np.empty((rows, nb), np.float32)
    lib().orc_quantize_blocks_absmax(_ptr(X), rows, cols, block, _ptr(Q), _ptr(a))
    return Q, a


def zeropoint_rows(X: np.ndarray):
    """(Q int8 [rows,cols], S float32 [rows], Z float32 [rows])."""
    X = _f16(X)
    rows, cols = X.shape
    Q = np.empty((rows, cols), np.int8)
    S = np.empty(rows, np.float32)
    Z = np.empty(rows, np.float32)
    lib().orc_zeropoint_rows(_ptr(X), rows, cols, _ptr(Q), _ptr(S), _ptr(Z))
    return Q, S, Z


def zeropoint_dequant(Q: np.ndarray, S: np.ndarray, Z: np.ndarray) -> np.ndarray:
    """X ~ (Q + Z) / S per row (fp64); a row with S == 0 dequantizes to Z."""
    S = S.astype(np.float64)[:, None]
    Z = Z.astype(np.float64)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        x = (Q.astype(np.float64) + Z) / S
    return np.where(S == 0, np.broadcast_to(Z, Q.shape), x)


def outlier_weights(CB: np.ndarray, SCB: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """fp16 [out, n_out]: the dequantized weight columns of the outlier dimensions."""
    CB = np.ascontiguousarray(CB, dtype=np.int8)
    SCB = np.ascontiguousarray(SCB, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    out, d = CB.shape
    W = np.empty((out, max(idx.size, 1)), np.uint16)
    lib().orc_outlier_weights(_ptr(CB), _ptr(SCB), out, d, _ptr(idx), idx.size, _ptr(W))
    return W[:, : idx.size].view(np.float16).copy()


def int8_matmul(X, CB, SCB, threshold=6.0, bias=None, rows=None, nthreads=None,
                want_acc=True):
    """The LLM.int8() matmul evaluated for the selected rows of X (all rows by default).

    Returns a dict: Y (fp64 [nrows,out]), acc (int64 [nrows,out] or None), Q (int8
    [nrows,in]), rowabs (fp32 [nrows]), idx (int32 outlier columns), rows (int64)."""
    X = _f16(X)
    T, d = X.shape
    CB = np.ascontiguousarray(CB, dtype=np.int8)
    SCB = np.ascontiguousarray(SCB, dtype=np.float32)
    out = CB.shape[0]
    assert CB.shape[1] == d
    b = None if bias is None else _f16(bias)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    nr = rows.size
    Y = np.empty((nr, out), np.float64)
    acc = np.empty((nr, out), np.int64) if want_acc else None
    Q = np.empty((nr, d), np.int8)
    ra = np.empty(nr, np.float32)
    idx = np.empty(max(d, 1), np.int32)
    n = lib().orc_int8_matmul(_ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(b),
                              _ptr(rows), nr, _ptr(Y), _ptr(acc), _ptr(Q), _ptr(ra), _ptr(idx),
                              int(nthreads or default_threads()))
    return {"Y": Y, "acc": acc, "Q": Q, "rowabs": ra, "idx": idx[:n].copy(), "rows": rows}



def int8_matmul_zeropoint(X, CB, SCB, threshold=6.0, bias=None, rows=None, nthreads=None,
                          want_acc=True):
    """The matmul with zeropoint activation codes for the selected rows of X.

    Returns a dict: Y (fp64), acc (int64, codes . CB^T over all columns, outlier codes 0),
    Q (int8), S and Z (fp32 per row), idx (outlier columns), rows."""
    X = _f16(X)
    T, d = X.shape
    CB = np.ascontiguousarray(CB, dtype=np.int8)
    SCB = np.ascontiguousarray(SCB, dtype=np.float32)
    out = CB.shape[0]
    assert CB.shape[1] == d
    b = None if bias is None else _f16(bias)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    nr = rows.size
    Y = np.empty((nr, out), np.float64)
    acc = np.empty((nr, out), np.int64) if want_acc else None
    Q = np.empty((nr, d), np.int8)
    S = np.empty(nr, np.float32)
    Z = np.empty(nr, np.float32)
    idx = np.empty(max(d, 1), np.int32)
    n = lib().orc_int8_matmul_zp(_ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold),
                                 _ptr(b), _ptr(rows), nr, _ptr(Y), _ptr(acc), _ptr(Q), _ptr(S),
                                 _ptr(Z), _ptr(idx), int(nthreads or default_threads()))
    return {"Y": Y, "acc": acc, "Q": Q, "S": S, "Z": Z, "idx": idx[:n].copy(), "rows": rows}

def activation_to_half(y: np.ndarray, relu: bool) -> np.ndarray:
    """fp16(act(y)) for fp64 y: ReLU (y <= 0 -> +0) or identity, one rounding to nearest."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    h = np.empty(y.shape, np.uint16)
    lib().orc_activation_to_half(_ptr(y), y.size, 1 if relu else 0, _ptr(h))
    return h.view(np.float16)


def ffn(X, CB_up, SCB_up, CB_down, SCB_down, threshold=6.0, bias_up=None, bias_down=None,
        act="relu", nthreads=None):
    """FFN block of two LLM.int8() matmuls: H = act(matmul(X, up)) rounded to fp16, then
    Y = matmul(H, down), each matmul with its own outlier decomposition.

    Returns a dict: H_exact (fp64 act of the first matmul's output), H (fp16, the second
    matmul's input), Y (fp64), up_idx and down_idx (the two outlier column sets)."""
    if act not in ("relu", "none"):
        raise ValueError(act)
    up = int8_matmul(X, CB_up, SCB_up, threshold, bias_up, nthreads=nthreads, want_acc=False)
    relu = act == "relu"
    H_exact = np.maximum(up["Y"], 0.0) if relu else up["Y"]
    H = activation_to_half(up["Y"], relu)
    down = int8_matmul(H, CB_down, SCB_down, threshold, bias_down, nthreads=nthreads,
                       want_acc=False)
    return {"H_exact": H_exact, "H": H, "Y": down["Y"], "up_idx": up["idx"],
            "down_idx": down["idx"]}
