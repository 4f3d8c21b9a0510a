"""Pins for the CPU oracle: checks against what the pages and plain mathematics fix.

None of these tests retypes the oracle's formulas to compare the oracle with itself. Each
compares it with a value the pages print, an exact rational computation, a closed-form
special case that reduces to an integer matmul (a library routine), an error bound, or a
brute-force enumeration on tiny inputs.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rne(fr: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even (exact)."""
    return round(fr)


# --------------------------------------------------------------------------- worked example
def test_absmax_worked_example_from_page():
    g = json.load(open(os.path.join(GOLDEN, "absmax_worked_example.json")))
    x = np.array([g["vector_printed"]], dtype=np.float16)
    Q, a = oracle.quantize_rows_absmax(x)
    # absmax is the fp16 value of the printed 5.4
    assert a[0] == np.float32(np.float16(g["absmax_printed"]))
    scale = 127.0 / float(a[0])
    assert abs(scale - g["scale_printed"]) <= 0.05
    lo, hi = g["code_range_printed"]
    assert Q.min() >= lo and Q.max() <= hi
    # the codes, derived in exact rational arithmetic from the fp16 inputs
    amax = Fraction(float(a[0]))
    expect = [rne(Fraction(float(v)) * 127 / amax) for v in x[0]]
    assert Q[0].tolist() == expect == [28, -12, -101, 127]


def test_int8_weight_footprint_matches_page_memory_example():
    """The page's 7B example stores the weights in a quarter of their fp32 bytes (the size
    estimator counts one byte per parameter). The quantized weight format's codes take the
    same quarter, inside the rounding of the printed sizes; its one fp32 scale per output
    feature comes on top (4 bytes per row of `in` codes)."""
    g = json.load(open(os.path.join(GOLDEN, "int8_memory_example.json")))
    lo = (g["fp32_gb_printed"] - 0.005) / (g["int8_gb_printed"] + 0.005)
    hi = (g["fp32_gb_printed"] + 0.005) / (g["int8_gb_printed"] - 0.005)
    assert lo <= g["ratio_printed"] <= hi
    rng = np.random.default_rng(11)
    out, d = 256, 4096  # rows of a 7B-class layer (hidden size 4096)
    W = (rng.standard_normal((out, d)) * 0.02).astype(np.float16)
    CB, SCB = oracle.quantize_weight(W)
    assert CB.dtype == np.int8 and CB.shape == (out, d)
    assert SCB.dtype == np.float32 and SCB.shape == (out,)
    ratio = (4 * W.size) / CB.nbytes
    assert lo <= ratio <= hi, ratio
    assert SCB.nbytes == 4 * out


# --------------------------------------------------------------------------- fp16 handling
def test_half_conversions_match_numpy():
    g = np.random.default_rng(7)
    f = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 100,
        g.standard_normal(2000).astype(np.float32) * 1e-6,           # subnormal halves
        np.array([65504, 65519.99, 65520, -65520, 1e6, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
                  0.0, -0.0, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11], np.float32),  # ties
    ])
    h = oracle.float_to_half(f)
    ref = f.astype(np.float16)
    assert np.array_equal(h.view(np.uint16), ref.view(np.uint16))
    allh = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    finite = np.isfinite(allh)
    back = oracle.half_to_float(allh[finite])
    assert np.array_equal(back, allh[finite].astype(np.float32))


# --------------------------------------------------------------------------- outlier columns
def brute_outliers(X, thr):
    T, d = X.shape
    return [j for j in range(d) if any(abs(float(X[i, j])) >= thr for i in range(T))]


def test_outlier_columns_threshold_edge_and_bruteforce():
    X = np.zeros((3, 9), np.float16)
    X[0, 1] = 6.0                       # exactly at the threshold: an outlier (>=)
    X[1, 2] = np.float16(5.99609375)    # largest fp16 below 6: not an outlier
    X[2, 4] = -6.0                      # magnitude counts, sign does not
    X[1, 7] = 100.0
    X[0, 8] = -5.0
    got = oracle.outlier_columns(X, 6.0).tolist()
    assert got == [1, 4, 7] == brute_outliers(X, 6.0)
    assert oracle.outlier_columns(X, math.inf).tolist() == []
    g = np.random.default_rng(3)
    for trial in range(30):
        T, d = g.integers(1, 6), g.integers(1, 12)
        Xr = (g.standard_normal((T, d)) * 4).astype(np.float16)
        thr = float(g.choice([0.5, 2.0, 6.0, 7.25]))
        assert oracle.outlier_columns(Xr, thr).tolist() == brute_outliers(Xr, thr)


def test_tiny_workload_outliers_are_the_planted_columns():
    w = synth.WORKLOADS["tiny"]
    X = synth.make_x(w)
    assert oracle.outlier_columns(X, w.threshold).tolist() == synth.outlier_columns(w).tolist()


# --------------------------------------------------------------------------- weights
def test_weight_quantization_roundtrip_bound_and_range():
    w = synth.WORKLOADS["tiny"]
    W = synth.make_w(w)
    W[5] = 0                                  # an all-zero row
    CB, SCB = oracle.quantize_weight(W)
    Wf = W.astype(np.float64)
    assert SCB[5] == 0 and not CB[5].any()
    np.testing.assert_array_equal(SCB, np.abs(Wf).max(axis=1).astype(np.float32))
    assert CB.min() >= -127 and CB.max() <= 127
    nz = SCB > 0
    assert (np.abs(CB[nz].astype(np.int32)).max(axis=1) == 127).all()
    err = np.abs(Wf - CB.astype(np.float64) * SCB[:, None].astype(np.float64) / 127.0)
    bound = SCB[:, None].astype(np.float64) * (1.0 / 254 + 2.0**-22)
    assert (err <= bound).all()


def test_weight_quantization_integer_rows_are_exact():
    W = synth.make_random_int(11, (6, 40), -127, 127)
    W[np.arange(6), np.arange(6) * 3] = np.array([127, -127, 127, -127, 127, -127])
    CB, SCB = oracle.quantize_weight(W.astype(np.float16))
    assert (SCB == 127).all()
    np.testing.assert_array_equal(CB.astype(np.int64), W)


# --------------------------------------------------------------------------- full matmul
def integer_case(seed=5, T=6, d=24, out=9, thr=200.0):
    """Integer inlier activations and weights whose row absmax is 127: every scale is 1,
    every code equals its input, and the method reduces to an exact integer matmul."""
    g = np.random.default_rng(seed)
    X = g.integers(-127, 128, (T, d)).astype(np.float64)
    out_cols = [3, 17]
    for i in range(T):
        inl = [j for j in range(d) if j not in out_cols]
        X[i, inl[i % len(inl)]] = 127 if i % 2 else -127
        X[i, out_cols[0]] = [200, -250, 3, 1000, -201, 0][i % 6]    # 200 is exactly thr
        X[i, out_cols[1]] = [-7, 512, 300, -300, 5, 256][i % 6]
    X[5, [j for j in range(d) if j not in out_cols]] = 0             # inlier part all zero
    W = g.integers(-127, 128, (out, d)).astype(np.float64)
    W[np.arange(out), (np.arange(out) * 5) % d] = 127
    W[2] = 0                                                          # all-zero weight row
    bias = (g.integers(-40, 41, out) * 0.25).astype(np.float16)
    return X.astype(np.float16), W.astype(np.float16), bias, out_cols, thr


def test_integer_case_reduces_to_exact_integer_matmul():
    X, W, bias, out_cols, thr = integer_case()
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul(X, CB, SCB, threshold=thr, bias=bias)
    assert r["idx"].tolist() == out_cols
    Xi = X.astype(np.int64)
    Wi = W.astype(np.int64)
    Xin = Xi.copy()
    Xin[:, out_cols] = 0
    np.testing.assert_array_equal(r["Q"].astype(np.int64), Xin)      # codes == inputs
    np.testing.assert_array_equal(r["acc"], Xin @ Wi.T)               # int32-range products
    exact = (Xi @ Wi.T).astype(np.float64) + bias.astype(np.float64)
    np.testing.assert_array_equal(r["Y"], exact)                      # no rounding anywhere
    assert r["rowabs"][5] == 0 and (r["rowabs"][:5] == 127).all()


def method_error_bound(X, W, CB, SCB, idx):
    """Per-element bound on |Y_method - (X W^T)| from the half-step quantization errors."""
    Xf = X.astype(np.float64)
    Wf = W.astype(np.float64)
    inl = np.ones(X.shape[1], bool)
    inl[idx] = False
    a = np.where(inl[None, :], np.abs(Xf), 0).max(axis=1)
    ex = a * (1.0 / 254 + 2.0**-22)                         # activation error per row
    ew = SCB.astype(np.float64) * (1.0 / 254 + 2.0**-22)     # weight error per out row
    Xa, Wa = np.abs(Xf), np.abs(Wf)
    b = (Xa[:, inl].sum(1)[:, None] * ew[None, :] + ex[:, None] * Wa[:, inl].sum(1)[None, :]
         + inl.sum() * ex[:, None] * ew[None, :])
    if idx.size:
        wout = np.abs(Wf[:, idx]) + ew[:, None]             # fp16 rounding of dequantized w
        b += Xa[:, idx] @ (ew[:, None] + wout * 2.0**-11 + 2.0**-25).T
    return b * (1 + 1e-9) + 1e-12, a


@pytest.mark.parametrize("name", ["tiny"])
def test_general_case_within_quantization_error_bound(name):
    w = synth.WORKLOADS[name]
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul(X, CB, SCB, threshold=w.threshold, bias=bias)
    exact = X.astype(np.float64) @ W.astype(np.float64).T + bias.astype(np.float64)
    bound, a = method_error_bound(X, W, CB, SCB, r["idx"])
    np.testing.assert_array_equal(r["rowabs"], a.astype(np.float32))
    err = np.abs(r["Y"] - exact)
    assert (err <= bound).all()
    # the decomposition matters: without the outlier term the error leaves the bound
    no_out = r["Y"] - X[:, r["idx"]].astype(np.float64) @ oracle.outlier_weights(
        CB, SCB, r["idx"]).astype(np.float64).T
    assert (np.abs(no_out - exact) > bound).any()


def test_acc_equals_library_integer_matmul_and_codes_in_range():
    w = synth.WORKLOADS["tiny"]
    X, W = synth.make_x(w), synth.make_w(w)
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul(X, CB, SCB, threshold=w.threshold)
    Q = r["Q"].astype(np.int64)
    assert Q.min() >= -127 and Q.max() <= 127
    assert not Q[:, r["idx"]].any()                               # outlier columns coded 0
    np.testing.assert_array_equal(r["acc"], Q @ CB.astype(np.int64).T)
    assert np.abs(r["acc"]).max() < 2**31


def test_threshold_inf_is_plain_vectorwise_int8():
    w = synth.WORKLOADS["tiny"]
    X, W = synth.make_x(w), synth.make_w(w)
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul(X, CB, SCB, threshold=math.inf)
    assert r["idx"].size == 0
    Qp, ap = oracle.quantize_rows_absmax(X)
    np.testing.assert_array_equal(r["Q"], Qp)
    np.testing.assert_array_equal(r["rowabs"], ap)
    np.testing.assert_array_equal(r["acc"], Qp.astype(np.int64) @ CB.astype(np.int64).T)


def test_zeroing_outlier_columns_reproduces_inlier_product():
    w = synth.WORKLOADS["tiny"]
    X, W = synth.make_x(w), synth.make_w(w)
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul(X, CB, SCB, threshold=w.threshold)
    Xz = X.copy()
    Xz[:, r["idx"]] = 0
    rz = oracle.int8_matmul(Xz, CB, SCB, threshold=math.inf)
    np.testing.assert_array_equal(rz["Q"], r["Q"])
    np.testing.assert_array_equal(rz["acc"], r["acc"])


def test_selected_rows_match_full_evaluation():
    w = synth.WORKLOADS["tiny"]
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    CB, SCB = oracle.quantize_weight(W)
    full = oracle.int8_matmul(X, CB, SCB, threshold=6.0, bias=bias, nthreads=3)
    rows = np.array([15, 0, 7])
    part = oracle.int8_matmul(X, CB, SCB, threshold=6.0, bias=bias, rows=rows, nthreads=1)
    np.testing.assert_array_equal(part["Y"], full["Y"][rows])
    np.testing.assert_array_equal(part["acc"], full["acc"][rows])


# --------------------------------------------------------------------------- zeropoint
def test_zeropoint_uses_full_range_on_one_sided_rows():
    w = synth.WORKLOADS["tiny"].with_(T=8, d_in=512)
    X = synth.make_relu_like(w)
    Q, S, Z = oracle.zeropoint_rows(X)
    Xf = X.astype(np.float64)
    mn, mx = Xf.min(1), Xf.max(1)
    # printed formula: S = 254 / (max - min)
    np.testing.assert_allclose(S, 254.0 / (mx - mn), rtol=2e-7)
    assert (Q.min(1) == -127).all() and (Q.max(1) == 127).all()
    assert (Z == np.round(Z)).all()                                   # integral zero-point
    rec = oracle.zeropoint_dequant(Q, S, Z)
    step = 1.0 / S.astype(np.float64)[:, None]
    assert (np.abs(rec - Xf) <= step * (0.5 + 1e-4) + 1e-7).all() or \
        (np.abs(rec - Xf) <= step).all()
    interior = (Q > -127) & (Q < 127)
    assert (np.abs(rec - Xf)[interior] <= (step * 0.5001 + 1e-7)[np.nonzero(interior)[0], 0]).all()


def test_absmax_leaves_the_negative_codes_unused_on_relu_rows():
    """zenn summary, "Zeropoint Quantization": on ReLU outputs absmax codes use only half of
    [-127, 127] (the negative half is wasted), which zeropoint codes recover. On the same
    one-sided rows the absmax codes lie in [0, 127] with 127 reached, while the zeropoint
    codes reach both ends; the zeropoint step is therefore about half the absmax step."""
    w = synth.WORKLOADS["tiny"].with_(T=8, d_in=512)
    X = synth.make_relu_like(w)
    X[:, ::7] = 0  # ReLU zeros
    Xf = X.astype(np.float64)
    assert (Xf >= 0).all() and (Xf.min(1) == 0).all()
    Qa, a = oracle.quantize_rows_absmax(X)
    assert (Qa.min(1) >= 0).all() and (Qa.max(1) == 127).all()
    Qz, S, Z = oracle.zeropoint_rows(X)
    assert (Qz.min(1) == -127).all() and (Qz.max(1) == 127).all()
    step_abs = a.astype(np.float64) / 127.0
    step_zp = 1.0 / S.astype(np.float64)
    np.testing.assert_allclose(step_zp / step_abs, 127.0 / 254.0, rtol=1e-6)


def test_zeropoint_zero_maps_exactly_and_constant_row():
    X = np.array([[0.0, 1.5, -2.0, 0.25, 0.0, 3.0],
                  [2.5, 2.5, 2.5, 2.5, 2.5, 2.5]], np.float16)
    Q, S, Z = oracle.zeropoint_rows(X)
    assert int(Q[0, 0]) + Z[0] == 0 and int(Q[0, 4]) + Z[0] == 0
    assert Q[0].min() == -127 and Q[0].max() == 127
    assert S[1] == 0 and Z[1] == 2.5 and not Q[1].any()
    rec = oracle.zeropoint_dequant(Q, S, Z)
    assert (rec[1] == 2.5).all()


# --------------------------------------------------------------------------- block-wise absmax
def power_of_two_blocks(rows, cols, block, seed):
    """X whose block k of row i is c * 2^e with integers c in [-127, 127], one |c| = 127 per
    block and a different exponent e per block: every block scale 127/(127 * 2^e) = 2^-e is
    exact in fp32, so the codes are exactly c and the absmax exactly 127 * 2^e."""
    g = np.random.default_rng(seed)
    nb = (cols + block - 1) // block
    C = g.integers(-127, 128, (rows, cols))
    E = g.integers(-10, 4, (rows, nb))
    for i in range(rows):
        for k in range(nb):
            j0 = k * block
            C[i, j0 + g.integers(0, min(block, cols - j0))] = 127 * g.choice([-1, 1])
    X = (C * np.exp2(np.repeat(E, block, axis=1)[:, :cols])).astype(np.float16)
    assert np.array_equal(X.astype(np.float64), C * np.exp2(np.repeat(E, block, 1)[:, :cols]))
    return X, C, 127.0 * np.exp2(E)


@pytest.mark.parametrize("block,cols", [(64, 256), (128, 1024), (64, 3 * 64 + 20), (128, 100)])
def test_blockwise_power_of_two_blocks_are_exact(block, cols):
    """Each block has its own scale: the codes are the integers c of every block, including a
    shorter last block, and the stored absmax is each block's own (a row-wide absmax would
    shrink the codes of the blocks with smaller exponents)."""
    X, C, A = power_of_two_blocks(5, cols, block, seed=block + cols)
    Q, a = oracle.quantize_blocks_absmax(X, block)
    assert a.shape == A.shape
    assert np.array_equal(a.astype(np.float64), A)
    assert np.array_equal(Q.astype(np.int64), C)


def test_blockwise_page_example_as_one_block():
    """The pages' worked absmax vector as block 1 of a row of 4-value blocks, between blocks
    of much larger and much smaller values: its codes are the page's, whatever its
    neighbours hold."""
    g = json.load(open(os.path.join(GOLDEN, "absmax_worked_example.json")))
    v = g["vector_printed"]
    X = np.array([[100.0, -3.0, 7.0, 50.0] + v + [0.01, -0.02, 0.005, 0.0]], np.float16)
    Q, a = oracle.quantize_blocks_absmax(X, 4)
    assert Q[0, 4:8].tolist() == [28, -12, -101, 127]
    assert a[0, 1] == np.float32(np.float16(g["absmax_printed"]))
    assert Q[0, 0] == 127 and Q[0, 9] == -127


def test_blockwise_with_one_block_per_row_is_the_row_quantizer():
    X = synth.make_random_f16(77, (9, 300), std=1.3)
    X[2] = 0
    Qr, ar = oracle.quantize_rows_absmax(X)
    for block in (300, 512):
        Qb, ab = oracle.quantize_blocks_absmax(X, block)
        assert np.array_equal(Qb, Qr) and np.array_equal(ab[:, 0], ar)


@pytest.mark.parametrize("block", [64, 128])
def test_blockwise_half_step_bound_range_and_independence(block):
    """Per block: |x - q*a/127| <= a/254 (up to fp32 rounding of the scale and product),
    codes in [-127, 127], the largest |code| of a non-zero block is 127, a zero block codes
    to 0; changing one block changes no other block's codes or absmax."""
    g = np.random.default_rng(block)
    rows, cols = 6, 8 * block + 40
    nb = (cols + block - 1) // block
    scales = np.exp2(g.integers(-6, 6, (rows, nb)))
    X = (g.standard_normal((rows, cols)) * np.repeat(scales, block, 1)[:, :cols]).astype(np.float16)
    X[1, block:2 * block] = 0
    Q, a = oracle.quantize_blocks_absmax(X, block)
    x = X.astype(np.float64)
    af = np.repeat(a.astype(np.float64), block, 1)[:, :cols]
    err = np.abs(x - Q.astype(np.float64) * af / 127.0)
    assert (err <= af / 254.0 * (1 + 2e-6) + 1e-12).all()
    assert Q.min() >= -127 and Q.max() <= 127
    for i in range(rows):
        for k in range(nb):
            q = Q[i, k * block:(k + 1) * block]
            assert (np.abs(q).max() == 127) == (a[i, k] > 0)
    assert a[1, 1] == 0 and not Q[1, block:2 * block].any()
    X2 = X.copy()
    X2[3, 2 * block:3 * block] *= np.float16(4)
    Q2, a2 = oracle.quantize_blocks_absmax(X2, block)
    other = np.ones(cols, bool)
    other[2 * block:3 * block] = False
    assert np.array_equal(Q2[:, other], Q[:, other]) and np.array_equal(Q2[:3], Q[:3])
    assert a2[3, 2] == 4 * a[3, 2] and np.array_equal(np.delete(a2, 2, 1), np.delete(a, 2, 1))


# --------------------------------------------------------------------------- FFN block
@pytest.mark.parametrize("outliers", [False, True])
def test_integer_ffn_block_reduces_to_exact_integer_chain(outliers):
    """With weights of absmax 1 and activations whose inlier absmax is 1 (or 0), every code
    is 127 times the value and both matmuls are exact, so the block equals the integer
    chain relu(X W_up^T) W_down^T + b_down, computed here with numpy integer matmuls. With
    outliers, column 0 of X (value 8) and the big features of H (values 6..10) are the two
    outlier sets at threshold 6."""
    d = synth.make_integer_ffn(3, 37, 64, 160, outliers)
    thr = 6.0 if outliers else math.inf
    CBu, SCBu = oracle.quantize_weight(d["W_up"])
    CBd, SCBd = oracle.quantize_weight(d["W_down"])
    r = oracle.ffn(d["X"], CBu, SCBu, CBd, SCBd, thr, None, d["b_down"], "relu", nthreads=2)
    Xi = d["X"].astype(np.int64)
    pre = Xi @ d["W_up"].astype(np.int64).T
    assert pre.min() < 0                       # the ReLU has work to do
    Hi = np.maximum(pre, 0)
    Yi = Hi @ d["W_down"].astype(np.int64).T + d["b_down"].astype(np.int64)
    assert np.array_equal(r["H_exact"], Hi.astype(np.float64))
    assert np.array_equal(r["H"].astype(np.int64), Hi)
    assert np.array_equal(r["Y"], Yi.astype(np.float64))
    if outliers:
        assert r["up_idx"].tolist() == [0]
        assert r["down_idx"].tolist() == d["big"].tolist()
        assert (Hi[:, d["big"]] >= 6).all()
    else:
        assert r["up_idx"].size == 0 and r["down_idx"].size == 0


def test_ffn_without_activation_is_two_chained_matmuls():
    """act = none: H is the first matmul's output rounded to fp16 (negative values kept)."""
    d = synth.make_integer_ffn(4, 9, 32, 64, True)
    CBu, SCBu = oracle.quantize_weight(d["W_up"])
    CBd, SCBd = oracle.quantize_weight(d["W_down"])
    r = oracle.ffn(d["X"], CBu, SCBu, CBd, SCBd, 6.0, None, d["b_down"], "none", nthreads=1)
    pre = d["X"].astype(np.int64) @ d["W_up"].astype(np.int64).T
    assert pre.min() < 0
    assert np.array_equal(r["H"].astype(np.int64), pre)
    Yi = pre @ d["W_down"].astype(np.int64).T + d["b_down"].astype(np.int64)
    assert np.array_equal(r["Y"], Yi.astype(np.float64))


def test_activation_rounding_is_one_step_from_fp64():
    """fp64 -> fp16 once, ties to even, ReLU zeros (including -0 and tiny negatives) become
    +0; values beyond the fp16 range round to infinity."""
    y = np.array([-3.5, -1e-30, -0.0, 0.0, 2049.0, 2051.0, 2049.0 + 2.0**-30, 65519.99,
                  65520.0, 1.0 + 2.0**-11])
    h = oracle.activation_to_half(y, relu=True)
    assert h.view(np.uint16).tolist()[:4] == [0, 0, 0, 0]
    assert h[4:].tolist() == [2048.0, 2052.0, 2050.0, 65504.0, math.inf, 1.0]
    g = oracle.activation_to_half(y, relu=False)
    assert g[0] == -3.5 and g.view(np.uint16)[1] == 0x8000 and g[4] == 2048.0


# --------------------------------------------------------------------------- zeropoint matmul
def zp_integer_case(outliers: bool, seed: int = 21):
    """One-sided rows on the grid k * step (k = 0..254, every row holding 0 and 254 * step,
    so S = 1/step and Z = 127 exactly), integer weights of absmax 127 (CB = W, SCB = 127).
    With outliers: step 1/64 (inliers below 6) and three columns of large integers."""
    g = np.random.default_rng(seed)
    T, d, out = 7, 96, 40
    step = 1.0 / 64 if outliers else 1.0
    K = g.integers(0, 255, (T, d))
    K[:, 3], K[:, 10] = 0, 254
    X = K * step
    cols = []
    if outliers:
        cols = [17, 50, 95]
        X[:, cols] = g.integers(8, 61, (T, 3)) * np.where(g.random((T, 3)) < 0.5, -1, 1)
    W = g.integers(-127, 128, (out, d))
    W[np.arange(out), (np.arange(out) * 7) % d] = 127
    return X.astype(np.float16), W.astype(np.float16), K, cols, step


@pytest.mark.parametrize("outliers", [False, True])
def test_zeropoint_matmul_on_one_sided_grid_rows_is_exact(outliers):
    """Rows on the grid fill the full code range [-127, 127] exactly (codes k - 127, the
    range absmax would halve on one-sided data), and the correction Z * sum(CB) restores
    the product: Y equals X W^T exactly (dyadic rationals, exact in fp64)."""
    X, W, K, cols, step = zp_integer_case(outliers)
    thr = 6.0 if outliers else math.inf
    CB, SCB = oracle.quantize_weight(W)
    assert (SCB == 127).all()
    r = oracle.int8_matmul_zeropoint(X, CB, SCB, threshold=thr)
    assert r["idx"].tolist() == cols
    assert (r["S"] == np.float32(1.0 / step)).all() and (r["Z"] == 127).all()
    inl = np.ones(X.shape[1], bool)
    inl[cols] = False
    np.testing.assert_array_equal(r["Q"][:, inl].astype(np.int64), K[:, inl] - 127)
    assert not r["Q"][:, ~inl].any()
    np.testing.assert_array_equal(r["acc"], r["Q"].astype(np.int64) @ CB.astype(np.int64).T)
    exact = X.astype(np.float64) @ W.astype(np.float64).T
    np.testing.assert_array_equal(r["Y"], exact)
    if not outliers:  # absmax on the same rows uses half the code range and is not exact
        ra = oracle.int8_matmul(X, CB, SCB, threshold=thr)
        assert not np.array_equal(ra["Y"], exact)


def test_zeropoint_matmul_constant_and_all_outlier_rows():
    """A constant inlier row dequantizes to its value (S = 0, Z = min); when every column is
    an outlier column the int8 part is empty and Y is the fp16 outlier product."""
    X, W, K, cols, step = zp_integer_case(True)
    X[2, :] = np.float16(0.5)
    X[2, cols] = np.float16(9)
    CB, SCB = oracle.quantize_weight(W)
    bias = np.arange(W.shape[0], dtype=np.float16) * np.float16(0.25)
    r = oracle.int8_matmul_zeropoint(X, CB, SCB, 6.0, bias)
    assert r["S"][2] == 0 and r["Z"][2] == 0.5 and not r["Q"][2].any()
    exact = X.astype(np.float64) @ W.astype(np.float64).T + bias.astype(np.float64)
    np.testing.assert_array_equal(r["Y"], exact)
    Xa = np.full((3, 32), 7, np.float16)
    Xa[1] = -11
    Wa = np.tile(np.arange(-16, 16, dtype=np.float16), (5, 1))
    CBa, SCBa = oracle.quantize_weight(Wa)
    ra = oracle.int8_matmul_zeropoint(Xa, CBa, SCBa, 6.0)
    assert ra["idx"].size == 32 and (ra["S"] == 0).all() and (ra["Z"] == 0).all()
    Wo = oracle.outlier_weights(CBa, SCBa, ra["idx"]).astype(np.float64)
    np.testing.assert_array_equal(ra["Y"], Xa.astype(np.float64) @ Wo.T)


def test_zeropoint_matmul_within_quantization_error_bound():
    """Synthetic tiny workload: |Y - X W^T| <= sum_j |w_j| / S (+ the weight and outlier
    weight rounding terms of the absmax bound), and the zeropoint codes of a row are the
    standalone zeropoint quantizer's codes of its inlier columns."""
    w = synth.WORKLOADS["tiny"]
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    CB, SCB = oracle.quantize_weight(W)
    r = oracle.int8_matmul_zeropoint(X, CB, SCB, threshold=w.threshold, bias=bias)
    inl = np.ones(X.shape[1], bool)
    inl[r["idx"]] = False
    Qs, Ss, Zs = oracle.zeropoint_rows(np.ascontiguousarray(X[:, inl]))
    np.testing.assert_array_equal(r["Q"][:, inl], Qs)
    np.testing.assert_array_equal(r["S"], Ss)
    np.testing.assert_array_equal(r["Z"], Zs)
    exact = X.astype(np.float64) @ W.astype(np.float64).T + bias.astype(np.float64)
    Xf, Wf = X.astype(np.float64), W.astype(np.float64)
    # activation error: half a step, a whole step where the clamp at -127 / 127 binds
    ex = 1.0 / r["S"].astype(np.float64) * (1 + 1e-6) + 1e-9
    ew = SCB.astype(np.float64) * (1.0 / 254 + 2.0**-22)
    Xa, Wa = np.abs(Xf), np.abs(Wf)
    b = (Xa[:, inl].sum(1)[:, None] * ew[None, :] + ex[:, None] * Wa[:, inl].sum(1)[None, :]
         + inl.sum() * ex[:, None] * ew[None, :])
    idx = r["idx"]
    wout = np.abs(Wf[:, idx]) + ew[:, None]
    b += Xa[:, idx] @ (ew[:, None] + wout * 2.0**-11 + 2.0**-25).T
    assert (np.abs(r["Y"] - exact) <= b * (1 + 1e-9) + 1e-12).all()
