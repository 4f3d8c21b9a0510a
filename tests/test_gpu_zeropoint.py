"""Parity of the zeropoint matmul (int8_matmul_zeropoint) with the CPU oracle: outlier sets,
zeropoint codes, S, Z and the int32 products bit for bit, Y within
|y - y_ref| <= 2e-2 + 2e-3 |y_ref|; the weight code sums bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 2e-3


@pytest.fixture(scope="module")
def i8():
    import int8_mixed_precision_03_b300 as m
    from int8_mixed_precision_03_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_and_compare(i8, X, W, bias, threshold, rows=None):
    CBo, SCBo = oracle.quantize_weight(W)
    CB, SCB = i8.int8_quantize_weight(dev(W))
    assert torch.equal(CB.cpu(), torch.from_numpy(CBo))
    sums = i8.int8_weight_code_sums(CB)
    assert np.array_equal(sums.cpu().numpy(), CBo.astype(np.int64).sum(axis=1))
    r = i8.int8_matmul_zeropoint_debug(dev(X), CB, SCB, sums, threshold,
                                       None if bias is None else dev(bias))
    assert i8.i8_get_status(r["workspace"]) == 0
    T = X.shape[0]
    rows = np.arange(T) if rows is None else rows
    ref = oracle.int8_matmul_zeropoint(X, CBo, SCBo, threshold, bias, rows=rows)
    assert r["idx"].cpu().numpy().tolist() == ref["idx"].tolist(), "outlier set differs"
    np.testing.assert_array_equal(r["Xq"].cpu().numpy()[rows], ref["Q"])
    np.testing.assert_array_equal(r["S"].cpu().numpy()[rows], ref["S"])
    np.testing.assert_array_equal(r["Z"].cpu().numpy()[rows], ref["Z"])
    np.testing.assert_array_equal(r["acc"].cpu().numpy()[rows].astype(np.int64), ref["acc"])
    Y = r["Y"].cpu().numpy()[rows].astype(np.float64)
    err = np.abs(Y - ref["Y"])
    bad = err > ATOL + RTOL * np.abs(ref["Y"])
    assert not bad.any(), f"{bad.sum()} outside tolerance, worst {err.max():.4g}"
    Y2 = i8.int8_matmul_zeropoint(dev(X), CB, SCB, sums, threshold,
                                  None if bias is None else dev(bias))
    assert torch.equal(Y2, r["Y"])
    return r, ref


def test_tiny_config(i8):
    w = synth.WORKLOADS["tiny"]
    r, _ = run_and_compare(i8, synth.make_x(w), synth.make_w(w), synth.make_bias(w), 6.0)
    assert r["n_out"] == 2


@pytest.mark.parametrize("T,d,out,k", [
    (1, 256, 300, 2), (8, 1024, 1000, 5), (13, 512, 129, 0), (64, 2064, 256, 17),
    (300, 3072, 640, 40), (257, 4096, 255, 2),
])
def test_ragged_shapes_all_on_the_tensor_core_kernel(i8, T, d, out, k):
    w = synth.Workload("zp", T, d, out, n_outlier_cols=k, row_frac=0.7, seed=T + 3 * d)
    run_and_compare(i8, synth.make_x(w), synth.make_w(w), synth.make_bias(w), 6.0)


def test_one_sided_rows_use_the_whole_code_range(i8):
    """ReLU-like rows (|N(0,1)| plus outlier columns): the codes reach -127 and 127."""
    w = synth.Workload("relu", 96, 1024, 512, n_outlier_cols=3, seed=8)
    X = np.abs(synth.make_x(w))
    r, ref = run_and_compare(i8, X, synth.make_w(w), synth.make_bias(w), 6.0)
    q = ref["Q"][:, np.setdiff1d(np.arange(1024), ref["idx"])]
    assert q.min() == -127 and q.max() == 127


def test_constant_and_all_outlier_rows(i8):
    w = synth.Workload("c", 24, 256, 200, n_outlier_cols=2, seed=9)
    X = synth.make_x(w)
    X[3, :] = np.float16(0.75)
    X[3, synth.outlier_columns(w)] = np.float16(20)
    X[5, :] = 0
    r, ref = run_and_compare(i8, X, synth.make_w(w), synth.make_bias(w), 6.0)
    assert ref["S"][3] == 0 and ref["Z"][3] == np.float32(0.75)
    Xa = np.full((4, 64), 9, np.float16)          # every column an outlier column
    Xa[2] = -7
    wa = synth.Workload("a", 4, 64, 48, seed=10)
    r, ref = run_and_compare(i8, Xa, synth.make_w(wa), None, 6.0)
    assert r["n_out"] == 64 and (ref["S"] == 0).all()


def test_threshold_inf_is_plain_vectorwise_zeropoint(i8):
    w = synth.WORKLOADS["tiny"]
    X = synth.make_x(w)
    r, ref = run_and_compare(i8, X, synth.make_w(w), None, float("inf"))
    Qs, Ss, Zs = oracle.zeropoint_rows(X)
    np.testing.assert_array_equal(ref["Q"], Qs)
    np.testing.assert_array_equal(ref["S"], Ss)


@pytest.mark.parametrize("name", ["ffn_6.7b_up", "ffn_13b_up"])
def test_full_size_sampled_rows(i8, name):
    """Full size: codes, S and Z of every row bit for bit (the oracle's zeropoint row
    quantizer over the inlier columns), the int32 products and Y on sampled rows."""
    w = synth.WORKLOADS[name]
    rows = np.array(sorted({0, 1, 255, 256, 1024, w.T - 1, 777}), np.int64)
    X = synth.make_x(w)
    r, ref = run_and_compare(i8, X, synth.make_w(w), synth.make_bias(w), w.threshold,
                             rows=rows)
    inl = np.setdiff1d(np.arange(w.d_in), ref["idx"])
    Qo, So, Zo = oracle.zeropoint_rows(np.ascontiguousarray(X[:, inl]))
    Q = r["Xq"].cpu().numpy()
    np.testing.assert_array_equal(Q[:, inl], Qo)
    assert not Q[:, ref["idx"]].any()
    np.testing.assert_array_equal(r["S"].cpu().numpy(), So)
    np.testing.assert_array_equal(r["Z"].cpu().numpy(), Zo)


def test_rows_far_from_zero_take_the_64_bit_correction(i8):
    """Inlier rows in [5, 5.015625]: S = 16256, Z = 81407, beyond the bound (16386 for
    in = 1024) up to which the epilogue adds Z * (code sum) in 32-bit integers; those tokens
    take the 64-bit path."""
    w = synth.Workload("far", 40, 1024, 384, n_outlier_cols=2, seed=12)
    X = synth.make_x(w)
    g = np.random.default_rng(5)
    inl = np.setdiff1d(np.arange(1024), synth.outlier_columns(w))
    for r in (0, 7, 39):
        X[r, inl] = (5.0 + g.integers(0, 3, inl.size) / 128.0).astype(np.float16)
        X[r, inl[:2]] = [5.0, 5.015625]
    r, ref = run_and_compare(i8, X, synth.make_w(w), synth.make_bias(w), 6.0)
    assert (ref["Z"][[0, 7, 39]] == 81407).all()
    assert np.abs(ref["Z"]).max() > (2**31 - 1 - 16129 * 1024) // (127 * 1024)
