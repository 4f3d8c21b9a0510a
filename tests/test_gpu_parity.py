"""Parity of the CUDA path (through the C-ABI) with the CPU oracle.

Bit-exact: outlier column sets, int8 codes, row absmax, CB/SCB, int32 accumulators,
zeropoint codes/S/Z. Floating point: |y - y_ref| <= 2e-2 + 2e-3 |y_ref| for the fp16 output
against the oracle's fp64 evaluation of the same quantized definition.
"""
import ctypes as C
import functools
import math

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


@functools.lru_cache(maxsize=2)
def _weights(d_out, d_in, w_std, seed):
    w = synth.Workload("w", 1, d_in, d_out, w_std=w_std, seed=seed)
    W = synth.make_w(w)
    return W, synth.make_bias(w), oracle.quantize_weight(W)


def weights(w):
    """W, bias and the oracle's CB/SCB, shared by configs with the same weight shape."""
    return _weights(w.d_out, w.d_in, w.w_std, w.seed)


def sample_rows(T, k=8, seed=0):
    g = np.random.default_rng(seed)
    base = {0, T - 1, T // 2}
    extra = g.choice(T, size=min(T, k), replace=False)
    return np.array(sorted(base | set(int(e) for e in extra)), dtype=np.int64)


def check_y(Y, ref):
    Y = Y.astype(np.float64)
    err = np.abs(Y - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; worst err "
                           f"{err.max():.4g} at ref {ref.flat[err.argmax()]:.4g}")


def outlier_mask(idx, d):
    m = np.zeros(d, np.uint8)
    m[np.asarray(idx, np.int64)] = 1
    return m


def run_and_compare(i8, X, W, bias, threshold, rows=None, CBo=None, SCBo=None,
                    check_weights=True, all_codes=True):
    """The CUDA path against the oracle: outlier set, codes and row absmax of every row
    (all_codes) or of the evaluated rows, and the int32 products and Y of the evaluated
    rows (all rows unless `rows` samples them)."""
    if CBo is None:
        CBo, SCBo = oracle.quantize_weight(W)
    Wd = dev(W)
    CB, SCB = i8.int8_quantize_weight(Wd)
    if check_weights:
        assert torch.equal(CB.cpu(), torch.from_numpy(CBo)), "CB codes differ"
        assert torch.equal(SCB.cpu(), torch.from_numpy(SCBo)), "SCB differs"
    r = i8.int8_matmul_debug(dev(X), CB, SCB, threshold,
                             None if bias is None else dev(bias))
    assert i8.i8_get_status(r["workspace"]) == 0
    T = X.shape[0]
    rows = np.arange(T) if rows is None else rows
    ref = oracle.int8_matmul(X, CBo, SCBo, threshold=threshold, bias=bias, rows=rows)
    assert r["idx"].cpu().numpy().tolist() == ref["idx"].tolist(), "outlier set differs"
    Xq_all = r["Xq"].cpu().numpy()
    ra_all = r["rowabs"].cpu().numpy()
    np.testing.assert_array_equal(Xq_all[rows], ref["Q"])
    np.testing.assert_array_equal(ra_all[rows], ref["rowabs"])
    if all_codes and len(rows) < T:
        # every row's codes and row absmax, from the oracle's row quantizer over the
        # inlier columns (the product is only evaluated on the sampled rows)
        Qo, ao = oracle.quantize_rows_absmax(X, outlier_mask(ref["idx"], X.shape[1]))
        np.testing.assert_array_equal(Xq_all, Qo)
        np.testing.assert_array_equal(ra_all, ao)
    acc = r["acc"].cpu().numpy()[rows].astype(np.int64)
    np.testing.assert_array_equal(acc, ref["acc"])
    check_y(r["Y"].cpu().numpy()[rows], ref["Y"])
    # the plain entry point gives the same output as the debug one
    Y2 = i8.int8_matmul(dev(X), CB, SCB, threshold, None if bias is None else dev(bias))
    assert torch.equal(Y2, r["Y"])
    return r, ref


# ----------------------------------------------------------------- small and ragged shapes
def test_tiny_config(i8):
    w = synth.WORKLOADS["tiny"]
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    r, ref = run_and_compare(i8, X, W, bias, w.threshold)
    assert r["n_out"] == 2


@pytest.mark.parametrize("T,d,out,k", [
    (1, 16, 1, 0), (2, 48, 7, 1), (7, 64, 129, 3), (8, 128, 100, 15), (9, 256, 257, 16),
    (63, 1040, 300, 17), (64, 2064, 128, 65), (65, 512, 384, 0), (129, 1024, 520, 5),
    (300, 3072, 640, 40), (257, 4096, 255, 2),
    # small token tiles (stages of four K blocks): a partial last int stage and outlier
    # counts whose last outlier stage is partly past the zero-padded slices
    (48, 1040, 272, 40), (17, 1536, 200, 100), (33, 4160, 136, 33),
])
def test_ragged_shapes(i8, T, d, out, k):
    w = synth.Workload("ragged", T, d, out, n_outlier_cols=k, row_frac=0.7, seed=T * 7 + d)
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    run_and_compare(i8, X, W, bias, 6.0)


@pytest.mark.parametrize("T,d,out,k", [
    (1, 14336, 3000, 14),     # 176B-like row length, CUDA-core decode kernel
    (8, 2048, 4100, 70),      # more outlier columns than the decode kernel's 64-column table
    (5, 1024, 20000, 3),      # many rows per CTA, odd T
    (8, 32768, 300, 2),       # T * in beyond the decode kernel's shared memory: tensor path
    (3, 16, 1, 1),            # one output feature, most warps idle
    (6, 14336, 2000, 14),     # dp4a decode kernel, 176B-like rows
    (9, 1040, 777, 20),       # mma.sync decode kernel, second token tile, K % 64 != 0
    (12, 4096, 3000, 70),     # outlier columns beyond the mma.sync kernel's table
    (16, 8192, 1000, 5),      # the largest decode tile
    (16, 14336, 500, 3),      # codes too large for shared memory: tensor path
])
def test_decode_sizes(i8, T, d, out, k):
    w = synth.Workload("decode", T, d, out, n_outlier_cols=k, row_frac=1.0, seed=T + d + out)
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    r, ref = run_and_compare(i8, X, W, bias, 6.0)
    assert r["n_out"] == len(ref["idx"])


def test_no_bias_zero_row_and_all_outlier_row(i8):
    w = synth.Workload("edge", 40, 512, 300, n_outlier_cols=6, row_frac=1.0, seed=3)
    X, W = synth.make_x(w), synth.make_w(w)
    X[5] = 0                                            # zero row: absmax 0, codes 0
    cols = synth.outlier_columns(w)
    X[9] = 0
    X[9, cols] = 50                                     # a row made only of outliers
    W[17] = 0                                           # zero weight row: SCB 0
    run_and_compare(i8, X, W, None, 6.0)


@pytest.mark.parametrize("thr,below,at", [
    (5.9, 5.8984375, 5.90234375),     # 5.9 lies between two fp16 values
    (6.01, 6.0078125, 6.01171875),
    (0.3, 0.2998046875, 0.30029296875),
])
def test_thresholds_that_are_not_fp16_values(i8, thr, below, at):
    """A threshold between two fp16 values: the largest fp16 below it is an inlier, the
    smallest above it an outlier (|x| >= threshold compared exactly). At 0.3 nearly every
    column of N(0,1) data is an outlier and the inlier codes are mostly zero."""
    w = synth.Workload("thr", 40, 256, 300, n_outlier_cols=2, seed=13)
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    c0, c1 = np.setdiff1d(np.arange(256), synth.outlier_columns(w))[[20, 21]]
    X[:, [c0, c1]] = np.clip(X[:, [c0, c1]], -0.1, 0.1)
    X[3, c0] = below
    X[7, c1] = -at
    r, ref = run_and_compare(i8, X, W, bias, thr)
    got = r["idx"].cpu().numpy().tolist()
    assert c1 in got and c0 not in got
    if thr < 1:
        assert r["n_out"] == 255


def test_threshold_inf_and_threshold_edge(i8):
    w = synth.Workload("thr", 33, 256, 200, n_outlier_cols=3, seed=11)
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    X[4, 10] = 6.0                                      # exactly at threshold: outlier
    X[6, 11] = np.float16(5.99609375)                   # just below: inlier
    r, _ = run_and_compare(i8, X, W, bias, 6.0)
    got = r["idx"].cpu().numpy().tolist()
    assert 10 in got and 11 not in got
    r, _ = run_and_compare(i8, X, W, bias, math.inf)
    assert r["n_out"] == 0


@pytest.mark.parametrize("pattern", ["same_sign", "alternating", "random"])
def test_int32_accumulator_exact_at_extreme_codes(i8, pattern):
    """Codes of +-127 everywhere make every fp32 chunk sum as large as the method allows
    (1024 * 127^2 < 2^24); the int32 result must still be exact."""
    T, d, out = 160, 4096, 256
    g = np.random.default_rng(5)
    if pattern == "same_sign":
        sx = np.ones((T, d)); sw = np.ones((out, d))
        sx[1::2] = -1
    elif pattern == "alternating":
        sx = np.where(np.arange(d) % 2 == 0, 1.0, -1.0)[None, :].repeat(T, 0)
        sw = np.where(np.arange(d) % 3 == 0, 1.0, -1.0)[None, :].repeat(out, 0)
    else:
        sx = g.choice([-1.0, 1.0], (T, d)); sw = g.choice([-1.0, 1.0], (out, d))
    # +-127 * 2^-10: every code is +-127 (the row scale cancels) and Y stays finite in fp16
    X = (127 * sx / 1024).astype(np.float16)
    W = (127 * sw / 1024).astype(np.float16)
    r, ref = run_and_compare(i8, X, W, None, math.inf)
    exact = (127 * sx).astype(np.int64) @ (127 * sw).astype(np.int64).T
    np.testing.assert_array_equal(r["acc"].cpu().numpy().astype(np.int64), exact)
    assert np.abs(exact).max() == 4096 * 127 * 127 or pattern != "same_sign"


def test_outlier_capacity_exceeded_sets_status(i8):
    w = synth.Workload("cap", 16, 1024, 128, n_outlier_cols=100, row_frac=1.0, seed=2)
    X, W = synth.make_x(w), synth.make_w(w)
    CB, SCB = i8.int8_quantize_weight(dev(W))
    ws = i8.alloc_workspace(16, 1024, 128, "cuda", max_outlier_cols=64)
    i8.int8_matmul(dev(X), CB, SCB, 6.0, workspace=ws)
    assert i8.i8_get_status(ws) == 6
    ws = i8.alloc_workspace(16, 1024, 128, "cuda", max_outlier_cols=128)
    i8.int8_matmul(dev(X), CB, SCB, 6.0, workspace=ws)
    assert i8.i8_get_status(ws) == 0


def test_workspace_reuse_across_calls(i8):
    """The header is reset per call: a second call on the same workspace is unaffected by
    the first one's outlier set."""
    wa = synth.Workload("a", 24, 512, 256, n_outlier_cols=9, seed=21)
    wb = synth.Workload("b", 24, 512, 256, n_outlier_cols=0, seed=22)
    ws = i8.alloc_workspace(24, 512, 256, "cuda")
    for w in (wa, wb, wa):
        X, W = synth.make_x(w), synth.make_w(w)
        CBo, SCBo = oracle.quantize_weight(W)
        CB, SCB = i8.int8_quantize_weight(dev(W))
        r = i8.int8_matmul_debug(dev(X), CB, SCB, 6.0, workspace=ws)
        ref = oracle.int8_matmul(X, CBo, SCBo, threshold=6.0)
        assert r["idx"].cpu().numpy().tolist() == ref["idx"].tolist()
        check_y(r["Y"].cpu().numpy(), ref["Y"])


# ----------------------------------------------------------------- standalone quantizers
@pytest.mark.parametrize("rows,cols", [(1024, 8192), (16384, 8192), (3, 7), (5, 1000),
                                       (17, 40), (2, 1)])
def test_absmax_rows_bit_exact(i8, rows, cols):
    X = synth.make_random_f16(rows * 31 + cols, (rows, cols), std=1.5)
    X[0, :] = 0
    Q, a = i8.absmax_quantize_rows(dev(X))
    Qo, ao = oracle.quantize_rows_absmax(X)
    np.testing.assert_array_equal(Q.cpu().numpy(), Qo)
    np.testing.assert_array_equal(a.cpu().numpy(), ao)


@pytest.mark.parametrize("rows,cols,block", [
    (1024, 8192, 64), (1024, 8192, 128),      # the sweep's X, the pages' block sizes
    (16384, 8192, 64),                         # the bench's large input
    (37, 1000, 64),                            # ragged last block (1000 = 15 * 64 + 40)
    (5, 200, 16), (3, 4104, 256), (9, 520, 32),
    (7, 100, 64),                              # cols % 8 != 0 (element path)
    (4, 96, 48), (2, 5, 3), (3, 64, 1000),     # other block sizes, one block per row
])
def test_absmax_blocks_bit_exact(i8, rows, cols, block):
    X = synth.make_random_f16(rows * 7 + cols + block, (rows, cols), std=1.5)
    g = np.random.default_rng(block)
    X *= np.exp2(g.integers(-4, 5, (rows, 1))).astype(np.float16)  # rows of different scales
    X[0, : min(cols, block)] = 0                                     # a zero block
    Q, a = i8.absmax_quantize_blocks(dev(X), block)
    Qo, ao = oracle.quantize_blocks_absmax(X, block)
    np.testing.assert_array_equal(Q.cpu().numpy(), Qo)
    np.testing.assert_array_equal(a.cpu().numpy(), ao)


@pytest.mark.parametrize("rows,cols", [(1024, 8192), (16384, 8192), (4, 9), (6, 1000), (3, 1)])
def test_zeropoint_rows_bit_exact(i8, rows, cols):
    w = synth.Workload("zp", rows, cols, 1)
    X = synth.make_relu_like(w)
    if rows > 3:
        X[3] = 2.5                       # constant row
        X[2] = -X[2]                     # a non-negative row turned non-positive
    Q, S, Z = i8.zeropoint_quantize_rows(dev(X))
    Qo, So, Zo = oracle.zeropoint_rows(X)
    np.testing.assert_array_equal(Q.cpu().numpy(), Qo)
    np.testing.assert_array_equal(S.cpu().numpy(), So)
    np.testing.assert_array_equal(Z.cpu().numpy(), Zo)


@pytest.mark.parametrize("out,d", [(1024, 256), (37, 100), (5, 16)])
def test_weight_quantize_bit_exact(i8, out, d):
    W = synth.make_random_f16(out + d, (out, d), std=0.02)
    CB, SCB = i8.int8_quantize_weight(dev(W))
    CBo, SCBo = oracle.quantize_weight(W)
    np.testing.assert_array_equal(CB.cpu().numpy(), CBo)
    np.testing.assert_array_equal(SCB.cpu().numpy(), SCBo)


@pytest.mark.parametrize("T,d,out", [(16, 256, 1024), (300, 1040, 520), (2048, 4096, 1024)])
def test_f16_matmul_comparator(i8, T, d, out):
    X = synth.make_random_f16(T + d, (T, d))
    W = synth.make_random_f16(out + d + 1, (out, d), std=0.02)
    b = synth.make_random_f16(out, (out,), std=0.01)
    Y = i8.f16_matmul(dev(X), dev(W), dev(b)).cpu().numpy().astype(np.float64)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    check_y(Y, ref)


# ----------------------------------------------------------------- full-size configurations
FULL = ["ffn_6.7b_up", "ffn_13b_up", "ffn_13b_down", "decode_176b_t1", "decode_176b_t8",
        "decode_176b_t64", "sweep_f0_thr6", "sweep_f0.1_thr6", "sweep_f0.5_thr6",
        "sweep_f2_thr6", "sweep_f0_thrinf", "sweep_f2_thrinf"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_config_sampled_rows(i8, name):
    """Every configuration at full size, in the launch configuration the benchmark times:
    the outlier set, the codes and the row absmax of all T rows bit for bit; the int32
    products and Y on sampled rows (the oracle's product of every row would take minutes)."""
    w = synth.WORKLOADS[name]
    X = synth.make_x(w)
    W, bias, (CBo, SCBo) = weights(w)
    rows = sample_rows(w.T)
    r, ref = run_and_compare(i8, X, W, bias, w.threshold, rows=rows, CBo=CBo, SCBo=SCBo)
    planted = synth.outlier_columns(w)
    if w.threshold == 6.0:
        assert set(planted.tolist()) <= set(ref["idx"].tolist())


@pytest.mark.parametrize("T", [64, 300])
def test_stalled_matmul_times_out_and_the_context_stays_usable(i8, T):
    """Every pipeline wait of the tensor-core matmul runs out (its loaders load nothing):
    the kernel records I8_ERR_TIMEOUT and returns; the next call on the stream is correct.
    64 tokens run on single CTAs, 300 (256-token tiles) on CTA pairs, whose two CTAs both
    unwind and leave together."""
    w = synth.Workload("stall", T, 256, 256, n_outlier_cols=2, seed=5)
    X, W, bias = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    Xd = dev(X)
    CB, SCB = i8.int8_quantize_weight(dev(W))
    ws = i8.alloc_workspace(w.T, w.d_in, w.d_out, "cuda")
    Y = torch.empty((w.T, w.d_out), dtype=torch.float16, device="cuda")
    ptr = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = i8.lib().i8_test_stalled_matmul(ptr(Xd), w.T, w.d_in, ptr(CB), ptr(SCB), w.d_out,
                                         ptr(Y), ptr(ws), ws.numel(), 20_000_000, stream)
    assert rc == 0
    assert i8.i8_get_status(ws) == 7  # I8_ERR_TIMEOUT
    run_and_compare(i8, X, W, bias, 6.0)


# ----------------------------------------------------------------- split schedule
@pytest.mark.parametrize("T,d,out,k", [
    (64, 2064, 128, 17),      # one tile cut into three single-chunk pieces
    (300, 3072, 640, 40),     # ten tiles over 30 CTAs
    (64, 14336, 8192, 14),    # decode-like tile of 64 tokens, 14 chunks per tile
    (200, 5120, 2560, 10),    # pieces of several chunks
])
def test_split_and_unsplit_schedules_agree_bit_for_bit(i8, T, d, out, k):
    """Tiles cut between CTAs (the split schedule, used with a full-size workspace) give the
    same Y, bit for bit, as whole tiles per CTA (the schedule a workspace without the split
    slots falls back to): the int32 sums are exact and each piece's outlier sums come
    from one CTA."""
    w = synth.Workload("split", T, d, out, n_outlier_cols=k, row_frac=0.8, seed=T + d + out)
    X, W, bias = dev(synth.make_x(w)), dev(synth.make_w(w)), dev(synth.make_bias(w))
    CB, SCB = i8.int8_quantize_weight(W)
    full = i8.int8_matmul_workspace_size(T, d, out, 64)
    ws_split = torch.empty(full, dtype=torch.uint8, device="cuda")
    ws_whole = torch.empty(full - 1, dtype=torch.uint8, device="cuda")
    Y1 = i8.int8_matmul(X, CB, SCB, 6.0, bias, workspace=ws_split)
    Y2 = i8.int8_matmul(X, CB, SCB, 6.0, bias, workspace=ws_whole)
    assert i8.i8_get_status(ws_split) == 0 and i8.i8_get_status(ws_whole) == 0
    assert torch.equal(Y1, Y2)
    sums = i8.int8_weight_code_sums(CB)
    Z1 = i8.int8_matmul_zeropoint(X, CB, SCB, sums, 6.0, bias, workspace=ws_split)
    Z2 = i8.int8_matmul_zeropoint(X, CB, SCB, sums, 6.0, bias, workspace=ws_whole)
    assert torch.equal(Z1, Z2)
