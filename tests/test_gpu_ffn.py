"""Parity of the FFN block (int8_ffn: up projection, ReLU, down projection, with the down
projection's column statistics taken in the up projection's epilogue) with the CPU oracle.

Bit-exact: the weight codes and the intermediate H on integer-valued blocks whose quantized
evaluation is exact (Y there rounds to the exact integer result), and the down
projection's outlier set. Floating point:
H and Y within |v - v_ref| <= 2e-2 + 2e-3 |v_ref| of the oracle's fp64 chain on the
synthetic blocks. At the 13B size the oracle evaluates sampled rows of H; the rest is
checked by properties: the outlier set is the set of columns of the emitted H that reach
the threshold, and the fused block equals the two-call composition on the GPU bit for bit.
"""
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


def check_close(v, ref, what):
    v = v.astype(np.float64)
    err = np.abs(v - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{err.max():.4g} at ref {ref.flat[err.argmax()]:.4g}")


def quantize_both(i8, W_up, W_down, check=True):
    CBu, SCBu = i8.int8_quantize_weight(dev(W_up))
    CBd, SCBd = i8.int8_quantize_weight(dev(W_down))
    ref = (oracle.quantize_weight(W_up), oracle.quantize_weight(W_down)) if check else None
    if check:
        for (CB, SCB), (CBo, SCBo) in zip(((CBu, SCBu), (CBd, SCBd)), ref):
            assert torch.equal(CB.cpu(), torch.from_numpy(CBo))
            assert torch.equal(SCB.cpu(), torch.from_numpy(SCBo))
    return (CBu, SCBu, CBd, SCBd), ref


def check_integer_y(Y: np.ndarray, ref: np.ndarray) -> None:
    """Y of an integer block: the fp32 epilogue sums exact integer terms, so the only error
    is the rounding of those sums (a residue of order 1e-7 where the terms cancel to 0)."""
    Y = Y.astype(np.float64)
    assert np.array_equal(np.rint(Y), ref), "Y does not round to the integer result"
    assert np.abs(Y - ref).max() <= 1e-3


def flagged_columns(H: np.ndarray, threshold: float) -> list:
    """Step 1 of the method applied to an fp16 matrix: columns with some |h| >= threshold."""
    return np.nonzero((np.abs(H.astype(np.float32)) >= threshold).any(axis=0))[0].tolist()


def unfused(i8, X, q, thr, b_up, b_down, act):
    """The same block as two int8_matmul calls with the activation in between."""
    CBu, SCBu, CBd, SCBd = q
    H = i8.int8_matmul(X, CBu, SCBu, thr, b_up)
    if act == "relu":
        H = torch.relu(H)
    return H, i8.int8_matmul(H, CBd, SCBd, thr, b_down)


# ----------------------------------------------------------------- exact integer blocks
@pytest.mark.parametrize("T,d,dff,outliers", [
    (37, 64, 160, True),     # tensor-core path in both matmuls
    (37, 64, 160, False),    # threshold inf: no decomposition anywhere
    (5, 64, 160, True),      # dp4a decode kernels (ReLU + flags in their epilogue)
    (13, 128, 256, True),    # mma.sync decode kernels
    (300, 256, 528, True),   # two token tiles, ragged d_ff (528 = 4 x 128 + 16)
])
def test_integer_block_is_exact(i8, T, d, dff, outliers):
    blk = synth.make_integer_ffn(T * 31 + dff, T, d, dff, outliers)
    thr = 6.0 if outliers else float("inf")
    q, ((CBuo, SCBuo), (CBdo, SCBdo)) = quantize_both(i8, blk["W_up"], blk["W_down"])
    r = i8.int8_ffn_debug(dev(blk["X"]), *q, thr, None, dev(blk["b_down"]), "relu")
    assert i8.i8_get_status(r["workspace"]) == 0
    ref = oracle.ffn(blk["X"], CBuo, SCBuo, CBdo, SCBdo, thr, None, blk["b_down"], "relu")
    H = r["H"].cpu().numpy()
    assert np.array_equal(H.view(np.uint16), ref["H"].view(np.uint16)), "H not bit-exact"
    check_integer_y(r["Y"].cpu().numpy(), ref["Y"])
    assert r["down_idx"].cpu().numpy().tolist() == ref["down_idx"].tolist()
    if outliers:
        assert ref["down_idx"].tolist() == blk["big"].tolist()


def test_integer_block_without_activation(i8):
    blk = synth.make_integer_ffn(11, 40, 64, 192, True)
    q, ((CBuo, SCBuo), (CBdo, SCBdo)) = quantize_both(i8, blk["W_up"], blk["W_down"])
    r = i8.int8_ffn_debug(dev(blk["X"]), *q, 6.0, None, dev(blk["b_down"]), "none")
    ref = oracle.ffn(blk["X"], CBuo, SCBuo, CBdo, SCBdo, 6.0, None, blk["b_down"], "none")
    H = r["H"].cpu().numpy()
    assert (H < 0).any()
    assert np.array_equal(H.astype(np.float64), ref["H"].astype(np.float64))
    check_integer_y(r["Y"].cpu().numpy(), ref["Y"])
    assert r["down_idx"].cpu().numpy().tolist() == ref["down_idx"].tolist()


# ----------------------------------------------------------------- synthetic blocks
@pytest.mark.parametrize("name", ["ffn_small", "ffn_decode_t8", "ffn_decode_t13"])
def test_synthetic_block_matches_oracle_chain(i8, name):
    f = synth.FFN_WORKLOADS[name]
    blk = synth.make_ffn(f)
    q, ((CBuo, SCBuo), (CBdo, SCBdo)) = quantize_both(i8, blk["W_up"], blk["W_down"])
    X, bu, bd = dev(blk["X"]), dev(blk["b_up"]), dev(blk["b_down"])
    r = i8.int8_ffn_debug(X, *q, f.threshold, bu, bd, "relu")
    assert i8.i8_get_status(r["workspace"]) == 0
    ref = oracle.ffn(blk["X"], CBuo, SCBuo, CBdo, SCBdo, f.threshold, blk["b_up"],
                     blk["b_down"], "relu")
    H = r["H"].cpu().numpy()
    check_close(H, ref["H_exact"], "H")
    check_close(r["Y"].cpu().numpy(), ref["Y"], "Y")
    idx = r["down_idx"].cpu().numpy().tolist()
    assert idx == ref["down_idx"].tolist() == blk["h_cols"].tolist()
    assert idx == flagged_columns(H, f.threshold)
    H2, Y2 = unfused(i8, X, q, f.threshold, bu, bd, "relu")
    assert torch.equal(H2, r["H"]) and torch.equal(Y2, r["Y"])
    # the plain entry point gives the same output as the debug one
    H3, Y3 = i8.int8_ffn(X, *q, f.threshold, bu, bd, "relu")
    assert torch.equal(H3, r["H"]) and torch.equal(Y3, r["Y"])


def test_13b_block_full_size(i8):
    """The benchmarked block [4096, 5120] -> 20480 -> 5120, in the launch configuration the
    benchmark times: H and Y of every row against the oracle's whole chain (about 20 s of
    CPU on 16 cores), the down projection's outlier set, and the fused block against the
    two-call composition bit for bit."""
    f = synth.FFN_WORKLOADS["ffn_13b_block"]
    blk = synth.make_ffn(f)
    q, ((CBuo, SCBuo), (CBdo, SCBdo)) = quantize_both(i8, blk["W_up"], blk["W_down"])
    X, bu, bd = dev(blk["X"]), dev(blk["b_up"]), dev(blk["b_down"])
    r = i8.int8_ffn_debug(X, *q, f.threshold, bu, bd, "relu")
    assert i8.i8_get_status(r["workspace"]) == 0
    H = r["H"].cpu().numpy()
    idx = r["down_idx"].cpu().numpy().tolist()
    assert idx == flagged_columns(H, f.threshold) == blk["h_cols"].tolist()
    H2, Y2 = unfused(i8, X, q, f.threshold, bu, bd, "relu")
    assert torch.equal(H2, r["H"]) and torch.equal(Y2, r["Y"])
    ref = oracle.ffn(blk["X"], CBuo, SCBuo, CBdo, SCBdo, f.threshold, blk["b_up"],
                     blk["b_down"], "relu")
    assert ref["down_idx"].tolist() == idx
    check_close(H, ref["H_exact"], "H")
    check_close(r["Y"].cpu().numpy(), ref["Y"], "Y")


# ----------------------------------------------------------------- edge cases
def test_empty_batch_is_a_noop(i8):
    blk = synth.make_integer_ffn(5, 4, 32, 64, False)
    q, _ = quantize_both(i8, blk["W_up"], blk["W_down"], check=False)
    X = torch.empty((0, 32), dtype=torch.float16, device="cuda")
    H, Y = i8.int8_ffn(X, *q, 6.0, act="relu")
    assert H.shape == (0, 64) and Y.shape == (0, 32)
    with pytest.raises(ValueError):
        i8.int8_ffn(dev(blk["X"]), *q, 6.0, act="gelu")


@pytest.mark.parametrize("where", ["up", "down"])
def test_outlier_capacity_error_reaches_the_one_status_word(i8, where):
    """More outlier columns than the 64-column capacity, in the first or the second
    matmul: i8_get_status(workspace) reports I8_ERR_OUTLIER_CAP either way."""
    T, d, dff = 20, 256, 512
    f = synth.FFN_WORKLOADS["ffn_small"].with_(T=T, d_model=d, d_ff=dff)
    if where == "up":
        f = f.with_(x_outlier_frac=0.4)          # ~100 outlier columns of X
    else:
        f = f.with_(h_outlier_frac=0.2)          # ~100 outlier features of H
    blk = synth.make_ffn(f)
    q, _ = quantize_both(i8, blk["W_up"], blk["W_down"], check=False)
    n = i8.int8_ffn_workspace_size(T, d, dff, 64)
    assert n < i8.int8_ffn_workspace_size(T, d, dff, 128)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    i8.int8_ffn(dev(blk["X"]), *q, 6.0, dev(blk["b_up"]), dev(blk["b_down"]), "relu",
                workspace=ws)
    assert i8.i8_get_status(ws) == 6
    # the same block with enough capacity is fine
    ws2 = torch.empty(i8.int8_ffn_workspace_size(T, d, dff, 0), dtype=torch.uint8,
                      device="cuda")
    i8.int8_ffn(dev(blk["X"]), *q, 6.0, dev(blk["b_up"]), dev(blk["b_down"]), "relu",
                workspace=ws2)
    assert i8.i8_get_status(ws2) == 0


# ----------------------------------------------------------------- fp16 comparator
def test_f16_ffn_is_two_f16_matmuls_with_relu(i8):
    f = synth.FFN_WORKLOADS["ffn_small"]
    blk = synth.make_ffn(f)
    X, Wu, Wd = dev(blk["X"]), dev(blk["W_up"]), dev(blk["W_down"])
    bu, bd = dev(blk["b_up"]), dev(blk["b_down"])
    H, Y = i8.f16_ffn(X, Wu, Wd, bu, bd, "relu")
    H2 = torch.relu(i8.f16_matmul(X, Wu, bu))
    assert torch.equal(H, H2)
    assert torch.equal(Y, i8.f16_matmul(H, Wd, bd))
    # against an fp64 evaluation of the same fp16 operands
    Hr = np.maximum(blk["X"].astype(np.float64) @ blk["W_up"].astype(np.float64).T
                    + blk["b_up"].astype(np.float64), 0.0)
    check_close(H.cpu().numpy(), Hr, "fp16 H")
