"""The method's quality against unquantized products, from the oracle (CPU): what the pages
say the decomposition and zeropoint quantization buy, measured rather than assumed.

"Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq), section "core
idea", and "LLM.int8() summary" (zenn), sections on outliers and decomposition: a few
large-magnitude feature columns wreck vector-wise int8 unless they are split off into fp16.
The zenn summary, section "Zeropoint Quantization": absmax leaves half of the code range
unused on one-sided (ReLU) data, which zeropoint quantization recovers.

The reference here is the product with the quantized weights, X (CB SCB / 127)^T + b, in
fp64, so the numbers isolate the activation side of the method (the weight rounding is
common to every variant)."""
import math

import numpy as np
import pytest

import oracle
import synth

CASES = [synth.WORKLOADS["tiny"],
         synth.Workload("q_small", 128, 1024, 512, n_outlier_cols=4, seed=1),
         synth.Workload("q_wide", 64, 4096, 256, n_outlier_cols=4, seed=2)]


def rel_rms(Y, ref):
    return float(np.sqrt(((Y - ref) ** 2).mean() / (ref ** 2).mean()))


def activation_errors(w, one_sided):
    X, W, b = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    if one_sided:
        X = np.abs(X)
    CB, SCB = oracle.quantize_weight(W)
    Wq = CB.astype(np.float64) * SCB.astype(np.float64)[:, None] / 127
    ref = X.astype(np.float64) @ Wq.T + b.astype(np.float64)
    absmax = oracle.int8_matmul(X, CB, SCB, 6.0, b, nthreads=4, want_acc=False)["Y"]
    plain = oracle.int8_matmul(X, CB, SCB, math.inf, b, nthreads=4, want_acc=False)["Y"]
    zp = oracle.int8_matmul_zeropoint(X, CB, SCB, 6.0, b, nthreads=4, want_acc=False)["Y"]
    return rel_rms(absmax, ref), rel_rms(plain, ref), rel_rms(zp, ref)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_decomposition_keeps_int8_precision_with_outlier_columns(w):
    e6, einf, _ = activation_errors(w, one_sided=False)
    print(f"{w.name}: relative rms error, threshold 6: {e6:.3e}, threshold inf: {einf:.3e}")
    assert einf > 5 * e6


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_zeropoint_halves_the_activation_error_on_one_sided_rows(w):
    e_abs, _, e_zp = activation_errors(w, one_sided=True)
    print(f"{w.name}: one-sided rows, absmax {e_abs:.3e}, zeropoint {e_zp:.3e}")
    assert 0.4 < e_zp / e_abs < 0.6          # half the step: half the rounding error
    e_abs2, _, e_zp2 = activation_errors(w, one_sided=False)
    assert 0.8 < e_zp2 / e_abs2 < 1.05       # two-sided rows: about the same
