"""int8_matmul_noalloc: the matmul for callers that cannot allocate device memory when they
call (applications whose device memory comes only from their own allocator, latency-critical
loops that must not call cudaMalloc). It runs on a scratch array built into the library.

This file is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest
import torch

import synth

ATOL, RTOL = 2e-2, 2e-3
A = 1 << 20  # 16-byte aligned fake address: rejected on the host, never dereferenced


@pytest.fixture(scope="module")
def i8():
    import int8_mixed_precision_03_b300 as m
    from int8_mixed_precision_03_b300 import build
    build.build()
    return m


def test_sizes_beyond_the_scratch_are_rejected_before_any_launch(i8):
    L = i8.lib()
    p = C.c_void_p(A)
    # activation codes alone need 2*4096*8192 bytes = 64 MiB > 32 MiB
    assert L.int8_matmul_noalloc(p, 4096, 8192, p, p, 1024, 6.0, None, p, None) == 8
    assert L.i8_status_string(8) == b"sizes exceed the built-in scratch of int8_matmul_noalloc"
    assert L.int8_matmul_noalloc(p, 16, 0, p, p, 64, 6.0, None, p, None) == 1  # bad size
    assert L.i8_last_launch_count() == 0


def _call_noalloc(i8, X, CB, SCB, thr, bias, Y):
    """One call through the C-ABI on the current stream."""
    T, d = X.shape
    out = CB.shape[0]
    ptr = lambda t: None if t is None else C.c_void_p(t.data_ptr())  # noqa: E731
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return i8.lib().int8_matmul_noalloc(ptr(X), T, d, ptr(CB), ptr(SCB), out, float(thr),
                                        ptr(bias), ptr(Y), stream)


@pytest.mark.gpu
def test_noalloc_matches_int8_matmul_on_two_calls_in_a_row(i8):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    cases = [synth.Workload("na1", 512, 4096, 2048, n_outlier_cols=4, seed=41),
             synth.Workload("na2", 300, 1040, 520, n_outlier_cols=17, row_frac=0.7, seed=42)]
    for k, w in enumerate(cases):
        X = torch.from_numpy(synth.make_x(w)).cuda()
        W = torch.from_numpy(synth.make_w(w)).cuda()
        bias = torch.from_numpy(synth.make_bias(w)).cuda() if k == 0 else None
        CB, SCB = i8.int8_quantize_weight(W)
        Y_ref = i8.int8_matmul(X, CB, SCB, 6.0, bias)          # workspace entry point
        Y = torch.full((w.T, w.d_out), float("nan"), dtype=torch.float16, device="cuda")
        assert _call_noalloc(i8, X, CB, SCB, 6.0, bias, Y) == 0
        torch.cuda.synchronize()
        y, ref = Y.cpu().double().numpy(), Y_ref.cpu().double().numpy()
        assert np.isfinite(y).all()
        assert (np.abs(y - ref) <= ATOL + RTOL * np.abs(ref)).all(), f"call {k + 1} differs"
