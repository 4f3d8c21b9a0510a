"""int8_matmul_noalloc: the matmul for callers that cannot allocate device memory when they
call (applications whose device memory comes only from their own allocator, latency-critical
loops that must not call cudaMalloc). It runs on a scratch array built into the library, and
i8_noalloc_status reads the device status word the last call left there.

This file is named so that pytest collects it last."""
import ctypes as C

import pytest
import torch

import synth

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
    assert L.int8_matmul_noalloc(p, 16, 0, p, p, 64, 6.0, None, p, None) == 1  # bad size
    assert L.int8_matmul_noalloc(p, 16, 24, p, p, 64, 6.0, None, p, None) == 2  # in % 16
    assert L.int8_matmul_noalloc(p, 16, 64, p, p, 64, float("nan"), None, p, None) == 1
    # activation codes alone need 2*4096*8192 bytes = 64 MiB > 32 MiB
    assert L.int8_matmul_noalloc(p, 4096, 8192, p, p, 1024, 6.0, None, p, None) == 8
    assert L.i8_status_string(8) == b"sizes exceed the built-in scratch of int8_matmul_noalloc"
    assert L.i8_last_launch_count() == 0


def _call_noalloc(i8, X, CB, SCB, thr, bias, Y):
    """One call through the C-ABI on the current stream."""
    T, d = X.shape
    out = CB.shape[0]
    ptr = lambda t: None if t is None else C.c_void_p(t.data_ptr())  # noqa: E731
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return i8.lib().int8_matmul_noalloc(ptr(X), T, d, ptr(CB), ptr(SCB), out, float(thr),
                                        ptr(bias), ptr(Y), stream)


def _status(i8):
    return i8.lib().i8_noalloc_status(C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_int8_matmul_bit_for_bit_on_calls_in_a_row(i8):
    """Both entry points run the same kernels (the schedules they may pick give the same Y
    bit for bit), so the outputs must be equal. The second call has more outlier columns
    than the first and the third fewer: what the scratch keeps from a call must not leak
    into the next one."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    cases = [synth.Workload("na1", 512, 4096, 2048, n_outlier_cols=4, seed=41),
             synth.Workload("na2", 300, 1040, 520, n_outlier_cols=40, row_frac=0.7, seed=42),
             synth.Workload("na3", 300, 1040, 520, n_outlier_cols=2, row_frac=0.7, seed=43),
             synth.Workload("na4", 5, 2048, 3000, n_outlier_cols=3, row_frac=1.0, seed=44)]
    for k, w in enumerate(cases):
        X = torch.from_numpy(synth.make_x(w)).cuda()
        W = torch.from_numpy(synth.make_w(w)).cuda()
        bias = torch.from_numpy(synth.make_bias(w)).cuda() if k % 2 == 0 else None
        CB, SCB = i8.int8_quantize_weight(W)
        Y_ref = i8.int8_matmul(X, CB, SCB, 6.0, bias)          # workspace entry point
        Y = torch.full((w.T, w.d_out), float("nan"), dtype=torch.float16, device="cuda")
        assert _call_noalloc(i8, X, CB, SCB, 6.0, bias, Y) == 0
        assert _status(i8) == 0
        assert torch.equal(Y, Y_ref), f"call {k + 1} differs from int8_matmul"


@pytest.mark.gpu
def test_noalloc_reports_outlier_capacity_on_the_device(i8):
    """With out = 131072 the outlier weight slice takes 256 KB per column, so the scratch
    holds a capacity of 64 columns; 100 outlier columns are recorded as I8_ERR_OUTLIER_CAP,
    readable through i8_noalloc_status, and the next call within capacity reads I8_OK."""
    T, d, out = 32, 256, 131072
    w = synth.Workload("cap", T, d, out, n_outlier_cols=100, row_frac=1.0, seed=45)
    X = torch.from_numpy(synth.make_x(w)).cuda()
    W = torch.from_numpy(synth.make_w(w)).cuda()
    CB, SCB = i8.int8_quantize_weight(W)
    del W
    Y = torch.empty((T, out), dtype=torch.float16, device="cuda")
    assert _call_noalloc(i8, X, CB, SCB, 6.0, None, Y) == 0  # accepted on the host
    assert _status(i8) == 6                                   # I8_ERR_OUTLIER_CAP
    assert i8.i8_noalloc_status() == 6                        # the binding reads the same
    X2 = torch.from_numpy(synth.make_x(w.with_(n_outlier_cols=5, seed=46))).cuda()
    assert _call_noalloc(i8, X2, CB, SCB, 6.0, None, Y) == 0
    assert _status(i8) == 0
    assert torch.equal(Y, i8.int8_matmul(X2, CB, SCB, 6.0))
