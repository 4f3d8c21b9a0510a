"""LLM.int8() mixed-precision matmul for NVIDIA B300 (sm_103a): Python binding.

The functions here have the names of the C-ABI calls in ``include/int8mm.h`` and only
marshal arguments: every step of the computation runs in the CUDA kernels of
``libint8mm.so``. PyTorch provides device memory and the current stream. There is no CPU
fallback: if the library is missing, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libint8mm.so")

I8_OK = 0
STATUS = {0: "I8_OK", 1: "I8_ERR_INVALID_ARG", 2: "I8_ERR_ALIGNMENT", 3: "I8_ERR_WORKSPACE",
          4: "I8_ERR_UNSUPPORTED_DEVICE", 5: "I8_ERR_CUDA", 6: "I8_ERR_OUTLIER_CAP",
          7: "I8_ERR_TIMEOUT", 8: "I8_ERR_SCRATCH_LIMIT"}

# Every symbol the header declares, with its ctypes signature.
_p, _i, _f, _sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
SIGNATURES = {
    "int8_quantize_weight": (_i, [_p, _i, _i, _p, _p, _p]),
    "int8_matmul_workspace_size": (_sz, [_i, _i, _i, _i]),
    "int8_matmul": (_i, [_p, _i, _i, _p, _p, _i, _f, _p, _p, _p, _sz, _p]),
    "int8_matmul_noalloc": (_i, [_p, _i, _i, _p, _p, _i, _f, _p, _p, _p]),
    "int8_matmul_debug": (_i, [_p, _i, _i, _p, _p, _i, _f, _p, _p, _p, _sz, _p,
                               _p, _p, _p, _p, _p]),
    "absmax_quantize_rows": (_i, [_p, _i, _i, _p, _p, _p]),
    "zeropoint_quantize_rows": (_i, [_p, _i, _i, _p, _p, _p, _p]),
    "f16_matmul": (_i, [_p, _i, _i, _p, _i, _p, _p, _p]),
    "i8_test_stalled_matmul": (_i, [_p, _i, _i, _p, _p, _i, _p, _p, _sz, C.c_uint64, _p]),
    "i8_get_status": (_i, [_p, _p]),
    "i8_status_string": (C.c_char_p, [_i]),
    "i8_last_launch_count": (_i, []),
    "i8_set_profile_events": (None, [_p]),
}

_lib = None


class Int8mmError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")


def lib() -> C.CDLL:
    """The loaded libint8mm.so (built in-tree by build.py). Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m "
                              "int8_mixed_precision_03_b300.build` (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(dev: torch.device) -> C.c_void_p:
    return C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(fn: str, code: int) -> None:
    if code != I8_OK:
        raise Int8mmError(fn, code)


def _need(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def int8_quantize_weight(W: torch.Tensor):
    """fp16 W [out, in] -> (CB int8 [out, in], SCB fp32 [out]) with W ~ CB*SCB/127."""
    _need(W, torch.float16, "W")
    out, d = W.shape
    CB = torch.empty((out, d), dtype=torch.int8, device=W.device)
    SCB = torch.empty(out, dtype=torch.float32, device=W.device)
    _check("int8_quantize_weight",
           lib().int8_quantize_weight(_ptr(W), out, d, _ptr(CB), _ptr(SCB), _stream(W.device)))
    return CB, SCB


def int8_matmul_workspace_size(T: int, d_in: int, d_out: int, max_outlier_cols: int = 0) -> int:
    return int(lib().int8_matmul_workspace_size(T, d_in, d_out, max_outlier_cols))


def alloc_workspace(T: int, d_in: int, d_out: int, device, max_outlier_cols: int = 0):
    n = int8_matmul_workspace_size(T, d_in, d_out, max_outlier_cols)
    if n == 0:
        raise ValueError("invalid sizes for int8_matmul")
    return torch.empty(n, dtype=torch.uint8, device=device)


def int8_matmul(X: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor, threshold: float = 6.0,
                bias: torch.Tensor | None = None, Y: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None) -> torch.Tensor:
    """LLM.int8() matmul: fp16 X [T, in], CB/SCB from int8_quantize_weight -> fp16 Y [T, out]."""
    _need(X, torch.float16, "X")
    _need(CB, torch.int8, "CB")
    _need(SCB, torch.float32, "SCB")
    T, d = X.shape
    out = CB.shape[0]
    if bias is not None:
        _need(bias, torch.float16, "bias")
    if Y is None:
        Y = torch.empty((T, out), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(T, d, out, X.device)
    _check("int8_matmul", lib().int8_matmul(
        _ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(bias), _ptr(Y),
        _ptr(workspace), workspace.numel(), _stream(X.device)))
    return Y


def int8_matmul_noalloc(X: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor,
                        threshold: float = 6.0, bias: torch.Tensor | None = None,
                        Y: torch.Tensor | None = None) -> torch.Tensor:
    """int8_matmul on the library's built-in device scratch instead of a workspace, for
    callers that cannot allocate device memory at call time (pass a preallocated Y)."""
    _need(X, torch.float16, "X")
    _need(CB, torch.int8, "CB")
    _need(SCB, torch.float32, "SCB")
    T, d = X.shape
    out = CB.shape[0]
    if Y is None:
        Y = torch.empty((T, out), dtype=torch.float16, device=X.device)
    _check("int8_matmul_noalloc", lib().int8_matmul_noalloc(
        _ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(bias), _ptr(Y),
        _stream(X.device)))
    return Y


def int8_matmul_debug(X, CB, SCB, threshold=6.0, bias=None, workspace=None):
    """int8_matmul plus its intermediates: dict of Y, idx (outlier columns), n_out, Xq,
    rowabs and acc (exact int32 products)."""
    _need(X, torch.float16, "X")
    T, d = X.shape
    out = CB.shape[0]
    dev = X.device
    Y = torch.empty((T, out), dtype=torch.float16, device=dev)
    idx = torch.full((d,), -1, dtype=torch.int32, device=dev)
    n = torch.zeros(4, dtype=torch.int32, device=dev)
    Xq = torch.empty((T, d), dtype=torch.int8, device=dev)
    rowabs = torch.empty(T, dtype=torch.float32, device=dev)
    acc = torch.empty((T, out), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(T, d, out, dev)
    _check("int8_matmul_debug", lib().int8_matmul_debug(
        _ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(bias), _ptr(Y),
        _ptr(workspace), workspace.numel(), _stream(dev), _ptr(idx), _ptr(n), _ptr(Xq),
        _ptr(rowabs), _ptr(acc)))
    n_out = int(n[0].item())
    return {"Y": Y, "idx": idx[:n_out], "n_out": n_out, "Xq": Xq, "rowabs": rowabs, "acc": acc,
            "workspace": workspace}


def absmax_quantize_rows(X: torch.Tensor):
    """fp16 X [rows, cols] -> (int8 Q, fp32 absmax [rows])."""
    _need(X, torch.float16, "X")
    rows, cols = X.shape
    Q = torch.empty((rows, cols), dtype=torch.int8, device=X.device)
    a = torch.empty(rows, dtype=torch.float32, device=X.device)
    _check("absmax_quantize_rows", lib().absmax_quantize_rows(
        _ptr(X), rows, cols, _ptr(Q), _ptr(a), _stream(X.device)))
    return Q, a


def zeropoint_quantize_rows(X: torch.Tensor):
    """fp16 X [rows, cols] -> (int8 Q, fp32 S [rows], fp32 Z [rows]); X ~ (Q + Z)/S."""
    _need(X, torch.float16, "X")
    rows, cols = X.shape
    Q = torch.empty((rows, cols), dtype=torch.int8, device=X.device)
    S = torch.empty(rows, dtype=torch.float32, device=X.device)
    Z = torch.empty(rows, dtype=torch.float32, device=X.device)
    _check("zeropoint_quantize_rows", lib().zeropoint_quantize_rows(
        _ptr(X), rows, cols, _ptr(Q), _ptr(S), _ptr(Z), _stream(X.device)))
    return Q, S, Z


def f16_matmul(X: torch.Tensor, W: torch.Tensor, bias: torch.Tensor | None = None,
               Y: torch.Tensor | None = None) -> torch.Tensor:
    """Our tcgen05 fp16 GEMM: Y = X W^T + bias (fp32 accumulation, fp16 out)."""
    _need(X, torch.float16, "X")
    _need(W, torch.float16, "W")
    T, d = X.shape
    out = W.shape[0]
    if Y is None:
        Y = torch.empty((T, out), dtype=torch.float16, device=X.device)
    _check("f16_matmul", lib().f16_matmul(_ptr(X), T, d, _ptr(W), out, _ptr(bias), _ptr(Y),
                                          _stream(X.device)))
    return Y


def i8_get_status(workspace: torch.Tensor) -> int:
    """Synchronizes the current stream and returns the workspace's device status code."""
    return int(lib().i8_get_status(_ptr(workspace), _stream(workspace.device)))


def i8_last_launch_count() -> int:
    return int(lib().i8_last_launch_count())


def i8_set_profile_events(events) -> None:
    """events: None, or 4 torch.cuda.Event(enable_timing=True) recorded around the three
    kernels of every following int8_matmul on this thread."""
    if events is None:
        lib().i8_set_profile_events(None)
        return
    for e in events:  # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record()
    arr = (C.c_void_p * 4)(*[C.c_void_p(e.cuda_event) for e in events])
    lib().i8_set_profile_events(C.cast(arr, C.c_void_p))
