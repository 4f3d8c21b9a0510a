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
ACT = {"none": 0, "relu": 1}  # I8_ACT_NONE, I8_ACT_RELU
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
    "i8_noalloc_status": (_i, [_p]),
    "int8_matmul_debug": (_i, [_p, _i, _i, _p, _p, _i, _f, _p, _p, _p, _sz, _p,
                               _p, _p, _p, _p, _p]),
    "absmax_quantize_rows": (_i, [_p, _i, _i, _p, _p, _p]),
    "absmax_quantize_blocks": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "zeropoint_quantize_rows": (_i, [_p, _i, _i, _p, _p, _p, _p]),
    "f16_matmul": (_i, [_p, _i, _i, _p, _i, _p, _p, _p]),
    "int8_weight_code_sums": (_i, [_p, _i, _i, _p, _p]),
    "int8_matmul_zeropoint": (_i, [_p, _i, _i, _p, _p, _p, _i, _f, _p, _p, _p, _sz, _p]),
    "int8_matmul_zeropoint_debug": (_i, [_p, _i, _i, _p, _p, _p, _i, _f, _p, _p, _p, _sz, _p,
                                         _p, _p, _p, _p, _p, _p]),
    "int8_ffn_workspace_size": (_sz, [_i, _i, _i, _i]),
    "int8_ffn": (_i, [_p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _f, _i, _p, _p, _p, _sz, _p]),
    "int8_ffn_debug": (_i, [_p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _f, _i, _p, _p, _p, _sz,
                            _p, _p, _p]),
    "f16_ffn": (_i, [_p, _i, _i, _i, _p, _p, _p, _p, _i, _p, _p, _p]),
    "i8_test_stalled_matmul": (_i, [_p, _i, _i, _p, _p, _i, _p, _p, _sz, C.c_uint64, _p]),
    "i8_get_status": (_i, [_p, _p]),
    "i8_status_string": (C.c_char_p, [_i]),
    "i8_last_launch_count": (_i, []),
    "i8_set_profile_events": (None, [_p]),
    "i8_set_profile_events_n": (None, [_p, _i]),
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


def _same_device(dev: torch.device, **tensors) -> None:
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, X on {dev}")


def _out(Y: torch.Tensor | None, shape: tuple, dev: torch.device) -> torch.Tensor:
    """The caller's output buffer after its checks, or a new one."""
    if Y is None:
        return torch.empty(shape, dtype=torch.float16, device=dev)
    _need(Y, torch.float16, "Y")
    if tuple(Y.shape) != tuple(shape):
        raise ValueError(f"Y must have shape {tuple(shape)}, got {tuple(Y.shape)}")
    return Y


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
    Y = _out(Y, (T, out), X.device)
    if workspace is None:
        workspace = alloc_workspace(T, d, out, X.device)
    _same_device(X.device, CB=CB, SCB=SCB, bias=bias, Y=Y, workspace=workspace)
    with torch.cuda.device(X.device):
        _check("int8_matmul", lib().int8_matmul(
            _ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(bias), _ptr(Y),
            _ptr(workspace), workspace.numel(), _stream(X.device)))
    return Y


def int8_matmul_noalloc(X: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor,
                        threshold: float = 6.0, bias: torch.Tensor | None = None,
                        Y: torch.Tensor | None = None) -> torch.Tensor:
    """int8_matmul on the library's built-in device scratch instead of a workspace, for
    callers that cannot allocate device memory at call time (pass a preallocated Y).
    Device-side errors of the call are read with i8_noalloc_status(X.device)."""
    _need(X, torch.float16, "X")
    _need(CB, torch.int8, "CB")
    _need(SCB, torch.float32, "SCB")
    if bias is not None:
        _need(bias, torch.float16, "bias")
    T, d = X.shape
    out = CB.shape[0]
    Y = _out(Y, (T, out), X.device)
    _same_device(X.device, CB=CB, SCB=SCB, bias=bias, Y=Y)
    with torch.cuda.device(X.device):
        _check("int8_matmul_noalloc", lib().int8_matmul_noalloc(
            _ptr(X), T, d, _ptr(CB), _ptr(SCB), out, float(threshold), _ptr(bias), _ptr(Y),
            _stream(X.device)))
    return Y


def i8_noalloc_status(device=None) -> int:
    """Synchronizes the device's current stream and returns the device status code of the
    last int8_matmul_noalloc on it (0 = I8_OK)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().i8_noalloc_status(_stream(dev)))


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


def absmax_quantize_blocks(X: torch.Tensor, block: int = 64):
    """fp16 X [rows, cols] -> (int8 Q, fp32 absmax [rows, ceil(cols / block)]): each block of
    `block` consecutive columns of a row quantized with its own absmax."""
    _need(X, torch.float16, "X")
    if block <= 0:
        raise ValueError("block must be positive")
    rows, cols = X.shape
    nb = (cols + block - 1) // block
    Q = torch.empty((rows, cols), dtype=torch.int8, device=X.device)
    a = torch.empty((rows, nb), dtype=torch.float32, device=X.device)
    with torch.cuda.device(X.device):
        _check("absmax_quantize_blocks", lib().absmax_quantize_blocks(
            _ptr(X), rows, cols, int(block), _ptr(Q), _ptr(a), _stream(X.device)))
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


def int8_weight_code_sums(CB: torch.Tensor) -> torch.Tensor:
    """int32 [out]: the sum of each weight row's codes (input of int8_matmul_zeropoint)."""
    _need(CB, torch.int8, "CB")
    out, d = CB.shape
    sums = torch.empty(out, dtype=torch.int32, device=CB.device)
    _check("int8_weight_code_sums",
           lib().int8_weight_code_sums(_ptr(CB), out, d, _ptr(sums), _stream(CB.device)))
    return sums


def int8_matmul_zeropoint(X, CB, SCB, CBsum, threshold: float = 6.0, bias=None, Y=None,
                          workspace=None) -> torch.Tensor:
    """The matmul with zeropoint activation codes: fp16 X [T, in] -> fp16 Y [T, out]."""
    _need(X, torch.float16, "X")
    _need(CB, torch.int8, "CB")
    _need(SCB, torch.float32, "SCB")
    _need(CBsum, torch.int32, "CBsum")
    T, d = X.shape
    out = CB.shape[0]
    if bias is not None:
        _need(bias, torch.float16, "bias")
    if Y is None:
        Y = torch.empty((T, out), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = alloc_workspace(T, d, out, X.device)
    _check("int8_matmul_zeropoint", lib().int8_matmul_zeropoint(
        _ptr(X), T, d, _ptr(CB), _ptr(SCB), _ptr(CBsum), out, float(threshold), _ptr(bias),
        _ptr(Y), _ptr(workspace), workspace.numel(), _stream(X.device)))
    return Y


def int8_matmul_zeropoint_debug(X, CB, SCB, CBsum, threshold: float = 6.0, bias=None,
                                workspace=None):
    """int8_matmul_zeropoint plus its intermediates: dict of Y, idx, n_out, Xq, S, Z, acc."""
    _need(X, torch.float16, "X")
    T, d = X.shape
    out = CB.shape[0]
    dev = X.device
    Y = torch.empty((T, out), dtype=torch.float16, device=dev)
    idx = torch.full((d,), -1, dtype=torch.int32, device=dev)
    n = torch.zeros(4, dtype=torch.int32, device=dev)
    Xq = torch.empty((T, d), dtype=torch.int8, device=dev)
    S = torch.empty(T, dtype=torch.float32, device=dev)
    Z = torch.empty(T, dtype=torch.float32, device=dev)
    acc = torch.empty((T, out), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(T, d, out, dev)
    _check("int8_matmul_zeropoint_debug", lib().int8_matmul_zeropoint_debug(
        _ptr(X), T, d, _ptr(CB), _ptr(SCB), _ptr(CBsum), out, float(threshold), _ptr(bias),
        _ptr(Y), _ptr(workspace), workspace.numel(), _stream(dev), _ptr(idx), _ptr(n),
        _ptr(Xq), _ptr(S), _ptr(Z), _ptr(acc)))
    n_out = int(n[0].item())
    return {"Y": Y, "idx": idx[:n_out], "n_out": n_out, "Xq": Xq, "S": S, "Z": Z, "acc": acc,
            "workspace": workspace}


def int8_ffn_workspace_size(T: int, d_model: int, d_ff: int, max_outlier_cols: int = 0) -> int:
    return int(lib().int8_ffn_workspace_size(T, d_model, d_ff, max_outlier_cols))


def _act(act: str) -> int:
    if act not in ACT:
        raise ValueError(f"act must be one of {sorted(ACT)}")
    return ACT[act]


def _ffn_args(X, CB_up, SCB_up, CB_down, SCB_down, bias_up, bias_down, H, Y, workspace):
    _need(X, torch.float16, "X")
    for t, dt, name in ((CB_up, torch.int8, "CB_up"), (SCB_up, torch.float32, "SCB_up"),
                        (CB_down, torch.int8, "CB_down"), (SCB_down, torch.float32, "SCB_down")):
        _need(t, dt, name)
    for t, name in ((bias_up, "bias_up"), (bias_down, "bias_down")):
        if t is not None:
            _need(t, torch.float16, name)
    T, d = X.shape
    d_ff = CB_up.shape[0]
    if CB_up.shape[1] != d or tuple(CB_down.shape) != (d, d_ff):
        raise ValueError("CB_up must be [d_ff, d_model] and CB_down [d_model, d_ff]")
    dev = X.device
    if H is None:
        H = torch.empty((T, d_ff), dtype=torch.float16, device=dev)
    if Y is None:
        Y = torch.empty((T, d), dtype=torch.float16, device=dev)
    if workspace is None:
        n = int8_ffn_workspace_size(T, d, d_ff)
        if n == 0:
            raise ValueError("invalid sizes for int8_ffn")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    return T, d, d_ff, H, Y, workspace


def int8_ffn(X, CB_up, SCB_up, CB_down, SCB_down, threshold: float = 6.0, bias_up=None,
             bias_down=None, act: str = "relu", H=None, Y=None, workspace=None):
    """FFN block of two LLM.int8() matmuls: H = act(X W_up^T + b_up), Y = H W_down^T + b_down,
    with the second matmul's column statistics taken in the first one's epilogue.
    Returns (H, Y)."""
    T, d, d_ff, H, Y, workspace = _ffn_args(X, CB_up, SCB_up, CB_down, SCB_down, bias_up,
                                            bias_down, H, Y, workspace)
    _check("int8_ffn", lib().int8_ffn(
        _ptr(X), T, d, d_ff, _ptr(CB_up), _ptr(SCB_up), _ptr(bias_up), _ptr(CB_down),
        _ptr(SCB_down), _ptr(bias_down), float(threshold), _act(act), _ptr(H), _ptr(Y),
        _ptr(workspace), workspace.numel(), _stream(X.device)))
    return H, Y


def int8_ffn_debug(X, CB_up, SCB_up, CB_down, SCB_down, threshold: float = 6.0, bias_up=None,
                   bias_down=None, act: str = "relu", workspace=None):
    """int8_ffn plus the second matmul's outlier columns: dict of H, Y, down_idx, down_n_out
    and the workspace."""
    T, d, d_ff, H, Y, workspace = _ffn_args(X, CB_up, SCB_up, CB_down, SCB_down, bias_up,
                                            bias_down, None, None, workspace)
    dev = X.device
    idx = torch.full((d_ff,), -1, dtype=torch.int32, device=dev)
    n = torch.zeros(4, dtype=torch.int32, device=dev)
    _check("int8_ffn_debug", lib().int8_ffn_debug(
        _ptr(X), T, d, d_ff, _ptr(CB_up), _ptr(SCB_up), _ptr(bias_up), _ptr(CB_down),
        _ptr(SCB_down), _ptr(bias_down), float(threshold), _act(act), _ptr(H), _ptr(Y),
        _ptr(workspace), workspace.numel(), _stream(dev), _ptr(idx), _ptr(n)))
    n_out = int(n[0].item()) if T > 0 else 0
    return {"H": H, "Y": Y, "down_idx": idx[:n_out], "down_n_out": n_out,
            "workspace": workspace}


def f16_ffn(X, W_up, W_down, bias_up=None, bias_down=None, act: str = "relu", H=None, Y=None):
    """The fp16 comparator of int8_ffn on our tcgen05 fp16 GEMM. Returns (H, Y)."""
    _need(X, torch.float16, "X")
    _need(W_up, torch.float16, "W_up")
    _need(W_down, torch.float16, "W_down")
    T, d = X.shape
    d_ff = W_up.shape[0]
    if H is None:
        H = torch.empty((T, d_ff), dtype=torch.float16, device=X.device)
    if Y is None:
        Y = torch.empty((T, d), dtype=torch.float16, device=X.device)
    _check("f16_ffn", lib().f16_ffn(_ptr(X), T, d, d_ff, _ptr(W_up), _ptr(bias_up),
                                    _ptr(W_down), _ptr(bias_down), _act(act), _ptr(H), _ptr(Y),
                                    _stream(X.device)))
    return H, Y


def i8_get_status(workspace: torch.Tensor) -> int:
    """Synchronizes the current stream and returns the workspace's device status code."""
    return int(lib().i8_get_status(_ptr(workspace), _stream(workspace.device)))


def i8_last_launch_count() -> int:
    return int(lib().i8_last_launch_count())


def i8_set_profile_events(events) -> None:
    """events: None, or 4 (int8_matmul) or 8 (int8_ffn: both matmuls)
    torch.cuda.Event(enable_timing=True), recorded around the kernels of every following
    call on this thread."""
    if events is None:
        lib().i8_set_profile_events_n(None, 0)
        return
    for e in events:  # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record()
    arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
    lib().i8_set_profile_events_n(C.cast(arr, C.c_void_p), len(events))
