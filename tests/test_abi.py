"""The C-ABI boundary without a GPU: the library loads, exports every symbol the header
declares, sizes workspaces, and rejects bad arguments on the host (nothing launched)."""
import ctypes as C
import math
import os
import re

import pytest

import int8_mixed_precision_03_b300 as i8
from int8_mixed_precision_03_b300 import build as i8build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "int8mm.h")


@pytest.fixture(scope="module")
def L():
    i8build.build()
    return i8.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", src)) - {"defined"})


def test_header_declares_the_pages_calls():
    names = declared_functions()
    for n in ["int8_quantize_weight", "int8_matmul", "absmax_quantize_rows",
              "zeropoint_quantize_rows"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(names) == set(i8.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(8):
        assert L.i8_status_string(code)
    assert L.i8_status_string(99) == b"unknown status"


def test_workspace_size(L):
    f = L.int8_matmul_workspace_size
    assert f(16, 256, 1024, 0) > 0
    assert f(16, 256, 1024, 0) == f(16, 256, 1024, 256)       # <= 0 means `in`
    assert f(16, 256, 1024, 1) == f(16, 256, 1024, 64)         # capacity rounds up to 64
    assert f(16, 256, 1024, 64) < f(16, 256, 1024, 0)
    assert f(-1, 256, 1024, 0) == 0 and f(16, 0, 1024, 0) == 0
    assert f(16, 262144, 1024, 0) == 0                          # above I8_MAX_IN
    # activation codes + both outlier slices dominate at the worst-case capacity
    T, d, o = 2048, 4096, 16384
    assert f(T, d, o, 0) >= 2 * T * d + 2 * (T + o) * d


def fake(addr):
    return C.c_void_p(addr)


A = 1 << 20  # a 16-byte aligned fake device address (never dereferenced: rejected first)


@pytest.mark.parametrize("kw,code", [
    (dict(X=None), 1),                 # null pointer
    (dict(threshold=float("nan")), 1),
    (dict(threshold=0.0), 1),
    (dict(threshold=-6.0), 1),
    (dict(T=-1), 1),
    (dict(d=0), 1),
    (dict(d=24), 2),                   # in not a multiple of 16
    (dict(X=A + 8), 2),                # misaligned pointer
    (dict(Y=A + 2), 2),
    (dict(bias=A + 4), 2),
    (dict(ws=None), 1),
])
def test_matmul_host_validation(L, kw, code):
    a = dict(X=A, T=16, d=256, CB=A, SCB=A, out=1024, threshold=6.0, bias=None, Y=A, ws=A,
             ws_bytes=1 << 30)
    a.update(kw)
    r = L.int8_matmul(fake(a["X"]) if a["X"] else None, a["T"], a["d"], fake(a["CB"]),
                      fake(a["SCB"]), a["out"], a["threshold"],
                      fake(a["bias"]) if a["bias"] else None, fake(a["Y"]),
                      fake(a["ws"]) if a["ws"] else None, a["ws_bytes"], None)
    assert r == code
    assert L.i8_last_launch_count() == 0


def test_matmul_workspace_too_small_and_empty_sizes(L):
    need = L.int8_matmul_workspace_size(16, 256, 1024, 64)
    args = (fake(A), 16, 256, fake(A), fake(A), 1024, 6.0, None, fake(A), fake(A))
    assert L.int8_matmul(*args, need - 1, None) == 3
    # T == 0 or out == 0: valid no-ops, nothing launched, no device needed
    assert L.int8_matmul(fake(A), 0, 256, fake(A), fake(A), 1024, 6.0, None, fake(A), fake(A),
                         1 << 30, None) == 0
    assert L.int8_matmul(fake(A), 16, 256, fake(A), fake(A), 0, math.inf, None, fake(A),
                         fake(A), 1 << 30, None) == 0
    assert L.i8_last_launch_count() == 0


def test_other_entry_points_validate(L):
    assert L.int8_quantize_weight(None, 4, 16, fake(A), fake(A), None) == 1
    assert L.int8_quantize_weight(fake(A + 1), 4, 16, fake(A), fake(A), None) == 2
    assert L.int8_quantize_weight(fake(A), 0, 16, fake(A), fake(A), None) == 0
    assert L.absmax_quantize_rows(fake(A), -1, 8, fake(A), fake(A), None) == 1
    assert L.absmax_quantize_rows(fake(A), 0, 8, fake(A), fake(A), None) == 0
    assert L.absmax_quantize_blocks(fake(A), 2, 8, 0, fake(A), fake(A), None) == 1
    assert L.absmax_quantize_blocks(fake(A), 2, 8, 64, fake(A), None, None) == 1
    assert L.absmax_quantize_blocks(fake(A), 2, 8, 64, fake(A + 2), fake(A), None) == 2
    assert L.absmax_quantize_blocks(fake(A), 0, 8, 64, fake(A), fake(A), None) == 0
    assert L.absmax_quantize_blocks(fake(A), 3, 0, 64, fake(A), fake(A), None) == 0
    assert L.zeropoint_quantize_rows(fake(A), 2, 8, None, fake(A), fake(A), None) == 1
    assert L.zeropoint_quantize_rows(fake(A), 2, 8, fake(A), fake(A + 4), fake(A), None) == 2
    assert L.f16_matmul(fake(A), 4, 20, fake(A), 8, None, fake(A), None) == 2
    assert L.f16_matmul(fake(A), 0, 32, fake(A), 8, None, fake(A), None) == 0
    assert L.i8_get_status(None, None) == 1


def test_stall_hook_rejects_decode_sizes_and_a_zero_limit_before_any_launch():
    L = i8.lib()
    p = C.c_void_p(1 << 20)
    # 8 tokens fit the decode kernels, which the hook does not cover
    assert L.i8_test_stalled_matmul(p, 8, 256, p, p, 64, p, p, 1 << 30, 1000, None) == 1
    assert L.i8_test_stalled_matmul(p, 64, 256, p, p, 64, p, p, 1 << 30, 0, None) == 1
    assert L.i8_last_launch_count() == 0


def test_ffn_workspace_size_is_both_matmuls(L):
    f, g = L.int8_ffn_workspace_size, L.int8_matmul_workspace_size
    T, d, dff = 200, 256, 1024
    both = g(T, dff, d, 0) + g(T, d, dff, 0)
    # the two sections are 256-byte aligned and each is a multiple of 256 bytes
    assert f(T, d, dff, 0) == both
    assert f(T, d, dff, 64) == g(T, dff, d, 64) + g(T, d, dff, 64)
    assert f(T, d, dff, 1) == f(T, d, dff, 64)
    # the capacity of each matmul is clamped to its own input width
    assert f(T, d, dff, 512) == g(T, dff, d, 512) + g(T, d, dff, 256)
    assert f(-1, d, dff, 0) == 0 and f(T, 0, dff, 0) == 0 and f(T, d, 0, 0) == 0
    assert f(T, d, 262144, 0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(act=2), 1),                  # unknown activation
    (dict(act=-1), 1),
    (dict(Y=None), 1),
    (dict(CBd=None), 1),
    (dict(dff=24), 2),                 # d_ff not a multiple of 16
    (dict(d=40), 2),                   # d_model not a multiple of 16
    (dict(CBd=A + 8), 2),
    (dict(bd=A + 2), 2),
    (dict(Y=A + 4), 2),
    (dict(threshold=0.0), 1),
    (dict(ws_bytes=1024), 3),
    (dict(T=0), 0),                    # a no-op: nothing launched, no device needed
])
def test_ffn_host_validation(L, kw, code):
    a = dict(X=A, T=16, d=256, dff=1024, CBu=A, SCBu=A, bu=None, CBd=A, SCBd=A, bd=None,
             threshold=6.0, act=1, H=A, Y=A, ws=A, ws_bytes=1 << 30)
    a.update(kw)
    p = lambda v: fake(v) if v else None  # noqa: E731
    r = L.int8_ffn(p(a["X"]), a["T"], a["d"], a["dff"], p(a["CBu"]), p(a["SCBu"]), p(a["bu"]),
                   p(a["CBd"]), p(a["SCBd"]), p(a["bd"]), a["threshold"], a["act"], p(a["H"]),
                   p(a["Y"]), p(a["ws"]), a["ws_bytes"], None)
    assert r == code
    assert L.i8_last_launch_count() == 0


def test_f16_ffn_validation(L):
    p = fake(A)
    assert L.f16_ffn(p, 4, 32, 64, p, None, p, None, 3, p, p, None) == 1
    assert L.f16_ffn(p, 4, 32, 40, p, None, p, None, 1, p, p, None) == 2
    assert L.f16_ffn(p, 4, 32, 64, p, None, p, None, 1, p, None, None) == 1
    assert L.f16_ffn(p, 0, 32, 64, p, None, p, None, 1, p, p, None) == 0


def test_zeropoint_entry_points_validate(L):
    p = fake(A)
    need = L.int8_matmul_workspace_size(16, 256, 1024, 0)
    # CBsum missing, misaligned; T == 0 is a no-op
    assert L.int8_matmul_zeropoint(p, 16, 256, p, p, None, 1024, 6.0, None, p, p, need,
                                   None) == 1
    assert L.int8_matmul_zeropoint(p, 16, 256, p, p, fake(A + 4), 1024, 6.0, None, p, p, need,
                                   None) == 2
    assert L.int8_matmul_zeropoint(p, 0, 256, p, p, p, 1024, 6.0, None, p, p, need, None) == 0
    assert L.int8_weight_code_sums(None, 4, 16, p, None) == 1
    assert L.int8_weight_code_sums(p, 4, 16, fake(A + 2), None) == 2
    assert L.int8_weight_code_sums(p, 0, 16, p, None) == 0
    assert L.i8_last_launch_count() == 0


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """No CPU fallback: with the shared library missing, the binding raises."""
    monkeypatch.setattr(i8, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(i8, "_lib", None)
    with pytest.raises(ImportError):
        i8.lib()
    import torch
    with pytest.raises((ImportError, ValueError)):
        i8.int8_matmul(torch.zeros(2, 16, dtype=torch.float16),
                       torch.zeros(4, 16, dtype=torch.int8), torch.ones(4))
