"""Guard canaries: every path writes only inside its workspace and its outputs. The
workspace, Y (and H for the FFN block) are slices of larger buffers whose guard bytes on
both sides hold a fixed pattern; after the call every guard byte must still hold it."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (a multiple of 256 keeps the slices aligned)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def i8():
    import int8_mixed_precision_03_b300 as m
    from int8_mixed_precision_03_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


class Guarded:
    """A uint8 buffer [guard | body | guard]; `body` views the middle with a dtype/shape."""

    def __init__(self, nbytes: int, dtype=torch.uint8, shape=None):
        self.n = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda")
        mid = self.buf[GUARD:GUARD + nbytes]
        self.body = mid.view(dtype).view(shape) if shape is not None else mid

    def intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.n:] == PATTERN).all())


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("T,d,out,k", [
    (1, 1024, 300, 2),        # dp4a decode kernel
    (13, 512, 200, 3),        # mma.sync decode kernel
    (37, 1040, 333, 17),      # ragged tiles, out % 8 != 0 (Y without TMA stores)
    (64, 2064, 128, 65),      # split schedule, two outlier K blocks
    (300, 3072, 640, 40),     # split schedule with 256-token tiles
    (520, 4096, 1000, 4),     # whole tiles, several waves of tokens
])
def test_matmul_paths_stay_inside_their_buffers(i8, T, d, out, k):
    w = synth.Workload("guard", T, d, out, n_outlier_cols=k, row_frac=0.8, seed=T * 3 + out)
    X, W, bias = dev(synth.make_x(w)), dev(synth.make_w(w)), dev(synth.make_bias(w))
    CB, SCB = i8.int8_quantize_weight(W)
    sums = i8.int8_weight_code_sums(CB)
    ws = Guarded(i8.int8_matmul_workspace_size(T, d, out, 0))
    for variant in ("absmax", "zeropoint"):
        Y = Guarded(2 * T * out, torch.float16, (T, out))
        if variant == "absmax":
            i8.int8_matmul(X, CB, SCB, 6.0, bias, Y=Y.body, workspace=ws.body)
        else:
            i8.int8_matmul_zeropoint(X, CB, SCB, sums, 6.0, bias, Y=Y.body, workspace=ws.body)
        torch.cuda.synchronize()
        assert i8.i8_get_status(ws.body) == 0
        assert ws.intact(), f"{variant}: workspace guard overwritten"
        assert Y.intact(), f"{variant}: Y guard overwritten"
        assert torch.isfinite(Y.body.float()).all()


@pytest.mark.parametrize("name", ["ffn_small", "ffn_decode_t8"])
def test_ffn_block_stays_inside_its_buffers(i8, name):
    f = synth.FFN_WORKLOADS[name]
    blk = synth.make_ffn(f)
    CBu, SCBu = i8.int8_quantize_weight(dev(blk["W_up"]))
    CBd, SCBd = i8.int8_quantize_weight(dev(blk["W_down"]))
    ws = Guarded(i8.int8_ffn_workspace_size(f.T, f.d_model, f.d_ff, 0))
    H = Guarded(2 * f.T * f.d_ff, torch.float16, (f.T, f.d_ff))
    Y = Guarded(2 * f.T * f.d_model, torch.float16, (f.T, f.d_model))
    i8.int8_ffn(dev(blk["X"]), CBu, SCBu, CBd, SCBd, f.threshold, dev(blk["b_up"]),
                dev(blk["b_down"]), "relu", H=H.body, Y=Y.body, workspace=ws.body)
    torch.cuda.synchronize()
    assert i8.i8_get_status(ws.body) == 0
    assert ws.intact() and H.intact() and Y.intact()
