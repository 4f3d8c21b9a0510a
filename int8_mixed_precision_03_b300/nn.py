"""`Linear8bitLt`, a drop-in `torch.nn.Linear` whose matmul is the LLM.int8() C-ABI call, and
`replace_8bit_linear`, which swaps the linear layers of a model for it.

"Hugging Face, LLM.int8() ... Transformers and Accelerate" (agentlenshq summary), section
"transformers integration": the 8-bit module takes (in_features, out_features, bias,
has_fp16_weights, threshold); with has_fp16_weights=False it keeps only the int8 weight
codes CB in [-127, 127] and their scales SCB (W ~ CB * SCB / 127), produced on the GPU
when the module is moved there; section "accelerate": the replacement walks the model
recursively and leaves the output head (`lm_head`) in 16 bit.

Everything numerical runs in the CUDA library (weight quantization and the matmul); this
module only keeps tensors and calls it. It fails on a CPU input: there is no CPU path.
"""
from __future__ import annotations

import math

import torch

from . import int8_matmul, int8_matmul_workspace_size, int8_quantize_weight

# One workspace per (device, stream), shared by every Linear8bitLt that runs there: the
# layers of a model run one after another on a stream, so they never use it at once.
_WORKSPACES: dict = {}


def _workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


class Linear8bitLt(torch.nn.Module):
    """y = LLM.int8() matmul of x with this layer's weight, plus bias (fp16 in and out).

    Before it is moved to a CUDA device the layer holds an fp16 `weight` [out, in]; on the
    device (or when it is loaded there) the weight is quantized once into int8 codes, kept
    as `weight` (int8), and `SCB` (fp32 [out]). With has_fp16_weights=True the fp16 weight is
    kept and quantized again at every call. State dicts hold `weight`, `SCB` (once
    quantized) and `bias`; an int8 state dict loads as it is, an fp16 one is quantized on
    load when the layer is on the GPU. `max_outlier_cols` bounds the outlier columns the
    workspace holds (0: all of `in_features`); more than that is reported in the workspace
    status word, not raised. A threshold <= 0 turns the decomposition off (stored as +inf,
    plain vector-wise int8), since the library takes only positive thresholds."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True,
                 has_fp16_weights: bool = False, threshold: float = 6.0, device=None,
                 max_outlier_cols: int = 0):
        super().__init__()
        if in_features % 16 != 0:
            raise ValueError("in_features must be a multiple of 16")
        self.in_features, self.out_features = in_features, out_features
        self.has_fp16_weights = has_fp16_weights
        self.threshold = float(threshold) if threshold > 0 else math.inf
        self.max_outlier_cols = max_outlier_cols
        w = torch.empty(out_features, in_features, dtype=torch.float16, device=device)
        if w.device.type != "meta":  # the initialisation of nn.Linear
            bound = 1.0 / math.sqrt(in_features)
            with torch.no_grad():
                w.copy_(torch.empty_like(w, dtype=torch.float32).uniform_(-bound, bound))
        self.weight = torch.nn.Parameter(w, requires_grad=has_fp16_weights)
        self.register_buffer("SCB", None)
        if bias:
            self.bias = torch.nn.Parameter(
                torch.zeros(out_features, dtype=torch.float16, device=device),
                requires_grad=has_fp16_weights)
        else:
            self.register_parameter("bias", None)

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, threshold: float = 6.0,
                    has_fp16_weights: bool = False) -> "Linear8bitLt":
        m = cls(linear.in_features, linear.out_features, linear.bias is not None,
                has_fp16_weights, threshold, device="meta")
        m.weight = torch.nn.Parameter(linear.weight.detach().to(torch.float16).contiguous(),
                                      requires_grad=has_fp16_weights)
        if linear.bias is not None:
            m.bias = torch.nn.Parameter(linear.bias.detach().to(torch.float16).contiguous(),
                                        requires_grad=has_fp16_weights)
        m._quantize_if_on_gpu()
        return m

    @property
    def quantized(self) -> bool:
        return self.SCB is not None

    def _quantize_if_on_gpu(self) -> None:
        if self.has_fp16_weights or self.quantized or self.weight.device.type != "cuda":
            return
        CB, SCB = int8_quantize_weight(self.weight.data.contiguous())
        self.weight = torch.nn.Parameter(CB, requires_grad=False)
        self.SCB = SCB

    def _apply(self, fn, recurse=True):
        super()._apply(fn, recurse)
        # the kernels' types, whatever a dtype conversion asked for: fp16 weight and bias,
        # fp32 scales (the int8 codes are not floating point and keep their type)
        if self.weight.dtype.is_floating_point and self.weight.dtype != torch.float16:
            self.weight.data = self.weight.data.to(torch.float16)
        if self.bias is not None and self.bias.dtype != torch.float16:
            self.bias.data = self.bias.data.to(torch.float16)
        if self.SCB is not None and self.SCB.dtype != torch.float32:
            self.SCB = self.SCB.to(torch.float32)
        self._quantize_if_on_gpu()
        return self

    def _load_from_state_dict(self, sd, prefix, local_metadata, strict, missing_keys,
                              unexpected_keys, error_msgs):
        wk, sk, bk = prefix + "weight", prefix + "SCB", prefix + "bias"
        dev = self.weight.device
        shape = (self.out_features, self.in_features)
        if wk not in sd:
            missing_keys.append(wk)
        elif tuple(sd[wk].shape) != shape:
            error_msgs.append(f"{wk}: shape {tuple(sd[wk].shape)}, expected {shape}")
        elif sd[wk].dtype == torch.int8:
            if sk not in sd:
                error_msgs.append(f"{wk} holds int8 codes but {sk} is missing")
            else:
                self.weight = torch.nn.Parameter(sd[wk].to(dev).contiguous(),
                                                 requires_grad=False)
                self.SCB = sd[sk].to(dev, torch.float32).contiguous()
        else:
            self.weight = torch.nn.Parameter(sd[wk].to(dev, torch.float16).contiguous(),
                                             requires_grad=self.has_fp16_weights)
            self.SCB = None
            self._quantize_if_on_gpu()
        if self.bias is not None:
            if bk in sd:
                self.bias.data = sd[bk].to(dev, torch.float16).contiguous()
            else:
                missing_keys.append(bk)
        if strict:
            known = {wk, sk, bk}
            for k in sd:
                if k.startswith(prefix) and "." not in k[len(prefix):] and k not in known:
                    unexpected_keys.append(k)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if not x.is_cuda:
            raise RuntimeError("Linear8bitLt runs on the GPU only: move the model to CUDA")
        if self.has_fp16_weights:
            CB, SCB = int8_quantize_weight(self.weight.data.contiguous())
        elif self.quantized:
            CB, SCB = self.weight, self.SCB
        else:
            raise RuntimeError("Linear8bitLt weight is not on the GPU: move the model first")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features).to(torch.float16).contiguous()
        T = x2.shape[0]
        n = int8_matmul_workspace_size(T, self.in_features, self.out_features,
                                       self.max_outlier_cols)
        ws = _workspace(n, x2.device)
        y = int8_matmul(x2, CB, SCB, self.threshold, self.bias, workspace=ws)
        return y.reshape(*lead, self.out_features).to(x.dtype)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, threshold={self.threshold}, "
                f"has_fp16_weights={self.has_fp16_weights}, quantized={self.quantized}")


def replace_8bit_linear(model: torch.nn.Module, threshold: float = 6.0,
                        modules_to_not_convert=("lm_head",)) -> torch.nn.Module:
    """Replaces, recursively and in place, every torch.nn.Linear whose attribute name is not
    in modules_to_not_convert by a Linear8bitLt holding the same weight and bias (quantized
    at once if the layer is already on the GPU). Returns the model."""
    for name, child in list(model.named_children()):
        if name in modules_to_not_convert:
            continue
        if isinstance(child, torch.nn.Linear) and not isinstance(child, Linear8bitLt):
            if child.in_features % 16 != 0:
                continue  # the int8 kernels need rows of 16-byte multiples: keep it
            setattr(model, name, Linear8bitLt.from_linear(child, threshold))
        else:
            replace_8bit_linear(child, threshold, modules_to_not_convert)
    return model
