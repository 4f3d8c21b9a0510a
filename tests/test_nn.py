"""Host-side behaviour of the Linear8bitLt module and the model rewrite (no GPU): types kept
through dtype conversions, state dicts in both forms, the recursive replacement and its
exclusions, and that nothing runs on a CPU tensor."""
import pytest
import torch

from int8_mixed_precision_03_b300.nn import Linear8bitLt, replace_8bit_linear


class Block(torch.nn.Module):
    def __init__(self):
        super().__init__()
        self.up = torch.nn.Linear(32, 64)
        self.act = torch.nn.ReLU()
        self.down = torch.nn.Linear(64, 32, bias=False)


class Model(torch.nn.Module):
    def __init__(self):
        super().__init__()
        self.blocks = torch.nn.ModuleList([Block(), Block()])
        self.odd = torch.nn.Linear(20, 8)          # in_features not a multiple of 16
        self.lm_head = torch.nn.Linear(32, 100)


def test_replacement_is_recursive_and_keeps_the_head():
    torch.manual_seed(0)
    m = Model().half()
    ref = {k: v.clone() for k, v in m.state_dict().items()}
    replace_8bit_linear(m, threshold=5.0)
    for b in m.blocks:
        assert isinstance(b.up, Linear8bitLt) and isinstance(b.down, Linear8bitLt)
        assert b.up.threshold == 5.0 and b.down.bias is None
    assert type(m.lm_head) is torch.nn.Linear and type(m.odd) is torch.nn.Linear
    sd = m.state_dict()
    for k, v in ref.items():   # same weights, not yet quantized (the model is on the CPU)
        assert torch.equal(sd[k], v), k
    assert not any(k.endswith("SCB") for k in sd)


def test_dtype_conversions_keep_the_kernel_types():
    m = Linear8bitLt(32, 48)
    m.float()
    assert m.weight.dtype == torch.float16 and m.bias.dtype == torch.float16
    codes = torch.randint(-127, 128, (48, 32), dtype=torch.int8)
    sd = {"weight": codes, "SCB": torch.rand(48, dtype=torch.float64), "bias": torch.zeros(48)}
    m.load_state_dict(sd)
    assert m.quantized and m.weight.dtype == torch.int8 and m.SCB.dtype == torch.float32
    m.half()
    assert m.weight.dtype == torch.int8 and m.SCB.dtype == torch.float32
    m.to(torch.float32)
    assert torch.equal(m.weight, codes) and m.bias.dtype == torch.float16
    sd2 = m.state_dict()
    assert set(sd2) == {"weight", "SCB", "bias"} and torch.equal(sd2["weight"], codes)


def test_state_dict_errors():
    m = Linear8bitLt(32, 48)
    with pytest.raises(RuntimeError):
        m.load_state_dict({"weight": torch.zeros(48, 16, dtype=torch.float16),
                           "bias": torch.zeros(48)})
    with pytest.raises(RuntimeError):      # int8 codes without their scales
        m.load_state_dict({"weight": torch.zeros(48, 32, dtype=torch.int8),
                           "bias": torch.zeros(48)})
    with pytest.raises(RuntimeError):      # unexpected key under strict loading
        m.load_state_dict({"weight": torch.zeros(48, 32), "bias": torch.zeros(48),
                           "extra": torch.zeros(1)})
    with pytest.raises(ValueError):
        Linear8bitLt(20, 8)


def test_meta_construction_and_no_cpu_path():
    m = Linear8bitLt(64, 128, device="meta")
    assert m.weight.is_meta
    c = Linear8bitLt(64, 128)
    with pytest.raises(RuntimeError):
        c(torch.zeros(2, 64, dtype=torch.float16))


def test_pages_example_two_64_by_64_layers_are_replaced():
    """The transformers-integration example: a model of two 64 x 64 linear layers, both
    replaced (neither is named lm_head), fp16 weights kept until the model moves to a GPU."""
    torch.manual_seed(3)
    fp16_model = torch.nn.Sequential(torch.nn.Linear(64, 64), torch.nn.Linear(64, 64)).half()
    ref = [m.weight.detach().clone() for m in fp16_model]
    int8_model = replace_8bit_linear(fp16_model, threshold=6.0)
    assert all(isinstance(m, Linear8bitLt) for m in int8_model)
    assert all(not m.quantized and m.weight.dtype == torch.float16 for m in int8_model)
    for m, w in zip(int8_model, ref):
        assert torch.equal(m.weight, w)


def test_threshold_zero_turns_the_decomposition_off():
    assert Linear8bitLt(32, 16, threshold=0.0).threshold == float("inf")
    assert Linear8bitLt(32, 16, threshold=-1.0).threshold == float("inf")
    assert Linear8bitLt(32, 16).threshold == 6.0
