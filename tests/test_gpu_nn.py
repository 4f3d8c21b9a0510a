"""Linear8bitLt on the GPU: the weight is quantized on the move to the device exactly as the
oracle quantizes it, the forward pass is the int8_matmul of the same tensors (any leading
shape), quantized state dicts round-trip, and a rewritten model keeps its fp16 head."""
import numpy as np
import pytest
import torch

import oracle
import synth
from int8_mixed_precision_03_b300.nn import Linear8bitLt, replace_8bit_linear

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 2e-3


@pytest.fixture(scope="module")
def i8():
    import int8_mixed_precision_03_b300 as m
    from int8_mixed_precision_03_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def make_layer(d_in=256, d_out=384, seed=3):
    w = synth.Workload("nn", 1, d_in, d_out, seed=seed)
    lin = torch.nn.Linear(d_in, d_out).half()
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(synth.make_w(w)))
        lin.bias.copy_(torch.from_numpy(synth.make_bias(w)))
    return lin


def test_quantized_on_the_move_and_forward_matches_oracle(i8):
    lin = make_layer()
    W = lin.weight.detach().numpy().copy()
    b = lin.bias.detach().numpy().copy()
    m = Linear8bitLt.from_linear(lin).cuda()
    assert m.quantized and m.weight.dtype == torch.int8
    CBo, SCBo = oracle.quantize_weight(W)
    assert np.array_equal(m.weight.cpu().numpy(), CBo)
    assert np.array_equal(m.SCB.cpu().numpy(), SCBo)
    w = synth.Workload("x", 2 * 17, 256, 384, n_outlier_cols=3, seed=5)
    X = synth.make_x(w)
    x = torch.from_numpy(X).cuda().reshape(2, 17, 256)
    y = m(x)
    assert y.shape == (2, 17, 384) and y.dtype == torch.float16
    y2 = i8.int8_matmul(x.reshape(-1, 256), m.weight, m.SCB, 6.0, m.bias)
    assert torch.equal(y.reshape(-1, 384), y2)
    ref = oracle.int8_matmul(X, CBo, SCBo, 6.0, b)
    err = np.abs(y.reshape(-1, 384).cpu().numpy().astype(np.float64) - ref["Y"])
    assert (err <= ATOL + RTOL * np.abs(ref["Y"])).all()
    # an fp32 input comes back fp32, from the same fp16 computation
    y3 = m(x.float())
    assert y3.dtype == torch.float32 and torch.equal(y3.half(), y)


def test_state_dict_round_trip_and_fp16_weights_mode(i8):
    lin = make_layer(seed=4)
    m = Linear8bitLt.from_linear(lin).cuda()
    sd = {k: v.cpu() for k, v in m.state_dict().items()}
    assert sd["weight"].dtype == torch.int8 and "SCB" in sd
    m2 = Linear8bitLt(256, 384).cuda()
    m2.load_state_dict(sd)
    x = torch.from_numpy(synth.make_random_f16(9, (40, 256))).cuda()
    assert torch.equal(m(x), m2(x))
    # fp16 weights kept: quantized again at every call, same result
    m3 = Linear8bitLt.from_linear(lin, has_fp16_weights=True).cuda()
    assert not m3.quantized and m3.weight.dtype == torch.float16
    assert torch.equal(m3(x), m(x))
    # an fp16 state dict loaded into a layer on the GPU is quantized on load
    m4 = Linear8bitLt(256, 384).cuda()
    m4.load_state_dict(lin.state_dict())
    assert m4.quantized and torch.equal(m4(x), m(x))


def test_rewritten_model_keeps_the_head_in_fp16(i8):
    torch.manual_seed(1)
    model = torch.nn.Sequential()
    model.add_module("fc1", torch.nn.Linear(128, 512))
    model.add_module("act", torch.nn.ReLU())
    model.add_module("fc2", torch.nn.Linear(512, 128))
    model.add_module("lm_head", torch.nn.Linear(128, 64))
    model = model.half()
    ref = {k: v.clone() for k, v in model.state_dict().items()}
    replace_8bit_linear(model)
    model.cuda()
    assert isinstance(model.fc1, Linear8bitLt) and model.fc1.quantized
    assert type(model.lm_head) is torch.nn.Linear
    x = torch.from_numpy(synth.make_random_f16(2, (30, 128))).cuda()
    y = model(x)
    # the same chain through the library calls
    CB1, S1 = i8.int8_quantize_weight(ref["fc1.weight"].cuda())
    CB2, S2 = i8.int8_quantize_weight(ref["fc2.weight"].cuda())
    h = torch.relu(i8.int8_matmul(x, CB1, S1, 6.0, ref["fc1.bias"].cuda()))
    h = i8.int8_matmul(h, CB2, S2, 6.0, ref["fc2.bias"].cuda())
    y2 = torch.nn.functional.linear(h, ref["lm_head.weight"].cuda(), ref["lm_head.bias"].cuda())
    assert torch.equal(y, y2)


def test_pages_example_two_64_by_64_layers(i8):
    """The two 64 x 64 layers of the transformers-integration example, moved to the GPU:
    each layer is quantized there and the model's output is the chain of the two calls."""
    torch.manual_seed(3)
    fp16_model = torch.nn.Sequential(torch.nn.Linear(64, 64), torch.nn.Linear(64, 64)).half()
    ref = {k: v.clone() for k, v in fp16_model.state_dict().items()}
    int8_model = replace_8bit_linear(fp16_model).to("cuda")
    assert all(m.quantized for m in int8_model)
    x = torch.from_numpy(synth.make_random_f16(4, (8, 64))).cuda()
    y = int8_model(x)
    CB0, S0 = i8.int8_quantize_weight(ref["0.weight"].cuda())
    CB1, S1 = i8.int8_quantize_weight(ref["1.weight"].cuda())
    h = i8.int8_matmul(x, CB0, S0, 6.0, ref["0.bias"].cuda())
    assert torch.equal(y, i8.int8_matmul(h, CB1, S1, 6.0, ref["1.bias"].cuda()))
