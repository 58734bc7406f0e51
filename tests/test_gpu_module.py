"""LowbitLinear and quantize_ on the GPU: every replaced layer against the
oracle's layer built from the oracle's own quantisation of the same weight."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bit_groupwise_weight_gb300 as lb
import synth
from oracle import Oracle
from parity import check_close, y_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _bf16_tensor(a32: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(synth.f32_to_bf16_bits(a32).view(np.int16)).view(torch.bfloat16).cuda()


def _oracle_layer(orc, layer: lb.LowbitLinear, w64: np.ndarray, bias: torch.Tensor | None, x_bits):
    codes, s, z = orc.quantize(w64, layer.bits, layer.group)
    b = None if bias is None else bias.detach().cpu().numpy().view(np.uint16)
    return orc.linear(x_bits, orc.pack(codes, layer.bits), s, z, b, w64.shape[1], layer.bits, layer.group)


def _make_model(seed: int):
    torch.manual_seed(seed)
    model = torch.nn.Sequential(
        torch.nn.Linear(1024, 768, bias=True), torch.nn.GELU(),
        torch.nn.Sequential(torch.nn.Linear(768, 512, bias=False), torch.nn.GELU(),
                            torch.nn.Linear(512, 200, bias=True)))
    for i, lin in enumerate(m for m in model.modules() if isinstance(m, torch.nn.Linear)):
        lin.weight.data = _bf16_tensor(synth.make_weights(seed, lin.out_features, lin.in_features, key=(i,))).cpu()
        if lin.bias is not None:
            lin.bias.data = torch.from_numpy(synth.make_bias(seed, lin.out_features, key=(i,)).view(np.int16)).view(torch.float16)
    return model.cuda()


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 64), (5, 128), (7, 256)])
def test_quantized_model_layers_match_oracle(orc, bits, group):
    model = _make_model(3)
    linears = [m for m in model.modules() if isinstance(m, torch.nn.Linear)]
    weights = [synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(l.weight.detach().float().cpu().numpy())).astype(np.float64)
               for l in linears]
    biases = [l.bias for l in linears]
    lb.quantize_(model, bits, group)
    lows = [m for m in model.modules() if isinstance(m, lb.LowbitLinear)]
    assert len(lows) == 3 and not any(isinstance(m, torch.nn.Linear) for m in model.modules())
    # Capture every layer's input and output on one forward pass.
    seen = []
    hooks = [m.register_forward_hook(lambda mod, inp, out: seen.append((mod, inp[0], out))) for m in lows]
    x = _bf16_tensor(synth.bf16_bits_to_f32(synth.make_x(3, 6, 1024)))
    y = model(x)
    torch.cuda.synchronize()
    for h in hooks:
        h.remove()
    assert y.shape == (6, 200) and y.dtype == torch.bfloat16
    for (mod, inp, out), w64, bias in zip(seen, weights, biases):
        x_bits = inp.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        ref = _oracle_layer(orc, mod, w64, bias, x_bits)
        check_close(y_to_f64(out), ref, f"{mod}")


def test_three_dimensional_inputs_and_filter(orc):
    model = _make_model(4)
    lb.quantize_(model, 4, 64, filter_fn=lambda layer, name: name != "2.2")
    assert isinstance(model[0], lb.LowbitLinear) and isinstance(model[2][0], lb.LowbitLinear)
    assert isinstance(model[2][2], torch.nn.Linear)
    x = _bf16_tensor(synth.bf16_bits_to_f32(synth.make_x(4, 2 * 5, 1024))).view(2, 5, 1024)
    y0 = model[0](x)
    assert y0.shape == (2, 5, 768)
    flat = model[0](x.reshape(10, 1024))
    assert torch.equal(y0.reshape(10, 768), flat)


@pytest.mark.parametrize("bits,group,bias", [(4, 64, True), (3, 128, False)])
def test_gate_up_module_matches_oracle(orc, bits, group, bias):
    """LowbitGateUp from two nn.Linear layers against the oracle's gated layer
    built from the oracle's own quantisation of the stacked weights."""
    K, F = 1024, 300
    torch.manual_seed(5)
    gate = torch.nn.Linear(K, F, bias=bias)
    up = torch.nn.Linear(K, F, bias=bias)
    ws = []
    for i, lin in enumerate((gate, up)):
        lin.weight.data = _bf16_tensor(synth.make_weights(8, F, K, key=(i, bits))).cpu()
        ws.append(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(lin.weight.detach().float().numpy()))
                  .astype(np.float64))
        if bias:
            lin.bias.data = torch.from_numpy(synth.make_bias(8, F, key=(i,)).view(np.int16)).view(torch.float16)
    gate, up = gate.cuda(), up.cuda()
    m = lb.LowbitGateUp.from_linears(gate, up, bits, group)
    x = _bf16_tensor(synth.bf16_bits_to_f32(synth.make_x(8, 2 * 3, K))).view(2, 3, K)
    h = m(x)
    assert h.shape == (2, 3, F) and h.dtype == torch.bfloat16
    w64 = np.concatenate(ws, axis=0)
    codes, s, z = orc.quantize(w64, bits, group)
    b = None if not bias else torch.cat([gate.bias, up.bias]).detach().cpu().numpy().view(np.uint16)
    x_bits = x.reshape(6, K).cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = orc.linear_swiglu(x_bits, orc.pack(codes, bits), s, z, b, K, bits, group)
    check_close(y_to_f64(h.reshape(6, F)), ref, f"gate_up module b={bits} g={group}")
