"""LowbitLinear / quantize_ host-side behaviour (no GPU needed)."""
import pytest
import torch

import bit_groupwise_weight_gb300 as lb


def test_buffers_and_shapes():
    m = lb.LowbitLinear(256, 48, bits=5, group=64, bias=True, device="cpu")
    sd = m.state_dict()
    assert sd["packed"].shape == (48, 256 * 5 // 8) and sd["packed"].dtype == torch.uint8
    assert sd["scales"].shape == (48, 4) and sd["scales"].dtype == torch.float16
    assert sd["zeros"].shape == (48, 4) and sd["bias"].shape == (48,)
    assert "bias" not in lb.LowbitLinear(256, 48, 5, 64, bias=False, device="cpu").state_dict()


@pytest.mark.parametrize("bits,group,k", [(0, 64, 256), (8, 64, 256), (4, 48, 240), (4, 64, 96)])
def test_bad_configuration_is_rejected(bits, group, k):
    with pytest.raises(ValueError):
        lb.LowbitLinear(k, 16, bits, group, device="cpu")


def test_forward_checks_inputs_before_any_call():
    m = lb.LowbitLinear(128, 16, 4, 64, device="cpu")
    with pytest.raises(ValueError, match="bf16"):
        m(torch.zeros(2, 128, dtype=torch.float32))
    with pytest.raises(ValueError, match="128"):
        m(torch.zeros(2, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        m(torch.zeros(2, 128, dtype=torch.bfloat16))


def test_from_linear_needs_a_cuda_layer():
    with pytest.raises(ValueError, match="CUDA"):
        lb.LowbitLinear.from_linear(torch.nn.Linear(128, 16), 4, 64)


def test_quantize_walks_the_tree_and_respects_the_filter():
    model = torch.nn.Sequential(torch.nn.Linear(128, 64), torch.nn.ReLU(),
                                torch.nn.Sequential(torch.nn.Linear(64, 32), torch.nn.Linear(32, 8)))
    seen = []

    def keep_all(layer, name):
        seen.append((name, layer.in_features))
        return False

    lb.quantize_(model, 4, 32, filter_fn=keep_all)
    assert seen == [("0", 128), ("2.0", 64), ("2.1", 32)]
    assert all(isinstance(m, torch.nn.Linear) for m in (model[0], model[2][0], model[2][1]))
    # The default filter takes every layer whose in_features the group divides;
    # on a CPU model that means a clear error from the first eligible layer.
    with pytest.raises(ValueError, match="CUDA"):
        lb.quantize_(model, 4, 32)


def test_gate_up_buffers_and_checks():
    m = lb.LowbitGateUp(256, 48, bits=3, group=64, bias=True, device="cpu")
    sd = m.state_dict()
    assert sd["inner.packed"].shape == (96, 256 * 3 // 8) and sd["inner.bias"].shape == (96,)
    with pytest.raises(ValueError, match="bf16"):
        m(torch.zeros(2, 256, dtype=torch.float32))
    with pytest.raises(ValueError, match="256"):
        m(torch.zeros(2, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        m(torch.zeros(2, 256, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="same shape"):
        lb.LowbitGateUp.from_linears(torch.nn.Linear(128, 16), torch.nn.Linear(128, 32), 4, 64)
    with pytest.raises(ValueError, match="bias"):
        lb.LowbitGateUp.from_linears(torch.nn.Linear(128, 16), torch.nn.Linear(128, 16, bias=False), 4, 64)
    with pytest.raises(ValueError, match="CUDA"):
        lb.LowbitGateUp.from_linears(torch.nn.Linear(128, 16), torch.nn.Linear(128, 16), 4, 64)
