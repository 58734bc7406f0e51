"""GPU parity of the gated decode call (lowbit_linear_swiglu) against the fp64
oracle: h = silu(x W[:F]^T + b[:F]) * (x W[F:]^T + b[F:]), rounded once to bf16.

Covers both CUDA-core kernels (the streaming decode kernel, and the generic
kernel for shapes the streaming kernel does not take), ragged F (not a
multiple of the rows a pass or a CTA covers), M above the two rows of x a
launch takes, bias on and off, every bit width, and the full Llama-3.1-8B
gate+up layer on sampled outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceLayer, check_close, y_to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_groupwise_weight_gb300 as lb  # noqa: E402
from bit_groupwise_weight_gb300 import build as lbuild  # noqa: E402

lbuild.build()
ORACLE = oracle.Oracle()


def _run(d: DeviceLayer, x=None):
    return lb.linear_swiglu(d.x if x is None else x, d.packed, d.scales, d.zeros, d.bias,
                            d.L.bits, d.L.group)


def _oracle_h(L):
    return ORACLE.linear_swiglu(L.x, ORACLE.pack(L.codes, L.bits), L.scales, L.zeros, L.bias,
                                L.K, L.bits, L.group)


# Streaming kernel: K % 1024 == 0 and K/group % 8 == 0.
@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("M,K,F,group,bias", [
    (1, 4096, 1000, 64, True),      # F not a multiple of the rows a pass holds
    (2, 2048, 777, 128, False),     # two rows of x in one launch
    (3, 4096, 513, 64, True),       # M = 3: a two-row launch, then a one-row launch
    (1, 8192, 96, 256, False),      # few outputs: fewer passes than CTAs
])
def test_swiglu_stream_kernel(bits, M, K, F, group, bias):
    L = synth.make_layer(40 + bits, M, K, 2 * F, bits, group, bias=bias)
    d = DeviceLayer(L)
    h = _run(d)
    assert h.shape == (M, F) and h.dtype == torch.bfloat16
    check_close(y_to_f64(h), _oracle_h(L), f"stream b={bits} M={M} K={K} F={F} g={group}")


# Generic kernel: K not a multiple of 1024, or too few groups per row.
@pytest.mark.parametrize("bits", [1, 3, 4, 7])
@pytest.mark.parametrize("M,K,F,group,bias", [
    (1, 1536, 301, 64, True),       # K % 1024 != 0
    (5, 1024, 130, 256, False),     # K/group = 4 groups: gated passes need 8; M in chunks of 4
    (4, 96, 7, 32, True),           # tiny K, odd F
])
def test_swiglu_generic_kernel(bits, M, K, F, group, bias):
    L = synth.make_layer(60 + bits, M, K, 2 * F, bits, group, bias=bias)
    d = DeviceLayer(L)
    check_close(y_to_f64(_run(d)), _oracle_h(L), f"generic b={bits} M={M} K={K} F={F} g={group}")


def test_swiglu_single_output():
    L = synth.make_layer(7, 1, 4096, 2, 4, 64, bias=True)
    d = DeviceLayer(L)
    check_close(y_to_f64(_run(d)), _oracle_h(L), "F = 1")


@pytest.mark.parametrize("bits", [2, 4, 7])
def test_swiglu_full_size_gate_up_sampled(bits):
    """Llama-3.1-8B gate+up (K = 4096, F = 14336, g = 64) at M = 1 and M = 2,
    in the configuration the decode benchmark runs; the oracle on sampled
    outputs, including the first and last."""
    K, N = synth.LLAMA_8B["gate_up"]
    F = N // 2
    L = synth.make_layer(3, 2, K, N, bits, 64, bias=True, outliers=True)
    d = DeviceLayer(L)
    fs = np.unique(np.concatenate([[0, F - 1], np.random.default_rng(bits).choice(F, 96, replace=False)]))
    packed = ORACLE.pack(L.codes, bits)
    for M in (1, 2):
        h = _run(d, d.x[:M].contiguous())
        ref = ORACLE.linear_swiglu_rows(L.x[:M], packed, L.scales, L.zeros, L.bias, K, bits, 64, fs)
        check_close(y_to_f64(h)[:, fs], ref, f"gate_up b={bits} M={M}")


def test_swiglu_matches_unfused_composition():
    """The fused call against the library's own linear followed by silu * up
    in fp32 from the bf16 outputs: equal up to the two extra bf16 roundings
    of the unfused path."""
    L = synth.make_layer(5, 1, 4096, 2 * 2048, 4, 64, bias=True)
    d = DeviceLayer(L)
    h = _run(d).float()
    y = lb.linear(d.x, d.packed, d.scales, d.zeros, d.bias, 4, 64, path=lb.PATH_QMV).float()
    a, u = y[:, :2048], y[:, 2048:]
    h2 = a * torch.sigmoid(a) * u
    err = (h - h2).abs()
    assert torch.all(err <= 2e-2 * (1 + h2.abs())), float(err.max())


def test_swiglu_empty_and_errors():
    L = synth.make_layer(1, 1, 1024, 8, 4, 64)
    d = DeviceLayer(L)
    x0 = torch.empty((0, 1024), dtype=torch.bfloat16, device="cuda")
    assert lb.linear_swiglu(x0, d.packed, d.scales, d.zeros, None, 4, 64).shape == (0, 4)
    with pytest.raises(ValueError):                       # odd row count
        lb.linear_swiglu(d.x, d.packed[:7].contiguous(), d.scales[:7].contiguous(),
                         d.zeros[:7].contiguous(), None, 4, 64)
    with pytest.raises(lb.LowbitError):                   # bits out of range
        lb.linear_swiglu(d.x, d.packed[:, :0].contiguous(), d.scales, d.zeros, None, 0, 64)
    torch.cuda.synchronize()
