"""GPU parity of the gated decode call (lowbit_linear_swiglu) against the fp64
oracle: h = silu(x W[:F]^T + b[:F]) * (x W[F:]^T + b[F:]), rounded once to bf16.

Covers the tensor-core decode kernel (K a multiple of 256, F a multiple of 16,
up to 8 rows of x per launch, K over a cluster), both CUDA-core kernels (the
streaming decode kernel, and the generic kernel for shapes the streaming
kernel does not take), ragged F (not a multiple of the rows a pass or a CTA
covers), M above the rows of x a launch takes, bias on and off, every bit
width, and the full Llama-3.1-8B gate+up layer on sampled outputs.  The
tolerance is derived below (check_gated).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import ATOL_REL, FROB_REL, DeviceLayer, y_to_f64

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


# Tolerance of the gated output.  The method's tolerance is stated for a linear
# output y; h = silu(g) * u is a function of two such sums that the kernel keeps
# in fp32 and rounds once, to h.  An error e in g reaches h multiplied by
# silu'(g) * u, which is large where |u| is (tens at b = 7) and silu(g) is small,
# so the bound is the y tolerance on h plus the first-order effect of an fp32
# accumulation error in g and u:
#     |h - h_ref| <= 2e-2 (1 + |h_ref|) + |silu'(g) u| e_g + |silu(g)| e_u,
#     e = 2^-19 (1 + sum_k |x_k W_nk|),
# 2^-19 being 32 units of fp32 rounding of the magnitude sum: a few times the
# log2(K) units that a blocked fp32 sum of K products can lose (measured: up to
# about 6 at b = 7, K = 4096), while one wrong or dropped 32-code block moves g
# or u by thousands of such units.
E_ACC = 2.0 ** -19


def check_gated(h: np.ndarray, L, fs, what: str, M=None):
    """h [M, len(fs)] (outputs fs of the gated layer) against the oracle."""
    F = L.N // 2
    M = L.M if M is None else M
    packed = ORACLE.pack(L.codes, L.bits)
    ref = ORACLE.linear_swiglu_rows(L.x[:M], packed, L.scales, L.zeros, L.bias, L.K, L.bits, L.group, fs)
    idx = np.concatenate([fs, F + fs])
    W = ORACLE.dequant(packed[idx], L.scales[idx], L.zeros[idx], L.K, L.bits, L.group)
    x = synth.bf16_bits_to_f32(L.x[:M]).astype(np.float64)
    y = x @ W.T
    if L.bias is not None:
        y += L.bias.view(np.float16).astype(np.float64)[idx]
    mag = 1.0 + np.abs(x) @ np.abs(W).T
    r = fs.size
    g, u = y[:, :r], y[:, r:]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    bound = ATOL_REL * (1.0 + np.abs(ref)) + E_ACC * (np.abs(dsilu * u) * mag[:, :r] + np.abs(g * sig) * mag[:, r:])
    err = np.abs(h - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(np.isfinite(h)), f"{what}: non-finite output"
    assert np.all(err <= bound), (f"{what}: element {worst} h={h[worst]} ref={ref[worst]} "
                                  f"err={err[worst]:.3e} > {bound[worst]:.3e}")
    frob = np.linalg.norm(h - ref) / max(np.linalg.norm(ref), 1e-30)
    assert frob <= FROB_REL, f"{what}: relative Frobenius error {frob:.3e}"


def check_h(h, L, what):
    check_gated(y_to_f64(h), L, np.arange(L.N // 2), what)


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
    check_h(h, L, f"stream b={bits} M={M} K={K} F={F} g={group}")


# Tensor-core decode kernel: K a multiple of 256 (over a cluster past 4096),
# F a multiple of 16, up to 2 / 4 / 8 rows of x per launch for g = 32 / 64 / 128+.
@pytest.mark.parametrize("bits", [1, 2, 4, 5, 7])
@pytest.mark.parametrize("M,K,F,group,bias", [
    (1, 4096, 1008, 64, True),
    (4, 2048, 400, 64, False),      # four rows: one launch
    (8, 1280, 208, 128, True),      # eight rows, two column sets per slice
    (6, 8192, 96, 256, True),       # cluster of two CTAs
    (3, 1024, 64, 32, False),       # g = 32: two launches
])
def test_swiglu_decode_kernel(bits, M, K, F, group, bias):
    L = synth.make_layer(80 + bits, M, K, 2 * F, bits, group, bias=bias, outliers=M > 1)
    d = DeviceLayer(L)
    check_h(_run(d), L, f"decode b={bits} M={M} K={K} F={F} g={group}")


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
    check_h(_run(d), L, f"generic b={bits} M={M} K={K} F={F} g={group}")


def test_swiglu_single_output():
    L = synth.make_layer(7, 1, 4096, 2, 4, 64, bias=True)
    d = DeviceLayer(L)
    check_h(_run(d), L, "F = 1")


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
    for M in (1, 2):
        h = _run(d, d.x[:M].contiguous())
        check_gated(y_to_f64(h)[:, fs], L, fs, f"gate_up b={bits} M={M}", M=M)


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
