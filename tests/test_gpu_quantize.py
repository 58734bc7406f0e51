"""GPU quantiser (lowbit_quantize_weights) against the oracle's reference
quantiser: packed bytes, scales and zeros bit-exact.

Both sides take every decision in fp64 on exactly the same weights, so the
codes, scales and zeros must agree bit for bit, including at exact rounding
ties, constant groups and signed-zero minima.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from oracle import Oracle

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "bf16", "f16"]


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _as_dtype(w32: np.ndarray, dtype: str):
    """(device tensor of `dtype`, exact float64 copy of the same values)."""
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(w32, dtype=np.float32))
        return t.cuda(), w32.astype(np.float64)
    if dtype == "bf16":
        bits = synth.f32_to_bf16_bits(w32)
        exact = synth.bf16_bits_to_f32(bits).astype(np.float64)
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda(), exact
    bits = synth.f16_bits(w32)
    exact = bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.float16).cuda(), exact


def _gpu_quantize(w_dev, bits, group):
    import bit_groupwise_weight_gb300 as lb
    packed, scales, zeros = lb.quantize_weights(w_dev, bits, group)
    torch.cuda.synchronize()
    return (packed.cpu().numpy(), scales.cpu().numpy().view(np.uint16),
            zeros.cpu().numpy().view(np.uint16))


def _check_exact(orc, w64, packed, scales, zeros, bits, group, what):
    codes_ref, s_ref, z_ref = orc.quantize(w64, bits, group)
    np.testing.assert_array_equal(scales, s_ref, err_msg=f"{what}: scales")
    np.testing.assert_array_equal(zeros, z_ref, err_msg=f"{what}: zeros")
    K = w64.shape[1]
    np.testing.assert_array_equal(orc.unpack(packed, K, bits), codes_ref, err_msg=f"{what}: codes")
    np.testing.assert_array_equal(packed, orc.pack(codes_ref, bits), err_msg=f"{what}: packed")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_quantize_bit_exact(orc, dtype, bits, group):
    # 37 rows (not a multiple of the 8 groups a block handles), several groups per row.
    w32 = synth.make_weights(0, 37, 512, key=(bits, group))
    w_dev, w64 = _as_dtype(w32, dtype)
    packed, scales, zeros = _gpu_quantize(w_dev, bits, group)
    _check_exact(orc, w64, packed, scales, zeros, bits, group, f"{dtype} b={bits} g={group}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits", [1, 3, 4, 6, 7])
@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_quantize_rows_with_partial_chunk(orc, dtype, bits, group):
    # Rows of one or more whole 1024-weight chunks of a warp and a partial
    # last one (K = 1344 or 1280), so that consecutive chunks of a warp cross
    # row ends at different offsets.
    K = 1344 if group <= 64 else 1280
    w32 = synth.make_weights(4, 29, K, key=(bits, group))
    w_dev, w64 = _as_dtype(w32, dtype)
    packed, scales, zeros = _gpu_quantize(w_dev, bits, group)
    _check_exact(orc, w64, packed, scales, zeros, bits, group, f"partial {dtype} b={bits} g={group}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bits", [3, 4])
def test_quantize_warps_stride_across_rows(orc, dtype, bits):
    # More chunks than resident warps, five chunks a row (K = 4416: four whole
    # and one partial): each warp walks several chunks and its stride carries
    # over row ends at changing chunk offsets.
    K, N = 4416, 1000
    w32 = synth.make_weights(5, N, K, key=(bits, 4416))
    w_dev, w64 = _as_dtype(w32, dtype)
    packed, scales, zeros = _gpu_quantize(w_dev, bits, 64)
    _check_exact(orc, w64, packed, scales, zeros, bits, 64, f"stride {dtype} b={bits}")


def _special_groups(bits: int, group: int) -> np.ndarray:
    """Rows of hand-built groups: each row is one group of `group` weights."""
    qmax = (1 << bits) - 1
    rows = []
    rows.append(np.full(group, 0.375))                        # constant group
    rows.append(np.full(group, -1.5))                         # constant, negative
    # Constant groups whose value is not an fp16 (as fp32 input): the scale must
    # cover min - zero, so that |w - W| <= scale / 2 still holds.
    rows.append(np.full(group, 0.3))
    rows.append(np.full(group, -0.3))
    rows.append(np.full(group, 1000.3))
    rows.append(np.full(group, 1e-6))
    rows.append(np.zeros(group))                              # all +0
    z = np.zeros(group); z[3] = -0.0; z[5] = 1.0              # +0 first, then -0
    rows.append(z)
    z = np.zeros(group); z[0] = -0.0; z[7] = 1.0              # -0 first
    rows.append(z)
    z = np.full(group, 0.5); z[9] = -0.0; z[2] = 0.0          # +0 at k=2 before -0 at k=9
    rows.append(z)
    # Exact ties: min 0 and max qmax * 2^-6 make scale exactly 2^-6 and zero 0,
    # so (j + 1/2) * 2^-6 lands exactly halfway between two codes.
    s0 = 2.0 ** -6
    t = np.array([(j % (qmax + 1) + 0.5) * s0 for j in range(group)])
    t[0], t[1] = 0.0, qmax * s0
    t = np.minimum(t, qmax * s0)
    rows.append(t)
    rows.append(-t)                                           # mirrored ties
    # One large outlier in an otherwise tiny group.
    o = np.linspace(-1e-3, 1e-3, group); o[group // 2] = 40.0
    rows.append(o)
    # Range just above qmax * h for an fp16 h: the scale quotient lies a hair
    # above h, where the fp32 bounds straddle an fp16 step (fp64 decides).
    h = 0.0078125 + 2 ** -17                                  # an fp16 value
    r = np.zeros(group, dtype=np.float32)
    r[1] = np.nextafter(np.float32(qmax * h), np.float32(1.0))
    r[2:] = np.linspace(0.0, qmax * h, group - 2, dtype=np.float32)
    rows.append(r.astype(np.float64))
    rows.append(np.linspace(-3.0, -2.0, group))               # all negative
    rows.append(np.linspace(1e-4, 2e-4, group))               # all positive, tiny range
    return np.stack(rows)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("group", [32, 256])
def test_quantize_special_groups(orc, dtype, bits, group):
    w = _special_groups(bits, group).astype(np.float32)
    # Two groups per row: the special group, then the same values reversed.
    w32 = np.ascontiguousarray(np.concatenate([w, w[:, ::-1]], axis=1))
    w_dev, w64 = _as_dtype(w32, dtype)
    # The signed zeros must survive the conversions.
    assert np.signbit(w64[7, 3]) and not np.signbit(w64[7, 0])
    packed, scales, zeros = _gpu_quantize(w_dev, bits, group)
    _check_exact(orc, w64, packed, scales, zeros, bits, group, f"special {dtype} b={bits} g={group}")
    # The quantiser's bound, on every weight of every special group.
    codes = orc.unpack(packed, w64.shape[1], bits).astype(np.float64)
    sf = np.repeat(scales.view(np.float16).astype(np.float64), group, axis=1)
    zf = np.repeat(zeros.view(np.float16).astype(np.float64), group, axis=1)
    assert np.all(np.abs(w64 - (sf * codes + zf)) <= sf / 2), f"bound {dtype} b={bits} g={group}"


@pytest.mark.parametrize("bits", [2, 3, 4, 6])
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_quantize_packed_any_alignment(orc, bits, offset):
    # The packed output may have any alignment (b = 2, 4, 6 store 16- or
    # 32-bit words only when it is aligned for them); the bytes must not change.
    import bit_groupwise_weight_gb300 as lb
    w32 = synth.make_weights(3, 21, 256, key=(bits, offset))
    w_dev, w64 = _as_dtype(w32, "bf16")
    ref, s_ref, z_ref = _gpu_quantize(w_dev, bits, 64)
    rb = 256 * bits // 8
    flat = torch.zeros(21 * rb + offset, dtype=torch.uint8, device=w_dev.device)
    packed = flat[offset:].view(21, rb)
    assert packed.data_ptr() % 4 != 0 or offset == 0
    lb.quantize_weights(w_dev, bits, 64, packed)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), ref), f"b={bits} offset={offset}"
    assert int(flat[:offset].sum().item()) == 0, "bytes before the output were written"


@pytest.mark.parametrize("bits,group", [(3, 64), (4, 128), (7, 32)])
def test_quantize_full_size_gate_up_sampled(orc, bits, group):
    """Llama 3.1 8B gate+up (K=4096, N=28672) in bf16, checked on sampled rows."""
    K, N = synth.LLAMA_8B["gate_up"]
    w32 = synth.make_weights(1, N, K, key=(bits, group))
    w_dev, w64 = _as_dtype(w32, "bf16")
    packed, scales, zeros = _gpu_quantize(w_dev, bits, group)
    rows = np.sort(synth.rng(1, 99, N).choice(N, size=64, replace=False))
    rows = np.unique(np.concatenate([[0, N - 1], rows]))
    _check_exact(orc, w64[rows], packed[rows], scales[rows], zeros[rows], bits, group,
                 f"gate_up b={bits} g={group}")


def test_quantize_then_linear_matches_oracle(orc):
    """The quantiser's outputs feed lowbit_linear directly: y agrees with the
    oracle's layer built from the oracle's own quantisation."""
    import bit_groupwise_weight_gb300 as lb
    from parity import check_close, dev_u16, y_to_f64
    M, K, N, bits, group = 3, 1024, 200, 5, 64
    w_dev, w64 = _as_dtype(synth.make_weights(2, N, K), "bf16")
    packed, scales, zeros = lb.quantize_weights(w_dev, bits, group)
    x = synth.make_x(2, M, K)
    y = lb.linear(dev_u16(x, torch.bfloat16), packed, scales, zeros, None, bits, group)
    codes_ref, s_ref, z_ref = orc.quantize(w64, bits, group)
    ref = orc.linear(x, orc.pack(codes_ref, bits), s_ref, z_ref, None, K, bits, group)
    check_close(y_to_f64(y), ref, "quantize -> linear")


def test_quantize_empty_and_errors():
    import bit_groupwise_weight_gb300 as lb
    w = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    packed, scales, zeros = lb.quantize_weights(w, 4, 64)
    assert packed.shape == (0, 32) and scales.shape == (0, 1) and zeros.shape == (0, 1)
    w = torch.zeros((4, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(lb.LowbitError):
        lb.quantize_weights(w, 4, 64)                  # K % group != 0
    with pytest.raises(lb.LowbitError):
        lb.quantize_weights(w[:, :64].contiguous(), 8, 64)   # bits out of range
