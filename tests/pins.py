"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` on a
mismatch.  The same pins run against the real oracle (tests/test_oracle_pins.py)
and against copies built with one planted mistake each, to show that every
planted mistake fails at least one pin.

What the pins rest on:
  * hand-derived packed bytes (tests/golden/pack_examples.txt), from the
    contiguous LSB-first rule of ao PR #2167 "metal lowbit kernels: qmv_fast
    optimization", Summary bullet 2;
  * the closed form "a packed row is the little-endian byte string of the
    integer sum_k q_k * 2^(k*b)" (Python big integers);
  * numpy's ``packbits(bitorder='little')`` on the code bits;
  * brute-force enumeration of codes on tiny K;
  * numpy's IEEE conversions for fp16 / bf16;
  * hand-derived worked examples of the layer (tests/golden/linear_worked.json);
  * special cases that reduce to a plain numpy matmul (scale = 1, zero = 0) or to
    group sums of x (scale = 0);
  * the quantise-then-dequantise invariant |w - W| <= scale/2.
"""
from __future__ import annotations

import json
from pathlib import Path

import math

import numpy as np

import synth

GOLDEN = Path(__file__).resolve().parent / "golden"

BF16_ONE = 0x3F80


# ---------------------------------------------------------------------------
# Independent helpers (numpy / Python ints; no oracle code).
# ---------------------------------------------------------------------------

def bigint_pack_row(codes_row, bits):
    v = 0
    for k, q in enumerate(codes_row):
        v |= (int(q) & ((1 << bits) - 1)) << (k * bits)
    return list(v.to_bytes(len(codes_row) * bits // 8, "little"))


def numpy_unpack(packed, K, bits):
    """Codes from packed rows via np.unpackbits (little bit order)."""
    N = packed.shape[0]
    stream = np.unpackbits(packed, axis=1, bitorder="little")[:, :K * bits]
    stream = stream.reshape(N, K, bits).astype(np.int64)
    return (stream << np.arange(bits)).sum(axis=2).astype(np.uint8)


def numpy_pack(codes, bits):
    N, K = codes.shape
    c = codes.astype(np.int64) & ((1 << bits) - 1)
    b = ((c[:, :, None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(N, K * bits)
    return np.packbits(b, axis=1, bitorder="little")


def f16(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def load_pack_examples():
    out = []
    for line in (GOLDEN / "pack_examples.txt").read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        b, codes, packed = (t.strip() for t in line.split(";"))
        out.append((int(b), [int(c) for c in codes.split()], [int(h, 16) for h in packed.split()]))
    return out


def _rule_vector(rule, K):
    kind = rule[0]
    k = np.arange(K)
    if kind == "const":
        return np.full(K, rule[1], dtype=np.float64)
    if kind == "mod":
        return (k % rule[1]) + rule[2]
    if kind == "rev_mod":
        return rule[2] - (k % rule[1])
    if kind == "iota":
        return k.astype(np.float64)
    if kind == "first_half":
        return np.where(k < K // 2, rule[1], 0.0)
    if kind == "second_half":
        return np.where(k >= K // 2, rule[1], 0.0)
    raise ValueError(kind)


def load_linear_cases():
    cases = json.loads((GOLDEN / "linear_worked.json").read_text())["cases"]
    out = []
    for c in cases:
        M, K, N = c["M"], c["K"], c["N"]
        codes = np.stack([_rule_vector(c["codes"][min(n, len(c["codes"]) - 1)], K)
                          for n in range(N)]).astype(np.uint8)
        x = np.stack([_rule_vector(c["x"][min(m, len(c["x"]) - 1)], K) for m in range(M)])
        out.append(dict(name=c["name"], M=M, K=K, N=N, bits=c["bits"], group=c["group"],
                        codes=codes, x=bf16(x), scales=f16(c["scales"]), zeros=f16(c["zeros"]),
                        bias=None if c["bias"] is None else f16(c["bias"]),
                        y=np.asarray(c["y"], dtype=np.float64)))
    return out


# ---------------------------------------------------------------------------
# Pins.
# ---------------------------------------------------------------------------

def pin_pack_golden(o):
    for b, codes, expect in load_pack_examples():
        got = o.pack(np.array([codes], np.uint8), b)[0].tolist()
        assert got == expect, f"b={b}: {got} != {expect}"
        back = o.unpack(np.array([expect], np.uint8), len(codes), b)[0].tolist()
        assert back == codes, f"b={b} unpack: {back} != {codes}"


def pin_pack_bigint(o):
    r = np.random.default_rng(11)
    for b in range(1, 8):
        for K in (8, 32, 40, 96, 256):
            codes = r.integers(0, 1 << b, size=(3, K), dtype=np.uint8)
            got = o.pack(codes, b)
            for n in range(3):
                assert got[n].tolist() == bigint_pack_row(codes[n], b), (b, K, n)


def pin_pack_numpy(o):
    r = np.random.default_rng(12)
    for b in range(1, 8):
        codes = r.integers(0, 1 << b, size=(5, 512), dtype=np.uint8)
        assert np.array_equal(o.pack(codes, b), numpy_pack(codes, b)), b
        packed = r.integers(0, 256, size=(5, 64 * b), dtype=np.uint8)
        assert np.array_equal(o.unpack(packed, 512, b), numpy_unpack(packed, 512, b)), b


def pin_roundtrip(o):
    r = np.random.default_rng(13)
    for b in range(1, 8):
        for K in (32, 64, 4096):
            codes = r.integers(0, 1 << b, size=(4, K), dtype=np.uint8)
            assert np.array_equal(o.unpack(o.pack(codes, b), K, b), codes), (b, K)


def pin_brute_force_single_code(o):
    for b in range(1, 8):
        for k in range(8):
            for v in range(1 << b):
                codes = np.zeros((1, 8), np.uint8)
                codes[0, k] = v
                packed = o.pack(codes, b)[0]
                expect = (v << (k * b)).to_bytes(b, "little")
                assert packed.tobytes() == expect, (b, k, v)


def pin_brute_force_identity(o):
    # b = 1, K = 8 and b = 2, K = 4: every code vector maps to one byte, and
    # all 256 vectors must give the 256 byte values, in order.
    for b, K in ((1, 8), (2, 4)):
        vecs = np.array([[(v >> (k * b)) & ((1 << b) - 1) for k in range(K)] for v in range(256)],
                        np.uint8)
        packed = o.pack(vecs, b)
        assert packed[:, 0].tolist() == list(range(256)), b
        assert np.array_equal(o.unpack(packed, K, b), vecs), b


def pin_code_masking(o):
    r = np.random.default_rng(14)
    for b in range(1, 8):
        codes = r.integers(0, 256, size=(2, 64), dtype=np.uint8)
        assert np.array_equal(o.pack(codes, b), o.pack(codes & ((1 << b) - 1), b)), b


def pin_half_decode(o):
    lib_vals = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([o.half_to_double(h) for h in range(0, 65536, 7)])
    ref = lib_vals[::7]
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def pin_bf16_decode(o):
    bits = np.arange(0, 65536, 5, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([o.bf16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


@np.errstate(over="ignore")
def pin_half_round(o):
    r = np.random.default_rng(15)
    vals = np.concatenate([r.standard_normal(3000) * 10.0 ** r.integers(-9, 5, 3000),
                           [65519.0, 65520.0, 1e-8, -3e-8, 2.0 ** -25, 0.5 + 2.0 ** -12]])
    for v in vals:
        rn = o.double_to_half(v, 0)
        assert rn == int(np.float16(v).view(np.uint16)), v
        dn = np.float64(np.uint16(o.double_to_half(v, 1)).view(np.float16))
        up = np.float64(np.uint16(o.double_to_half(v, 2)).view(np.float16))
        assert dn <= v <= up, v
        if dn != up:
            assert np.nextafter(np.float16(dn), np.float16(np.inf)) == np.float16(up), v


def pin_linear_worked(o):
    for c in load_linear_cases():
        packed = numpy_pack(c["codes"], c["bits"])
        y = o.linear(c["x"], packed, c["scales"], c["zeros"], c["bias"], c["K"], c["bits"], c["group"])
        assert np.array_equal(y, c["y"]), (c["name"], y, c["y"])


def pin_linear_integer_matmul(o):
    # scale = 1, zero = 0: W = q exactly, so y = x @ q^T (a plain numpy matmul).
    r = np.random.default_rng(16)
    for b, g in ((1, 32), (3, 64), (4, 128), (7, 256)):
        M, K, N = 3, 512, 17
        codes = r.integers(0, 1 << b, size=(N, K), dtype=np.uint8)
        x = synth.make_x(3, M, K)
        ones, zeros = f16(np.ones((N, K // g))), f16(np.zeros((N, K // g)))
        y = o.linear(x, numpy_pack(codes, b), ones, zeros, None, K, b, g)
        xf = synth.bf16_bits_to_f32(x).astype(np.float64)
        ref = xf @ codes.astype(np.float64).T
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-12), (b, g)


def pin_linear_zero_only(o):
    # scale = 0: W[n,k] = zero[n, k//g], so y[m,n] = sum_g zero[n,g] * sum_{k in g} x[m,k].
    r = np.random.default_rng(17)
    M, K, N, g, b = 2, 1024, 9, 128, 5
    codes = r.integers(0, 1 << b, size=(N, K), dtype=np.uint8)
    x = synth.make_x(4, M, K)
    z = f16(r.uniform(-1, 1, size=(N, K // g)))
    y = o.linear(x, numpy_pack(codes, b), f16(np.zeros((N, K // g))), z, None, K, b, g)
    xs = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(M, K // g, g).sum(axis=2)
    ref = xs @ z.view(np.float16).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def pin_linear_one_group(o):
    # Only group j has a non-zero scale and zero; every other group contributes 0.
    # A one-hot x at column k then gives W[n,k] when k is in group j, else 0.
    r = np.random.default_rng(18)
    N, K, g, b = 5, 512, 64, 4
    G = K // g
    codes = r.integers(0, 1 << b, size=(N, K), dtype=np.uint8)
    packed = numpy_pack(codes, b)
    for j in (0, 3, G - 1):
        s = np.zeros((N, G)); z = np.zeros((N, G))
        s[:, j] = r.uniform(0.5, 2.0, N); z[:, j] = r.uniform(-3, 3, N)
        sh, zh = f16(s), f16(z)
        for k in (0, 70, j * g, j * g + g - 1, K - 1):
            x = np.zeros((1, K), np.uint16); x[0, k] = BF16_ONE
            y = o.linear(x, packed, sh, zh, None, K, b, g)[0]
            if k // g == j:
                ref = (sh[:, j].view(np.float16).astype(np.float64) * codes[:, k]
                       + zh[:, j].view(np.float16).astype(np.float64))
            else:
                ref = np.zeros(N)
            assert np.array_equal(y, ref), (j, k, y, ref)


def pin_linear_bias_and_rows(o):
    # bias adds per output column n; linear_rows equals the selected columns of linear.
    L = synth.make_layer(5, 3, 256, 11, 6, 32, bias=True)
    packed = numpy_pack(L.codes, 6)
    y = o.linear(L.x, packed, L.scales, L.zeros, L.bias, 256, 6, 32)
    y0 = o.linear(L.x, packed, L.scales, L.zeros, None, 256, 6, 32)
    assert np.array_equal(y - y0, np.broadcast_to(L.bias.view(np.float16).astype(np.float64), y.shape))
    rows = np.array([10, 0, 4])
    yr = o.linear_rows(L.x, packed, L.scales, L.zeros, L.bias, 256, 6, 32, rows)
    assert np.array_equal(yr, y[:, rows])


def pin_linear_numpy_matmul(o):
    # A generic layer against numpy: codes via np.unpackbits, W = s*q + z via
    # numpy broadcasting, then a float64 matmul.
    for b, g in ((2, 32), (5, 64), (6, 256)):
        L = synth.make_layer(6, 4, 768 if g != 256 else 1024, 13, b, g, bias=True)
        K = L.x.shape[1]
        packed = numpy_pack(L.codes, b)
        y = o.linear(L.x, packed, L.scales, L.zeros, L.bias, K, b, g)
        q = numpy_unpack(packed, K, b).astype(np.float64)
        s = np.repeat(L.scales.view(np.float16).astype(np.float64), g, axis=1)
        z = np.repeat(L.zeros.view(np.float16).astype(np.float64), g, axis=1)
        W = s * q + z
        ref = synth.bf16_bits_to_f32(L.x).astype(np.float64) @ W.T + L.bias.view(np.float16)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12), (b, g)


def pin_linearity(o):
    # Homogeneity y(2x) - bias = 2 (y(x) - bias), and additivity over x1, x2 with
    # disjoint column supports (so that x1 + x2 is exact in bf16).
    L = synth.make_layer(7, 2, 256, 6, 3, 64, bias=True)
    packed = numpy_pack(L.codes, 3)
    bias = L.bias.view(np.float16).astype(np.float64)

    def y_of(x):
        return o.linear(x, packed, L.scales, L.zeros, L.bias, 256, 3, 64) - bias

    x = L.x
    x2 = bf16(synth.bf16_bits_to_f32(x) * 2.0)
    assert np.allclose(y_of(x2), 2.0 * y_of(x), rtol=1e-13, atol=1e-13)
    x1 = x.copy(); x1[:, 100:] = 0
    xb = x.copy(); xb[:, :100] = 0
    assert np.allclose(y_of(x), y_of(x1) + y_of(xb), rtol=1e-12, atol=1e-12)


def pin_dequant(o):
    # dequant agrees with the layer on one-hot x (every column recovered) and
    # with the scale=1/zero=0 special case (W equals the codes).
    L = synth.make_layer(8, 1, 128, 7, 7, 32)
    packed = numpy_pack(L.codes, 7)
    W = o.dequant(packed, L.scales, L.zeros, 128, 7, 32)
    for k in (0, 31, 32, 127):
        x = np.zeros((1, 128), np.uint16); x[0, k] = BF16_ONE
        assert np.array_equal(o.linear(x, packed, L.scales, L.zeros, None, 128, 7, 32)[0], W[:, k])
    G = 128 // 32
    Wq = o.dequant(packed, f16(np.ones((7, G))), f16(np.zeros((7, G))), 128, 7, 32)
    assert np.array_equal(Wq, L.codes.astype(np.float64))


def pin_quantizer_invariant(o):
    r = np.random.default_rng(19)
    for b in range(1, 8):
        for g in (32, 64, 128, 256):
            N, K = 4, 512
            w = r.standard_normal((N, K))
            codes, s, z = o.quantize(w, b, g)
            assert codes.max() < (1 << b)
            W = o.dequant(numpy_pack(codes, b), s, z, K, b, g)
            sf = np.repeat(s.view(np.float16).astype(np.float64), g, axis=1)
            assert np.all(np.abs(w - W) <= sf / 2 * (1 + 1e-12)), (b, g)
            # zero never above the group minimum, scale covers the range
            wg = w.reshape(N, K // g, g)
            zf = z.view(np.float16).astype(np.float64)
            assert np.all(zf <= wg.min(axis=2))
            assert np.all(s.view(np.float16).astype(np.float64) * ((1 << b) - 1) + zf >= wg.max(axis=2))


def _f16_down(v: float) -> float:
    """Largest fp16 <= v (numpy's float16, stepped down when it rounded up)."""
    h = np.float16(v)
    if float(h) > v:
        h = np.nextafter(h, np.float16(-np.inf))
    return float(h)


def _f16_up(v: float) -> float:
    """Smallest fp16 >= v."""
    h = np.float16(v)
    if float(h) < v:
        h = np.nextafter(h, np.float16(np.inf))
    return float(h)


def pin_quantizer_constant_group(o):
    # A constant group: every code 0, zero = largest fp16 <= w, scale = the
    # larger of 2^-14 and the smallest fp16 >= 2 (w - zero), so that the
    # weight is recovered within scale / 2 even when w is not an fp16 (fp32 or
    # fp64 input).  Directed rounding here comes from numpy's float16.
    for v in (0.3, -0.3, 0.1, -1.5, 1000.3, 1e-6, -3e-7, float(np.float32(0.3)),
              float(np.float32(-7.7)), 0.0, -0.0):
        for b in (1, 4, 7):
            codes, s, z = o.quantize(np.full((1, 64), v), b, 32)
            assert codes.max() == 0
            zf = _f16_down(v)
            sf = max(2.0 ** -14, _f16_up(2.0 * (v - zf)))
            assert np.all(z.view(np.float16).astype(np.float64) == zf), (v, b)
            assert np.all(s.view(np.float16).astype(np.float64) == sf), (v, b)
            assert abs(v - zf) <= sf / 2, (v, b)
            assert np.all(np.signbit(z.view(np.float16)) == np.signbit(zf)), (v, b)


def _golden_values(field: str) -> list[float]:
    out = []
    for tok in field.split():
        if "*" in tok:
            v, n = tok.split("*")
            out += [float(v)] * int(n)
        else:
            out.append(float(tok))
    return out


def pin_quantizer_golden(o):
    """Hand-derived groups (tests/golden/quantize_worked.txt): exact ties
    (round half to even), signed-zero minima (first zero in k order) and
    constant groups, each with its codes, scale and zero worked out by hand."""
    cases = 0
    for line in (GOLDEN / "quantize_worked.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        bits_f, w_f, q_f, s_f, z_f = (f.strip() for f in line.split(";"))
        b = int(bits_f)
        w = np.array(_golden_values(w_f))
        q = np.array(_golden_values(q_f), dtype=np.int64)
        assert w.size == 32 and q.size == 32, line[:40]
        codes, s, z = o.quantize(w[None, :], b, 32)
        assert codes[0].tolist() == q.tolist(), (line[:40], codes[0].tolist())
        assert int(s[0, 0]) == int(s_f, 16), (line[:40], hex(int(s[0, 0])))
        assert int(z[0, 0]) == int(z_f, 16), (line[:40], hex(int(z[0, 0])))
        cases += 1
    assert cases == 7


def pin_silu_closed_forms(o):
    """sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4 exactly, so silu(+-ln 3) are
    +-ln 3 * (3/4, 1/4); silu(0) = 0; the product is linear in u."""
    l3 = math.log(3.0)
    y = np.array([[l3, -l3, 0.0, 2.5, 1.0, 1.0, 7.0, -3.0]])   # gates | ups (F = 4)
    h = o.silu_mul(y)
    want = [l3 * 0.75 * 1.0, -l3 * 0.25 * 1.0, 0.0, 2.5 * (1.0 / (1.0 + math.exp(-2.5))) * -3.0]
    assert h.shape == (1, 4)
    np.testing.assert_allclose(h[0, :2], want[:2], rtol=1e-15)
    assert h[0, 2] == 0.0
    # Doubling u doubles h.
    y2 = y.copy(); y2[0, 4:] *= 2.0
    np.testing.assert_allclose(o.silu_mul(y2), 2.0 * h, rtol=1e-15)


def pin_silu_odd_identity(o):
    """silu(a) - silu(-a) = a for every a (sigma(a) + sigma(-a) = 1), and the
    tails: silu(a) -> a for large a, -> 0 for very negative a."""
    a = np.array([-30.0, -4.0, -0.5, 0.25, 1.0, 6.0, 30.0])
    F = a.size
    pos = o.silu_mul(np.concatenate([a, np.ones(F)])[None, :])[0]
    neg = o.silu_mul(np.concatenate([-a, np.ones(F)])[None, :])[0]
    np.testing.assert_allclose(pos - neg, a, rtol=1e-14, atol=1e-14)
    assert abs(pos[-1] - 30.0) < 1e-11 and abs(pos[0]) < 1e-11


def pin_silu_layout(o):
    """h[m, f] takes its gate from column f and its up value from column F + f
    of the same row m (not interleaved, not transposed): gates drawn from
    {ln 3, -ln 3, 0}, whose silu values are closed forms, and distinct ups."""
    M, F = 3, 5
    l3 = math.log(3.0)
    silu_of = {0: l3 * 0.75, 1: -l3 * 0.25, 2: 0.0}
    pick = np.array([[(3 * m + 2 * f) % 3 for f in range(F)] for m in range(M)])
    gates = np.choose(pick, [l3, -l3, 0.0])
    ups = np.arange(1, M * F + 1, dtype=np.float64).reshape(M, F) * 1.5
    h = o.silu_mul(np.concatenate([gates, ups], axis=1))
    want = np.vectorize(silu_of.get)(pick) * ups
    np.testing.assert_allclose(h, want, rtol=1e-15, atol=0)


PINS = [
    pin_pack_golden, pin_pack_bigint, pin_pack_numpy, pin_roundtrip,
    pin_brute_force_single_code, pin_brute_force_identity, pin_code_masking,
    pin_half_decode, pin_bf16_decode, pin_half_round,
    pin_linear_worked, pin_linear_integer_matmul, pin_linear_zero_only, pin_linear_one_group,
    pin_linear_bias_and_rows, pin_linear_numpy_matmul, pin_linearity, pin_dequant,
    pin_quantizer_invariant, pin_quantizer_constant_group, pin_quantizer_golden,
    pin_silu_closed_forms, pin_silu_odd_identity, pin_silu_layout,
]
