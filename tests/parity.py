"""Shared helpers for the GPU parity tests: device copies of seeded inputs and
the tolerance check.

Tolerance for bf16 outputs against the fp64 oracle (stated with the method's
target): element-wise |y - y_ref| <= 2e-2 * (1 + |y_ref|), and relative
Frobenius error ||y - y_ref|| / ||y_ref|| <= 5e-3.  The library multiplies the
exact codes (on the tensor cores as bf16 128 + q), accumulates in fp32 and
rounds once to bf16 (relative error 2^-9 ~ 2e-3 per element), so both bounds
leave room for fp32 summation order and the final rounding.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

ATOL_REL = 2e-2
FROB_REL = 5e-3


def dev_u16(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype).cuda()


class DeviceLayer:
    def __init__(self, L: synth.Layer, packed: torch.Tensor | None = None):
        import bit_groupwise_weight_gb300 as lb
        self.L = L
        self.x = dev_u16(L.x, torch.bfloat16)
        self.codes = torch.from_numpy(L.codes).cuda()
        self.packed = packed if packed is not None else lb.pack_weights(self.codes, L.bits)
        self.scales = dev_u16(L.scales, torch.float16)
        self.zeros = dev_u16(L.zeros, torch.float16)
        self.bias = None if L.bias is None else dev_u16(L.bias, torch.float16)

    def run(self, path=0, x=None):
        import bit_groupwise_weight_gb300 as lb
        return lb.linear(self.x if x is None else x, self.packed, self.scales, self.zeros,
                         self.bias, self.L.bits, self.L.group, path=path)


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def check_close(y: np.ndarray, ref: np.ndarray, what: str = ""):
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    bound = ATOL_REL * (1.0 + np.abs(ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: element {worst} y={y[worst]} ref={ref[worst]} "
                                  f"err={err[worst]:.3e} > {bound[worst]:.3e}")
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(y - ref) / nref
        assert rel <= FROB_REL, f"{what}: relative Frobenius error {rel:.3e} > {FROB_REL}"
