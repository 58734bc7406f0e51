"""nn.Linear replacement holding groupwise low-bit weights, and a model
transform that swaps every eligible linear layer for it.

The pages' user-facing pieces (ao issue #3446 "Revamp int4 MPS support in
torchao": the `UIntxWeightOnlyQuantizedLinear` module and the recursive
`_replace_linear_with_quantized_linear_mps` walk behind `quant_api.quantize`,
which calls the per-bit-width pack op for every linear; the same issue asks for
bias support) sit above the C ABI here: `LowbitLinear.from_linear` quantises
and packs a layer's weight on the GPU (`lowbit_quantize_weights`) and
`forward` calls `lowbit_linear`.  `LowbitGateUp` holds a gated MLP's gate
and up projections as one packed weight and calls `lowbit_linear_swiglu`.
Only argument marshalling happens in Python; every step runs in the
library's kernels.
"""
from __future__ import annotations

from typing import Callable

import torch

from . import _abi


class LowbitLinear(torch.nn.Module):
    """y = x @ W^T + bias with W[n,k] = scales[n,k//g] * q[n,k] + zeros[n,k//g],
    q packed b bits per code (contiguous, LSB-first).

    Buffers: ``packed`` uint8 [out, in*bits/8], ``scales`` and ``zeros`` fp16
    [out, in/group], ``bias`` fp16 [out] or None.  Inputs are bf16 [..., in]
    on the module's device; outputs are bf16 [..., out].
    """

    def __init__(self, in_features: int, out_features: int, bits: int, group: int,
                 bias: bool = True, device=None):
        super().__init__()
        if not 1 <= bits <= 7:
            raise ValueError(f"bits must be in 1..7, got {bits}")
        if group not in (32, 64, 128, 256) or in_features % group != 0:
            raise ValueError(f"group must be 32, 64, 128 or 256 and divide in_features "
                             f"({in_features}), got {group}")
        self.in_features, self.out_features = in_features, out_features
        self.bits, self.group = bits, group
        G = in_features // group
        self.register_buffer("packed", torch.zeros((out_features, in_features * bits // 8),
                                                   dtype=torch.uint8, device=device))
        self.register_buffer("scales", torch.zeros((out_features, G), dtype=torch.float16, device=device))
        self.register_buffer("zeros", torch.zeros((out_features, G), dtype=torch.float16, device=device))
        if bias:
            self.register_buffer("bias", torch.zeros(out_features, dtype=torch.float16, device=device))
        else:
            self.bias = None

    @classmethod
    @torch.no_grad()
    def from_linear(cls, linear: torch.nn.Linear, bits: int, group: int) -> "LowbitLinear":
        """Quantise a CUDA nn.Linear (fp32, bf16 or fp16 weight) with the min/max
        groupwise quantiser and pack it; the bias, if any, is converted to fp16
        once, here."""
        w = linear.weight
        if not w.is_cuda:
            raise ValueError("from_linear needs the layer on a CUDA device")
        m = cls(linear.in_features, linear.out_features, bits, group,
                bias=linear.bias is not None, device=w.device)
        _abi.quantize_weights(w.detach().contiguous(), bits, group, m.packed, m.scales, m.zeros)
        if linear.bias is not None:
            m.bias.copy_(linear.bias.detach())          # stored as fp16 (load time, once)
        return m

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise ValueError(f"LowbitLinear takes bf16 inputs, got {x.dtype}")
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected inputs [..., {self.in_features}], got {tuple(x.shape)}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        if not x2.is_contiguous():
            raise ValueError("inputs must be contiguous in their last dimension")
        y = _abi.linear(x2, self.packed, self.scales, self.zeros, self.bias, self.bits, self.group)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bits={self.bits}, group={self.group}, bias={self.bias is not None}")


class LowbitGateUp(torch.nn.Module):
    """silu(x @ Wg^T + bg) * (x @ Wu^T + bu): the gate and up projections of a
    gated MLP held as one packed weight of 2F rows (gate rows, then up rows)
    and run as one call (``lowbit_linear_swiglu``).

    Buffers: ``packed`` uint8 [2F, in*bits/8], ``scales`` and ``zeros`` fp16
    [2F, in/group], ``bias`` fp16 [2F] or None.  Inputs bf16 [..., in];
    outputs bf16 [..., F].
    """

    def __init__(self, in_features: int, hidden_features: int, bits: int, group: int,
                 bias: bool = False, device=None):
        super().__init__()
        self.inner = LowbitLinear(in_features, 2 * hidden_features, bits, group, bias=bias, device=device)
        self.in_features, self.hidden_features = in_features, hidden_features

    @classmethod
    @torch.no_grad()
    def from_linears(cls, gate: torch.nn.Linear, up: torch.nn.Linear, bits: int, group: int) -> "LowbitGateUp":
        """Quantise two CUDA nn.Linear layers of the same shape into one gated
        layer (the gate's and up's rows quantised group by group exactly as
        LowbitLinear.from_linear would quantise each)."""
        if gate.weight.shape != up.weight.shape:
            raise ValueError(f"gate and up must have the same shape, got {tuple(gate.weight.shape)} "
                             f"and {tuple(up.weight.shape)}")
        if (gate.bias is None) != (up.bias is None):
            raise ValueError("gate and up must both have a bias or both have none")
        if not gate.weight.is_cuda or not up.weight.is_cuda:
            raise ValueError("from_linears needs both layers on a CUDA device")
        m = cls(gate.in_features, gate.out_features, bits, group, bias=gate.bias is not None,
                device=gate.weight.device)
        w = torch.cat([gate.weight.detach(), up.weight.detach()], dim=0).contiguous()
        i = m.inner
        _abi.quantize_weights(w, bits, group, i.packed, i.scales, i.zeros)
        if gate.bias is not None:
            i.bias.copy_(torch.cat([gate.bias.detach(), up.bias.detach()]))   # fp16, once
        return m

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise ValueError(f"LowbitGateUp takes bf16 inputs, got {x.dtype}")
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected inputs [..., {self.in_features}], got {tuple(x.shape)}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        if not x2.is_contiguous():
            raise ValueError("inputs must be contiguous in their last dimension")
        i = self.inner
        h = _abi.linear_swiglu(x2, i.packed, i.scales, i.zeros, i.bias, i.bits, i.group)
        return h.reshape(*lead, self.hidden_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, hidden_features={self.hidden_features}, "
                f"bits={self.inner.bits}, group={self.inner.group}, bias={self.inner.bias is not None}")


def quantize_(model: torch.nn.Module, bits: int, group: int,
              filter_fn: Callable[[torch.nn.Linear, str], bool] | None = None) -> torch.nn.Module:
    """Replace, in place and recursively, every nn.Linear of `model` that
    `filter_fn(layer, qualified_name)` accepts (default: every layer whose
    in_features is a multiple of `group`) by a LowbitLinear with `bits`-bit
    codes.  Returns `model`."""
    def walk(mod: torch.nn.Module, prefix: str):
        for name, child in list(mod.named_children()):
            full = f"{prefix}.{name}" if prefix else name
            if isinstance(child, torch.nn.Linear):
                ok = filter_fn(child, full) if filter_fn is not None else child.in_features % group == 0
                if ok:
                    setattr(mod, name, LowbitLinear.from_linear(child, bits, group))
            else:
                walk(child, full)
    walk(model, "")
    return model
