"""bit_groupwise_weight_gb300 -- groupwise low-bit weight-only linear layer on GB300.

Python binding of liblowbit (include/lowbit.h).  This module only marshals
arguments: it hands device pointers from torch tensors and the current CUDA
stream to the C ABI.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and every function raises
if the compiled library is missing.

    packed = pack_weights(codes, bits)            # codes: uint8 [N, K] on cuda
    packed, scales, zeros = quantize_weights(w, bits=4, group=64)   # w: float [N, K]
    y = linear(x, packed, scales, zeros, bias, bits=4, group=64)
    h = linear_swiglu(x, packed_gate_up, scales, zeros, bias, bits=4, group=64)   # silu(gate) * up
    quantize_(model, bits=4, group=64)             # nn.Linear -> LowbitLinear, in place
"""
from __future__ import annotations

from ._abi import (  # noqa: F401
    LowbitError,
    PATH_AUTO,
    PATH_QMM,
    PATH_QMV,
    abi,
    linear,
    linear_ptr,
    linear_swiglu,
    linear_swiglu_ptr,
    pack_weights,
    packed_bytes,
    quantize_weights,
    select_path,
    selftest_wait_timeout,
    status_string,
    unpack_weights,
    wait_timeouts,
)
from .module import LowbitGateUp, LowbitLinear, quantize_  # noqa: F401

__all__ = [
    "LowbitError", "LowbitGateUp", "LowbitLinear", "PATH_AUTO", "PATH_QMM", "PATH_QMV", "abi", "linear", "linear_ptr",
    "linear_swiglu", "linear_swiglu_ptr",
    "pack_weights", "packed_bytes", "quantize_weights", "select_path", "selftest_wait_timeout", "status_string", "unpack_weights",
    "quantize_", "wait_timeouts",
]
