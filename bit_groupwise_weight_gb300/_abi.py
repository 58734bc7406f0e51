"""ctypes binding of liblowbit: same names as the C ABI in include/lowbit.h.

Argument marshalling only.  Tensors must already live on the GPU with the
dtypes and layouts the C ABI documents; this module checks dtypes and shapes,
passes raw pointers and ``torch.cuda.current_stream()``, and turns a non-zero
status into ``LowbitError``.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import build as _build

LOWBIT_OK, LOWBIT_EINVAL, LOWBIT_EUNSUPPORTED, LOWBIT_ECUDA = 0, 1, 2, 3
PATH_AUTO, PATH_QMV, PATH_QMM = 0, 1, 2
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2

_lib = None


class LowbitError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def _bind(lib):
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.lowbit_status_string.argtypes = [ci]
    lib.lowbit_status_string.restype = ctypes.c_char_p
    lib.lowbit_packed_bytes.argtypes = [i64, i64, ci]
    lib.lowbit_packed_bytes.restype = ctypes.c_size_t
    lib.lowbit_pack_weights.argtypes = [vp, vp, i64, i64, ci, vp]
    lib.lowbit_pack_weights.restype = ci
    lib.lowbit_unpack_weights.argtypes = [vp, vp, i64, i64, ci, vp]
    lib.lowbit_unpack_weights.restype = ci
    lib.lowbit_quantize_weights.argtypes = [vp, ci, vp, vp, vp, i64, i64, ci, ci, vp]
    lib.lowbit_quantize_weights.restype = ci
    lib.lowbit_linear.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, vp]
    lib.lowbit_linear.restype = ci
    lib.lowbit_linear_ex.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, vp]
    lib.lowbit_linear_ex.restype = ci
    lib.lowbit_linear_swiglu.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, vp]
    lib.lowbit_linear_swiglu.restype = ci
    lib.lowbit_select_path.argtypes = [i64, i64, i64, ci, ci]
    lib.lowbit_select_path.restype = ci
    lib.lowbit_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32), ci]
    lib.lowbit_wait_timeouts.restype = ci
    lib.lowbit_selftest_wait_timeout.argtypes = [vp, vp]
    lib.lowbit_selftest_wait_timeout.restype = ci
    return lib


def library_path() -> Path:
    """The in-tree build of the library (the only one this binding loads)."""
    return _build.LIB


def abi():
    """The loaded liblowbit (ctypes.CDLL).  Raises ImportError if it was never built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not path.exists():
            raise ImportError(
                f"liblowbit is not built ({path} missing); run bit_groupwise_weight_gb300.build.build()")
        _lib = _bind(ctypes.CDLL(str(path)))
    return _lib


def status_string(status: int) -> str:
    return abi().lowbit_status_string(int(status)).decode()


def packed_bytes(N: int, K: int, bits: int) -> int:
    return int(abi().lowbit_packed_bytes(N, K, bits))


def select_path(M: int, K: int, N: int, bits: int, group: int) -> int:
    return int(abi().lowbit_select_path(M, K, N, bits, group))


def wait_timeouts(reset: bool = False) -> int:
    """Device-side count of bounded waits that gave up (0 in normal operation)."""
    n = ctypes.c_uint32(0)
    _check(abi().lowbit_wait_timeouts(ctypes.byref(n), int(reset)), "lowbit_wait_timeouts")
    return int(n.value)


def selftest_wait_timeout(gave_up: torch.Tensor) -> None:
    """Enqueue the bounded-wait self-test: a kernel whose wait nothing completes
    gives up after the wait limit (about one second), writes 1 to ``gave_up``
    (a CUDA uint32/int32 tensor of one element) and counts one timeout."""
    if not isinstance(gave_up, torch.Tensor) or not gave_up.is_cuda or gave_up.numel() != 1 \
            or gave_up.element_size() != 4:
        raise ValueError("gave_up must be a one-element 32-bit CUDA tensor")
    with torch.cuda.device(gave_up.device):
        _check(abi().lowbit_selftest_wait_timeout(gave_up.data_ptr(), _stream(gave_up.device)),
               "lowbit_selftest_wait_timeout")


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, what: str):
    if status != LOWBIT_OK:
        raise LowbitError(status, what)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _device_of(*tensors) -> torch.device:
    """The one device every given tensor (None entries skipped) lives on; the
    C call is then made with that device current."""
    dev = tensors[0].device
    for t in tensors[1:]:
        if t is not None and t.device != dev:
            raise ValueError(f"all tensors must be on one device, got {dev} and {t.device}")
    return dev


def pack_weights(codes: torch.Tensor, bits: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """codes uint8 [N, K] (one code per byte) -> packed uint8 [N, K*bits/8]."""
    N, K = codes.shape
    _need(codes, "codes", torch.uint8, (N, K))
    if out is None:
        out = torch.empty((N, K * bits // 8), dtype=torch.uint8, device=codes.device)
    _need(out, "out", torch.uint8, (N, K * bits // 8))
    dev = _device_of(codes, out)
    with torch.cuda.device(dev):
        _check(abi().lowbit_pack_weights(codes.data_ptr(), out.data_ptr(), N, K, bits, _stream(dev)),
               "lowbit_pack_weights")
    return out


def unpack_weights(packed: torch.Tensor, K: int, bits: int, out: torch.Tensor | None = None) -> torch.Tensor:
    N = packed.shape[0]
    _need(packed, "packed", torch.uint8, (N, K * bits // 8))
    if out is None:
        out = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    _need(out, "out", torch.uint8, (N, K))
    dev = _device_of(packed, out)
    with torch.cuda.device(dev):
        _check(abi().lowbit_unpack_weights(packed.data_ptr(), out.data_ptr(), N, K, bits, _stream(dev)),
               "lowbit_unpack_weights")
    return out


_W_DTYPES = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}


def quantize_weights(w: torch.Tensor, bits: int, group: int, packed: torch.Tensor | None = None,
                     scales: torch.Tensor | None = None, zeros: torch.Tensor | None = None):
    """w float32/bfloat16/float16 [N, K] -> (packed uint8 [N, K*bits/8],
    scales fp16 [N, K/group], zeros fp16 [N, K/group]), min/max asymmetric."""
    N, K = w.shape
    if w.dtype not in _W_DTYPES:
        raise ValueError(f"w must be float32, bfloat16 or float16, got {w.dtype}")
    _need(w, "w", w.dtype, (N, K))
    G = K // group if group else 0
    if packed is None:
        packed = torch.empty((N, K * bits // 8), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, G), dtype=torch.float16, device=w.device)
    if zeros is None:
        zeros = torch.empty((N, G), dtype=torch.float16, device=w.device)
    _need(packed, "packed", torch.uint8, (N, K * bits // 8))
    _need(scales, "scales", torch.float16, (N, G))
    _need(zeros, "zeros", torch.float16, (N, G))
    dev = _device_of(w, packed, scales, zeros)
    with torch.cuda.device(dev):
        _check(abi().lowbit_quantize_weights(w.data_ptr(), _W_DTYPES[w.dtype], packed.data_ptr(),
                                             scales.data_ptr(), zeros.data_ptr(), N, K, bits, group,
                                             _stream(dev)), "lowbit_quantize_weights")
    return packed, scales, zeros


def linear(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
           bias: torch.Tensor | None, bits: int, group: int, out: torch.Tensor | None = None,
           path: int = PATH_AUTO) -> torch.Tensor:
    """y = x @ W^T + bias with W[n,k] = scales[n,k//g]*q[n,k] + zeros[n,k//g].

    x bf16 [M, K]; packed_w uint8 [N, K*bits/8]; scales, zeros fp16 [N, K/group];
    bias fp16 [N] or None.  Returns bf16 [M, N] (or writes ``out``).
    """
    M, K = x.shape
    N = packed_w.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed_w, "packed_w", torch.uint8, (N, K * bits // 8))
    G = K // group if group else 0
    _need(scales, "scales", torch.float16, (N, G))
    _need(zeros, "zeros", torch.float16, (N, G))
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (M, N))
    dev = _device_of(x, packed_w, scales, zeros, bias, out)
    with torch.cuda.device(dev):
        _check(abi().lowbit_linear_ex(x.data_ptr(), packed_w.data_ptr(), scales.data_ptr(),
                                      zeros.data_ptr(), None if bias is None else bias.data_ptr(),
                                      out.data_ptr(), M, K, N, bits, group, path, _stream(dev)),
               "lowbit_linear")
    return out


def linear_swiglu(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                  bias: torch.Tensor | None, bits: int, group: int,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """silu(x @ W[:F]^T + bias[:F]) * (x @ W[F:]^T + bias[F:]) for a packed
    weight of 2F rows (gate rows, then up rows).

    x bf16 [M, K]; packed_w uint8 [2F, K*bits/8]; scales, zeros fp16
    [2F, K/group]; bias fp16 [2F] or None.  Returns bf16 [M, F] (or writes ``out``).
    """
    M, K = x.shape
    N = packed_w.shape[0]
    if N % 2:
        raise ValueError(f"packed_w must hold 2F rows (gate, then up), got {N}")
    F = N // 2
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed_w, "packed_w", torch.uint8, (N, K * bits // 8))
    G = K // group if group else 0
    _need(scales, "scales", torch.float16, (N, G))
    _need(zeros, "zeros", torch.float16, (N, G))
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,))
    if out is None:
        out = torch.empty((M, F), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (M, F))
    dev = _device_of(x, packed_w, scales, zeros, bias, out)
    with torch.cuda.device(dev):
        _check(abi().lowbit_linear_swiglu(x.data_ptr(), packed_w.data_ptr(), scales.data_ptr(),
                                          zeros.data_ptr(), None if bias is None else bias.data_ptr(),
                                          out.data_ptr(), M, K, F, bits, group, _stream(dev)),
               "lowbit_linear_swiglu")
    return out


def linear_swiglu_ptr(x: int, packed_w: int, scales: int, zeros: int, bias: int | None, y: int,
                      M: int, K: int, F: int, bits: int, group: int, stream: int) -> None:
    """The gated C call on raw device pointers (for CUDA-graph capture and timing loops)."""
    _check(abi().lowbit_linear_swiglu(x, packed_w, scales, zeros, bias, y, M, K, F, bits, group, stream),
           "lowbit_linear_swiglu")


def linear_ptr(x: int, packed_w: int, scales: int, zeros: int, bias: int | None, y: int,
               M: int, K: int, N: int, bits: int, group: int, stream: int,
               path: int = PATH_AUTO) -> None:
    """The C call on raw device pointers (for CUDA-graph capture and timing loops)."""
    _check(abi().lowbit_linear_ex(x, packed_w, scales, zeros, bias, y, M, K, N, bits, group, path,
                                  stream), "lowbit_linear")
