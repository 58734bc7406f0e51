"""CPU oracle for the groupwise low-bit weight-only linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  The product
path (the CUDA library and its Python binding) never imports it, and the two
share no code: the arithmetic lives in ``oracle.c`` (plain C, fp64), this file
only marshals numpy arrays into it.

Functions follow the pages' definitions:

* ``pack`` / ``unpack`` -- contiguous LSB-first bit packing, a code spilling
  into the next byte when the current one is full (ao PR #2167
  "metal lowbit kernels: qmv_fast optimization", Summary, bullet 2).
* ``dequant`` -- W[n,k] = scale[n,k//g]*q[n,k] + zero[n,k//g], scales and
  zeros N x num_groups (same page, Summary, bullet 1).
* ``linear`` / ``linear_rows`` -- y = x W^T + bias in fp64 (torchchat PR #1415
  "Add torchao mps ops": weight-only quantization, bit width 1..7, group
  size 32..256; ao issue #3446: bias).
* ``silu_mul`` / ``linear_swiglu`` -- silu(gate) * up over a layer whose
  first half of rows is the gate projection and second half the up
  projection (the MLP of the Llama decode the pages time; written out here).
* ``quantize`` -- a min/max asymmetric reference quantiser (the pages name a
  ``_quantize`` function without defining it; ao PR #2167 Summary bullet 1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"

RN, RD, RU = 0, 1, 2

_lib = None


def build(force: bool = False, defines: tuple[str, ...] = (), out: Path | None = None) -> Path:
    """Compile oracle.c into a shared library with gcc (-O2, no fast-math).

    ``defines`` and ``out`` exist for the pin-strength tests, which compile
    copies with a deliberate mistake planted under a macro.
    """
    target = Path(out) if out is not None else _LIB_PATH
    if target.exists() and not force and not defines:
        if target.stat().st_mtime >= _SRC.stat().st_mtime:
            return target
    target.parent.mkdir(parents=True, exist_ok=True)
    tmp = target.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra"]
    cmd += [f"-D{d}" for d in defines]
    cmd += [str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


def _bind(lib):
    i64, u8p, u16p, f64p, i64p = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p)
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_row_bytes.argtypes = [i64, ctypes.c_int]
    lib.oracle_row_bytes.restype = i64
    lib.oracle_pack.argtypes = [u8p, u8p, i64, i64, ctypes.c_int]
    lib.oracle_unpack.argtypes = [u8p, u8p, i64, i64, ctypes.c_int]
    lib.oracle_dequant.argtypes = [u8p, u16p, u16p, i64, i64, ctypes.c_int, ctypes.c_int, f64p]
    lib.oracle_linear.argtypes = [u16p, u8p, u16p, u16p, u16p, i64, i64, i64,
                                  ctypes.c_int, ctypes.c_int, f64p, f64p]
    lib.oracle_linear_rows.argtypes = [u16p, u8p, u16p, u16p, u16p, i64, i64, i64,
                                       ctypes.c_int, ctypes.c_int, i64p, i64, f64p, f64p]
    lib.oracle_quantize.argtypes = [f64p, i64, i64, ctypes.c_int, ctypes.c_int, u8p, u16p, u16p]
    lib.oracle_silu_mul.argtypes = [f64p, i64, i64, f64p]
    for name in ("oracle_pack", "oracle_unpack", "oracle_dequant", "oracle_linear",
                 "oracle_linear_rows", "oracle_quantize", "oracle_silu_mul"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load(path: Path | None = None):
    """Load (building first if needed) the oracle library; returns a ctypes CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(build())))
    return _lib


class Oracle:
    """numpy-facing wrapper around one build of the oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data

    def _check(self, rc, what):
        if rc != 0:
            raise ValueError(f"oracle {what}: invalid arguments (status {rc})")

    # -- number formats -----------------------------------------------------
    def half_to_double(self, h: int) -> float:
        return self.lib.oracle_half_to_double(int(h))

    def bf16_to_double(self, b: int) -> float:
        return self.lib.oracle_bf16_to_double(int(b))

    def double_to_half(self, v: float, mode: int = RN) -> int:
        return int(self.lib.oracle_double_to_half(float(v), int(mode)))

    # -- packing ------------------------------------------------------------
    def pack(self, codes: np.ndarray, bits: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, K = codes.shape
        out = np.empty((N, K * bits // 8), dtype=np.uint8)
        self._check(self.lib.oracle_pack(self._ptr(codes), self._ptr(out), N, K, bits), "pack")
        return out

    def unpack(self, packed: np.ndarray, K: int, bits: int) -> np.ndarray:
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        N = packed.shape[0]
        out = np.empty((N, K), dtype=np.uint8)
        self._check(self.lib.oracle_unpack(self._ptr(packed), self._ptr(out), N, K, bits), "unpack")
        return out

    # -- dequantisation and the layer -----------------------------------------
    def dequant(self, packed, scales, zeros, K: int, bits: int, group: int) -> np.ndarray:
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        zeros = np.ascontiguousarray(zeros, dtype=np.uint16)
        N = packed.shape[0]
        W = np.empty((N, K), dtype=np.float64)
        self._check(self.lib.oracle_dequant(self._ptr(packed), self._ptr(scales), self._ptr(zeros),
                                            N, K, bits, group, self._ptr(W)), "dequant")
        return W

    def linear(self, x, packed, scales, zeros, bias, K: int, bits: int, group: int) -> np.ndarray:
        """fp64 y [M, N].  x: bf16 bit patterns (uint16) [M, K]; scales/zeros/bias: fp16
        bit patterns (uint16); bias may be None."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        zeros = np.ascontiguousarray(zeros, dtype=np.uint16)
        bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
        M = x.shape[0]
        N = packed.shape[0]
        y = np.empty((M, N), dtype=np.float64)
        tmp = np.empty(K, dtype=np.float64)
        self._check(self.lib.oracle_linear(self._ptr(x), self._ptr(packed), self._ptr(scales),
                                           self._ptr(zeros), self._ptr(bias), M, K, N, bits, group,
                                           self._ptr(y), self._ptr(tmp)), "linear")
        return y

    def linear_rows(self, x, packed, scales, zeros, bias, K: int, bits: int, group: int,
                    rows, N: int | None = None) -> np.ndarray:
        """fp64 y [M, len(rows)] for the listed output rows n only."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        zeros = np.ascontiguousarray(zeros, dtype=np.uint16)
        bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        M = x.shape[0]
        N = packed.shape[0] if N is None else N
        y = np.empty((M, rows.size), dtype=np.float64)
        tmp = np.empty(K, dtype=np.float64)
        self._check(self.lib.oracle_linear_rows(self._ptr(x), self._ptr(packed), self._ptr(scales),
                                                self._ptr(zeros), self._ptr(bias), M, K, N, bits,
                                                group, self._ptr(rows), rows.size, self._ptr(y),
                                                self._ptr(tmp)), "linear_rows")
        return y

    def silu_mul(self, y: np.ndarray) -> np.ndarray:
        """fp64 h [M, F] = silu(y[:, :F]) * y[:, F:] for y [M, 2F]."""
        y = np.ascontiguousarray(y, dtype=np.float64)
        M, N = y.shape
        if N % 2:
            raise ValueError("silu_mul needs an even number of columns")
        h = np.empty((M, N // 2), dtype=np.float64)
        self._check(self.lib.oracle_silu_mul(self._ptr(y), M, N // 2, self._ptr(h)), "silu_mul")
        return h

    def linear_swiglu(self, x, packed, scales, zeros, bias, K: int, bits: int, group: int) -> np.ndarray:
        """fp64 h [M, F] for a 2F-row layer (gate rows, then up rows)."""
        return self.silu_mul(self.linear(x, packed, scales, zeros, bias, K, bits, group))

    def linear_swiglu_rows(self, x, packed, scales, zeros, bias, K: int, bits: int, group: int,
                           fs) -> np.ndarray:
        """fp64 h [M, len(fs)] for the listed outputs f only."""
        fs = np.asarray(fs, dtype=np.int64)
        F = packed.shape[0] // 2
        y = self.linear_rows(x, packed, scales, zeros, bias, K, bits, group, np.concatenate([fs, F + fs]))
        return self.silu_mul(y)

    def quantize(self, w: np.ndarray, bits: int, group: int):
        """Returns (codes uint8 [N,K], scales uint16 fp16 bits [N,K/g], zeros ditto)."""
        w = np.ascontiguousarray(w, dtype=np.float64)
        N, K = w.shape
        codes = np.empty((N, K), dtype=np.uint8)
        scales = np.empty((N, K // group), dtype=np.uint16)
        zeros = np.empty((N, K // group), dtype=np.uint16)
        self._check(self.lib.oracle_quantize(self._ptr(w), N, K, bits, group, self._ptr(codes),
                                             self._ptr(scales), self._ptr(zeros)), "quantize")
        return codes, scales, zeros
