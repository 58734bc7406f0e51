"""Host-side checks of the C ABI (no GPU needed).

The library must build, load, and export every function include/lowbit.h
declares; argument validation and path selection are host logic and are
checked here without touching CUDA (every call below is rejected before the
library makes its first CUDA call, or is pure arithmetic).
"""
import ctypes
import re
from pathlib import Path

import pytest

import bit_groupwise_weight_gb300 as lb
from bit_groupwise_weight_gb300 import build as lbuild

ROOT = Path(__file__).resolve().parent.parent
EINVAL = 1


@pytest.fixture(scope="module")
def lib():
    lbuild.build()
    return lb.abi()


def declared_functions():
    text = "\n".join(p.read_text() for p in sorted((ROOT / "include").glob("*.h")))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"LOWBIT_API\s+[\w\s\*]*?\b(lowbit_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for fn in ("lowbit_pack_weights", "lowbit_linear", "lowbit_unpack_weights",
               "lowbit_packed_bytes", "lowbit_status_string", "lowbit_linear_ex",
               "lowbit_select_path", "lowbit_wait_timeouts", "lowbit_linear_swiglu"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(str(lbuild.LIB))
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_packed_bytes(lib):
    assert lb.packed_bytes(4096, 4096, 4) == 4096 * 2048
    assert lb.packed_bytes(3, 8, 3) == 9
    assert lb.packed_bytes(28672, 4096, 7) == 28672 * 4096 * 7 // 8
    assert lb.packed_bytes(1, 12, 3) == 0        # 36 bits: not whole bytes
    assert lb.packed_bytes(1, 32, 0) == 0
    assert lb.packed_bytes(1, 32, 8) == 0
    assert lb.packed_bytes(-1, 32, 4) == 0
    assert lb.packed_bytes(0, 32, 4) == 0
    assert lb.packed_bytes(1, 1 << 62, 7) == 0    # beyond the size limit, no overflow
    assert lb.packed_bytes(1 << 40, 64, 4) == 0


def test_status_strings(lib):
    for s in range(4):
        assert lb.status_string(s)
    assert "invalid" in lb.status_string(1)
    assert lb.status_string(99) == "unknown status"


def test_select_path(lib):
    assert lb.select_path(1, 4096, 4096, 4, 64) == lb.PATH_QMV
    assert lb.select_path(0, 4096, 4096, 4, 64) == lb.PATH_QMV
    assert lb.select_path(128, 4096, 4096, 4, 64) == lb.PATH_QMM
    # Measured crossovers.  The tensor-core decode kernel takes 2 / 4 / 8 rows of x
    # per launch for g = 32 / 64 / >= 128 and wins in up to 128 / g launches (one
    # for g >= 128), twice as many for N >= 24576; with K > 8192 (K split over
    # clusters of three or more CTAs) only up to 4 / 6 / 8 rows.
    assert lb.select_path(8, 4096, 4096, 4, 64) == lb.PATH_QMV        # 2 launches
    assert lb.select_path(9, 4096, 4096, 4, 64) == lb.PATH_QMM
    assert lb.select_path(8, 4096, 6144, 4, 128) == lb.PATH_QMV
    assert lb.select_path(9, 4096, 6144, 4, 128) == lb.PATH_QMM
    assert lb.select_path(4, 14336, 4096, 7, 256) == lb.PATH_QMV
    assert lb.select_path(5, 14336, 4096, 7, 256) == lb.PATH_QMM
    assert lb.select_path(4, 14336, 4096, 4, 128) == lb.PATH_QMV
    assert lb.select_path(5, 14336, 4096, 4, 128) == lb.PATH_QMM
    assert lb.select_path(6, 14336, 4096, 4, 64) == lb.PATH_QMV
    assert lb.select_path(7, 14336, 4096, 4, 64) == lb.PATH_QMM
    assert lb.select_path(8, 14336, 4096, 4, 32) == lb.PATH_QMV
    assert lb.select_path(9, 14336, 4096, 4, 32) == lb.PATH_QMM
    assert lb.select_path(8, 8192, 3072, 4, 128) == lb.PATH_QMV
    assert lb.select_path(8, 8192, 3072, 4, 32) == lb.PATH_QMV        # K = 8192: no row cap
    assert lb.select_path(8, 4096, 4096, 4, 32) == lb.PATH_QMV        # 4 launches
    assert lb.select_path(9, 4096, 4096, 4, 32) == lb.PATH_QMM
    assert lb.select_path(16, 4096, 28672, 4, 128) == lb.PATH_QMV     # 2 launches, N >= 24576
    assert lb.select_path(17, 4096, 28672, 4, 128) == lb.PATH_QMM
    assert lb.select_path(16, 4096, 28672, 4, 64) == lb.PATH_QMV      # 4 launches
    assert lb.select_path(17, 4096, 28672, 4, 64) == lb.PATH_QMM
    assert lb.select_path(16, 4096, 28672, 4, 32) == lb.PATH_QMV      # 8 launches
    assert lb.select_path(17, 4096, 28672, 4, 32) == lb.PATH_QMM
    assert lb.select_path(9, 4096, 16384, 4, 128) == lb.PATH_QMM
    assert lb.select_path(16, 4096, 16384, 4, 128) == lb.PATH_QMM
    assert lb.select_path(9, 4096, 28672, 7, 256) == lb.PATH_QMM      # g = 256: one launch
    # Shapes the decode kernel does not take: the CUDA-core kernel's crossover
    # (K % 256 != 0; K / group not a multiple of 8).
    assert lb.select_path(2, 4096 + 128, 4096, 4, 64) == lb.PATH_QMV
    assert lb.select_path(3, 4096 + 128, 4096, 4, 64) == lb.PATH_QMM
    assert lb.select_path(6, 4096 + 128, 28672, 4, 64) == lb.PATH_QMV
    assert lb.select_path(7, 4096 + 128, 28672, 4, 64) == lb.PATH_QMM
    assert lb.select_path(3, 3072, 3072, 4, 256) == lb.PATH_QMM
    assert lb.select_path(128, 4096 + 64, 4096, 4, 64) == lb.PATH_QMV
    for bad in ((1, 4096, 4096, 0, 64), (1, 4096, 4096, 8, 64), (1, 4096, 4096, 4, 48),
                (1, 4000, 4096, 4, 64), (1, 0, 4096, 4, 64), (-1, 4096, 4096, 4, 64)):
        assert lb.select_path(*bad) == lb.PATH_AUTO


LINEAR_ARGS = dict(x=16, w=16, s=2, z=2, bias=0, y=2, M=1, K=64, N=8, bits=4, group=32, path=0)


def call_linear(lib, **kw):
    a = dict(LINEAR_ARGS, **kw)
    bias = a["bias"] or None
    return lib.lowbit_linear_ex(a["x"] or None, a["w"] or None, a["s"] or None, a["z"] or None,
                                bias, a["y"] or None, a["M"], a["K"], a["N"], a["bits"],
                                a["group"], a["path"], None)


@pytest.mark.parametrize("kw", [
    dict(bits=0), dict(bits=8), dict(group=16), dict(group=512), dict(K=80),
    dict(K=0), dict(M=-1), dict(N=-3), dict(x=0), dict(w=0), dict(s=0), dict(z=0),
    dict(y=0), dict(x=8), dict(w=24), dict(s=1), dict(z=3), dict(y=5), dict(bias=7),
    dict(path=3), dict(K=1 << 31),
])
def test_linear_rejects_bad_arguments(lib, kw):
    # The pointer values are fake; every case fails validation before CUDA is touched.
    assert call_linear(lib, **kw) == EINVAL


def test_linear_empty_is_noop(lib):
    assert call_linear(lib, M=0) == 0
    assert call_linear(lib, N=0) == 0
    assert call_linear(lib, M=0, x=0, w=0, s=0, z=0, y=0) == 0


def call_swiglu(lib, **kw):
    a = dict(LINEAR_ARGS, **kw)
    F = a.get("F", 4)
    return lib.lowbit_linear_swiglu(a["x"] or None, a["w"] or None, a["s"] or None, a["z"] or None,
                                    a["bias"] or None, a["y"] or None, a["M"], a["K"], F, a["bits"],
                                    a["group"], None)


@pytest.mark.parametrize("kw", [
    dict(bits=0), dict(bits=8), dict(group=16), dict(K=80), dict(K=0), dict(M=-1), dict(F=-1),
    dict(F=1 << 30), dict(x=0), dict(w=0), dict(s=0), dict(z=0), dict(y=0), dict(x=8), dict(w=24),
    dict(s=1), dict(z=3), dict(y=5), dict(bias=7),
])
def test_swiglu_rejects_bad_arguments(lib, kw):
    assert call_swiglu(lib, **kw) == EINVAL


def test_swiglu_empty_is_noop(lib):
    assert call_swiglu(lib, M=0) == 0
    assert call_swiglu(lib, F=0) == 0
    assert call_swiglu(lib, F=0, x=0, w=0, s=0, z=0, y=0) == 0


@pytest.mark.parametrize("args", [
    (16, 16, 8, 32, 0), (16, 16, 8, 32, 8), (16, 16, 8, 12, 3), (0, 16, 8, 32, 4),
    (16, 0, 8, 32, 4), (12, 16, 8, 32, 4), (16, 16, -1, 32, 4),
])
def test_pack_rejects_bad_arguments(lib, args):
    codes, packed, N, K, bits = args
    assert lib.lowbit_pack_weights(codes or None, packed or None, N, K, bits, None) == EINVAL
    assert lib.lowbit_unpack_weights(packed or None, codes or None, N, K, bits, None) == EINVAL


def test_pack_empty_is_noop(lib):
    assert lib.lowbit_pack_weights(None, None, 0, 64, 3, None) == 0
    assert lib.lowbit_unpack_weights(None, None, 5, 0, 3, None) == 0


# (w, dtype, packed, scales, zeros, N, K, bits, group); pointers are fake but
# suitably aligned unless the case is about alignment: argument checks come
# before any CUDA call, so none of these touches a device.
_Q_OK = (4096, 0, 8192, 16384, 24576, 4, 256, 4, 64)


@pytest.mark.parametrize("change", [
    {7: 0}, {7: 8}, {8: 48}, {8: 512}, {6: 96}, {6: 0}, {5: -1}, {1: 3}, {1: -1},
    {0: 0}, {2: 0}, {3: 0}, {4: 0}, {0: 4098}, {0: 4097, 1: 1}, {3: 16385}, {4: 24577},
])
def test_quantize_rejects_bad_arguments(lib, change):
    args = list(_Q_OK)
    for i, v in change.items():
        args[i] = v
    w, dt, p, s, z, N, K, bits, group = args
    assert lib.lowbit_quantize_weights(w or None, dt, p or None, s or None, z or None,
                                       N, K, bits, group, None) == EINVAL


def test_quantize_empty_is_noop(lib):
    assert lib.lowbit_quantize_weights(None, 1, None, None, None, 0, 256, 3, 128, None) == 0


def test_wait_timeouts_rejects_null(lib):
    assert lib.lowbit_wait_timeouts(None, 0) == EINVAL


def test_wait_selftest_rejects_bad_pointers(lib):
    assert lib.lowbit_selftest_wait_timeout(None, None) == EINVAL
    assert lib.lowbit_selftest_wait_timeout(0x1002, None) == EINVAL   # not 4-byte aligned


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import bit_groupwise_weight_gb300._abi as abi_mod
    monkeypatch.setattr(abi_mod, "_lib", None)
    monkeypatch.setattr(abi_mod, "library_path", lambda: tmp_path / "missing.so")
    with pytest.raises(ImportError):
        abi_mod.abi()


def test_plain_c_client_links_and_runs(lib, tmp_path):
    """A C program built against include/lowbit.h and linked to the shared
    library (no Python in between) runs the host-side entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_host_check"
    libdir = lbuild.LIB.parent
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", str(ROOT / "include"),
                    str(ROOT / "tests" / "c" / "abi_host_check.c"), "-o", str(exe),
                    "-L", str(libdir), "-llowbit", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout


def test_binding_requires_one_device():
    from types import SimpleNamespace
    from bit_groupwise_weight_gb300 import _abi
    a, b = SimpleNamespace(device="cuda:0"), SimpleNamespace(device="cuda:1")
    assert _abi._device_of(a, None, a) == "cuda:0"
    with pytest.raises(ValueError, match="one device"):
        _abi._device_of(a, b)
