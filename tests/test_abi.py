"""The C ABI on a CPU-only host: the library loads, exports every entry point
declared in include/w4a16.h with a matching binding, and rejects bad
arguments synchronously, before touching any device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from w4a16_weight_only_gemm_gb300 import _native, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.lib()


def declared_functions() -> set[str]:
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(w4a16_\w+)\s*\(", text))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("w4a16_quantize", "w4a16_repack", "w4a16_unrepack", "w4a16_gemm",
                     "w4a16_repacked_bytes", "w4a16_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert names == set(_native.SIGNATURES), names ^ set(_native.SIGNATURES)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in _native.STATUS_NAMES.items():
        assert lib.w4a16_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.w4a16_status_string(99)
    assert lib.w4a16_version() >= 100


def test_repacked_bytes(lib):
    assert lib.w4a16_repacked_bytes(4096, 4096) == 4096 * 2048
    assert lib.w4a16_repacked_bytes(130, 256) == 256 * 128
    assert lib.w4a16_repacked_bytes(1, 128) == 128 * 64
    assert lib.w4a16_repacked_bytes(10, 100) == -1
    assert lib.w4a16_repacked_bytes(0, 128) == -1


FAKE = 0x10000  # an aligned non-null pointer value; never dereferenced here
MISALIGNED = 0x10008


def test_quantize_argument_errors(lib):
    q = lib.w4a16_quantize
    assert q(None, 8, 128, 128, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 128, 64, FAKE, FAKE, None) == 2     # group must be 128
    assert q(FAKE, 8, 200, 128, FAKE, FAKE, None) == 2    # K % 128
    assert q(FAKE, 0, 128, 128, FAKE, FAKE, None) == 2
    assert q(MISALIGNED, 8, 128, 128, FAKE, FAKE, None) == 3


def test_quantize_ex_argument_errors(lib):
    q = lib.w4a16_quantize_ex
    assert q(FAKE, 8, 128, 128, 1, FAKE, FAKE, None, None) == 1   # asymmetric needs zeros
    assert q(FAKE, 8, 128, 16, 0, FAKE, FAKE, None, None) == 2    # group 16
    assert q(FAKE, 8, 256, 96, 0, FAKE, FAKE, None, None) == 2    # group 96
    assert q(FAKE, 8, 128, 128, 2, FAKE, FAKE, FAKE, None) == 2   # asymmetric flag
    assert q(FAKE, 8, 200, -1, 0, FAKE, FAKE, None, None) == 2    # K % 128
    assert q(FAKE, 8, 128, 32, 1, FAKE, FAKE, MISALIGNED, None) == 3


def test_repack_argument_errors(lib):
    assert lib.w4a16_repack(None, 8, 128, FAKE, None) == 1
    assert lib.w4a16_repack(FAKE, 8, 96, FAKE, None) == 2
    assert lib.w4a16_unrepack(FAKE, 8, 128, MISALIGNED, None) == 3


def test_gemm_argument_errors(lib):
    g = lib.w4a16_gemm
    assert g(FAKE, FAKE, None, FAKE, 1, 8, 128, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 8, 128, None) == 2
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 130, None) == 2
    assert g(FAKE, FAKE, FAKE, FAKE, 1, -3, 128, None) == 2
    assert g(FAKE, MISALIGNED, FAKE, FAKE, 1, 8, 128, None) == 3
    assert g(FAKE, FAKE, FAKE, MISALIGNED, 1, 8, 128, None) == 3


def test_gemm_ex_argument_errors(lib):
    g = lib.w4a16_gemm_ex
    assert g(FAKE, None, FAKE, None, None, FAKE, 1, 8, 128, 32, None) == 1
    assert g(FAKE, None, FAKE, FAKE, None, FAKE, 1, 8, 128, 16, None) == 2     # group 16
    assert g(FAKE, None, FAKE, FAKE, FAKE, FAKE, 0, 8, 128, 32, None) == 2     # M >= 1
    assert g(FAKE, FAKE, FAKE, FAKE, None, FAKE, (1 << 22) + 1, 8, 128, 128, None) == 2
    assert g(FAKE, None, FAKE, FAKE, None, FAKE, 1, 8, 192, 128, None) == 2    # K % 128
    assert g(FAKE, None, FAKE, FAKE, MISALIGNED, FAKE, 1, 8, 128, 32, None) == 3
    assert g(FAKE, MISALIGNED, FAKE, FAKE, None, FAKE, 1, 8, 128, 32, None) == 3


def test_gemm_ex_plan_argument_errors(lib):
    p = lib.w4a16_gemm_ex_plan
    out = [ctypes.c_int(0) for _ in range(4)]
    refs = [ctypes.byref(o) for o in out]
    assert p(17, 8, 128, 32, 1, 0, None, *refs[1:]) == 1
    assert p(0, 8, 128, 32, 1, 0, *refs) == 2
    assert p(17, 8, 128, 48, 0, 0, *refs) == 2                                 # group 48
    assert p(17, 8, 130, 32, 0, 1, *refs) == 2


def test_q4_0_argument_errors(lib):
    assert lib.w4a16_quantize_q4_0(None, 8, 256, FAKE, None) == 1
    assert lib.w4a16_quantize_q4_0(FAKE, 8, 384, FAKE, None) == 2   # K % 256
    assert lib.w4a16_gemm_q4_0(FAKE, FAKE, FAKE, 17, 8, 256, None) == 2
    assert lib.w4a16_gemm_q4_0(FAKE, MISALIGNED, FAKE, 1, 8, 256, None) == 3


def test_w8_argument_errors(lib):
    assert lib.w4a16_quantize_w8(None, 8, 128, FAKE, FAKE, None) == 1
    assert lib.w4a16_quantize_w8(FAKE, 8, 200, FAKE, FAKE, None) == 2
    assert lib.w4a16_gemm_w8(FAKE, FAKE, FAKE, FAKE, 17, 8, 128, None) == 2   # M <= 16
    assert lib.w4a16_gemm_w8(FAKE, MISALIGNED, FAKE, FAKE, 1, 8, 128, None) == 3


def test_device_status_rejects_null(lib):
    assert lib.w4a16_device_status(None) == 1


def test_python_layer_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "_LIB", None)
    monkeypatch.setattr(_native, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _native.lib()


def test_operands_on_one_device():
    """The wrappers launch on the operands' device: operands on different
    devices (or an explicit stream on another device) are refused before any
    call into the library."""
    from types import SimpleNamespace

    import torch

    from w4a16_weight_only_gemm_gb300 import ops

    d0, d1 = torch.device("cuda:0"), torch.device("cuda:1")
    a, b = SimpleNamespace(device=d0), SimpleNamespace(device=d1)
    assert ops._device_of(None, ("x", a), ("scales", a), ("out", None)) == d0
    with pytest.raises(ValueError, match="scales"):
        ops._device_of(None, ("x", a), ("scales", b))
    with pytest.raises(ValueError, match="stream"):
        ops._device_of(SimpleNamespace(device=d1), ("x", a))
