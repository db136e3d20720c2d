"""CPU oracle for the W4A16 group-wise path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement of what the path
computes, used to check the CUDA library.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it.  The product library never imports, links or calls it, and it imports
nothing from the product package.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, binary32 quantizer,
binary64 dequantizer and GEMM); this module compiles it with gcc on first use
and marshals numpy arrays through ctypes.  Sources, cited by page title and
section:

* "LLM quantization from IEEE 754 to GPTQ/AWQ/GGUF" tutorial (qaqbuyan.com
  article 126), chapter "量化的数学基石": §1 FP16 bit layout, §2 symmetric
  and asymmetric quantization formulas, §3 quantization granularity
  (per-channel, per-group with group 128 or 32) and the per-group
  quantizer/dequantizer functions.
* "W4A16 量化算子解码性能基准跑分与端侧大模型推理显存实测报告" (mhpq.cn):
  §一 format (group 128, symmetric INT4, fp16 scales), §二/§五 the decode
  product y = x W^T from the packed weights.

Parity status of each function is stated in its docstring.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

GROUP = 128

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fopenmp"]


def _lib_path(src: str = _SRC) -> str:
    with open(src, "rb") as f:
        digest = hashlib.sha1(f.read() + " ".join(_CFLAGS).encode()
                              + os.uname().machine.encode()).hexdigest()[:12]
    return os.path.join(_BUILD_DIR, f"liboracle_{digest}.so")


def build(src: str = _SRC, out: str | None = None, verbose: bool = False) -> str:
    """Compile the oracle C source with gcc (idempotent); return the .so path.

    ``src``/``out`` let the tests compile deliberately broken copies of the
    oracle (planted mistakes) to show that the pins catch them."""
    path = out or _lib_path(src)
    if os.path.exists(path):
        return path
    os.makedirs(os.path.dirname(path), exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, "-o", tmp, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _bind(lib):
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_float_to_half.argtypes = [ctypes.c_float]
    lib.orc_float_to_half.restype = ctypes.c_uint16
    lib.orc_half_to_double_n.argtypes = [p, i64, p]
    lib.orc_float_to_half_n.argtypes = [p, i64, p]
    lib.orc_quantize.argtypes = [p, i64, i64, i64, p, p]
    lib.orc_quantize.restype = ctypes.c_int
    lib.orc_quantize_asym.argtypes = [p, i64, i64, i64, p, p, p]
    lib.orc_quantize_asym.restype = ctypes.c_int
    lib.orc_dequantize.argtypes = [p, p, p, i64, i64, i64, p]
    lib.orc_dequantize.restype = ctypes.c_int
    lib.orc_dequantize_f16.argtypes = [p, p, p, i64, i64, i64, p]
    lib.orc_dequantize_f16.restype = ctypes.c_int
    lib.orc_gemm.argtypes = [p, i64, i64, p, p, p, i64, i64, p]
    lib.orc_gemm.restype = ctypes.c_int
    lib.orc_gemm_rows.argtypes = [p, i64, i64, p, p, p, i64, i64, p, i64, p]
    lib.orc_gemm_rows.restype = ctypes.c_int
    lib.orc_scale_activations.argtypes = [p, i64, i64, p, p]
    lib.orc_pack_q4_0.argtypes = [p, p, i64, i64, p]
    lib.orc_pack_q4_0.restype = ctypes.c_int
    lib.orc_dequantize_q4_0.argtypes = [p, i64, i64, p]
    lib.orc_dequantize_q4_0.restype = ctypes.c_int
    lib.orc_quantize_w8.argtypes = [p, i64, i64, p, p]
    lib.orc_quantize_w8.restype = ctypes.c_int
    lib.orc_dequantize_w8.argtypes = [p, p, i64, i64, p]
    lib.orc_dequantize_w8.restype = ctypes.c_int
    lib.orc_gemm_rows_w8.argtypes = [p, i64, i64, p, p, i64, p, i64, p]
    lib.orc_gemm_rows_w8.restype = ctypes.c_int
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _zptr(zeros) -> int | None:
    return None if zeros is None else zeros.ctypes.data


def _group(group: int, K: int) -> int:
    """group = -1 means per-channel: one group spanning the row."""
    return K if group == -1 else group


class Oracle:
    """One loaded build of the oracle library (the real one, or a test mutant)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    def num_threads(self) -> int:
        return int(self._lib.orc_num_threads())

    def set_num_threads(self, n: int) -> None:
        self._lib.orc_set_num_threads(int(n))

    # ------------------------------------------------------------------
    # FP16 bit layout (tutorial §1).  Pinned: exhaustive / random
    # comparison with numpy's IEEE float16 conversion.
    # ------------------------------------------------------------------
    def half_to_double(self, h: np.ndarray) -> np.ndarray:
        """Exact binary64 value of fp16 bit patterns (uint16 array)."""
        h = _c(h, np.uint16)
        out = np.empty(h.shape, dtype=np.float64)
        self._lib.orc_half_to_double_n(_ptr(h), h.size, _ptr(out))
        return out

    def float_to_half(self, f: np.ndarray) -> np.ndarray:
        """fp16 bits (uint16) of binary32 values, round to nearest even."""
        f = _c(f, np.float32)
        out = np.empty(f.shape, dtype=np.uint16)
        self._lib.orc_float_to_half_n(_ptr(f), f.size, _ptr(out))
        return out

    # ------------------------------------------------------------------
    # Quantizer (tutorial §2 formula, §3 per_group_symmetric_quantize).
    # Pinned: +-amax -> +-7, all-zero group, tie cases, small-scale clamp,
    # round-trip bound, nearest-level brute force, scale through numpy,
    # nibble-order fixture.
    # ------------------------------------------------------------------
    def quantize(self, W16: np.ndarray, group: int = GROUP):
        """Group-wise symmetric RTN INT4 quantization of fp16 weights.

        ``W16``: uint16 fp16 bit patterns, shape [N, K] (rows = out_features).
        ``group``: weights per scale along K; -1 = per-channel (one group per row).
        Returns ``(qweight uint8 [N, K/2], scales uint16 fp16 bits [N, K/group])``.
        """
        W16 = _c(W16, np.uint16)
        if W16.ndim != 2:
            raise ValueError("W must be 2-D [N, K]")
        N, K = W16.shape
        group = _group(group, K)
        if group <= 0 or K % group:
            raise ValueError(f"K={K} is not a multiple of group={group}")
        q = np.empty((N, K // 2), dtype=np.uint8)
        s = np.empty((N, K // group), dtype=np.uint16)
        rc = self._lib.orc_quantize(_ptr(W16), N, K, group, _ptr(q), _ptr(s))
        if rc != 0:
            raise ValueError(f"oracle quantize rejected shape N={N} K={K} group={group}")
        return q, s

    # ------------------------------------------------------------------
    # Asymmetric quantizer (tutorial §2 asymmetric formula).  Pinned:
    # integer-grid fixtures (min -> 0, max -> 15, z exact), constant and
    # all-zero groups, nearest-level and nearest-zero-point brute force,
    # round-trip bound, scale through numpy.
    # ------------------------------------------------------------------
    def quantize_asym(self, W16: np.ndarray, group: int = GROUP):
        """Group-wise asymmetric RTN INT4 quantization of fp16 weights.

        Returns ``(qweight uint8 [N, K/2] holding q in [0, 15],
        scales uint16 fp16 bits [N, K/group], zeros uint8 [N, K/group])``."""
        W16 = _c(W16, np.uint16)
        if W16.ndim != 2:
            raise ValueError("W must be 2-D [N, K]")
        N, K = W16.shape
        group = _group(group, K)
        if group <= 0 or K % group:
            raise ValueError(f"K={K} is not a multiple of group={group}")
        q = np.empty((N, K // 2), dtype=np.uint8)
        s = np.empty((N, K // group), dtype=np.uint16)
        z = np.empty((N, K // group), dtype=np.uint8)
        rc = self._lib.orc_quantize_asym(_ptr(W16), N, K, group, _ptr(q), _ptr(s), _ptr(z))
        if rc != 0:
            raise ValueError(f"oracle quantize_asym rejected shape N={N} K={K} group={group}")
        return q, s, z

    # ------------------------------------------------------------------
    # Dequantizer (tutorial §3 per_group_symmetric_dequantize).  Pinned:
    # closed forms and the round-trip bound against the master weights.
    # ------------------------------------------------------------------
    def dequantize(self, qweight: np.ndarray, scales: np.ndarray,
                   group: int = GROUP, zeros: np.ndarray | None = None) -> np.ndarray:
        """Exact dequantized weights (nibble - z) * scale16 in binary64, [N, K];
        z = zeros[n, k / group] (asymmetric) or 8 (symmetric, zeros None)."""
        qweight = _c(qweight, np.uint8)
        scales = _c(scales, np.uint16)
        zeros = None if zeros is None else _c(zeros, np.uint8)
        N, K2 = qweight.shape
        K = 2 * K2
        group = _group(group, K)
        out = np.empty((N, K), dtype=np.float64)
        rc = self._lib.orc_dequantize(_ptr(qweight), _ptr(scales), _zptr(zeros), N, K, group,
                                      _ptr(out))
        if rc != 0:
            raise ValueError("oracle dequantize rejected shape")
        return out

    def dequantize_f16(self, qweight: np.ndarray, scales: np.ndarray,
                       group: int = GROUP, zeros: np.ndarray | None = None) -> np.ndarray:
        """The tutorial's own fp16 dequantized weight fp16(float(q) * float(s)).

        Returns uint16 fp16 bits [N, K].  Pinned by the hand-derived fixture
        ``tests/golden/dequant_f16.txt`` (ties, subnormals, overflow, zero
        points) and by numpy's single float16 rounding of the exact binary64
        dequantized value on random codes."""
        qweight = _c(qweight, np.uint8)
        scales = _c(scales, np.uint16)
        zeros = None if zeros is None else _c(zeros, np.uint8)
        N, K2 = qweight.shape
        K = 2 * K2
        group = _group(group, K)
        out = np.empty((N, K), dtype=np.uint16)
        rc = self._lib.orc_dequantize_f16(_ptr(qweight), _ptr(scales), _zptr(zeros), N, K,
                                          group, _ptr(out))
        if rc != 0:
            raise ValueError("oracle dequantize_f16 rejected shape")
        return out

    # ------------------------------------------------------------------
    # GGUF Q4_0 blocks (tutorial GGUF section).  Pinned: a hand-derived
    # block fixture; decode of packed blocks equals the group-32 dequantizer.
    # ------------------------------------------------------------------
    def quantize_q4_0(self, W16: np.ndarray) -> np.ndarray:
        """Q4_0 blocks uint8 [N, K/32 * 18] (group-32 symmetric codes)."""
        q, s = self.quantize(W16, 32)
        return self.pack_q4_0(q, s)

    def pack_q4_0(self, qweight: np.ndarray, scales: np.ndarray) -> np.ndarray:
        qweight = _c(qweight, np.uint8)
        scales = _c(scales, np.uint16)
        N, K = qweight.shape[0], 2 * qweight.shape[1]
        out = np.empty((N, K // 32 * 18), dtype=np.uint8)
        if self._lib.orc_pack_q4_0(_ptr(qweight), _ptr(scales), N, K, _ptr(out)) != 0:
            raise ValueError("oracle pack_q4_0 rejected shape")
        return out

    def dequantize_q4_0(self, blocks: np.ndarray, K: int) -> np.ndarray:
        blocks = _c(blocks, np.uint8)
        N = blocks.shape[0]
        out = np.empty((N, K), dtype=np.float64)
        if self._lib.orc_dequantize_q4_0(_ptr(blocks), N, K, _ptr(out)) != 0:
            raise ValueError("oracle dequantize_q4_0 rejected shape")
        return out

    def gemm_q4_0(self, x16: np.ndarray, blocks: np.ndarray, rows=None) -> np.ndarray:
        """Columns ``rows`` (default all) of y = x Wd^T with Wd decoded from Q4_0 blocks."""
        x16 = _c(x16, np.uint16)
        K = x16.shape[1]
        blocks = _c(blocks, np.uint8)
        sel = blocks if rows is None else blocks[np.asarray(rows)]
        wd = self.dequantize_q4_0(sel, K)
        return x16.view(np.float16).astype(np.float64) @ wd.T

    # ------------------------------------------------------------------
    # W8A16 per-channel INT8 (tutorial §2 formula with b = 8, INT8 section).
    # Pinned: +-amax -> +-127, scale through numpy, nearest-level brute
    # force, round-trip bound, numpy GEMM.
    # ------------------------------------------------------------------
    def quantize_w8(self, W16: np.ndarray):
        """(q8 uint8 [N, K] holding q + 128, scales uint16 fp16 bits [N])."""
        W16 = _c(W16, np.uint16)
        N, K = W16.shape
        q8 = np.empty((N, K), dtype=np.uint8)
        s = np.empty((N,), dtype=np.uint16)
        if self._lib.orc_quantize_w8(_ptr(W16), N, K, _ptr(q8), _ptr(s)) != 0:
            raise ValueError("oracle quantize_w8 rejected shape")
        return q8, s

    def dequantize_w8(self, q8: np.ndarray, scales: np.ndarray) -> np.ndarray:
        q8 = _c(q8, np.uint8)
        scales = _c(scales, np.uint16)
        N, K = q8.shape
        out = np.empty((N, K), dtype=np.float64)
        self._lib.orc_dequantize_w8(_ptr(q8), _ptr(scales), N, K, _ptr(out))
        return out

    def gemm_rows_w8(self, x16: np.ndarray, q8: np.ndarray, scales: np.ndarray,
                     rows=None) -> np.ndarray:
        """Columns ``rows`` (default all) of y = x Wd^T, binary64 [M, len(rows)]."""
        x16 = _c(x16, np.uint16)
        q8 = _c(q8, np.uint8)
        scales = _c(scales, np.uint16)
        M, K = x16.shape
        N = q8.shape[0]
        rows = _c(np.arange(N) if rows is None else np.asarray(rows), np.int64)
        y = np.empty((M, rows.size), dtype=np.float64)
        if self._lib.orc_gemm_rows_w8(_ptr(x16), M, K, _ptr(q8), _ptr(scales), N, _ptr(rows),
                                      rows.size, _ptr(y)) != 0:
            raise ValueError("oracle gemm_rows_w8 rejected arguments")
        return y

    # ------------------------------------------------------------------
    # AWQ activation scaling (tutorial AWQ section).  Pinned: numpy's exact
    # binary32 product and IEEE fp16 conversion; alpha = 1 is the identity;
    # alpha acts per input channel (one-hot alpha against numpy matmul).
    # ------------------------------------------------------------------
    def scale_activations(self, x16: np.ndarray, alpha16: np.ndarray) -> np.ndarray:
        """x~[m, k] = fp16_rne(x[m, k] * alpha[k]); uint16 fp16 bits [M, K]."""
        x16 = _c(x16, np.uint16)
        alpha16 = _c(alpha16, np.uint16)
        M, K = x16.shape
        if alpha16.shape != (K,):
            raise ValueError("alpha must be [K]")
        out = np.empty((M, K), dtype=np.uint16)
        self._lib.orc_scale_activations(_ptr(x16), M, K, _ptr(alpha16), _ptr(out))
        return out

    # ------------------------------------------------------------------
    # GEMM y = x W^T in binary64 (report §二/§五).  Pinned: numpy float64
    # matmul of the dequantized weights on tiny shapes; closed form q = 1,
    # s = 1 gives y = sum_k x exactly.
    # ------------------------------------------------------------------
    def gemm(self, x16: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
             group: int = GROUP, zeros: np.ndarray | None = None) -> np.ndarray:
        """y[m, n] = sum_k x[m, k] * Wd[n, k], binary64, unrounded.  x16: uint16 [M, K]."""
        x16 = _c(x16, np.uint16)
        qweight = _c(qweight, np.uint8)
        scales = _c(scales, np.uint16)
        zeros = None if zeros is None else _c(zeros, np.uint8)
        M, K = x16.shape
        N = qweight.shape[0]
        if qweight.shape[1] * 2 != K:
            raise ValueError("x and qweight disagree on K")
        group = _group(group, K)
        y = np.empty((M, N), dtype=np.float64)
        rc = self._lib.orc_gemm(_ptr(x16), M, K, _ptr(qweight), _ptr(scales), _zptr(zeros), N,
                                group, _ptr(y))
        if rc != 0:
            raise ValueError("oracle gemm rejected shape")
        return y

    def gemm_rows(self, x16: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
                  rows, group: int = GROUP, zeros: np.ndarray | None = None) -> np.ndarray:
        """Columns ``rows`` of y only: returns [M, len(rows)] binary64."""
        x16 = _c(x16, np.uint16)
        qweight = _c(qweight, np.uint8)
        scales = _c(scales, np.uint16)
        zeros = None if zeros is None else _c(zeros, np.uint8)
        rows = _c(np.asarray(rows), np.int64)
        M, K = x16.shape
        N = qweight.shape[0]
        if qweight.shape[1] * 2 != K:
            raise ValueError("x and qweight disagree on K")
        group = _group(group, K)
        y = np.empty((M, rows.size), dtype=np.float64)
        rc = self._lib.orc_gemm_rows(_ptr(x16), M, K, _ptr(qweight), _ptr(scales), _zptr(zeros),
                                     N, group, _ptr(rows), rows.size, _ptr(y))
        if rc != 0:
            raise ValueError("oracle gemm_rows rejected arguments")
        return y


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = Oracle(build())
    return _LIB


def half_to_double(h):
    return default().half_to_double(h)


def float_to_half(f):
    return default().float_to_half(f)


def quantize(W16, group: int = GROUP):
    return default().quantize(W16, group)


def quantize_asym(W16, group: int = GROUP):
    return default().quantize_asym(W16, group)


def quantize_q4_0(W16):
    return default().quantize_q4_0(W16)


def pack_q4_0(qweight, scales):
    return default().pack_q4_0(qweight, scales)


def dequantize_q4_0(blocks, K):
    return default().dequantize_q4_0(blocks, K)


def gemm_q4_0(x16, blocks, rows=None):
    return default().gemm_q4_0(x16, blocks, rows)


def quantize_w8(W16):
    return default().quantize_w8(W16)


def dequantize_w8(q8, scales):
    return default().dequantize_w8(q8, scales)


def gemm_rows_w8(x16, q8, scales, rows=None):
    return default().gemm_rows_w8(x16, q8, scales, rows)


def scale_activations(x16, alpha16):
    return default().scale_activations(x16, alpha16)


def dequantize(qweight, scales, group: int = GROUP, zeros=None):
    return default().dequantize(qweight, scales, group, zeros)


def dequantize_f16(qweight, scales, group: int = GROUP, zeros=None):
    return default().dequantize_f16(qweight, scales, group, zeros)


def gemm(x16, qweight, scales, group: int = GROUP, zeros=None):
    return default().gemm(x16, qweight, scales, group, zeros)


def gemm_rows(x16, qweight, scales, rows, group: int = GROUP, zeros=None):
    return default().gemm_rows(x16, qweight, scales, rows, group, zeros)


def num_threads() -> int:
    return default().num_threads()


def set_num_threads(n: int) -> None:
    default().set_num_threads(n)
