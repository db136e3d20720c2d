"""The bit-level encodings the CUDA kernels rely on, checked on the CPU with
numpy (no GPU, no oracle): each is a fact about IEEE binary16 / binary32 that
a kernel's arithmetic depends on, so a wrong constant fails here first."""
from __future__ import annotations

import numpy as np


def f16(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_exact_codes_from_the_mantissa_of_1024():
    """The decode GEMV ORs a nibble n into fp16 1024.0 (0x6400): at bits 0..3
    it reads 1024 + n, and minus 1032 gives q = n - 8; at bits 4..7 it reads
    1024 + 16 n, and times 1/16 minus 72 gives q -- every step exact in fp16
    (the hardware's half2 subtract and fma, emulated with numpy float16)."""
    n = np.arange(16)
    lo = f16(0x6400 | n)
    hi = f16(0x6400 | (n << 4))
    assert np.array_equal(lo, 1024.0 + n)
    assert np.array_equal(hi, 1024.0 + 16 * n)
    q_lo = (lo.astype(np.float16) - np.float16(1032)).astype(np.float64)
    q_hi = (hi.astype(np.float16) * np.float16(1 / 16) + np.float16(-72)).astype(np.float64)
    assert np.array_equal(q_lo, n - 8) and np.array_equal(q_hi, n - 8)


def test_magic_1024_minus_offset_gives_nib_minus_z():
    """The format kernels: (1024 + nib) - (1024 + z) and
    (1024 + 16 nib) / 16 - (64 + z) are both nib - z, exactly."""
    for z in range(16):
        for nib in range(16):
            lo = f16(0x6400 | nib)
            hi = f16(0x6400 | (nib << 4))
            assert lo - (1024 + z) == nib - z
            assert np.float16(hi * np.float16(1 / 16)) - (64 + z) == nib - z


def test_w8_codes_in_the_mantissa_of_1024():
    """The W8A16 GEMV's prmt puts a code byte c under exponent byte 0x64:
    fp16 1024 + c, and minus 1152 gives q = c - 128 exactly."""
    c = np.arange(256)
    v = f16((0x64 << 8) | c)
    assert np.array_equal(v, 1024.0 + c)
    assert np.array_equal(v - 1152.0, c - 128.0)


def test_q4_0_byte_to_pair():
    """The Q4_0 GEMV: byte b -> halves (0x6400 | lo, 0x6400 | hi << 4), one
    fma by (1, 1/16) plus (-1032, -72) gives (lo - 8, hi - 8) exactly."""
    for b in range(256):
        lo, hi = b & 15, b >> 4
        h0 = f16(0x6400 | lo)
        h1 = f16(0x6400 | (hi << 4))
        r0 = np.float16(h0 * 1.0 + np.float16(-1032.0))
        r1 = np.float16(h1 * np.float16(1 / 16) + np.float16(-72.0))
        assert r0 == lo - 8 and r1 == hi - 8


def test_quantizer_round_constant():
    """kRound = 1.5 * 2^23 + 8: t = RN(r + kRound) in binary32 rounds r to
    the nearest integer with ties to even and leaves q + 8 in the low 4 bits
    of t, for |r| < 8."""
    k_round = np.float32(12582920.0)
    assert float(k_round) == 1.5 * 2 ** 23 + 8
    r = np.concatenate([np.linspace(-7.49, 7.49, 4001), np.arange(-7, 8) + 0.5,
                        np.arange(-7, 7) - 0.5]).astype(np.float32)
    t = (r + k_round).astype(np.float32)
    q = np.rint(r.astype(np.float64))  # numpy rint: nearest, ties to even
    q = np.clip(q, -8, 7)
    low = t.view(np.uint32) & 0xF
    keep = np.abs(r) < 7.5
    assert np.array_equal(low[keep], (q[keep] + 8).astype(np.uint32))
    assert np.all((t.view(np.uint32)[keep] >> 4) == (0x4B400000 >> 4))
