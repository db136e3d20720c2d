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
    (1024 + 16 nib) / 16 - (64 + z) are both nib - z, exactly.  The decode
    GEMV builds its offsets without a conversion: 1024 + z is the bit pattern
    0x6400 + z, and 64 + z is the fp16 difference (0x6400 + z) - 960, exact
    for every byte z."""
    for z in range(16):
        for nib in range(16):
            lo = f16(0x6400 | nib)
            hi = f16(0x6400 | (nib << 4))
            assert lo - (1024 + z) == nib - z
            assert np.float16(hi * np.float16(1 / 16)) - (64 + z) == nib - z
    z = np.arange(256)
    assert np.array_equal(f16(0x6400 + z), 1024.0 + z)
    assert f16(0x6380) == 960.0
    diff = (f16(0x6400 + z).astype(np.float16) - np.float16(960.0)).astype(np.float64)
    assert np.array_equal(diff, 64.0 + z)


def test_w8_codes_in_the_mantissa_of_1024():
    """The W8A16 GEMV's prmt puts a code byte c under exponent byte 0x64:
    fp16 1024 + c, and minus 1152 gives q = c - 128 exactly."""
    c = np.arange(256)
    v = f16((0x64 << 8) | c)
    assert np.array_equal(v, 1024.0 + c)
    assert np.array_equal(v - 1152.0, c - 128.0)


def _prmt(a: int, b: int, sel: int) -> int:
    """PTX prmt.b32 (default mode): byte k of the result is byte
    (sel >> 4k) & 7 of the 8-byte value b:a."""
    src = (b << 32) | a
    out = 0
    for k in range(4):
        idx = (sel >> (4 * k)) & 7
        out |= ((src >> (8 * idx)) & 0xFF) << (8 * k)
    return out


def _halves(w: int) -> tuple[float, float]:
    return float(f16(w & 0xFFFF)), float(f16(w >> 16))


def test_q4_0_word_decode_and_x_pairing():
    """The Q4_0 GEMV: a lane's 32-bit quant word (byte i: element 2i low,
    2i + 1 high) -> four fp16 pairs by lop3 into 0x64006400 with the masks
    0x000F000F / 0x00F000F0 (of w and w >> 8), then - 1032 or * 1/16 - 72:
    exactly (e - 8, e' - 8) for (e0, e4), (e1, e5), (e2, e6), (e3, e7).  x is
    permuted per 8 elements by prmt 0x5410 / 0x7632 into the same pairing,
    so the pairwise products sum to the block's dot product."""
    rng = np.random.default_rng(5)
    for _ in range(500):
        w = int(rng.integers(0, 2 ** 32))
        nib = [(w >> (4 * i)) & 15 for i in range(8)]  # element e = nibble e
        magic = 0x64006400
        lo0 = (w & 0x000F000F) | magic
        hi0 = (w & 0x00F000F0) | magic
        lo1 = ((w >> 8) & 0x000F000F) | magic
        hi1 = ((w >> 8) & 0x00F000F0) | magic
        f1032, f16th, fm72 = np.float16(1032), np.float16(1 / 16), np.float16(-72)
        pairs = []
        for v, is_hi in ((lo0, False), (hi0, True), (lo1, False), (hi1, True)):
            h = [np.float16(x) for x in _halves(v)]
            pairs.append(tuple(float(np.float16(x * f16th + fm72)) if is_hi else float(x - f1032)
                               for x in h))
        q = [n - 8 for n in nib]
        assert pairs == [(q[0], q[4]), (q[1], q[5]), (q[2], q[6]), (q[3], q[7])]
        # x: eight fp16 values in four 32-bit words, permuted as the kernel does
        xs = rng.standard_normal(8).astype(np.float16)
        xw = [int(xs[2 * i].view(np.uint16)) | (int(xs[2 * i + 1].view(np.uint16)) << 16)
              for i in range(4)]
        o = [_prmt(xw[0], xw[2], 0x5410), _prmt(xw[0], xw[2], 0x7632),
             _prmt(xw[1], xw[3], 0x5410), _prmt(xw[1], xw[3], 0x7632)]
        got = sum(a * b for pr, ow in zip(pairs, o) for a, b in zip(pr, _halves(ow)))
        want = sum(float(qq) * float(xx) for qq, xx in zip(q, xs))
        assert got == want


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
