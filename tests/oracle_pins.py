"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Every function here takes an ``oracle.Oracle`` (the real build, or a mutant
with a planted mistake) and raises ``AssertionError`` when the oracle breaks
the pinned fact.  None of them re-types the oracle's own arithmetic: each is
a hand-derived fixture, a closed form, an invariant, a library routine
(numpy's IEEE float16 conversion and float64 matmul) on a special case, or a
brute-force enumeration on tiny inputs.

Sources: qaqbuyan.com quantization tutorial, chapter "量化的数学基石"
(§1 FP16 bit layout; §2 symmetric and asymmetric formulas and the
rounding-error model |error| <= s/2; §3 granularity -- per-channel,
per-group 128 and 32 -- and the per-group quantizer and dequantizer); W4A16
benchmark report (mhpq.cn) §二/§五 for y = x W^T.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GROUP = 128


def _read_fixture(name: str) -> list[list[str]]:
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _f16_bits(values) -> np.ndarray:
    return np.asarray(values, dtype=np.float16).view(np.uint16)


def _nibbles(qweight: np.ndarray) -> np.ndarray:
    """Unpack bytes into stored nibbles in k order (low nibble first)."""
    lo = qweight & 0x0F
    hi = qweight >> 4
    return np.stack([lo, hi], axis=-1).reshape(qweight.shape[0], -1).astype(np.int16)


def _random_weights(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    w = rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02)
    mask = rng.random((N, K)) < 0.001
    w[mask] *= np.float32(20.0)
    return w.astype(np.float16).view(np.uint16)


# --------------------------------------------------------------------------
# FP16 bit layout
# --------------------------------------------------------------------------

def pin_half_to_double_exhaustive(o) -> None:
    """All 65536 fp16 patterns decode to numpy's IEEE float16 value."""
    h = np.arange(65536, dtype=np.uint16)
    got = o.half_to_double(h)
    ref = h.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"{(~same).sum()} fp16 patterns decode wrongly"
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def pin_float_to_half_numpy(o) -> None:
    """binary32 -> fp16 RNE agrees with numpy on boundaries and random floats."""
    rng = np.random.default_rng(1234)
    boundary = np.array([
        0.0, -0.0, 65504.0, 65505.0, 65519.996, 65520.0, 65536.0, 1e9, -65520.0,
        2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14,
        2.0 ** -14 - 2.0 ** -25, 2.0 ** -14 - 2.0 ** -26, 1.0 + 2.0 ** -11,
        1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -11 + 2.0 ** -23, 1e-8, 5.96e-8,
        np.inf, -np.inf, 0.1, 1.0 / 3.0, 2047.5, 2048.5, 4095.0,
    ], dtype=np.float32)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    rand_bits = bits.view(np.float32)
    rand_bits = rand_bits[np.isfinite(rand_bits)]
    rand_mid = (rng.standard_normal(400_000) * np.exp(rng.uniform(-20, 12, 400_000))
                ).astype(np.float32)
    for f in (boundary, rand_bits, rand_mid):
        got = o.float_to_half(f)
        with np.errstate(over="ignore"):
            ref = f.astype(np.float16).view(np.uint16)
        assert np.array_equal(got, ref), (
            f"float->half differs on {np.count_nonzero(got != ref)} values, e.g. "
            f"{f[got != ref][:4]}")


def pin_half_round_trip(o) -> None:
    """Every finite fp16 value survives half -> double -> float -> half."""
    h = np.arange(65536, dtype=np.uint16)
    finite = (h & 0x7C00) != 0x7C00
    h = h[finite]
    back = o.float_to_half(o.half_to_double(h).astype(np.float32))
    assert np.array_equal(back, h)


# --------------------------------------------------------------------------
# Quantizer
# --------------------------------------------------------------------------

def pin_nibble_order_fixture(o) -> None:
    rows = {r[0]: r[1:] for r in _read_fixture("nibble_order_group128.txt")}
    c = [int(v) for v in rows["c"]] + [0] * int(rows["c_rest"][1])
    assert len(c) == GROUP
    w = _f16_bits(np.array(c, dtype=np.float64) * 2.0 ** -6).reshape(1, GROUP)
    expect = [int(b, 16) for b in rows["bytes"]]
    expect += [int(rows["bytes_rest"][0], 16)] * int(rows["bytes_rest"][1])
    q, s = o.quantize(w, GROUP)
    assert q.tolist() == [expect], f"packed bytes {q[0, :8].tolist()}"
    assert s.tolist() == [[int(rows["scale_bits"][0], 16)]]


def pin_ties_to_even(o) -> None:
    rows = _read_fixture("ties_pow2_scale.txt")
    amax = float(rows[0][1])
    cases = [(float(r[1]), int(r[2])) for r in rows[1:]]
    vals = [amax] + [r for r, _ in cases]
    vals += [0.0] * (GROUP - len(vals))
    w = _f16_bits(np.array(vals) * 2.0 ** -6).reshape(1, GROUP)
    q, s = o.quantize(w, GROUP)
    nib = _nibbles(q)[0] - 8
    assert nib[0] == 7
    for i, (r, expect) in enumerate(cases, start=1):
        assert nib[i] == expect, f"r={r}: q={nib[i]}, expected {expect}"
    assert s[0, 0] == _f16_bits([2.0 ** -6])[0]


def pin_tiny_scale_clamp(o) -> None:
    rows = {r[0]: r[1:] for r in _read_fixture("tiny_scale_clamp.txt")}
    w = np.full((1, GROUP), int(rows["w_bits"][0], 16), dtype=np.uint16)
    q, s = o.quantize(w, GROUP)
    assert (q == int(rows["bytes"][0], 16)).all(), f"bytes {q[0, :4]}"
    assert s[0, 0] == int(rows["scale_bits"][0], 16)


def pin_all_zero_group(o) -> None:
    """An all-zero group packs to 0x88 bytes, a +0 scale, and dequantizes to 0."""
    w = np.zeros((3, 2 * GROUP), dtype=np.uint16)
    w[1, GROUP:] = _f16_bits(np.linspace(-1, 1, GROUP))  # one live group
    w[2, :] = 0x8000                                      # negative zeros
    q, s = o.quantize(w, GROUP)
    assert (q[0] == 0x88).all() and (q[2] == 0x88).all() and (q[1, :GROUP // 2] == 0x88).all()
    assert s[0].tolist() == [0, 0] and s[2].tolist() == [0, 0] and s[1, 0] == 0
    wd = o.dequantize(q, s, GROUP)
    assert (wd[0] == 0).all() and (wd[2] == 0).all() and (wd[1, :GROUP] == 0).all()


def pin_amax_maps_to_seven(o) -> None:
    """The largest |w| of every group quantizes to +-7 with w's sign, and no
    |q| exceeds 7 (symmetric quantization never reaches -8)."""
    rng = np.random.default_rng(7)
    w16 = _random_weights(rng, 64, 1024)
    q, s = o.quantize(w16, GROUP)
    qv = _nibbles(q) - 8
    w = w16.view(np.float16).astype(np.float64)
    wg = w.reshape(64, -1, GROUP)
    qg = qv.reshape(64, -1, GROUP)
    idx = np.abs(wg).argmax(axis=-1)
    amax_q = np.take_along_axis(qg, idx[..., None], axis=-1)[..., 0]
    amax_w = np.take_along_axis(wg, idx[..., None], axis=-1)[..., 0]
    assert (amax_q == 7 * np.sign(amax_w)).all()
    assert np.abs(qv).max() == 7


def _round_exact(x, frac_bits: int, min_exp: int):
    """Round a non-negative Fraction to the nearest binary floating-point value
    with `frac_bits` fraction bits and minimum normal exponent `min_exp`
    (ties to even), in exact rational arithmetic; returns a Fraction."""
    from fractions import Fraction
    if x == 0:
        return Fraction(0)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    quantum = Fraction(2) ** (max(e, min_exp) - frac_bits)
    m = x / quantum
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return lo * quantum


def pin_scale_is_fp16_of_amax_over_7(o) -> None:
    """For every finite non-negative fp16 absmax a (31,744 groups, one each),
    the stored scale is binary16-RNE of max(binary32-RNE(a / 7), binary32-RNE
    (1e-8)) -- the tutorial §3 reading (fp32 arithmetic, fp16 scale at the
    end) -- evaluated here in exact rational arithmetic, not with hardware
    division."""
    from fractions import Fraction
    amax_bits = np.arange(0, 0x7C00, dtype=np.uint16)
    n = amax_bits.size
    w16 = np.zeros((n, GROUP), dtype=np.uint16)
    w16[:, 5] = amax_bits
    w16[:, 77] = amax_bits ^ 0x8000  # the same magnitude negative
    _, s = o.quantize(w16, GROUP)
    floor32 = _round_exact(Fraction(1, 10 ** 8), 23, -126)
    want = np.empty(n, dtype=np.uint16)
    for i, b in enumerate(amax_bits.tolist()):
        a = Fraction(np.uint16(b).view(np.float16).item())
        s32 = max(_round_exact(a / 7, 23, -126), floor32)
        s16 = _round_exact(s32, 10, -14)
        want[i] = np.float16(float(s16)).view(np.uint16)  # exact: s16 is an fp16 value
    np.testing.assert_array_equal(s[:, 0], want)


def pin_nearest_level_brute_force(o) -> None:
    """On tiny inputs, q is the level j in [-8, 7] nearest to fp32(w)/fp32(s),
    ties to the even level, found by enumerating all 16 levels."""
    rng = np.random.default_rng(9)
    w16 = _random_weights(rng, 4, 2 * GROUP)
    q, _ = o.quantize(w16, GROUP)
    qv = _nibbles(q) - 8
    w32 = w16.view(np.float16).astype(np.float32)
    levels = np.arange(-8, 8, dtype=np.float64)
    for n in range(w32.shape[0]):
        for g in range(w32.shape[1] // GROUP):
            blk = w32[n, g * GROUP:(g + 1) * GROUP]
            s32 = max(np.float32(np.abs(blk).max()) / np.float32(7.0), np.float32(1e-8))
            for i, wv in enumerate(blk):
                r = float(np.float32(wv) / np.float32(s32))
                d = np.abs(levels - r)
                best = levels[d == d.min()]
                j = best[0] if best.size == 1 else best[np.fmod(best, 2) == 0][0]
                assert qv[n, g * GROUP + i] == j, (n, g, i, r, qv[n, g * GROUP + i])


def pin_round_trip_bound(o) -> None:
    """Rounding-error model (tutorial §2): every element comes back within
    half a step.  With the stored fp16 scale s16 (|s16 - s32| <= 2^-11 s32 in
    the normal range) the bound is s16 (1 + 2^-10) (1/2 + 2^-21 + 8 * 2^-11)."""
    rng = np.random.default_rng(10)
    w16 = _random_weights(rng, 128, 4096)
    q, s = o.quantize(w16, GROUP)
    wd = o.dequantize(q, s, GROUP)
    w = w16.view(np.float16).astype(np.float64)
    s64 = o.half_to_double(s)
    assert (s64 >= 2.0 ** -14).all()
    bound = np.repeat(s64, GROUP, axis=1) * (1 + 2.0 ** -10) * (0.5 + 2.0 ** -21 + 8 * 2.0 ** -11)
    err = np.abs(w - wd)
    assert (err <= bound).all(), float((err / bound).max())
    # the error is a half-step uniform noise on average (|U| with U ~ U(-1/2, 1/2))
    rel = (err / np.repeat(s64, GROUP, axis=1)).mean()
    assert 0.2 < rel < 0.3, rel


# --------------------------------------------------------------------------
# Dequantizer and GEMM
# --------------------------------------------------------------------------

def pin_dequant_closed_forms(o) -> None:
    """Nibble 9 with scale 1.0 is +1; nibble 0 is -8 * scale; nibble 8 is 0."""
    N, K = 3, 2 * GROUP
    q = np.full((N, K // 2), 0x99, dtype=np.uint8)
    q[1] = 0x00
    q[2] = 0x08  # low nibble 8 (0), high nibble 0 (-8)
    s = np.full((N, K // GROUP), 0x3C00, dtype=np.uint16)   # 1.0
    s[1, 1] = 0x4000                                         # 2.0 in group 1
    s[2] = _f16_bits([0.25, 0.5])
    wd = o.dequantize(q, s, GROUP)
    assert (wd[0] == 1.0).all()
    assert (wd[1, :GROUP] == -8.0).all() and (wd[1, GROUP:] == -16.0).all()
    assert (wd[2, 0::2] == 0.0).all()
    assert (wd[2, 1:GROUP:2] == -2.0).all() and (wd[2, GROUP + 1::2] == -4.0).all()


def pin_gemm_numpy_tiny(o) -> None:
    """Tiny shapes: y equals numpy's float64 matmul x @ Wd^T (Wd pinned above)."""
    rng = np.random.default_rng(11)
    for M, N, K in ((1, 1, 128), (2, 3, 256), (16, 8, 128), (3, 5, 384)):
        w16 = _random_weights(rng, N, K)
        q, s = o.quantize(w16, GROUP)
        x16 = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
        y = o.gemm(x16, q, s, GROUP)
        ref = x16.view(np.float16).astype(np.float64) @ o.dequantize(q, s, GROUP).T
        assert y.shape == (M, N)
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        rows = np.array([N - 1, 0])
        np.testing.assert_array_equal(o.gemm_rows(x16, q, s, rows, GROUP), y[:, rows])


def pin_gemm_closed_form(o) -> None:
    """q = 1 and scale s[n, g] = 2^-(n+g) give y[m, n] = sum_g 2^-(n+g) sum_{k in g} x[m, k],
    which binary64 holds exactly (fp16 x, at most a few hundred terms)."""
    rng = np.random.default_rng(12)
    M, N, K = 3, 4, 3 * GROUP
    x16 = rng.standard_normal((M, K)).astype(np.float16)
    q = np.full((N, K // 2), 0x99, dtype=np.uint8)
    s = np.array([[2.0 ** -(n + g) for g in range(K // GROUP)] for n in range(N)])
    y = o.gemm(x16.view(np.uint16), q, _f16_bits(s), GROUP)
    xs = x16.astype(np.float64)
    for m in range(M):
        for n in range(N):
            expect = math.fsum(
                s[n, g] * math.fsum(xs[m, g * GROUP:(g + 1) * GROUP]) for g in range(K // GROUP))
            assert y[m, n] == expect, (m, n, y[m, n], expect)


# --------------------------------------------------------------------------
# Asymmetric quantizer (tutorial §2 asymmetric formula) and other group sizes
# (tutorial §3: per-group 128 and 32, per-channel)
# --------------------------------------------------------------------------

def pin_asym_integer_grid(o) -> None:
    """Weights on an integer grid from min = -5 to max = 10 (times 2^-4): the
    step is exactly (10 + 5) / 15 = one grid unit, z = 5, and every weight v
    quantizes to v + 5 -- the minimum to 0, the maximum to 15."""
    rng = np.random.default_rng(21)
    for group in (32, 64, 128):
        v = rng.integers(-5, 11, size=(2, 4 * group))
        v[:, ::group] = -5   # every group holds the minimum ...
        v[:, 1::group] = 10  # ... and the maximum
        q, s, z = o.quantize_asym(_f16_bits(v * 2.0 ** -4), group)
        assert (z == 5).all(), z
        assert (s == _f16_bits([2.0 ** -4])[0]).all()
        assert np.array_equal(_nibbles(q), v + 5)


def pin_asym_range_includes_zero(o) -> None:
    """The zero point is the code of 0.0, so 0 is in every group's range: an
    all-positive group 0.5 j (j = 1..15) gets step 0.5 and z = 0 (q = j); the
    all-negative -0.5 j gets z = 15 (q = 15 - j)."""
    j = np.concatenate([np.arange(1, 16), np.ones(GROUP - 15, dtype=np.int64)])
    q, s, z = o.quantize_asym(_f16_bits(np.stack([0.5 * j, -0.5 * j])), GROUP)
    assert z[:, 0].tolist() == [0, 15]
    assert (s == _f16_bits([0.5])[0]).all()
    nib = _nibbles(q)
    assert np.array_equal(nib[0], j) and np.array_equal(nib[1], 15 - j)


def pin_asym_constant_and_zero_groups(o) -> None:
    """A constant group c > 0 stores q = 15, z = 0 and s = fp16(c / 15); c < 0
    stores q = 0, z = 15; an all-zero group stores q = 0, z = 0 and comes back
    as exact zeros."""
    w = np.zeros((3, GROUP), dtype=np.uint16)
    w[0] = _f16_bits([3.0])[0]
    w[1] = _f16_bits([-0.75])[0]
    q, s, z = o.quantize_asym(w, GROUP)
    nib = _nibbles(q)
    assert (nib[0] == 15).all() and z[0, 0] == 0 and s[0, 0] == _f16_bits([0.2])[0]
    assert (nib[1] == 0).all() and z[1, 0] == 15 and s[1, 0] == _f16_bits([0.05])[0]
    assert (nib[2] == 0).all() and z[2, 0] == 0
    wd = o.dequantize(q, s, GROUP, zeros=z)
    assert (wd[2] == 0).all()
    assert np.allclose(wd[0], 3.0, rtol=2e-3) and np.allclose(wd[1], -0.75, rtol=2e-3)


def pin_asym_nearest_level_brute_force(o) -> None:
    """Tiny inputs, with s32 = max(fp32(max' - min') / 15, 1e-8) over the group
    and 0 (a numpy float32 restatement of the step only): -z is the integer
    nearest to min'/s32 and q is the level j in [0, 15] whose j - z is nearest
    to fp32(w) / s32, ties to even, both found by enumerating all 16 codes."""
    rng = np.random.default_rng(22)
    codes = np.arange(16, dtype=np.float64)
    for group in (32, 128):
        w16 = _random_weights(rng, 4, 2 * group)
        w16[0] = _f16_bits(np.abs(w16[0].view(np.float16).astype(np.float64)))  # all >= 0
        q, _, z = o.quantize_asym(w16, group)
        nib = _nibbles(q)
        w32 = w16.view(np.float16).astype(np.float32)
        for n in range(w32.shape[0]):
            for g in range(w32.shape[1] // group):
                blk = w32[n, g * group:(g + 1) * group]
                mn = min(np.float32(blk.min()), np.float32(0.0))
                mx = max(np.float32(blk.max()), np.float32(0.0))
                s32 = max(np.float32(mx - mn) / np.float32(15.0), np.float32(1e-8))
                r0 = float(np.float32(mn) / s32)
                d0 = np.abs(-codes - r0)
                cand = codes[d0 == d0.min()]
                zb = cand[0] if cand.size == 1 else cand[np.fmod(cand, 2) == 0][0]
                zz = int(z[n, g])
                assert zz == zb, (n, g, zz, r0)
                for i, wv in enumerate(blk):
                    r = float(np.float32(wv) / s32)
                    d = np.abs((codes - zz) - r)
                    best = codes[d == d.min()]
                    jb = best[0] if best.size == 1 else best[np.fmod(best - zz, 2) == 0][0]
                    assert nib[n, g * group + i] == jb, (n, g, i, r, zz)


def pin_asym_round_trip_bound(o) -> None:
    """Every element comes back within one step (half a step of rounding, at
    most half a step more where the rounded zero point pushes it to a clamped
    end), and on average within a quarter step (uniform rounding noise)."""
    rng = np.random.default_rng(23)
    w16 = _random_weights(rng, 128, 4096)
    w = w16.view(np.float16).astype(np.float64)
    for group in (32, 128):
        q, s, z = o.quantize_asym(w16, group)
        s64 = np.repeat(o.half_to_double(s), group, axis=1)
        err = np.abs(w - o.dequantize(q, s, group, zeros=z))
        assert (err <= s64 * (1 + 2.0 ** -6)).all(), float((err / s64).max())
        rel = (err / s64).mean()
        assert 0.2 < rel < 0.3, rel


def pin_asym_gemm_numpy_tiny(o) -> None:
    """With zero points, y equals numpy's float64 x @ ((nibble - z) * s)^T,
    nibbles, zero points and scales decoded by numpy."""
    rng = np.random.default_rng(24)
    for M, N, K, group in ((1, 1, 128, 128), (2, 3, 256, 64), (3, 5, 384, 32), (2, 2, 256, 256)):
        q, s, z = o.quantize_asym(_random_weights(rng, N, K), group)
        x16 = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
        wd = (_nibbles(q) - np.repeat(z.astype(np.int16), group, axis=1)) * np.repeat(
            s.view(np.float16).astype(np.float64), group, axis=1)
        np.testing.assert_array_equal(o.dequantize(q, s, group, zeros=z), wd)
        y = o.gemm(x16, q, s, group, zeros=z)
        np.testing.assert_allclose(y, x16.view(np.float16).astype(np.float64) @ wd.T,
                                   rtol=1e-12, atol=1e-12)
        rows = np.array([N - 1, 0])
        np.testing.assert_array_equal(o.gemm_rows(x16, q, s, rows, group, zeros=z), y[:, rows])


def pin_group_sizes_symmetric(o) -> None:
    """Groups of 32 and 64 and one group per row (per-channel, rows up to
    8192): every group's largest |w| maps to +-7, its scale is numpy's
    fp16(max(fp32(amax) / 7, 1e-8)), and dequantization uses the group's own
    scale."""
    rng = np.random.default_rng(25)
    for K, group in ((1024, 32), (1024, 64), (4096, -1), (8192, -1)):
        g = K if group == -1 else group
        w16 = _random_weights(rng, 16, K)
        q, s = o.quantize(w16, group)
        assert s.shape == (16, K // g)
        w = w16.view(np.float16)
        wg = w.astype(np.float64).reshape(16, -1, g)
        qg = (_nibbles(q) - 8).reshape(16, -1, g)
        idx = np.abs(wg).argmax(axis=-1)[..., None]
        assert (np.take_along_axis(qg, idx, -1) == 7 * np.sign(np.take_along_axis(wg, idx, -1))).all()
        a = np.abs(w.astype(np.float32)).reshape(16, -1, g).max(-1)
        ref = np.maximum(a / np.float32(7.0), np.float32(1e-8)).astype(np.float16).view(np.uint16)
        assert np.array_equal(s, ref)
        wd = o.dequantize(q, s, group)
        s64 = np.repeat(o.half_to_double(s), g, axis=1)
        np.testing.assert_array_equal(wd, (_nibbles(q) - 8) * s64)


# --------------------------------------------------------------------------
# AWQ activation scaling (tutorial AWQ section: x~_j = x_j * alpha_j)
# --------------------------------------------------------------------------

def pin_awq_scale_numpy(o) -> None:
    """x~ is numpy's IEEE fp16 conversion of the exact binary32 product x * alpha
    (subnormal, tie and overflow-free ranges included); alpha = 1 is the identity."""
    rng = np.random.default_rng(31)
    M, K = 5, 384
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-12, 4, (M, K)))).astype(np.float16)
    a = rng.uniform(0.5, 2.0, K).astype(np.float16)
    a[:4] = [1.0, 2.0 ** -3, 1.0 + 2.0 ** -10, 1.5]
    x[0, :4] = [1.0 + 2.0 ** -10, 3.0, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10]
    got = o.scale_activations(x.view(np.uint16), a.view(np.uint16))
    ref = (x.astype(np.float32) * a.astype(np.float32)).astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    # (1 + 2^-10)^2 rounds down to 1 + 2^-9; 1.5 (1 + 2^-10) is a tie -> even mantissa
    assert got[0, 2] == 0x3C02 and got[0, 3] == 0x3E02
    ones = np.full(K, 0x3C00, dtype=np.uint16)
    assert np.array_equal(o.scale_activations(x.view(np.uint16), ones), x.view(np.uint16))


def pin_awq_scale_per_input_channel(o) -> None:
    """alpha acts on input channel k: a one-hot alpha (2 at channel j) changes y by
    exactly x[:, j] * Wd[:, j], the dequantised column j (numpy)."""
    rng = np.random.default_rng(32)
    M, N, K = 3, 6, 256
    q, s = o.quantize(_random_weights(rng, N, K), GROUP)
    x16 = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    j = 77
    a = np.full(K, 0x3C00, dtype=np.uint16)
    a[j] = 0x4000  # 2.0
    y0 = o.gemm(x16, q, s, GROUP)
    y1 = o.gemm(o.scale_activations(x16, a), q, s, GROUP)
    wd = o.dequantize(q, s, GROUP)
    np.testing.assert_allclose(y1 - y0, np.outer(x16.view(np.float16)[:, j].astype(np.float64), wd[:, j]),
                               rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# W8A16 per-channel INT8 (tutorial §2 formula with b = 8, INT8 section)
# --------------------------------------------------------------------------

def pin_w8_amax_and_scale(o) -> None:
    """Every row's largest |w| maps to +-127 (code 128 +- 127), the scale is
    numpy's fp16(max(fp32(amax) / 127, 1e-8)); an all-zero row stays zero."""
    rng = np.random.default_rng(41)
    w16 = _random_weights(rng, 24, 640)
    w16[5] = 0
    q8, s = o.quantize_w8(w16)
    q = q8.astype(np.int64) - 128
    w = w16.view(np.float16).astype(np.float64)
    idx = np.abs(w).argmax(axis=1)
    live = np.abs(w).max(axis=1) > 0
    assert (q[live, idx[live]] == 127 * np.sign(w[live, idx[live]])).all()
    assert (q[5] == 0).all()
    a = np.abs(w16.view(np.float16).astype(np.float32)).max(axis=1)
    ref = np.maximum(a / np.float32(127.0), np.float32(1e-8)).astype(np.float16).view(np.uint16)
    assert np.array_equal(s, ref)


def pin_w8_nearest_level(o) -> None:
    """q is the integer nearest to fp32(w) / s32 (ties to even), checked by
    rounding numpy's float32 quotient with numpy's round-half-even."""
    rng = np.random.default_rng(42)
    w16 = _random_weights(rng, 6, 256)
    w16[0, :4] = _f16_bits([0.5, -1.5, 2.5, 127.0 * 2.0 ** -8])  # ties when s = 2^-8
    w16[0, 4] = _f16_bits([127.0 * 2.0 ** -8])[0]
    w16[0, 5:] = 0
    q8, _ = o.quantize_w8(w16)
    w32 = w16.view(np.float16).astype(np.float32)
    s32 = np.maximum(np.abs(w32).max(axis=1) / np.float32(127.0), np.float32(1e-8))
    ref = np.clip(np.rint(w32 / s32[:, None]), -128, 127).astype(np.int64)
    assert np.array_equal(q8.astype(np.int64) - 128, ref)


def pin_w8_round_trip_and_gemm(o) -> None:
    """Round trip within half a step of the binary32 scale; against the stored
    fp16 scale (|s16 - s32| <= 2^-11 s32) and |q| <= 128 that is
    s16 (1 + 2^-10) (1/2 + 2^-21 + 128 * 2^-11).  y equals numpy's float64
    matmul of the dequantised rows (decoded by numpy) on tiny shapes."""
    rng = np.random.default_rng(43)
    w16 = _random_weights(rng, 16, 512)
    q8, s = o.quantize_w8(w16)
    s64 = s.view(np.float16).astype(np.float64)
    wd = (q8.astype(np.float64) - 128) * s64[:, None]
    np.testing.assert_array_equal(o.dequantize_w8(q8, s), wd)
    err = np.abs(w16.view(np.float16).astype(np.float64) - wd)
    assert (err <= s64[:, None] * (1 + 2.0 ** -10) * (0.5 + 2.0 ** -21 + 2.0 ** -4)).all()
    assert 0.2 < (err / s64[:, None]).mean() < 0.3
    x16 = rng.standard_normal((3, 512)).astype(np.float16).view(np.uint16)
    y = o.gemm_rows_w8(x16, q8, s)
    np.testing.assert_allclose(y, x16.view(np.float16).astype(np.float64) @ wd.T, rtol=1e-12,
                               atol=1e-12)


def pin_dequant_f16_fixture(o) -> None:
    """The tutorial's fp16 dequantized weight matches hand-derived bits:
    exact products, ties to even (up and down), subnormal results, overflow
    to infinity, and the asymmetric zero point subtracted from the nibble."""
    for row in _read_fixture("dequant_f16.txt"):
        nib, z, sbits, ebits = int(row[1]), row[2], int(row[3], 16), int(row[4], 16)
        q = np.full((1, 64), nib | (nib << 4), dtype=np.uint8)  # K = 128, one group
        s = np.array([[sbits]], dtype=np.uint16)
        zeros = None if z == "-" else np.array([[int(z)]], dtype=np.uint8)
        out = o.dequantize_f16(q, s, GROUP, zeros)
        assert out.shape == (1, 128)
        assert (out == ebits).all(), f"nib {nib} z {z} s {sbits:#06x}: {out[0, 0]:#06x} != {ebits:#06x}"
    # two groups with different scales: each element takes its own group's scale
    q = np.full((1, 128), 0xFF, dtype=np.uint8)  # nibble 15 (q = 7), K = 256
    s = _f16_bits([[0.5, 0.25]])
    out = o.dequantize_f16(q, s, GROUP)
    assert (out[0, :128] == 0x4300).all() and (out[0, 128:] == 0x3F00).all()  # 3.5, 1.75


def pin_dequant_f16_single_rounding(o) -> None:
    """On random codes and scales the fp16 dequantized weight is numpy's IEEE
    float16 rounding of the exact binary64 dequantized value (the binary32
    product of an fp16 scale and |q| <= 15 is exact, so one rounding is all
    there is), symmetric and asymmetric, for groups of 32 and 128."""
    rng = np.random.default_rng(61)
    for group, asym in ((128, False), (32, True)):
        N, K = 5, 256
        q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        s = _f16_bits(rng.uniform(-3.0, 3.0, size=(N, K // group)) * 10.0 ** rng.integers(
            -4, 3, size=(N, K // group)))
        zeros = rng.integers(0, 16, size=(N, K // group), dtype=np.uint8) if asym else None
        nib = _nibbles(q).astype(np.float64)
        zz = 8.0 if zeros is None else np.repeat(zeros.astype(np.float64), group, axis=1)
        exact = (nib - zz) * np.repeat(s.view(np.float16).astype(np.float64), group, axis=1)
        want = exact.astype(np.float16).view(np.uint16)
        np.testing.assert_array_equal(o.dequantize_f16(q, s, group, zeros), want)


# --------------------------------------------------------------------------
# GGUF Q4_0 blocks (tutorial GGUF section)
# --------------------------------------------------------------------------

def pin_q4_0_block_fixture(o) -> None:
    """A hand-derived 18-byte block decodes to the fixture's values."""
    rows = {r[0]: r[1:] for r in _read_fixture("q4_0_block.txt")}
    blk = np.array([[int(b, 16) for b in rows["block"]]], dtype=np.uint8)
    expect = [float(v) for v in rows["values"]] + [float(rows["values_rest"][0])] * int(
        rows["values_rest"][1])
    assert o.dequantize_q4_0(blk, 32).tolist() == [expect]
    # and packing the same codes and scale gives the same block
    q = blk[:, 2:]
    s = np.array([[int(blk[0, 0]) | (int(blk[0, 1]) << 8)]], dtype=np.uint16)
    assert np.array_equal(o.pack_q4_0(q, s), blk)


def pin_q4_0_matches_group32(o) -> None:
    """Blocks of group-32 symmetric codes decode to exactly the group-32
    dequantized weights, 18 bytes per 32 weights; the GEMM follows."""
    rng = np.random.default_rng(51)
    w16 = _random_weights(rng, 7, 512)
    q, s = o.quantize(w16, 32)
    blocks = o.quantize_q4_0(w16)
    assert blocks.shape == (7, 512 // 32 * 18)
    np.testing.assert_array_equal(o.dequantize_q4_0(blocks, 512), o.dequantize(q, s, 32))
    x16 = rng.standard_normal((2, 512)).astype(np.float16).view(np.uint16)
    np.testing.assert_allclose(o.gemm_q4_0(x16, blocks), o.gemm(x16, q, s, 32), rtol=1e-12,
                               atol=1e-12)


ALL_PINS = (
    pin_half_to_double_exhaustive,
    pin_float_to_half_numpy,
    pin_half_round_trip,
    pin_nibble_order_fixture,
    pin_ties_to_even,
    pin_tiny_scale_clamp,
    pin_all_zero_group,
    pin_amax_maps_to_seven,
    pin_scale_is_fp16_of_amax_over_7,
    pin_nearest_level_brute_force,
    pin_round_trip_bound,
    pin_dequant_closed_forms,
    pin_gemm_numpy_tiny,
    pin_gemm_closed_form,
    pin_asym_integer_grid,
    pin_asym_range_includes_zero,
    pin_asym_constant_and_zero_groups,
    pin_asym_nearest_level_brute_force,
    pin_asym_round_trip_bound,
    pin_asym_gemm_numpy_tiny,
    pin_group_sizes_symmetric,
    pin_awq_scale_numpy,
    pin_awq_scale_per_input_channel,
    pin_w8_amax_and_scale,
    pin_q4_0_block_fixture,
    pin_q4_0_matches_group32,
    pin_w8_nearest_level,
    pin_w8_round_trip_and_gemm,
    pin_dequant_f16_fixture,
    pin_dequant_f16_single_rounding,
)
