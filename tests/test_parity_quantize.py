"""GPU quantizer vs the CPU oracle: packed bytes and fp16 scale bits must be
identical (the quantizer's result is unique under its definition)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits16, from_bits16
from parity_data import quantized
import w4a16_weight_only_gemm_gb300 as w4

pytestmark = pytest.mark.gpu


def _check(w16: np.ndarray, q_ref=None, s_ref=None):
    if q_ref is None:
        q_ref, s_ref = oracle.quantize(w16)
    q, s = w4.quantize(from_bits16(w16))
    torch.cuda.synchronize()
    q_np = q.cpu().numpy()
    s_np = bits16(s)
    bad_q = np.count_nonzero(q_np != q_ref)
    bad_s = np.count_nonzero(s_np != s_ref)
    assert bad_q == 0 and bad_s == 0, f"{bad_q} packed bytes and {bad_s} scales differ"


@pytest.mark.parametrize("N,K", [(1, 128), (3, 256), (130, 384), (1000, 1152), (4096, 4096)])
def test_random_outlier_weights(w4lib, N, K):
    w16, q, s = quantized(N, K, 100 + N)
    _check(w16, q, s)


def test_special_groups(w4lib):
    """All-zero, negative-zero, subnormal (scale clamp), power-of-two ties,
    +-amax, single-outlier and full-range groups in one matrix."""
    rng = np.random.default_rng(5)
    K = 128 * 12
    rows = []
    rows.append(np.zeros(K))
    rows.append(np.full(K, -0.0))
    rows.append(np.full(K, 2.0 ** -24))                         # amax/7 < 1e-8
    ties = np.array([7, 0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, -0.5, -1.5, -2.5, -3.5,
                     -4.5, -5.5, -6.5, -7] * 8) * 2.0 ** -6
    rows.append(np.tile(ties, K // 128))
    r = rng.standard_normal(K) * 1e-3
    r[::128] = 1.0                                              # one outlier per group
    rows.append(r)
    rows.append(rng.uniform(-65504, 65504, K))                  # full fp16 range
    rows.append(rng.standard_normal(K) * 2.0 ** -20)            # subnormal weights
    rows.append(-np.abs(rng.standard_normal(K)))                # negative amax
    w16 = np.stack(rows).astype(np.float16).view(np.uint16)
    _check(w16)


def test_random_fp16_bit_patterns(w4lib):
    rng = np.random.default_rng(6)
    bits = rng.integers(0, 65536, size=(64, 1024), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7C00) == 0x7C00] = 0x3C00                   # finite inputs only
    _check(bits)


def _all_below(amax: float) -> np.ndarray:
    """Every finite fp16 bit pattern with |value| <= amax, in groups of 127
    that each get amax itself as element 0 (so every group has that scale)."""
    vals = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = vals[(vals & 0x7C00) != 0x7C00]                      # finite patterns only
    vals = vals[np.abs(vals.view(np.float16).astype(np.float64)) <= amax]
    pad = (-len(vals)) % 127
    vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 127)
    head = np.full((vals.shape[0], 1), np.float16(amax).view(np.uint16), np.uint16)
    return np.concatenate([head, vals], axis=1)


# 0.2002, 0.024566650390625 and 3.14453125 are scales at which rounding
# w * fl(1 / s) instead of fl(w / s) changes some codes (found by scanning
# fp16 absmax values on the CPU); the others are plain and boundary scales.
@pytest.mark.parametrize("amax", [1.0, 0.0123, 3.7, 0.2002, 0.024566650390625, 3.14453125,
                                  65504.0, 2.0 ** -14, 7.0 * 2.0 ** -10])
def test_every_fp16_value_per_scale(w4lib, amax):
    """Each rounding decision w / s for all fp16 w of one scale: exact ties
    and values a few ulps either side of a half-integer included."""
    groups = _all_below(amax)
    K = 128 * 8
    rows = -(-groups.shape[0] // 8)
    full = np.zeros((rows * 8, 128), np.uint16)
    full[: groups.shape[0]] = groups
    _check(full.reshape(rows, K))


def test_every_fp16_absmax(w4lib):
    """One group per finite fp16 absmax a (both signs of it), the other 127
    weights spread over [-a, a]: every scale RN(a / 7) the quantizer can
    produce, and codes at each of those scales."""
    bits = np.arange(0x7C00, dtype=np.uint32).astype(np.uint16)
    a = bits.view(np.float16).astype(np.float64)
    frac = np.linspace(-1.0, 1.0, 127)
    body = (a[:, None] * frac[None, :]).astype(np.float16).view(np.uint16)
    sign = np.where(np.arange(len(bits)) % 2 == 1, 0x8000, 0).astype(np.uint16)
    groups = np.concatenate([(bits | sign)[:, None], body], axis=1)
    groups = groups[: len(groups) // 8 * 8]
    _check(groups.reshape(-1, 128 * 8))


@pytest.mark.parametrize("N,K", [(14336, 4096), (128256, 4096), (4096, 14336)])
def test_full_size(w4lib, N, K):
    """The quantizer workload [14336, 4096] plus the largest decode shapes."""
    w16, q, s = quantized(N, K, 4000 + N)
    _check(w16, q, s)


def test_round_trip_on_device(w4lib):
    """Dequantising the GPU result stays within half a step of the master."""
    w16, _, _ = quantized(256, 1024, 77)
    q, s = w4.quantize(from_bits16(w16))
    wd = oracle.dequantize(q.cpu().numpy(), bits16(s))
    w = w16.view(np.float16).astype(np.float64)
    s64 = np.repeat(oracle.half_to_double(bits16(s)), 128, axis=1)
    assert (np.abs(w - wd) <= s64 * (1 + 2.0 ** -10) * (0.5 + 2.0 ** -21 + 8 * 2.0 ** -11)).all()


# --------------------------------------------------------------------------
# Format variants: groups of 32 / 64 / per-channel, asymmetric with zero points
# --------------------------------------------------------------------------

def _special_rows(K: int, rng: np.random.Generator) -> np.ndarray:
    """Rows exercising the variant-specific edge cases: all-zero, constant
    positive / negative, all-positive and all-negative, integer-grid ties,
    subnormals, and random outlier weights."""
    rows = [
        np.zeros(K),
        np.full(K, 3.0),
        np.full(K, -0.75),
        np.abs(rng.standard_normal(K)) * 0.02,
        -np.abs(rng.standard_normal(K)) * 0.02,
        (rng.integers(-5, 11, size=K) * 2.0 ** -4),
        rng.integers(-3, 4, size=K) * 2.0 ** -20,
        rng.standard_normal(K) * 0.02 * np.where(rng.random(K) < 0.001, 20.0, 1.0),
    ]
    return np.stack(rows).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("group,K", [(32, 1024), (64, 1152), (128, 640), (w4.PER_CHANNEL, 4096),
                                     (w4.PER_CHANNEL, 4224), (w4.PER_CHANNEL, 14336)])
def test_format_variants_bit_exact(w4lib, group, K, asym):
    """Packed codes, fp16 scales and zero points identical to the oracle."""
    rng = np.random.default_rng(200 + K)
    w16 = np.concatenate([_special_rows(K, rng), quantized(130, K, 201)[0]])
    if asym:
        q_ref, s_ref, z_ref = oracle.quantize_asym(w16, group)
    else:
        q_ref, s_ref = oracle.quantize(w16, group)
    q, s, z = w4.quantize_ex(from_bits16(w16), group, asymmetric=asym)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref), np.count_nonzero(q.cpu().numpy() != q_ref)
    assert np.array_equal(bits16(s), s_ref)
    if asym:
        assert np.array_equal(z.cpu().numpy(), z_ref)
    else:
        assert z is None


def test_variant_group128_symmetric_is_the_default_quantizer(w4lib):
    w16 = quantized(64, 1024, 202)[0]
    q0, s0 = w4.quantize(from_bits16(w16))
    q1, s1, _ = w4.quantize_ex(from_bits16(w16), 128)
    torch.cuda.synchronize()
    assert torch.equal(q0, q1) and torch.equal(s0, s1)
