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
