"""W8A16 (per-channel symmetric INT8 weights, fp16 activations) vs the CPU
oracle: codes and scales bit-exact; the GEMV within the GEMV bar (products
q * x are exact, only FP32 sums and the final fp16 rounding of y round)."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits16, from_bits16, u8
from parity_data import acts, quantized, sample_rows
import w4a16_weight_only_gemm_gb300 as w4
from w4a16_weight_only_gemm_gb300 import synthetic, workloads

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=16)
def quantized_w8(N: int, K: int, seed: int):
    w16 = quantized(N, K, seed)[0]
    return w16, *oracle.quantize_w8(w16)


@pytest.mark.parametrize("N,K", [(1, 128), (130, 384), (1000, 2048), (4096, 14336)])
def test_quantizer_bit_exact(w4lib, N, K):
    w16, q_ref, s_ref = quantized_w8(N, K, 500 + N)
    w16 = w16.copy()
    w16[0] = 0  # an all-zero row
    q_ref, s_ref = oracle.quantize_w8(w16)
    q, s = w4.quantize_w8(from_bits16(w16))
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(bits16(s), s_ref)


@pytest.mark.parametrize("N,K", [(1000, 2048), (4136, 1152), (300, 4096), (37, 128)])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_gemv_every_row(w4lib, M, N, K):
    _, q, s = quantized_w8(N, K, 510 + K)
    x16 = acts(M, K, 511 + M)
    y = w4.gemm_w8(from_bits16(x16), u8(q), from_bits16(s))
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), oracle.gemm_rows_w8(x16, q, s), f"w8 M={M} N={N} K={K}")
    assert w4.device_status() == 0


def test_out_is_checked(w4lib):
    """A caller's y of the wrong shape or dtype is refused before any launch."""
    _, q, s = quantized_w8(64, 256, 520)
    x = from_bits16(acts(2, 256, 521))
    for bad in (torch.empty((2, 65), dtype=torch.float16, device="cuda"),
                torch.empty((2, 64), dtype=torch.float32, device="cuda"),
                torch.empty((64, 2), dtype=torch.float16, device="cuda").t()):
        with pytest.raises(ValueError):
            w4.gemm_w8(x, u8(q), from_bits16(s), out=bad)
    assert w4.device_status() == 0


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA3_8B)))
def test_llama3_8b_shapes_m1(w4lib, idx):
    lin = workloads.LLAMA3_8B[idx]
    sw, sx = synthetic.seeds("llama3_8b_decode", idx)
    _, q, s = quantized_w8(lin.N, lin.K, sw)
    x16 = acts(1, lin.K, sx)
    y = w4.gemm_w8(from_bits16(x16), u8(q), from_bits16(s))
    torch.cuda.synchronize()
    rows = sample_rows(lin.N, 256, sw)
    assert_close(y[:, rows].float().cpu().numpy(), oracle.gemm_rows_w8(x16, q, s, rows), lin.name)


def _fuzz_cases():
    """Seeded W8A16 calls across the unit plans, ragged N and K tails."""
    rng = np.random.default_rng(20261207)
    cases = []
    for _ in range(8):
        M = int(rng.choice([1, 3, 8, 9, 16]))
        K = 128 * int(rng.integers(1, 60))
        N = int(rng.integers(50, max(100, min(100000, 20_000_000 // K))))
        cases.append((M, N, K))
    return cases


@pytest.mark.parametrize("M,N,K", _fuzz_cases())
def test_w8_plans_fuzz(w4lib, M, N, K):
    """Whatever unit plan a call gets: no wait times out, sampled rows meet
    the bar, and a repeat call is bit-identical."""
    q8, s8 = oracle.quantize_w8(bits16(synthetic.master_weight(N, K, 640)))
    x16 = acts.__wrapped__(M, K, 641 + M)
    qt, st = u8(q8), from_bits16(s8)
    x = from_bits16(x16)
    w4.device_status()  # clear
    y1 = w4.gemm_w8(x, qt, st)
    y2 = w4.gemm_w8(x, qt, st)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    y = y1.float().cpu().numpy()
    assert np.array_equal(y, y2.float().cpu().numpy())
    rows = sample_rows(N, 96, 642)
    assert_close(y[:, rows], oracle.gemm_rows_w8(x16, q8, s8, rows), f"w8 M={M} N={N} K={K}")
