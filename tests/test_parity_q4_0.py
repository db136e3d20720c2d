"""GGUF Q4_0 blocks (32 weights in 18 bytes, inline fp16 scale) vs the CPU
oracle: blocks bit-exact; the GEMV within the GEMV bar (q * x products exact,
one FP32 rescale per block, FP32 sums, y rounded once)."""
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
def blocks_of(N: int, K: int, seed: int):
    w16 = quantized(N, K, seed)[0]
    return w16, oracle.quantize_q4_0(w16)


@pytest.mark.parametrize("N,K", [(1, 256), (130, 512), (1000, 2048), (4096, 14336)])
def test_quantizer_bit_exact(w4lib, N, K):
    w16, ref = blocks_of(N, K, 600 + N)
    w16 = w16.copy()
    w16[0, :64] = 0  # two all-zero blocks
    ref = oracle.quantize_q4_0(w16)
    got = w4.quantize_q4_0(from_bits16(w16))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("N,K", [(1000, 2048), (4136, 1280), (300, 4096), (37, 256)])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_gemv_every_row(w4lib, M, N, K):
    _, blocks = blocks_of(N, K, 610 + K)
    x16 = acts(M, K, 611 + M)
    y = w4.gemm_q4_0(from_bits16(x16), u8(blocks))
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), oracle.gemm_q4_0(x16, blocks), f"q4_0 M={M} N={N} K={K}")
    assert w4.device_status() == 0


@pytest.mark.parametrize("M", [1, 9])
def test_many_units_every_row(w4lib, M):
    """More units than one wave of CTAs holds, the last one ragged
    (N = 60001); a repeat call is bit-identical."""
    N, K = 60001, 1024
    _, blocks = blocks_of(N, K, 620)
    x16 = acts(M, K, 621 + M)
    y = w4.gemm_q4_0(from_bits16(x16), u8(blocks))
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), oracle.gemm_q4_0(x16, blocks), f"q4_0 M={M}")
    assert np.array_equal(w4.gemm_q4_0(from_bits16(x16), u8(blocks)).cpu().numpy(),
                          y.cpu().numpy())
    assert w4.device_status() == 0


def test_out_is_checked(w4lib):
    """A caller's y of the wrong shape or dtype is refused before any launch."""
    _, blocks = blocks_of(64, 256, 530)
    x = from_bits16(acts(2, 256, 531))
    for bad in (torch.empty((2, 65), dtype=torch.float16, device="cuda"),
                torch.empty((2, 64), dtype=torch.float32, device="cuda"),
                torch.empty((64, 2), dtype=torch.float16, device="cuda").t()):
        with pytest.raises(ValueError):
            w4.gemm_q4_0(x, u8(blocks), out=bad)
    assert w4.device_status() == 0


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA3_8B)))
def test_llama3_8b_shapes_m1(w4lib, idx):
    lin = workloads.LLAMA3_8B[idx]
    sw, sx = synthetic.seeds("llama3_8b_decode", idx)
    _, blocks = blocks_of(lin.N, lin.K, sw)
    x16 = acts(1, lin.K, sx)
    y = w4.gemm_q4_0(from_bits16(x16), u8(blocks))
    torch.cuda.synchronize()
    rows = sample_rows(lin.N, 256, sw)
    assert_close(y[:, rows].float().cpu().numpy(), oracle.gemm_q4_0(x16, blocks, rows), lin.name)


def _fuzz_cases():
    """Seeded Q4_0 calls across the unit plans (16 to 128 rows per CTA, one
    or several waves), M = 1 (the odd-column skip) and M > 1, ragged N."""
    rng = np.random.default_rng(20261206)
    cases = []
    for _ in range(10):
        M = int(rng.choice([1, 1, 2, 4, 8, 9, 16]))
        K = 256 * int(rng.integers(1, 40))
        N = int(rng.integers(50, max(100, min(150000, 30_000_000 // K))))
        cases.append((M, N, K))
    return cases


@pytest.mark.parametrize("M,N,K", _fuzz_cases())
def test_q4_0_plans_fuzz(w4lib, M, N, K):
    """Whatever unit plan a call gets: no wait times out, sampled rows meet
    the bar, and a repeat call is bit-identical."""
    w16 = bits16(synthetic.master_weight(N, K, 630))
    blocks = oracle.quantize_q4_0(w16)
    x16 = acts.__wrapped__(M, K, 631 + M)
    bt = u8(blocks)
    x = from_bits16(x16)
    w4.device_status()  # clear
    y1 = w4.gemm_q4_0(x, bt)
    y2 = w4.gemm_q4_0(x, bt)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    y = y1.float().cpu().numpy()
    assert np.array_equal(y, y2.float().cpu().numpy())
    rows = sample_rows(N, 96, 632)
    assert_close(y[:, rows], oracle.gemm_q4_0(x16, blocks, rows), f"q4_0 M={M} N={N} K={K}")
