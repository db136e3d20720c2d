"""Prefill GEMM (M > 16, tcgen05 tensor cores) vs the binary64 oracle.

The kernel stages fp16(q * scale) -- the tutorial's own fp16 dequantized
weight, one rounding of at most 2^-11 relative -- and accumulates in FP32 in
tensor memory; together with the final fp16 rounding of y that stays inside
the same bar as the GEMV: max|y - y_ref| <= 2e-3 max|y_ref| and
||y - y_ref|| <= 1e-3 ||y_ref||."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits16, from_bits16
from parity_data import acts, as_device, quantized, sample_rows
import w4a16_weight_only_gemm_gb300 as w4
from w4a16_weight_only_gemm_gb300 import synthetic, workloads

pytestmark = pytest.mark.gpu


def run_gemm(x16, q, s):
    qt, st = as_device(q, s)
    y = w4.gemm(from_bits16(x16), w4.repack(qt), st)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M", [17, 31, 64, 128, 130, 256, 300])
def test_m_values(w4lib, M):
    N, K = 256, 512
    w16, q, s = quantized(N, K, 61)
    x16 = acts(M, K, 62 + M)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M}")


@pytest.mark.parametrize("N,K", [(128, 128), (200, 384), (1000, 1152), (4168, 640), (136, 18944),
                                 (136, 32768)])
@pytest.mark.parametrize("M", [20, 144])
def test_shapes_and_tails(w4lib, M, N, K):
    w16, q, s = quantized(N, K, 71)
    x16 = acts(M, K, 72)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(300, 14336, 1152), (512, 14336, 512), (300, 2000, 18944),
                                   (512, 4096, 14336), (290, 977, 4096)])
def test_pairs_of_96_row_ctas(w4lib, M, N, K):
    """CTA pairs with two x tiles and 96 weight rows per CTA (N = 192 MMAs;
    a CTA's six tiles straddle kernel-layout blocks in two of every four
    CTAs), with and without a K split over the cluster; ragged N leaves the
    last CTAs partly or wholly past N.  Every output, and a repeat call is
    bit-identical."""
    plan = w4.gemm_plan(M, N, K)
    if plan["rows_per_cta"] != 96:
        pytest.skip(f"planner chose {plan} for this shape on this device")
    w16, q, s = quantized(N, K, 73)
    x16 = acts(M, K, 74)
    y = run_gemm(x16, q, s)
    assert_close(y, oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")
    assert np.array_equal(run_gemm(x16, q, s), y)


def test_pairs_of_96_row_ctas_covered(w4lib):
    """The cases above reach the 96-row CTAs both unsplit and split."""
    plans = [w4.gemm_plan(M, N, K) for M, N, K in
             [(300, 14336, 1152), (512, 14336, 512), (300, 2000, 18944), (512, 4096, 14336),
              (290, 977, 4096)]]
    picked = [p for p in plans if p["rows_per_cta"] == 96]
    assert any(p["splits"] == 2 for p in picked) and any(p["splits"] > 2 for p in picked), plans


@pytest.mark.parametrize("kind", synthetic.OFFSET_KINDS)
@pytest.mark.parametrize("M,N,K", [(40, 1000, 1152), (300, 512, 4096)])
def test_offset_activations(w4lib, kind, M, N, K):
    """Activations with a large common offset, every output."""
    w16, q, s = quantized(N, K, 75)
    x16 = bits16(synthetic.activations_offset(M, K, 76, kind))
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"{kind} M={M} N={N} K={K}")


def test_every_nibble_value(w4lib):
    rng = np.random.default_rng(81)
    N, K, M = 384, 1024, 96
    q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = (rng.uniform(0.5, 2.0, size=(N, K // 128)) * 2.0 ** rng.integers(-12, 2, size=(N, K // 128))
         ).astype(np.float16).view(np.uint16)
    x16 = acts(M, K, 82)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), "nibbles")


def test_guard_bands(w4lib):
    N, K, M = 200, 256, 70
    w16, q, s = quantized(N, K, 91)
    x = from_bits16(acts(M, K, 92))
    qt, st = as_device(q, s)
    r = w4.repack(qt)
    pad = 64
    buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    w4.gemm(x, r, st, out=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()
    x16 = x.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_close(y.float().cpu().numpy(), oracle.gemm(x16, q, s), "guard")


@pytest.mark.parametrize("M,N,K", [(300, 19000, 384), (200, 19300, 256), (512, 38400, 128)])
def test_cta_pair_path(w4lib, M, N, K):
    """Tiles on CTA pairs (2-CTA MMAs): 512 x 256 and 256 x 256, an odd
    number of 128-row weight blocks (the last pair's odd CTA holds none),
    ragged M; every output compared."""
    plan = w4.gemm_plan(M, N, K)
    assert plan["path"] == "tensor_core" and plan["splits"] == 2, plan
    w16, q, s = quantized(N, K, 81)
    x16 = acts(M, K, 82)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")


@pytest.mark.parametrize("M,N,K,cluster", [(300, 8000, 1920, 4), (300, 4000, 16384, 6),
                                           (300, 1000, 18944, 8), (300, 136, 18944, 8)])
def test_split_k_path(w4lib, M, N, K, cluster):
    """CTA pairs splitting K two, three or four ways, the splits of a tile reducing
    through the cluster's shared memory (ragged M; a pair whose odd CTA holds
    no weights): every output compared, and two calls give the same bits
    (the reduction order is fixed)."""
    plan = w4.gemm_plan(M, N, K)
    assert plan["path"] == "tensor_core" and plan["splits"] == cluster, plan
    w16, q, s = quantized(N, K, 91)
    x16 = acts(M, K, 92)
    qt, st = as_device(q, s)
    r = w4.repack(qt)
    x = from_bits16(x16)
    y1 = w4.gemm(x, r, st)
    y2 = w4.gemm(x, r, st)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert_close(y1.float().cpu().numpy().astype(np.float64), oracle.gemm(x16, q, s),
                 f"M={M} N={N} K={K} {plan}")
    assert w4.device_status() == 0


@pytest.mark.parametrize("idx", range(len(workloads.PREFILL)))
def test_prefill_full_size(w4lib, idx):
    """M = 512 prompt pass on the two prefill shapes; oracle on sampled rows."""
    lin = workloads.PREFILL[idx]
    sw, sx = synthetic.seeds("prefill", idx)
    w16, q, s = quantized(lin.N, lin.K, sw)
    x16 = acts(workloads.PREFILL_M, lin.K, sx)
    y = run_gemm(x16, q, s)
    rows = sample_rows(lin.N, 96, sw)
    assert_close(y[:, rows], oracle.gemm_rows(x16, q, s, rows), lin.name)


def _fuzz_cases():
    """Seeded prefill shapes across the tile plans: single CTAs, CTA pairs of
    128- and 96-row CTAs, K split over clusters; ragged M, N and K tails."""
    rng = np.random.default_rng(20261204)
    cases = []
    for _ in range(12):
        M = int(rng.integers(17, 700))
        K = 128 * int(rng.integers(1, 65))
        N = int(rng.integers(100, max(200, min(30000, 40_000_000 // K))))
        cases.append((M, N, K))
    return cases


@pytest.mark.parametrize("M,N,K", _fuzz_cases())
def test_tile_plans_fuzz(w4lib, M, N, K):
    """Whatever tile plan a shape gets: no wait times out, sampled columns
    (the first and last weight rows of a block included) meet the bar for
    every x row, and a repeat call is bit-identical."""
    w16, q, s = quantized.__wrapped__(N, K, 95)
    x16 = acts.__wrapped__(M, K, 96)
    qt, st = as_device(q, s)
    r = w4.repack(qt)
    x = from_bits16(x16)
    w4.device_status()  # clear
    y1 = w4.gemm(x, r, st)
    y2 = w4.gemm(x, r, st)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    y = y1.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y2.float().cpu().numpy().astype(np.float64))
    rows = sample_rows(N, 96, 97)
    assert_close(y[:, rows], oracle.gemm_rows(x16, q, s, rows), f"M={M} N={N} K={K}")
