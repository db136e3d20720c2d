"""Decode GEMV (M = 1..16) vs the binary64 oracle.

Bar (floating point, from the accuracy target of the path): max|y - y_ref| <=
2e-3 max|y_ref| and ||y - y_ref|| <= 1e-3 ||y_ref||.  The budget is the final
fp16 rounding of y (2^-11 relative, ~2.8e-4 RMS); products q*x are exact and
sums are FP32."""
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


def run_gemm(x16: np.ndarray, q: np.ndarray, s: np.ndarray) -> np.ndarray:
    qt, st = as_device(q, s)
    y = w4.gemm(from_bits16(x16), w4.repack(qt), st)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_every_m_small(w4lib, M):
    """Several row blocks, a ragged row tail, K split over a cluster."""
    N, K = 1000, 1152
    w16, q, s = quantized(N, K, 11)
    x16 = acts(M, K, 12 + M)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M}")


@pytest.mark.parametrize("N,K", [(1, 128), (8, 128), (16, 256), (136, 384), (200, 1024),
                                 (4168, 4096), (264, 18944), (4096, 640)])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_shapes_and_tails(w4lib, M, N, K):
    w16, q, s = quantized(N, K, 21)
    x16 = acts(M, K, 22)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M} N={N} K={K}")


def test_every_nibble_value(w4lib):
    """Hand-made packed data covering all 16 nibbles, including 0 (q = -8),
    which the quantizer never emits, and varied fp16 scales."""
    rng = np.random.default_rng(31)
    N, K = 520, 1024
    q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = (rng.uniform(0.5, 2.0, size=(N, K // 128)) * 2.0 ** rng.integers(-12, 2, size=(N, K // 128))
         ).astype(np.float16).view(np.uint16)
    for M in (1, 5, 16):
        x16 = acts(M, K, 32)
        assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"nibbles M={M}")


def test_output_guard_bands(w4lib):
    """Nothing is written outside y: sentinels around the output survive."""
    N, K, M = 136, 512, 3
    w16, q, s = quantized(N, K, 41)
    x = from_bits16(acts(M, K, 42))
    qt, st = as_device(q, s)
    r = w4.repack(qt)
    pad = 64
    buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    w4.gemm(x, r, st, out=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()
    assert_close(y.float().cpu().numpy(), oracle.gemm(bits16(x), q, s), "guard")


def test_single_gemv_4096(w4lib):
    """The single 4096x4096 M=1 GEMV, compared in full."""
    sw, sx = synthetic.seeds("gemv_4096")
    w16, q, s = quantized(4096, 4096, sw)
    x16 = acts(1, 4096, sx)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), "gemv_4096")


@pytest.mark.parametrize("M", [1, 5, 9, 16])
@pytest.mark.parametrize("N,K", [(70001, 1152), (50000, 4096)])
def test_persistent_path_all_rows(w4lib, M, N, K):
    """More 128-row blocks than CTA slots: each CTA walks several blocks with
    its ring running across block boundaries; every row checked."""
    plan = w4.gemm_plan(M, N, K)
    assert plan["path"] == "gemv" and plan["blocks_per_cta"] > 1, plan
    w16, q, s = quantized(N, K, 51)
    x16 = acts(M, K, 52)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("K", [256, 1152])
@pytest.mark.parametrize("tail_rows", [16, 32, 64])
def test_persistent_tail_units_all_rows(w4lib, M, K, tail_rows):
    """A persistent launch whose last round is partial runs those blocks as
    units of 16, 32 or 64 rows, one per CTA after its whole blocks.  The
    shape puts R left-over blocks on G CTAs (R * 128 / tail_rows <= G) and
    ends in a ragged block (91 rows), so some tail units are partly or
    wholly beyond N; K = 1152 ends the units' streams in a partial stage.
    Every row is checked, and a repeat call is bit-identical."""
    G = w4.gemm_plan(M, 200_000, K)["ctas"]
    rem = {16: G // 8, 32: G // 4, 64: G // 2}[tail_rows]
    N = 128 * (G + rem) - 37
    plan = w4.gemm_plan(M, N, K)
    tail = w4.gemm_plan_tail(M, N, K)
    assert plan["blocks_per_cta"] > 1 and plan["ctas"] == G, plan
    assert tail == {"tail_rows": tail_rows, "tail_units": rem * 128 // tail_rows}, (tail, plan)
    w16, q, s = quantized(N, K, 71)
    x16 = acts(M, K, 72 + M)
    y = run_gemm(x16, q, s)
    assert_close(y, oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan} {tail}")
    assert np.array_equal(run_gemm(x16, q, s), y)


@pytest.mark.parametrize("M", [1, 4, 9, 16])
def test_persistent_short_k_many_blocks_all_rows(w4lib, M):
    """A persistent launch at K = 256 (one ring stage per block) whose CTAs
    walk three or more blocks: the producer reuses a scale-slab buffer before
    its ring wraps, so it must have issued x (M <= 4: the CTA-wide slice;
    M > 4: the boxes of the stages issued so far) before it waits for the
    consumers to free that buffer.  N ends in a ragged block; every row is
    checked."""
    K = 256
    G = w4.gemm_plan(M, 200_000, K)["ctas"]
    N = 128 * (3 * G) + 128 * (G // 5) - 37
    plan = w4.gemm_plan(M, N, K)
    assert plan["blocks_per_cta"] >= 3 and plan["ctas"] == G, plan
    w16, q, s = quantized(N, K, 75)
    x16 = acts(M, K, 76 + M)
    w4.device_status()  # clear
    y = run_gemm(x16, q, s)
    assert w4.device_status() == 0  # no wait timed out
    assert_close(y, oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")


@pytest.mark.parametrize("M", [5, 9, 16])
@pytest.mark.parametrize("K", [256, 1152])
def test_persistent_x_in_ring_all_rows(w4lib, M, K):
    """With M > 4 a whole-block launch streams x with every ring stage (a
    swizzled box of 4 chunks x M rows) instead of one CTA-wide slice, and a
    partial last round runs as whole blocks.  K = 1152 ends each block in a
    half stage whose box reaches past K (filled with zeros); N ends in a
    ragged block.  Every row is checked, and a repeat call is bit-identical."""
    G = w4.gemm_plan(M, 200_000, K)["ctas"]
    N = 128 * (G + G // 3) - 37
    plan = w4.gemm_plan(M, N, K)
    assert plan["blocks_per_cta"] == 2 and plan["ctas"] == G, plan
    assert w4.gemm_plan_tail(M, N, K) == {"tail_rows": 0, "tail_units": 0}
    w16, q, s = quantized(N, K, 73)
    x16 = acts(M, K, 74 + M)
    y = run_gemm(x16, q, s)
    assert_close(y, oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")
    assert np.array_equal(run_gemm(x16, q, s), y)


# Activations with a large common offset (real decode activations are not
# zero-mean) make the group sums of x large; a decode that fed biased codes to
# the MMAs and removed bias * sum(x) afterwards would lose the dot product's
# low bits there.  Each kind of launch on such activations.
# (Persistent launches take, at M <= 4, the decode of unbiased codes whose x
# sums are removed after the MMAs.)
OFFSET_CANDIDATES = {
    "unit": [(4096, 4096), (6144, 4096), (1000, 2048), (16384, 2048), (8000, 1920), (16384, 1024),
             (4096, 512)],
    "split": [(264, 18944), (136, 18944), (1000, 1152), (4096, 4096), (4096, 14336)],
    "persistent": [(50000, 1152), (70001, 1152)],
}


def _launch_of(plan) -> str:
    if plan["blocks_per_cta"] > 1:
        return "persistent"
    if plan["splits"] > 1:
        return "split"
    return "unit" if plan["rows_per_cta"] < 128 else "whole"


# (At M = 1 the planner no longer splits K for these shapes: one CTA's x
# slice is small, and units skip the cluster reduction.  The split kernel at
# M = 1 is the one at M = 3.)
OFFSET_LAUNCHES = [(launch, M) for launch in ("unit", "split", "persistent")
                   for M in (1, 3, 9, 16) if (launch, M) != ("split", 1)]


@pytest.mark.parametrize("kind", synthetic.OFFSET_KINDS)
@pytest.mark.parametrize("launch,M", OFFSET_LAUNCHES)
def test_offset_activations_all_rows(w4lib, kind, M, launch):
    """The first candidate shape the planner launches this way, every row."""
    shapes = [(N, K) for N, K in OFFSET_CANDIDATES[launch]
              if _launch_of(w4.gemm_plan(M, N, K)) == launch]
    assert shapes, (launch, M, [w4.gemm_plan(M, N, K) for N, K in OFFSET_CANDIDATES[launch]])
    N, K = shapes[0]
    w16, q, s = quantized(N, K, 81)
    x16 = bits16(synthetic.activations_offset(M, K, 82 + M, kind))
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s),
                 f"{kind} M={M} {launch} N={N} K={K} {w4.gemm_plan(M, N, K)}")


# Unit launches at M <= 4 whose warps each see 16 or more groups per round
# of the x-sum pass (ceil(8 G M / 256) rounds, G = K / 128) take the decode of
# unbiased codes.
LONG_UNIT_CANDIDATES = [(28672, 4096), (14336, 4096), (4096, 14336), (8192, 14336)]


@pytest.mark.parametrize("kind", ("normal",) + synthetic.OFFSET_KINDS)
@pytest.mark.parametrize("M", [1])
def test_long_units_all_rows(w4lib, kind, M):
    """The first candidate the planner runs as such units, every row."""
    def long_unit(N, K):
        p = w4.gemm_plan(M, N, K)
        G, T = K // 128, p["rows_per_cta"] // 16
        return _launch_of(p) == "unit" and G * T // 8 >= 16 * -(-G * M * 8 // 256)
    shapes = [(N, K) for N, K in LONG_UNIT_CANDIDATES if long_unit(N, K)]
    assert shapes, (M, [w4.gemm_plan(M, N, K) for N, K in LONG_UNIT_CANDIDATES])
    N, K = shapes[0]
    w16, q, s = quantized(N, K, 83)
    x = (synthetic.activations(M, K, 84 + M) if kind == "normal"
         else synthetic.activations_offset(M, K, 84 + M, kind))
    x16 = bits16(x)
    assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s),
                 f"{kind} M={M} N={N} K={K} {w4.gemm_plan(M, N, K)}")


# Launches made of sub-block units (16, 32 or 64 weight rows per CTA over the
# whole K range): ragged row tails inside a tile, and K ranges that end in a
# partial ring stage (K = 11008: 172 chunks; K = 1920: 30).
SUB_BLOCK_CASES = [(1000, 2048, 1), (1000, 2048, 4), (4096, 4096, 1),
                   (4096, 4096, 2), (6144, 4096, 1), (4136, 11008, 1), (8000, 1920, 1),
                   (8000, 1920, 4), (24000, 1024, 1), (24000, 1024, 3), (16384, 2048, 2),
                   # x slices of 8 rows (M = 5..8 units: 16-row units beat K splits there)
                   (4096, 4096, 8), (3584, 3584, 8), (4608, 3584, 7)]


@pytest.mark.parametrize("N,K,M", SUB_BLOCK_CASES)
def test_sub_block_units_all_rows(w4lib, N, K, M):
    """Every row of launches whose CTAs own 1, 2 or 4 tiles and split K over
    their warps, reducing in shared memory."""
    plan = w4.gemm_plan(M, N, K)
    assert plan["path"] == "gemv" and plan["splits"] == 1 and plan["rows_per_cta"] < 128, plan
    w16, q, s = quantized(N, K, 61)
    x16 = acts(M, K, 62 + M)
    y = run_gemm(x16, q, s)
    assert_close(y, oracle.gemm(x16, q, s), f"M={M} N={N} K={K} {plan}")
    # the in-CTA reduction runs in a fixed order: a repeat call is bit-identical
    assert np.array_equal(run_gemm(x16, q, s), y)


def test_sub_block_unit_sizes_covered(w4lib):
    """The cases above exercise all three unit sizes."""
    rows = {w4.gemm_plan(M, N, K)["rows_per_cta"] for N, K, M in SUB_BLOCK_CASES}
    assert {16, 32, 64} <= rows, rows


def test_sub_block_units_two_n8_tiles(w4lib):
    """Sub-block units with M > 8 (two n8 tiles per MMA step): the launches
    among these shapes that the planner makes of units, every row."""
    cands = [(16384, 2048, 12), (8000, 1920, 9), (16384, 2048, 9), (12000, 1536, 10)]
    picked = [(N, K, M) for N, K, M in cands if w4.gemm_plan(M, N, K)["rows_per_cta"] < 128]
    assert picked, [w4.gemm_plan(M, N, K) for N, K, M in cands]
    for N, K, M in picked[:2]:
        w16, q, s = quantized(N, K, 63)
        x16 = acts(M, K, 64)
        assert_close(run_gemm(x16, q, s), oracle.gemm(x16, q, s), f"M={M} N={N} K={K}")


def _sampled(lin, M, workload, idx):
    sw, sx = synthetic.seeds(workload, idx)
    w16, q, s = quantized(lin.N, lin.K, sw)
    x16 = acts(M, lin.K, sx)
    y = run_gemm(x16, q, s)
    rows = sample_rows(lin.N, 384, sw)
    y_ref = oracle.gemm_rows(x16, q, s, rows)
    assert_close(y[:, rows], y_ref, f"{lin.name} M={M}")


@pytest.mark.parametrize("idx", range(len(workloads.LLAMA3_8B)))
def test_llama3_8b_decode_shapes(w4lib, idx):
    _sampled(workloads.LLAMA3_8B[idx], 1, "llama3_8b_decode", idx)


@pytest.mark.parametrize("M", workloads.DECODE_SWEEP_M)
@pytest.mark.parametrize("idx", range(len(workloads.LLAMA3_8B) + len(workloads.QWEN25_7B)))
def test_decode_sweep(w4lib, M, idx):
    shapes = workloads.LLAMA3_8B + workloads.QWEN25_7B
    _sampled(shapes[idx], M, "decode_sweep", idx)


def _fuzz_cases():
    """Seeded shapes across the planner's regimes: unit launches, K splits,
    persistent grids with and without partial last rounds, short and long K
    (weights kept under ~60 M so the oracle quantizes them in a second)."""
    rng = np.random.default_rng(20261203)
    ks = [128, 256, 384, 512, 768, 1152, 2048, 3584, 4096]
    cases = []
    for _ in range(24):
        M = int(rng.integers(1, 17))
        K = int(rng.choice(ks))
        N = int(rng.integers(1000, max(4096, 60_000_000 // K)))
        cases.append((M, N, K))
    return cases


@pytest.mark.parametrize("M,N,K", _fuzz_cases())
def test_planner_regimes_fuzz(w4lib, M, N, K):
    """Whatever launch the planner picks: no wait times out, sampled rows
    (the first and last of a block included) meet the bar, and a repeat call
    is bit-identical."""
    plan = w4.gemm_plan(M, N, K)
    w16, q, s = quantized.__wrapped__(N, K, 90 + M)
    x16 = acts.__wrapped__(M, K, 91 + M)
    w4.device_status()  # clear
    qt, st = as_device(q, s)
    r = w4.repack(qt)
    x = from_bits16(x16)
    y1 = w4.gemm(x, r, st)
    y2 = w4.gemm(x, r, st)
    torch.cuda.synchronize()
    assert w4.device_status() == 0, plan
    y = y1.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y2.float().cpu().numpy().astype(np.float64)), plan
    rows = sample_rows(N, 192, 92 + M)
    assert_close(y[:, rows], oracle.gemm_rows(x16, q, s, rows), f"M={M} N={N} K={K} {plan}")
