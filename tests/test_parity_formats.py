"""Format variants of the decode GEMV (w4a16_gemm_ex: groups of 32, 64, 128
or per-channel, symmetric or asymmetric codes) vs the binary64 oracle, on the
oracle's own codes, scales and zero points.

Bar: the same as the default GEMV (max|dy| <= 2e-3 max|y_ref|, relative L2
<= 1e-3).  The variants round (q - z) * scale once to fp16 per weight (the
tutorial's own fp16 dequantised weight): about 2^-12 relative per weight,
random in sign, well inside the L2 budget next to the final fp16 rounding."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, from_bits16, u8
from parity_data import acts, sample_rows
import w4a16_weight_only_gemm_gb300 as w4
from w4a16_weight_only_gemm_gb300 import synthetic, workloads

pytestmark = pytest.mark.gpu

FORMATS = [(32, False), (32, True), (64, False), (64, True), (128, True), (w4.PER_CHANNEL, False),
           (w4.PER_CHANNEL, True)]


@functools.lru_cache(maxsize=32)
def quantized_fmt(N: int, K: int, seed: int, group: int, asym: bool):
    w16 = synthetic.master_weight(N, K, seed).contiguous().view(torch.int16).numpy().view(np.uint16)
    if asym:
        return oracle.quantize_asym(w16, group)
    q, s = oracle.quantize(w16, group)
    return q, s, None


def run_fmt(x16, q, s, z, group):
    r = w4.repack(u8(q))
    st = from_bits16(s)
    zt = u8(z) if z is not None else None
    y = w4.gemm_ex(from_bits16(x16), r, st, zt, group)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("N,K", [(1000, 2048), (4136, 1152), (300, 4096)])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_formats_every_row(w4lib, M, N, K, group, asym):
    q, s, z = quantized_fmt(N, K, 300 + K, group, asym)
    x16 = acts(M, K, 301 + M)
    y = run_fmt(x16, q, s, z, group)
    assert_close(y, oracle.gemm(x16, q, s, group, zeros=z), f"g={group} asym={asym} M={M}")
    assert w4.device_status() == 0


@pytest.mark.parametrize("kind", synthetic.OFFSET_KINDS)
@pytest.mark.parametrize("group,asym", [(32, False), (128, True), (w4.PER_CHANNEL, True)])
@pytest.mark.parametrize("M", [1, 9, 16])
def test_formats_offset_activations(w4lib, M, group, asym, kind):
    """Activations with a large common offset (4 + N(0,1), |N(0,3)|, one group
    of 468.75) on the variant decode GEMV, every row."""
    N, K = 1000, 2048
    q, s, z = quantized_fmt(N, K, 310, group, asym)
    from gpu_util import bits16
    x16 = bits16(synthetic.activations_offset(M, K, 311 + M, kind))
    y = run_fmt(x16, q, s, z, group)
    assert_close(y, oracle.gemm(x16, q, s, group, zeros=z), f"{kind} g={group} asym={asym} M={M}")


@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("idx", range(len(workloads.LLAMA3_8B)))
def test_formats_llama3_8b_m1(w4lib, idx, group, asym):
    """The Llama-3-8B decode shapes at M = 1, sampled rows."""
    lin = workloads.LLAMA3_8B[idx]
    sw, sx = synthetic.seeds("llama3_8b_decode", idx)
    q, s, z = quantized_fmt(lin.N, lin.K, sw, group, asym)
    x16 = acts(1, lin.K, sx)
    y = run_fmt(x16, q, s, z, group)
    rows = sample_rows(lin.N, 256, sw)
    assert_close(y[:, rows], oracle.gemm_rows(x16, q, s, rows, group, zeros=z),
                 f"{lin.name} g={group} asym={asym}")


def test_group128_symmetric_is_the_default_gemm(w4lib):
    q, s, _ = quantized_fmt(512, 1024, 310, 128, False)
    x = from_bits16(acts(3, 1024, 311))
    r = w4.repack(u8(q))
    st = from_bits16(s)
    assert torch.equal(w4.gemm_ex(x, r, st, None, 128), w4.gemm(x, r, st))


def test_shape_beyond_the_gemv_runs_on_tensor_cores(w4lib):
    """M = 16 with K = 14336: x[16, K] does not fit beside the GEMV's ring, so
    the call takes the tensor-core GEMM; every output compared."""
    N, K, M = 256, 14336, 16
    assert w4.gemm_ex_plan(M, N, K, 32, True)["path"] == "tensor_core"
    q, s, z = quantized_fmt(N, K, 312, 32, True)
    x16 = acts(M, K, 313)
    assert_close(run_fmt(x16, q, s, z, 32), oracle.gemm(x16, q, s, 32, zeros=z), "M=16 K=14336")
    assert w4.device_status() == 0


# --------------------------------------------------------------------------
# Prefill (M > 16): the tcgen05 GEMM with the variants' dequantisers
# --------------------------------------------------------------------------

@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("M,N,K", [(20, 1000, 1152), (200, 4136, 384), (300, 2000, 2048)])
def test_formats_prefill_every_output(w4lib, M, N, K, group, asym):
    assert w4.gemm_ex_plan(M, N, K, group, asym)["path"] == "tensor_core"
    q, s, z = quantized_fmt(N, K, 500 + M, group, asym)
    x16 = acts(M, K, 501 + M)
    assert_close(run_fmt(x16, q, s, z, group), oracle.gemm(x16, q, s, group, zeros=z),
                 f"prefill M={M} N={N} K={K} g={group} asym={asym}")
    assert w4.device_status() == 0


@pytest.mark.parametrize("group,asym", [(32, True), (w4.PER_CHANNEL, False), (64, False)])
def test_formats_prefill_launch_shapes(w4lib, group, asym):
    """One CTA per 128 x 128 tile, CTA pairs (2-CTA MMAs, an odd last block),
    and pairs splitting K through the cluster, with ragged M: every output
    compared, and two calls of a split launch give the same bits."""
    seen = set()
    for M, N, K in [(20, 1000, 1152), (200, 19300, 256), (300, 19000, 384), (300, 8000, 1920),
                    (300, 4000, 16384), (300, 1000, 18944)]:
        plan = w4.gemm_ex_plan(M, N, K, group, asym)
        assert plan["path"] == "tensor_core", plan
        seen.add(plan["splits"])
        q, s, z = quantized_fmt(N, K, 600, group, asym)
        x16 = acts(M, K, 601)
        r = w4.repack(u8(q))
        st, zt = from_bits16(s), (u8(z) if z is not None else None)
        x = from_bits16(x16)
        y1 = w4.gemm_ex(x, r, st, zt, group)
        y2 = w4.gemm_ex(x, r, st, zt, group)
        torch.cuda.synchronize()
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
        assert_close(y1.float().cpu().numpy().astype(np.float64),
                     oracle.gemm(x16, q, s, group, zeros=z), f"M={M} N={N} K={K} {plan}")
        del r, st, zt, x, y1, y2
    assert {1, 2} <= seen and seen & {4, 6, 8}, seen
    assert w4.device_status() == 0


@pytest.mark.parametrize("M,N,K,group,asym", [
    (17, 1, 128, 32, True),                    # one weight row, one k-block pair
    (129, 130, 32768, w4.PER_CHANNEL, True),   # the largest K, per-channel zero points
    (130, 257, 32768, 32, False),              # the largest K at group 32 (1024 groups a row)
    (1500, 384, 256, 64, True),                # many x tiles, few k-blocks
])
def test_formats_prefill_edges(w4lib, M, N, K, group, asym):
    q, s, z = quantized_fmt(N, K, 700 + N, group, asym)
    x16 = acts(M, K, 701)
    assert_close(run_fmt(x16, q, s, z, group), oracle.gemm(x16, q, s, group, zeros=z),
                 f"edge M={M} N={N} K={K} g={group} asym={asym}")
    assert w4.device_status() == 0


@pytest.mark.parametrize("idx", range(len(workloads.PREFILL)))
def test_formats_prefill_full_size(w4lib, idx):
    """M = 512 prompt pass on the prefill shapes with group-32 asymmetric
    codes; oracle on sampled rows."""
    lin = workloads.PREFILL[idx]
    sw, sx = synthetic.seeds("prefill", idx)
    q, s, z = quantized_fmt(lin.N, lin.K, sw, 32, True)
    x16 = acts(workloads.PREFILL_M, lin.K, sx)
    y = run_fmt(x16, q, s, z, 32)
    rows = sample_rows(lin.N, 96, sw)
    assert_close(y[:, rows], oracle.gemm_rows(x16, q, s, rows, 32, zeros=z), lin.name)


# --------------------------------------------------------------------------
# AWQ activation scale in the prologue: y = fp16(x * alpha) @ dequant(Q(W / alpha))^T
# --------------------------------------------------------------------------

def _awq_case(N, K, seed, group, asym):
    """Weights divided by a per-input-channel alpha before quantization (the
    AWQ transform, done here in numpy), alpha in [0.5, 2]."""
    rng = np.random.default_rng(seed)
    alpha = rng.uniform(0.5, 2.0, K).astype(np.float16)
    w = synthetic.master_weight(N, K, seed).float().numpy()
    w16 = (w / alpha.astype(np.float32)).astype(np.float16).view(np.uint16)
    if asym:
        q, s, z = oracle.quantize_asym(w16, group)
    else:
        (q, s), z = oracle.quantize(w16, group), None
    return alpha.view(np.uint16), q, s, z


@pytest.mark.parametrize("group,asym", [(128, False), (128, True), (32, True), (w4.PER_CHANNEL, False)])
@pytest.mark.parametrize("M", [1, 7, 16, 40, 200, 300])
def test_awq_activation_scale(w4lib, M, group, asym):
    """Decode (M <= 16) and prefill: one CTA per tile (40), CTA pairs (200),
    pairs with two x tiles splitting K (300)."""
    N, K = 1000, 2048
    alpha16, q, s, z = _awq_case(N, K, 400, group, asym)
    x16 = acts(M, K, 401 + M)
    r = w4.repack(u8(q))
    y = w4.gemm_ex(from_bits16(x16), r, from_bits16(s), u8(z) if z is not None else None, group,
                   alpha=from_bits16(alpha16))
    torch.cuda.synchronize()
    y_ref = oracle.gemm(oracle.scale_activations(x16, alpha16), q, s, group, zeros=z)
    assert_close(y.float().cpu().numpy(), y_ref, f"awq g={group} asym={asym} M={M}")


def test_awq_llama3_8b_gate_up_m1(w4lib):
    lin = workloads.LLAMA3_8B[2]
    sw, sx = synthetic.seeds("llama3_8b_decode", 2)
    alpha16, q, s, z = _awq_case(lin.N, lin.K, sw, 128, False)
    x16 = acts(1, lin.K, sx)
    y = w4.gemm_ex(from_bits16(x16), w4.repack(u8(q)), from_bits16(s), None, 128,
                   alpha=from_bits16(alpha16))
    torch.cuda.synchronize()
    rows = sample_rows(lin.N, 256, sw)
    y_ref = oracle.gemm_rows(oracle.scale_activations(x16, alpha16), q, s, rows, 128)
    assert_close(y[:, rows].float().cpu().numpy(), y_ref, "awq gate_up")


def _fuzz_cases():
    """Seeded format calls across the unit plans (16/32/64-row units, 2- to
    6-stage rings, group-blocked and row-major slabs) and, for M > 16, the
    tensor-core path; ragged N, every group size."""
    rng = np.random.default_rng(20261205)
    groups = [32, 64, 128, w4.PER_CHANNEL]
    cases = []
    for _ in range(16):
        M = int(rng.choice([1, 2, 3, 4, 7, 8, 9, 13, 16, 40, 300]))
        group = int(rng.choice(groups))
        asym = bool(rng.integers(0, 2))
        K = 128 * int(rng.integers(1, 48))
        N = int(rng.integers(100, max(200, min(60000, 30_000_000 // K))))
        cases.append((M, N, K, group, asym))
    return cases


@pytest.mark.parametrize("M,N,K,group,asym", _fuzz_cases())
def test_formats_plans_fuzz(w4lib, M, N, K, group, asym):
    """Whatever launch a format call gets: no wait times out, sampled rows
    meet the bar, and a repeat call is bit-identical."""
    q, s, z = quantized_fmt.__wrapped__(N, K, 310, group, asym)
    x16 = acts.__wrapped__(M, K, 311 + M)
    r = w4.repack(u8(q))
    st = from_bits16(s)
    zt = u8(z) if z is not None else None
    x = from_bits16(x16)
    w4.device_status()  # clear
    y1 = w4.gemm_ex(x, r, st, zt, group)
    y2 = w4.gemm_ex(x, r, st, zt, group)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    y = y1.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y2.float().cpu().numpy().astype(np.float64))
    rows = sample_rows(N, 96, 312)
    y_ref = oracle.gemm_rows(x16, q, s, rows, group, zeros=z)
    assert_close(y[:, rows], y_ref, f"g={group} asym={asym} M={M} N={N} K={K}")
