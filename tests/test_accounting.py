"""Byte accounting of the path against the pages' own figures.

* W4A16 benchmark report (mhpq.cn) §二: weight memory of a 7-8B model is
  14.8 GB in FP16 and 3.9 GB in W4A16; §三: arithmetic intensity is below
  0.5 "FLOP/Byte" for FP16 and about 2.0 for W4A16 (the figures match if one
  fused multiply-add is counted as one operation).
* qaqbuyan.com quantization tutorial, "量化的数学基石" §3: one fp16 scale
  per 128 INT4 weights costs 2 / 64 bytes = 3.1 % extra storage.
"""
from __future__ import annotations

from w4a16_weight_only_gemm_gb300 import workloads as wl


def _stack_weights() -> int:
    return sum(lin.N * lin.K for lin in wl.stack_8b())


def test_stack_weight_count():
    # 32 x (6144 + 4096 + 28672) x 4096 + 32 x 4096 x 14336 + 128256 x 4096
    assert _stack_weights() == 7_504_658_432


def test_fp16_bytes_match_report():
    fp16 = 2 * _stack_weights()
    assert abs(fp16 / 14.8e9 - 1) < 0.015          # 15.01 GB vs 14.8 GB


def test_w4a16_bytes_match_report():
    w4 = sum(wl.algorithmic_bytes(1, l.N, l.K) - 2 * l.K - 2 * l.N for l in wl.stack_8b())
    assert w4 == 3_752_329_216 + 117_260_288       # packed nibbles + fp16 scales
    assert abs(w4 / 3.9e9 - 1) < 0.01              # 3.874 GB vs 3.9 GB
    assert sum(wl.algorithmic_bytes(1, l.N, l.K) for l in wl.stack_8b()) == 3_874_310_656


def test_scale_overhead_matches_tutorial():
    N, K = 4096, 4096
    packed, scales = N * K // 2, 2 * N * (K // 128)
    assert scales / packed == 2 / 64               # 3.125 % ~ "3.1 %"


def test_intensity_matches_report():
    N, K = 4096, 4096
    fma = N * K
    w4 = wl.algorithmic_bytes(1, N, K)
    fp16 = 2 * N * K + 2 * K + 2 * N
    assert 1.9 < fma / w4 < 2.0                    # ~2.0 "FLOP/B" (FMA counted once)
    assert fma / fp16 <= 0.5                       # "< 0.5" for FP16


def test_single_gemv_bytes():
    assert wl.algorithmic_bytes(1, 4096, 4096) == 8_667_136
