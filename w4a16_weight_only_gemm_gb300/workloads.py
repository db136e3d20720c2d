"""Workload shapes and byte accounting for the W4A16 decode/prefill path.

Shapes follow the models named by the W4A16 benchmark report (mhpq.cn, §一:
LLaMA-3-8B and Qwen-2.5-7B, prompt 512).  Byte accounting follows the same
report's §二 memory table (FP16 vs W4A16 weight bytes) and the per-group
scale overhead of the qaqbuyan.com quantization tutorial ("量化的数学基石" §3:
2 bytes of fp16 scale per 128 INT4 weights).
"""
from __future__ import annotations

from dataclasses import dataclass

@dataclass(frozen=True)
class Linear:
    """One linear layer y[M, N] = x[M, K] W[N, K]^T."""
    name: str
    N: int
    K: int


# Llama-3-8B decode linear shapes: hidden 4096, intermediate 14336,
# 32 query heads and 8 KV heads of 128, vocabulary 128256, 32 layers.
LLAMA3_8B = (
    Linear("qkv", 6144, 4096),
    Linear("o_proj", 4096, 4096),
    Linear("gate_up", 28672, 4096),
    Linear("down", 4096, 14336),
    Linear("lm_head", 128256, 4096),
)
LLAMA3_8B_LAYERS = 32

# Qwen-2.5-7B linear shapes from hidden 3584 and intermediate 18944
# (28 query heads, 4 KV heads of 128).
QWEN25_7B = (
    Linear("qkv", 4608, 3584),
    Linear("o_proj", 3584, 3584),
    Linear("gate_up", 37888, 3584),
    Linear("down", 3584, 18944),
)

SINGLE_GEMV = Linear("gemv_4096", 4096, 4096)
PREFILL_M = 512
PREFILL = (
    Linear("prefill_up", 14336, 4096),
    Linear("prefill_down", 4096, 14336),
)
QUANTIZER_SHAPE = (14336, 4096)
DECODE_SWEEP_M = (2, 4, 8, 16)


def stack_8b() -> list[Linear]:
    """The 129 GEMVs of one decode token of the 8B linear stack."""
    layers = [lin for _ in range(LLAMA3_8B_LAYERS) for lin in LLAMA3_8B[:4]]
    return layers + [LLAMA3_8B[4]]


def algorithmic_bytes(M: int, N: int, K: int, group: int = 128, zero_points: bool = False) -> int:
    """Bytes one call must move: packed weights + fp16 scales (+ one byte of
    zero point per group) + x + y.  group = -1: one group per row."""
    g = K if group == -1 else group
    return N * K // 2 + (3 if zero_points else 2) * N * (K // g) + 2 * M * K + 2 * M * N
