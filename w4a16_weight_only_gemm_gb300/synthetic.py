"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module draws random numbers and nothing else: it holds none of the
quantizer's or the GEMM's arithmetic, so both the CUDA path and the CPU oracle
can be fed from it without sharing any of the method.

Distributions stand in for the decode workloads of the W4A16 benchmark report
(mhpq.cn, §一: LLaMA-3-8B and Qwen-2.5-7B, prompt 512, decode 512 tokens);
no model weights or datasets are used:

* master weights ``W = 0.02 * N(0, 1)`` in fp32, with an independent
  Bernoulli(0.001) outlier mask (second generator, seed + 1) whose entries are
  multiplied by 20, then rounded to fp16;
* activations ``x = N(0, 1)`` in fp32 rounded to fp16.

CPU generation (``device="cpu"``) is bit-reproducible on any host and is what
the parity tests use.  ``device="cuda"`` draws the same distributions from the
CUDA generator (different numbers, same law) for the large benchmark stack.
"""
from __future__ import annotations

import torch

WEIGHT_STD = 0.02
OUTLIER_PROB = 0.001
OUTLIER_GAIN = 20.0


def master_weight(N: int, K: int, seed: int, device: str = "cpu") -> torch.Tensor:
    """fp16 [N, K] master weight matrix (rows = out_features)."""
    g = torch.Generator(device=device).manual_seed(seed)
    w = torch.randn(N, K, generator=g, dtype=torch.float32, device=device)
    w.mul_(WEIGHT_STD)
    g2 = torch.Generator(device=device).manual_seed(seed + 1)
    mask = torch.rand(N, K, generator=g2, dtype=torch.float32, device=device) < OUTLIER_PROB
    w = torch.where(mask, w * OUTLIER_GAIN, w)
    return w.half()


def activations(M: int, K: int, seed: int, device: str = "cpu") -> torch.Tensor:
    """fp16 [M, K] activations ~ N(0, 1)."""
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(M, K, generator=g, dtype=torch.float32, device=device).half()


# Activation laws with a large common offset, as real decode activations have
# (they are not zero-mean): the group sums of x are then far from 0.
OFFSET_KINDS = ("shift4", "abs3", "big_group")


def activations_offset(M: int, K: int, seed: int, kind: str, device: str = "cpu") -> torch.Tensor:
    """fp16 [M, K] activations with a common offset:

    * ``shift4``: 4 + N(0, 1);
    * ``abs3``: |N(0, 3)| (all positive, like the output of a SiLU gate);
    * ``big_group``: N(0, 1) with the first 128 values of every row set to
      60000 / 128 = 468.75 (one group summing to 60000, still finite in fp16).
    """
    g = torch.Generator(device=device).manual_seed(seed)
    z = torch.randn(M, K, generator=g, dtype=torch.float32, device=device)
    if kind == "shift4":
        x = z + 4.0
    elif kind == "abs3":
        x = (z * 3.0).abs()
    elif kind == "big_group":
        x = z.clone()
        x[:, :128] = 60000.0 / 128.0
    else:
        raise ValueError(f"unknown activation kind {kind!r}")
    return x.half()


# Base seed of each workload; tensor i of a workload uses seed_W = base + 10*i
# and seed_x = seed_W + 2.  The single 4096x4096 GEMV uses (0, 2).
WORKLOAD_SEED_BASE = {
    "gemv_4096": None,
    "llama3_8b_decode": 1000,
    "stack_8b": 2000,
    "decode_sweep": 3000,
    "prefill": 4000,
}


def seeds(workload: str, tensor_index: int = 0) -> tuple[int, int]:
    """(seed_W, seed_x) for tensor ``tensor_index`` of the named workload."""
    base = WORKLOAD_SEED_BASE[workload]
    if base is None:
        return 0, 2
    sw = base + 10 * tensor_index
    return sw, sw + 2
