"""Seeded inputs and oracle results for the GPU parity tests (cached per
session).  Inputs come from the shared synthetic generators; expected values
come only from the CPU oracle."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from gpu_util import bits16
from w4a16_weight_only_gemm_gb300 import synthetic


@functools.lru_cache(maxsize=64)
def quantized(N: int, K: int, seed: int):
    """(W16 bits, qweight, scales bits) for a synthetic master weight; oracle-quantized."""
    W = synthetic.master_weight(N, K, seed)
    w16 = bits16(W)
    q, s = oracle.quantize(w16)
    return w16, q, s


@functools.lru_cache(maxsize=32)
def acts(M: int, K: int, seed: int) -> np.ndarray:
    return bits16(synthetic.activations(M, K, seed))


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(count, N), replace=False).tolist())
    rows |= {0, N - 1, min(N - 1, 127), min(N - 1, 128)}
    return np.array(sorted(rows), dtype=np.int64)


def as_device(q: np.ndarray, s: np.ndarray):
    qt = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    st = torch.from_numpy(np.ascontiguousarray(s).view(np.int16)).view(torch.float16).cuda()
    return qt, st
