"""Helpers shared by the GPU parity tests (conversion and tolerance checks)."""
from __future__ import annotations

import numpy as np
import torch

# Acceptance bars for floating-point outputs against the exact (binary64)
# oracle: max-abs error relative to max |y_ref|, and relative L2 error.
MAX_REL = 2e-3
L2_REL = 1e-3


def bits16(t: torch.Tensor) -> np.ndarray:
    """fp16 tensor -> uint16 bit patterns (numpy, CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).to(device)


def u8(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def assert_close(y: np.ndarray, y_ref: np.ndarray, what: str = "") -> tuple[float, float]:
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    denom = np.abs(y_ref).max()
    max_rel = float(err.max() / denom) if denom > 0 else float(err.max())
    l2 = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300))
    assert max_rel <= MAX_REL, f"{what}: max rel err {max_rel:.3e} > {MAX_REL}"
    assert l2 <= L2_REL, f"{what}: L2 rel err {l2:.3e} > {L2_REL}"
    return max_rel, l2
