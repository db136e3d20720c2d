"""Repack: a bijective re-layout.  Checked by round trip (byte-identical) and
against the layout documented in include/w4a16.h written out in numpy."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import w4a16_weight_only_gemm_gb300 as w4

pytestmark = pytest.mark.gpu


def documented_layout(q: np.ndarray, N: int, K: int) -> np.ndarray:
    """Kernel layout per the header: ((b*(K/64) + c)*8 + i)*512 + 16*L, word s
    nibble positions (r0,k') (r1,k') (r0,k'+2) (r1,k'+2) (r0,k'+1) (r1,k'+1)
    (r0,k'+3) (r1,k'+3), padding rows hold nibble 8."""
    Npad = -(-N // 128) * 128
    nib = np.full((Npad, K), 8, dtype=np.uint32)
    nib[:N, 0::2] = q & 0xF
    nib[:N, 1::2] = q >> 4
    out = np.zeros(Npad * K // 8, dtype=np.uint32)   # 32-bit words
    C = K // 64
    for b in range(Npad // 128):
        for c in range(C):
            for i in range(8):
                for L in range(32):
                    g, t = L // 4, L % 4
                    r0, r1 = b * 128 + i * 16 + g, b * 128 + i * 16 + g + 8
                    for s in range(4):
                        k = c * 64 + 16 * t + 4 * s
                        order = [(r0, k), (r1, k), (r0, k + 2), (r1, k + 2),
                                 (r0, k + 1), (r1, k + 1), (r0, k + 3), (r1, k + 3)]
                        word = 0
                        for p, (r, kk) in enumerate(order):
                            word |= int(nib[r, kk]) << (4 * p)
                        out[(((b * C + c) * 8 + i) * 512 + 16 * L) // 4 + s] = word
    return out.view(np.uint8)


@pytest.mark.parametrize("N,K", [(1, 128), (100, 256), (130, 384), (256, 1024), (4168, 4096)])
def test_round_trip(w4lib, N, K):
    rng = np.random.default_rng(N + K)
    q = torch.from_numpy(rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)).cuda()
    r = w4.repack(q)
    assert r.numel() == w4.repacked_bytes(N, K)
    back = w4.unrepack(r, N, K)
    assert torch.equal(back, q)


@pytest.mark.parametrize("N,K", [(16, 128), (130, 256)])
def test_matches_documented_layout(w4lib, N, K):
    rng = np.random.default_rng(3)
    q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    r = w4.repack(torch.from_numpy(q).cuda()).cpu().numpy()
    assert np.array_equal(r, documented_layout(q, N, K))
