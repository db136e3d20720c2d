"""Failure detection without faulting the GPU: a kernel waits on an mbarrier
that nothing arrives on, gives up after a short bound, records a time-out in
the device status word and exits normally; the context stays usable."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, from_bits16
from parity_data import acts, as_device, quantized
import w4a16_weight_only_gemm_gb300 as w4

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout(w4lib):
    assert w4.device_status() == 0
    w4.selftest_wait_timeout(2_000_000)          # 2 ms
    assert w4.device_status() == 5               # W4A16_ERR_TIMEOUT
    assert w4.device_status() == 0               # read clears it


def test_context_usable_after_timeout(w4lib):
    w4.selftest_wait_timeout(1_000_000)
    assert w4.device_status() == 5
    w16, q, s = quantized(256, 512, 51)
    x16 = acts(2, 512, 52)
    qt, st = as_device(q, s)
    y = w4.gemm(from_bits16(x16), w4.repack(qt), st)
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), oracle.gemm(x16, q, s), "after timeout")
    assert w4.device_status() == 0


def test_shape_errors_raise(w4lib):
    from w4a16_weight_only_gemm_gb300._native import W4A16Error
    with pytest.raises(W4A16Error) as e:
        w4.quantize(torch.zeros(4, 200, dtype=torch.float16, device="cuda"))
    assert e.value.code == 2
