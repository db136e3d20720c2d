"""GB300 (sm_103a) W4A16 weight-only INT4 GEMV/GEMM behind a C ABI.

The CUDA library is ``libw4a16.so`` (sources in ``csrc/``, ABI in
``include/w4a16.h``); ``ops`` wraps it for torch tensors.  Importing this
package does not load the library; the first call does, and fails loudly if
it has not been built.
"""
from .ops import (GROUP, PER_CHANNEL, W4A16Linear, device_status, gemm, gemm_ex, gemm_ex_plan,
                  gemm_plan, gemm_plan_tail, gemm_q4_0, gemm_w8, quantize, quantize_ex, quantize_q4_0, quantize_w8, repack,
                  repacked_bytes, selftest_wait_timeout, set_wait_timeout_ns, unrepack)

__all__ = ["GROUP", "PER_CHANNEL", "W4A16Linear", "device_status", "gemm", "gemm_ex", "gemm_ex_plan",
           "gemm_plan", "gemm_plan_tail", "gemm_q4_0", "gemm_w8", "quantize", "quantize_ex", "quantize_q4_0", "quantize_w8",
           "repack",
           "repacked_bytes", "selftest_wait_timeout", "set_wait_timeout_ns", "unrepack"]
