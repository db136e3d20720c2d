"""Python entry points over the C ABI, for torch tensors.

Each function validates shapes/dtypes, allocates outputs with torch (device
memory is torch's), and calls the library on the current CUDA stream.  No
arithmetic of the method happens here.
"""
from __future__ import annotations

import ctypes
import functools

import torch

from . import _native

GROUP = 128


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, device: torch.device | None = None) -> int:
    """The cudaStream_t of `stream`, else of the current stream of `device`
    (the raw-handle query costs a fraction of building a Stream object: a
    decode call is a few microseconds of host time)."""
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_stream is not None and device is not None and device.index is not None:
        return int(_raw_stream(device.index))
    return int(torch.cuda.current_stream().cuda_stream)


def _device_of(stream, *named) -> torch.device:
    """The one device of the named tensors (None entries skipped), checked to
    be shared by all of them and by an explicit `stream`; the library launches
    on the current device, so a mix would hand it foreign pointers."""
    dev = None
    for name, t in named:
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other operands on {dev}")
    if stream is not None and dev is not None and getattr(stream, "device", dev) != dev:
        raise ValueError(f"stream is on {stream.device}, the operands on {dev}")
    return dev


def _call(dev: torch.device, fn, *args) -> int:
    """fn(*args) with `dev` the current CUDA device (switched only when it is
    not already current: the common case costs one device query)."""
    idx = dev.index
    if idx is None or idx == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(idx):
        return fn(*args)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def quantize(W: torch.Tensor, group: int = GROUP, stream=None):
    """W fp16 [N, K] -> (qweight uint8 [N, K/2], scales fp16 [N, K/128])."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    dev = _device_of(stream, ("W", W))
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((N, K // GROUP), dtype=torch.float16, device=dev)
    rc = _call(dev, _native.lib().w4a16_quantize, W.data_ptr(), N, K, group, q.data_ptr(),
               s.data_ptr(), _stream_ptr(stream, dev))
    _native.check(rc, "w4a16_quantize")
    return q, s


PER_CHANNEL = -1


def quantize_ex(W: torch.Tensor, group: int = GROUP, asymmetric: bool = False, stream=None):
    """Format variants: W fp16 [N, K] -> (qweight uint8 [N, K/2], scales fp16
    [N, K/g], zeros uint8 [N, K/g] or None), g = group (32, 64, 128) or K for
    PER_CHANNEL; asymmetric codes hold q in [0, 15] with a zero point per group."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    g = K if group == PER_CHANNEL else group
    if g <= 0 or K % g:
        raise ValueError(f"K={K} is not a multiple of group={group}")
    dev = _device_of(stream, ("W", W))
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((N, K // g), dtype=torch.float16, device=dev)
    z = torch.empty((N, K // g), dtype=torch.uint8, device=dev) if asymmetric else None
    rc = _call(dev, _native.lib().w4a16_quantize_ex, W.data_ptr(), N, K, group, int(asymmetric),
               q.data_ptr(), s.data_ptr(), z.data_ptr() if asymmetric else None,
               _stream_ptr(stream, dev))
    _native.check(rc, "w4a16_quantize_ex")
    return q, s, z


@functools.lru_cache(maxsize=1024)
def repacked_bytes(N: int, K: int) -> int:
    n = _native.lib().w4a16_repacked_bytes(N, K)
    if n < 0:
        raise ValueError(f"unsupported shape N={N} K={K}")
    return int(n)


def repack(qweight: torch.Tensor, stream=None) -> torch.Tensor:
    """Canonical [N, K/2] packed bytes -> kernel-layout bytes (1-D uint8)."""
    _need(qweight, torch.uint8, "qweight")
    N, K2 = qweight.shape
    dev = _device_of(stream, ("qweight", qweight))
    out = torch.empty(repacked_bytes(N, 2 * K2), dtype=torch.uint8, device=dev)
    rc = _call(dev, _native.lib().w4a16_repack, qweight.data_ptr(), N, 2 * K2, out.data_ptr(),
               _stream_ptr(stream, dev))
    _native.check(rc, "w4a16_repack")
    return out


def unrepack(repacked: torch.Tensor, N: int, K: int, stream=None) -> torch.Tensor:
    """Kernel-layout bytes -> canonical [N, K/2] packed bytes."""
    _need(repacked, torch.uint8, "repacked")
    if repacked.numel() != repacked_bytes(N, K):
        raise ValueError("repacked buffer size does not match N, K")
    dev = _device_of(stream, ("repacked", repacked))
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    rc = _call(dev, _native.lib().w4a16_unrepack, repacked.data_ptr(), N, K, q.data_ptr(),
               _stream_ptr(stream, dev))
    _native.check(rc, "w4a16_unrepack")
    return q


def _out_tensor(out: torch.Tensor | None, M: int, N: int, device) -> torch.Tensor:
    """`out` checked to be a contiguous fp16 CUDA [M, N] tensor (the kernels
    write exactly M x N halves there), or a new one."""
    if out is None:
        return torch.empty((M, N), dtype=torch.float16, device=device)
    _need(out, torch.float16, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out must be [{M}, {N}], got {tuple(out.shape)}")
    return out


def _check_weights(repacked: torch.Tensor, scales: torch.Tensor) -> tuple[int, int]:
    _need(repacked, torch.uint8, "repacked")
    _need(scales, torch.float16, "scales")
    N, G = scales.shape
    if repacked.numel() != repacked_bytes(N, G * GROUP):
        raise ValueError("repacked buffer size does not match the scales' N, K")
    return N, G * GROUP


def _gemm(x: torch.Tensor, repacked: torch.Tensor, scales: torch.Tensor, N: int, K: int,
          out: torch.Tensor | None, stream) -> torch.Tensor:
    _need(x, torch.float16, "x")
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError(f"x must be [M, {K}]")
    dev = _device_of(stream, ("x", x), ("repacked", repacked), ("scales", scales), ("out", out))
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _need(out, torch.float16, "out")
        if tuple(out.shape) != (M, N):
            raise ValueError("out has the wrong shape")
    rc = _call(dev, _native.lib().w4a16_gemm, x.data_ptr(), repacked.data_ptr(), scales.data_ptr(),
               out.data_ptr(), M, N, K, _stream_ptr(stream, dev))
    if rc:
        _native.check(rc, "w4a16_gemm")
    return out


def gemm(x: torch.Tensor, repacked: torch.Tensor, scales: torch.Tensor,
         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ dequant(W)^T; W given as kernel-layout bytes + scales [N, K/128]."""
    N, K = _check_weights(repacked, scales)
    return _gemm(x, repacked, scales, N, K, out, stream)


def gemm_ex(x: torch.Tensor, repacked: torch.Tensor, scales: torch.Tensor,
            zeros: torch.Tensor | None = None, group: int = GROUP,
            out: torch.Tensor | None = None, stream=None,
            alpha: torch.Tensor | None = None) -> torch.Tensor:
    """y = x~ @ dequant(W)^T for the format variants of quantize_ex: scales
    [N, K/g] fp16, zeros [N, K/g] uint8 (asymmetric) or None, g = group or K
    for PER_CHANNEL; x~ = x, or fp16(x * alpha) with an AWQ activation scale
    alpha [K] fp16."""
    _need(x, torch.float16, "x")
    if alpha is not None:
        _need(alpha, torch.float16, "alpha")
        if alpha.shape != (x.shape[-1],):
            raise ValueError("alpha must be [K]")
    _need(repacked, torch.uint8, "repacked")
    _need(scales, torch.float16, "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, "zeros")
        if zeros.shape != scales.shape:
            raise ValueError("zeros and scales differ in shape")
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    N = scales.shape[0]
    g = K if group == PER_CHANNEL else group
    if g <= 0 or K % g or scales.shape[1] != K // g:
        raise ValueError(f"scales must be [N, {K}/{g}]")
    if repacked.numel() != repacked_bytes(N, K):
        raise ValueError("repacked buffer size does not match N, K")
    dev = _device_of(stream, ("x", x), ("alpha", alpha), ("repacked", repacked),
                     ("scales", scales), ("zeros", zeros), ("out", out))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _need(out, torch.float16, "out")
        if tuple(out.shape) != (M, N):
            raise ValueError("out has the wrong shape")
    rc = _call(dev, _native.lib().w4a16_gemm_ex, x.data_ptr(),
               alpha.data_ptr() if alpha is not None else None, repacked.data_ptr(),
               scales.data_ptr(), zeros.data_ptr() if zeros is not None else None,
               out.data_ptr(), M, N, K, group, _stream_ptr(stream, dev))
    _native.check(rc, "w4a16_gemm_ex")
    return out


def quantize_q4_0(W: torch.Tensor, stream=None) -> torch.Tensor:
    """W fp16 [N, K] -> GGUF Q4_0 blocks uint8 [N, K/32 * 18] (K % 256 == 0)."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    dev = _device_of(stream, ("W", W))
    blocks = torch.empty((N, K // 32 * 18), dtype=torch.uint8, device=dev)
    _native.check(_call(dev, _native.lib().w4a16_quantize_q4_0, W.data_ptr(), N, K,
                        blocks.data_ptr(), _stream_ptr(stream, dev)), "w4a16_quantize_q4_0")
    return blocks


def gemm_q4_0(x: torch.Tensor, blocks: torch.Tensor, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ decode(blocks)^T for GGUF Q4_0 blocks [N, K/32 * 18], M <= 16."""
    _need(x, torch.float16, "x")
    _need(blocks, torch.uint8, "blocks")
    N = blocks.shape[0]
    K = x.shape[-1]
    if x.dim() != 2 or blocks.shape[1] != K // 32 * 18:
        raise ValueError(f"x must be [M, K] and blocks [N, K/32*18]")
    M = x.shape[0]
    dev = _device_of(stream, ("x", x), ("blocks", blocks), ("out", out))
    out = _out_tensor(out, M, N, dev)
    _native.check(_call(dev, _native.lib().w4a16_gemm_q4_0, x.data_ptr(), blocks.data_ptr(),
                        out.data_ptr(), M, N, K, _stream_ptr(stream, dev)), "w4a16_gemm_q4_0")
    return out


def quantize_w8(W: torch.Tensor, stream=None):
    """W8A16: W fp16 [N, K] -> (codes uint8 [N, K] holding q + 128, scales fp16 [N])."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    dev = _device_of(stream, ("W", W))
    codes = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s = torch.empty((N,), dtype=torch.float16, device=dev)
    _native.check(_call(dev, _native.lib().w4a16_quantize_w8, W.data_ptr(), N, K, codes.data_ptr(),
                        s.data_ptr(), _stream_ptr(stream, dev)), "w4a16_quantize_w8")
    return codes, s


def gemm_w8(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """W8A16 GEMV: y[M, N] = x[M, K] @ ((codes - 128) * scales[:, None])^T, M <= 16."""
    _need(x, torch.float16, "x")
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float16, "scales")
    N, K = codes.shape
    if x.dim() != 2 or x.shape[1] != K or scales.shape != (N,):
        raise ValueError(f"x must be [M, {K}] and scales [{N}]")
    M = x.shape[0]
    dev = _device_of(stream, ("x", x), ("codes", codes), ("scales", scales), ("out", out))
    out = _out_tensor(out, M, N, dev)
    _native.check(_call(dev, _native.lib().w4a16_gemm_w8, x.data_ptr(), codes.data_ptr(),
                        scales.data_ptr(), out.data_ptr(), M, N, K, _stream_ptr(stream, dev)),
                  "w4a16_gemm_w8")
    return out


def gemm_plan(M: int, N: int, K: int) -> dict:
    """The launch gemm() makes for (M, N, K) on the current device:
    {"path": "gemv" | "tensor_core", "splits", "ctas", "blocks_per_cta", "rows_per_cta"}."""
    out = [ctypes.c_int(0) for _ in range(5)]
    _native.check(_native.lib().w4a16_gemm_plan(int(M), int(N), int(K),
                                                *[ctypes.byref(o) for o in out]),
                  "w4a16_gemm_plan")
    path = {1: "gemv", 2: "tensor_core"}[out[0].value]
    return {"path": path, "splits": out[1].value, "ctas": out[2].value,
            "blocks_per_cta": out[3].value, "rows_per_cta": out[4].value}


def gemm_plan_tail(M: int, N: int, K: int) -> dict:
    """The partial last round of a persistent decode launch for (M, N, K):
    {"tail_rows": rows per tail unit (0: no such round), "tail_units": count}."""
    out = [ctypes.c_int(0) for _ in range(2)]
    _native.check(_native.lib().w4a16_gemm_plan_tail(int(M), int(N), int(K),
                                                     *[ctypes.byref(o) for o in out]),
                  "w4a16_gemm_plan_tail")
    return {"tail_rows": out[0].value, "tail_units": out[1].value}


def gemm_ex_plan(M: int, N: int, K: int, group: int, asymmetric: bool = False,
                 alpha: bool = False) -> dict:
    """The launch gemm_ex() makes for (M, N, K) with this group, zero points
    (asymmetric) and AWQ scale (alpha): {"path": "gemv" | "tensor_core",
    "splits", "ctas", "rows_per_cta"}."""
    out = [ctypes.c_int(0) for _ in range(4)]
    _native.check(_native.lib().w4a16_gemm_ex_plan(int(M), int(N), int(K), int(group),
                                                   int(bool(asymmetric)), int(bool(alpha)),
                                                   *[ctypes.byref(o) for o in out]),
                  "w4a16_gemm_ex_plan")
    path = {1: "gemv", 2: "tensor_core"}[out[0].value]
    return {"path": path, "splits": out[1].value, "ctas": out[2].value,
            "rows_per_cta": out[3].value}


def device_status() -> int:
    """Synchronise and return (and clear) the kernels' recorded status code."""
    st = ctypes.c_int(0)
    _native.check(_native.lib().w4a16_device_status(ctypes.byref(st)), "w4a16_device_status")
    return st.value


def set_wait_timeout_ns(ns: int) -> None:
    _native.lib().w4a16_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    rc = _native.lib().w4a16_selftest_wait_timeout(int(timeout_ns), _stream_ptr(stream))
    _native.check(rc, "w4a16_selftest_wait_timeout")


class W4A16Linear:
    """A quantized linear layer y = x W^T held as kernel-layout weights + scales."""

    def __init__(self, W: torch.Tensor):
        self.N, self.K = W.shape
        q, self.scales = quantize(W)
        self.repacked = repack(q)

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
        # the weights were checked when they were made: only x / out here
        return _gemm(x, self.repacked, self.scales, self.N, self.K, out, stream)
