"""GB300 (sm_103a) fused linear cross entropy: Python binding of libflce03.so.

The functions named like the C ABI (``flce_fwd_bwd``, ``ce_fwd_bwd``,
``flce_workspace_size`` ...) marshal their arguments and call the library:
pointer arguments accept a torch tensor (its ``data_ptr()``), an integer
address or ``None``.  ``fused_linear_cross_entropy`` and ``cross_entropy``
add output / workspace allocation with torch and raise on an error status.
Every step of the computation runs in the library's CUDA kernels; there is
no fallback.  If the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "REDUCTIONS", "DTYPES", "STATUS_BIT_TARGET_RANGE", "STATUS_BIT_TIMEOUT", "KERNEL_NAMES",
    "library_path", "lib", "flce_status_string", "flce_version", "flce_default_chunk",
    "flce_workspace_size", "flce_workspace_size_typed", "flce_fwd_bwd", "flce_fwd_bwd_typed", "ce_workspace_size", "ce_fwd_bwd", "ce_fwd_bwd_noalloc",
    "flce_vp_workspace_size", "flce_vp_forward", "flce_vp_backward", "ce_vp_partials", "ce_vp_backward",
    "flce_set_wait_timeout_ns", "flce_selftest_wait_timeout", "flce_kernel_name",
    "flce_profile_enable", "flce_profile_disable", "flce_profile_read",
    "fused_linear_cross_entropy", "cross_entropy", "FlceError",
]

REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}
DTYPES = {"bf16": 0, "fp32": 1, "fp16": 2, "fp32_rounded": 3}
STATUS_BIT_TARGET_RANGE = 0x1
STATUS_BIT_TIMEOUT = 0x2
KERNEL_NAMES = ("count_targets", "gemm_forward", "row_finalize", "grad_logits", "gemm_backward",
                "loss_reduce", "ce_rows", "zero", "bias_reduce", "gh_reduce")

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libflce03.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGNATURES = {
    "flce_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "flce_version": (ctypes.c_int, []),
    "flce_default_chunk": (_I64, [_I64, _I64, _I64]),
    "flce_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, ctypes.c_int]),
    "flce_workspace_size_typed": (_SZ, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int]),
    "flce_fwd_bwd": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_int, _I64,
                                    ctypes.c_float, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P,
                                    _P, _SZ, _P, _P]),
    "flce_fwd_bwd_typed": (ctypes.c_int, [ctypes.c_int, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_int,
                                          _I64, ctypes.c_float, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P,
                                          _P, _SZ, _P, _P]),
    "ce_workspace_size": (_SZ, [_I64, _I64, ctypes.c_int, ctypes.c_int]),
    "ce_fwd_bwd": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _I64, _I64, _I64, ctypes.c_int,
                                  ctypes.c_float, _P, _P, _P, _SZ, _P, _P]),
    "ce_fwd_bwd_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _I64, _I64, _I64, ctypes.c_int,
                                          ctypes.c_float, _P, _P, _P, _P]),
    "flce_vp_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "flce_vp_forward": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _SZ,
                                       _P, _P]),
    "flce_vp_backward": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P,
                                        ctypes.c_int, _P, _SZ, _P, _P]),
    "ce_vp_partials": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P]),
    "ce_vp_backward": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P]),
    "flce_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "flce_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_uint64, _P]),
    "flce_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
    "flce_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "flce_profile_disable": (None, []),
    "flce_profile_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float),
                                         ctypes.c_int]),
}


class FlceError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {flce_status_string(status)}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(or linear_cross_entropy_03_gb300/_build.py); there is no fallback implementation")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _red(reduction) -> int:
    return REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)


# ------------------------------------------------------------------ raw ABI

def flce_status_string(status: int) -> str:
    return lib().flce_status_string(int(status)).decode()


def flce_version() -> int:
    return lib().flce_version()


def flce_default_chunk(N: int, H: int, V: int) -> int:
    return lib().flce_default_chunk(N, H, V)


def flce_workspace_size(N: int, H: int, V: int, chunk: int = 0, reduction="mean") -> int:
    return lib().flce_workspace_size(N, H, V, chunk, _red(reduction))


def flce_workspace_size_typed(dtype, N: int, H: int, V: int, chunk: int = 0, reduction="mean") -> int:
    return lib().flce_workspace_size_typed(_dt(dtype), N, H, V, chunk, _red(reduction))


def flce_fwd_bwd(hidden, weight, bias, target, N, H, V, ignore_index, reduction, chunk, grad_scale,
                 grad_out_none, loss, grad_hidden, grad_weight, grad_bias, accumulate, n_valid_out,
                 lse_out, target_logit_out, workspace, workspace_bytes, status_dev, stream=None) -> int:
    return lib().flce_fwd_bwd(
        _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(target), N, H, V, ignore_index, _red(reduction),
        chunk, float(grad_scale), _ptr(grad_out_none), _ptr(loss), _ptr(grad_hidden), _ptr(grad_weight),
        _ptr(grad_bias), int(accumulate), _ptr(n_valid_out), _ptr(lse_out), _ptr(target_logit_out),
        _ptr(workspace), int(workspace_bytes), _ptr(status_dev), _stream(stream))


def flce_fwd_bwd_typed(dtype, hidden, weight, bias, target, N, H, V, ignore_index, reduction, chunk, grad_scale,
                       grad_out_none, loss, grad_hidden, grad_weight, grad_bias, accumulate, n_valid_out,
                       lse_out, target_logit_out, workspace, workspace_bytes, status_dev, stream=None) -> int:
    return lib().flce_fwd_bwd_typed(
        _dt(dtype), _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(target), N, H, V, ignore_index,
        _red(reduction), chunk, float(grad_scale), _ptr(grad_out_none), _ptr(loss), _ptr(grad_hidden),
        _ptr(grad_weight), _ptr(grad_bias), int(accumulate), _ptr(n_valid_out), _ptr(lse_out),
        _ptr(target_logit_out), _ptr(workspace), int(workspace_bytes), _ptr(status_dev), _stream(stream))


def ce_workspace_size(N: int, V: int, dtype="bf16", reduction="mean") -> int:
    return lib().ce_workspace_size(N, V, DTYPES[dtype] if isinstance(dtype, str) else int(dtype),
                                   _red(reduction))


def ce_fwd_bwd(logits, dtype, grad_logits, target, N, V, ignore_index, reduction, grad_scale,
               grad_out_none, loss, workspace, workspace_bytes, status_dev, stream=None) -> int:
    return lib().ce_fwd_bwd(
        _ptr(logits), DTYPES[dtype] if isinstance(dtype, str) else int(dtype), _ptr(grad_logits),
        _ptr(target), N, V, ignore_index, _red(reduction), float(grad_scale), _ptr(grad_out_none),
        _ptr(loss), _ptr(workspace), int(workspace_bytes), _ptr(status_dev), _stream(stream))


NOALLOC_MAX_ROWS = 65536


def ce_fwd_bwd_noalloc(logits, dtype, grad_logits, target, N, V, ignore_index, reduction, grad_scale,
                       grad_out_none, loss, status_dev, stream=None) -> int:
    """ce_fwd_bwd without a workspace: the library's own fixed scratch array is
    used, so nothing is allocated.  For callers that may not allocate device
    memory; calls must not overlap on the GPU (they share that array)."""
    return lib().ce_fwd_bwd_noalloc(
        _ptr(logits), DTYPES[dtype] if isinstance(dtype, str) else int(dtype), _ptr(grad_logits),
        _ptr(target), N, V, ignore_index, _red(reduction), float(grad_scale), _ptr(grad_out_none),
        _ptr(loss), _ptr(status_dev), _stream(stream))


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def flce_vp_workspace_size(C: int, H: int, V_shard: int) -> int:
    return lib().flce_vp_workspace_size(C, H, V_shard)


def flce_vp_forward(hidden, weight_shard, bias_shard, target, C, H, V_shard, vocab_offset, ignore_index,
                    lse_shard, lse16_shard, target_logit_shard, workspace, workspace_bytes, status_dev,
                    stream=None) -> int:
    return lib().flce_vp_forward(
        _ptr(hidden), _ptr(weight_shard), _ptr(bias_shard), _ptr(target), C, H, V_shard, vocab_offset,
        ignore_index, _ptr(lse_shard), _ptr(lse16_shard), _ptr(target_logit_shard), _ptr(workspace),
        int(workspace_bytes), _ptr(status_dev), _stream(stream))


def flce_vp_backward(hidden, weight_shard, target, C, H, V_shard, vocab_offset, ignore_index, lse16,
                     row_scale, grad_hidden_partial, grad_weight_shard, grad_bias_shard, accumulate, workspace,
                     workspace_bytes, status_dev, stream=None) -> int:
    return lib().flce_vp_backward(
        _ptr(hidden), _ptr(weight_shard), _ptr(target), C, H, V_shard, vocab_offset, ignore_index,
        _ptr(lse16), _ptr(row_scale), _ptr(grad_hidden_partial), _ptr(grad_weight_shard), _ptr(grad_bias_shard),
        int(accumulate), _ptr(workspace), int(workspace_bytes), _ptr(status_dev), _stream(stream))


def ce_vp_partials(logits, dtype, target, N, V_shard, vocab_offset, ignore_index, lse_shard,
                   target_logit_shard, status_dev, stream=None) -> int:
    return lib().ce_vp_partials(_ptr(logits), _dt(dtype), _ptr(target), N, V_shard, vocab_offset, ignore_index,
                                _ptr(lse_shard), _ptr(target_logit_shard), _ptr(status_dev), _stream(stream))


def ce_vp_backward(logits, dtype, grad_logits, target, N, V_shard, vocab_offset, ignore_index, lse, row_scale,
                   status_dev, stream=None) -> int:
    return lib().ce_vp_backward(_ptr(logits), _dt(dtype), _ptr(grad_logits), _ptr(target), N, V_shard,
                                vocab_offset, ignore_index, _ptr(lse), _ptr(row_scale), _ptr(status_dev),
                                _stream(stream))


def flce_set_wait_timeout_ns(ns: int) -> None:
    lib().flce_set_wait_timeout_ns(int(ns))


def flce_selftest_wait_timeout(status_dev, timeout_ns: int, stream=None) -> int:
    return lib().flce_selftest_wait_timeout(_ptr(status_dev), int(timeout_ns), _stream(stream))


def flce_kernel_name(kernel_id: int) -> str:
    return lib().flce_kernel_name(int(kernel_id)).decode()


def flce_profile_enable(capacity: int) -> int:
    return lib().flce_profile_enable(int(capacity))


def flce_profile_disable() -> None:
    lib().flce_profile_disable()


def flce_profile_read(max_records: int = 4096):
    """[(kernel name, ms)] for the launches recorded since flce_profile_enable."""
    ids = (ctypes.c_int * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = lib().flce_profile_read(ids, ms, max_records)
    return [(flce_kernel_name(ids[i]), float(ms[i])) for i in range(n)]


# ------------------------------------------------------------------ tensor API

def _check(status: int, where: str):
    if status != 0:
        raise FlceError(status, where)


def fused_linear_cross_entropy(hidden, weight, target, bias=None, *, ignore_index: int = -100,
                               reduction="mean", chunk: int = 0, grad_scale: float = 1.0,
                               grad_out=None, grad_hidden: bool = True, grad_weight: bool = True,
                               grad_weight_out=None, grad_bias_out=None, accumulate: bool = False,
                               row_stats: bool = False, fp32_mode: str = "split", workspace=None, status=None,
                               stream=None) -> dict:
    """Loss and gradients of cross_entropy(hidden @ weight.T + bias, target).

    hidden [N, H] and weight [V, H] bf16, fp16 or fp32 (both the same), bias
    [V] of that type or None, target [N] int64, all on one CUDA device and
    contiguous.  Returns a dict with ``loss`` (fp32 [N] or []),
    ``grad_hidden`` ([N, H], the input type), ``grad_weight``
    (fp32 [V, H]), ``grad_bias`` (fp32 [V]), ``n_valid`` (int32 [1]) and, with
    ``row_stats``, ``lse`` and ``target_logit`` (fp32 [N]).  fp32 operands
    run split into bf16 hi + lo (``fp32_mode="split"``, three products) or
    rounded to bf16 once (``"rounded"``).  Asynchronous on ``stream``
    (default: the current stream); ``status`` is the device status word
    (int32 [1]).
    """
    import torch
    n, h = hidden.shape
    v = weight.shape[0]
    dev = hidden.device
    red = _red(reduction)
    loss = torch.empty(n if red == 0 else 1, dtype=torch.float32, device=dev)
    dtype = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}.get(hidden.dtype)
    if dtype is None or weight.dtype != hidden.dtype or (bias is not None and bias.dtype != hidden.dtype):
        raise FlceError(2, "fused_linear_cross_entropy: hidden, weight and bias must share one of bf16/fp16/fp32")
    if dtype == "fp32" and fp32_mode == "rounded":
        dtype = "fp32_rounded"
    elif dtype == "fp32" and fp32_mode != "split":
        raise FlceError(1, f"fused_linear_cross_entropy: fp32_mode {fp32_mode!r}")
    gh = torch.empty(n, h, dtype=hidden.dtype, device=dev) if grad_hidden else None
    gw = grad_weight_out if grad_weight_out is not None else (
        torch.empty(v, h, dtype=torch.float32, device=dev) if grad_weight else None)
    gb = grad_bias_out if grad_bias_out is not None else (
        torch.empty(v, dtype=torch.float32, device=dev) if bias is not None else None)
    nv = torch.zeros(1, dtype=torch.int32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev) if row_stats else None
    tl = torch.empty(n, dtype=torch.float32, device=dev) if row_stats else None
    ws_bytes = flce_workspace_size_typed(dtype, n, h, v, chunk, red)
    if ws_bytes == 0:
        raise FlceError(1, "flce_workspace_size_typed")
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = flce_fwd_bwd_typed(dtype, hidden, weight, bias, target, n, h, v, ignore_index, red, chunk, grad_scale,
                            grad_out, loss, gh, gw, gb, accumulate, nv, lse, tl, workspace, ws_bytes,
                            status, stream)
    _check(st, "flce_fwd_bwd_typed")
    out = dict(loss=loss if red == 0 else loss[0], grad_hidden=gh, grad_weight=gw, grad_bias=gb,
               n_valid=nv, status=status, workspace=workspace)
    if row_stats:
        out.update(lse=lse, target_logit=tl)
    return out


def cross_entropy(logits, target, *, ignore_index: int = -100, reduction="mean", grad_scale: float = 1.0,
                  grad_out=None, in_place: bool = False, want_grad: bool = True, grad_out_buffer=None,
                  workspace=None, status=None, stream=None) -> dict:
    """Loss and grad_logits of cross_entropy(logits, target) on [N, V] bf16/fp16/fp32 logits.

    ``in_place`` writes the gradient over ``logits``.  Returns a dict with
    ``loss``, ``grad_logits`` (or None) and ``status``.
    """
    import torch
    n, v = logits.shape
    dt = {torch.bfloat16: "bf16", torch.float32: "fp32", torch.float16: "fp16"}.get(logits.dtype)
    if dt is None:
        raise FlceError(2, "cross_entropy")
    red = _red(reduction)
    dev = logits.device
    loss = torch.empty(n if red == 0 else 1, dtype=torch.float32, device=dev)
    if not want_grad:
        grad = None
    elif in_place:
        grad = logits
    else:
        grad = grad_out_buffer if grad_out_buffer is not None else torch.empty_like(logits)
    ws_bytes = ce_workspace_size(n, v, dt, red)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = ce_fwd_bwd(logits, dt, grad, target, n, v, ignore_index, red, grad_scale, grad_out, loss,
                    workspace, ws_bytes, status, stream)
    _check(st, "ce_fwd_bwd")
    return dict(loss=loss if red == 0 else loss[0], grad_logits=grad, status=status)
