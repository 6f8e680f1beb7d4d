"""Helpers shared by the GPU parity tests: moving the generator's bytes to the
device, running the library, and the comparison rule.

Comparison rule (the method's stated tolerances): loss relative error
<= 2e-3 (for reduction none: max |diff| <= 2e-3 * max |ref|); every gradient
max |diff| <= 1e-2 * max |ref|; the ignore mask exact (ignored rows have loss
0 and zero gradient rows) and the valid-target count exact.
"""
from __future__ import annotations

import numpy as np
import torch

import linear_cross_entropy_03_gb300 as flce

LOSS_RTOL = 2e-3
GRAD_RTOL = 1e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev16(a: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16), float16 or float32 values on the GPU, as
    bf16 / fp16 / fp32."""
    if a.dtype in (np.float16, np.float32):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev_bf16(a)


def host(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_flce(inp, *, reduction="mean", chunk=0, use_bias=True, grad_scale=1.0, grad_out=None,
             accumulate=False, grad_weight_init=None, grad_bias_init=None, ignore_index=None,
             grads=True, keep_f32=False, fp32_mode="split"):
    h = dev16(inp.hidden)
    w = dev16(inp.weight)
    b = dev16(inp.bias) if (use_bias and inp.bias is not None) else None
    t = torch.from_numpy(inp.target).cuda()
    go = torch.from_numpy(grad_out).cuda() if grad_out is not None else None
    gw0 = torch.from_numpy(grad_weight_init.astype(np.float32)).cuda() if grad_weight_init is not None else None
    gb0 = torch.from_numpy(grad_bias_init.astype(np.float32)).cuda() if grad_bias_init is not None else None
    out = flce.fused_linear_cross_entropy(
        h, w, t, b, ignore_index=inp.ignore_index if ignore_index is None else ignore_index,
        reduction=reduction, chunk=chunk, grad_scale=grad_scale, grad_out=go, grad_hidden=grads,
        grad_weight=grads, grad_weight_out=gw0, grad_bias_out=gb0 if b is not None else None,
        accumulate=accumulate, row_stats=True, fp32_mode=fp32_mode)
    torch.cuda.synchronize()
    conv = (lambda x: x.float().cpu().numpy()) if keep_f32 else host
    res = {k: (conv(v) if isinstance(v, torch.Tensor) and k not in ("status", "n_valid", "workspace") else v)
           for k, v in out.items() if v is not None}
    if keep_f32 and "loss" in res and np.ndim(res["loss"]) == 0:
        res["loss"] = float(res["loss"])
    res["status"] = int(out["status"].item())
    res["n_valid"] = int(out["n_valid"].item())
    return res


def assert_loss(got, ref, reduction):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if reduction == "none":
        assert got.shape == ref.shape
        err = np.abs(got - ref).max() if ref.size else 0.0
        assert err <= LOSS_RTOL * max(np.abs(ref).max() if ref.size else 0.0, 1e-30), f"loss err {err}"
    elif np.isnan(ref):
        assert np.isnan(got), f"loss {got}, expected NaN"
    else:
        assert abs(float(got) - float(ref)) <= LOSS_RTOL * abs(float(ref)) + 1e-30, f"loss {got} vs {ref}"


def assert_grad(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(got - ref).max() if ref.size else 0.0
    if scale == 0.0:
        assert err == 0.0, f"{name}: expected exact zeros, max |got| {err}"
    else:
        assert err <= GRAD_RTOL * scale, f"{name}: max err {err:.3e} > {GRAD_RTOL} * {scale:.3e}"


def assert_flce_parity(res, ref, reduction, *, check_grads=True, row_rtol=1e-5):
    """row_rtol bounds the per-row lse / target logit error relative to the
    largest |lse|: 1e-5 when the oracle sees the very operands the tensor
    cores multiply (fp32 accumulation is all that differs), the loss
    tolerance when the kernel rounds the operands first (fp32 inputs)."""
    assert res["status"] == 0, f"device status {res['status']:#x}"
    assert res["n_valid"] == ref["n_valid"]
    assert_loss(res["loss"], ref["loss"], reduction)
    valid = ref["valid"]
    lse_scale = max(1.0, np.abs(ref["lse"]).max())
    assert np.abs(res["lse"] - ref["lse"]).max() <= row_rtol * lse_scale
    assert np.abs(res["target_logit"][valid] - ref["target_logit"][valid]).max(initial=0) <= row_rtol * lse_scale
    assert np.all(res["target_logit"][~valid] == 0.0)
    if reduction == "none":
        assert np.all(res["loss"][~valid] == 0.0), "ignored rows must carry exactly zero loss"
    if check_grads:
        assert_grad(res["grad_hidden"], ref["grad_hidden"], "grad_hidden")
        assert np.all(res["grad_hidden"][~valid] == 0.0), "ignored rows must have zero grad_hidden"
        assert_grad(res["grad_weight"], ref["grad_weight"], "grad_weight")
        if ref.get("grad_bias") is not None and "grad_bias" in res:
            assert_grad(res["grad_bias"], ref["grad_bias"], "grad_bias")
