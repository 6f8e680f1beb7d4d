"""GPU parity of flce_fwd_bwd against the fp64 oracle, element by element, on
shapes the oracle finishes in seconds: the tiny and small workloads, ragged
tails in N, H, V and the chunk, every reduction, bias, accumulation, upstream
gradients and the degenerate cases."""
import math

import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_flce_parity, assert_grad, assert_loss, run_flce

pytestmark = pytest.mark.gpu


def _ref(inp, reduction, use_bias=True, **kw):
    return O.flce_reference(inp.hidden, inp.weight, inp.bias if use_bias else None, inp.target,
                            ignore_index=inp.ignore_index, reduction=reduction, **kw)


@pytest.mark.parametrize("chunk", [0, 100])
def test_tiny_config(chunk):
    inp = si.config_inputs("tiny")
    ref = _ref(inp, "mean")
    res = run_flce(inp, reduction="mean", chunk=chunk)
    assert_flce_parity(res, ref, "mean")


@pytest.mark.parametrize("v", [32768, 65536])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_small_tp_shard_config(v, reduction):
    name = "small_v32k" if v == 32768 else "small_v64k"
    inp = si.config_inputs(name)
    ref = _ref(inp, reduction)
    res = run_flce(inp, reduction=reduction)
    assert_flce_parity(res, ref, reduction)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("shape,chunk", [((300, 136, 1000), 128), ((257, 64, 777), 100),
                                         ((130, 8, 300), 0), ((513, 264, 2049), 256)])
def test_ragged_with_bias(shape, chunk, reduction):
    n, h, v = shape
    inp = si.make_flce_inputs(n, h, v, 40 + n, w_std=0.05, bias_std=0.1, ignore_frac=0.1)
    go = si.make_grad_out(n, 7) if reduction == "none" else None
    ref = _ref(inp, reduction, grad_scale=0.5, grad_out=go)
    res = run_flce(inp, reduction=reduction, chunk=chunk, grad_scale=0.5, grad_out=go)
    assert_flce_parity(res, ref, reduction)


def test_accumulate_into_existing_gradients():
    inp = si.make_flce_inputs(200, 128, 3000, 5, bias_std=0.1, ignore_frac=0.05)
    gw0 = si.bf16_to_float32(si.normal_bf16(5, 11, (3000, 128), 0.01)).astype(np.float64)
    gb0 = si.bf16_to_float32(si.normal_bf16(5, 12, (3000,), 0.01)).astype(np.float64)
    ref = _ref(inp, "sum", grad_weight_init=gw0, grad_bias_init=gb0)
    res = run_flce(inp, reduction="sum", chunk=64, accumulate=True, grad_weight_init=gw0, grad_bias_init=gb0)
    assert_flce_parity(res, ref, "sum")


def test_index_encoding_gathers_target_logit_exactly():
    # H[n] = (1, 256, 0...), W[v] = (v mod 256, v div 256, 0...) => z[n, v] = v exactly
    n, h, v = 384, 64, 65536
    hid = np.zeros((n, h), dtype=np.float32)
    hid[:, 0], hid[:, 1] = 1.0, 256.0
    w = np.zeros((v, h), dtype=np.float32)
    ids = np.arange(v)
    w[:, 0], w[:, 1] = ids % 256, ids // 256
    t = si.uniform_targets(3, 1, n, v)
    t[::7] = -100
    inp = si.FlceInputs(si.float32_to_bf16_bits(hid), si.float32_to_bf16_bits(w), None, t)
    res = run_flce(inp, reduction="none", chunk=128, use_bias=False, grads=False)
    valid = t != -100
    assert res["status"] == 0
    assert np.array_equal(res["target_logit"][valid], t[valid].astype(np.float64))
    assert np.all(res["target_logit"][~valid] == 0.0)
    assert np.all(res["loss"][~valid] == 0.0)
    lse_expect = (v - 1) - math.log1p(-math.exp(-1.0))
    assert np.abs(res["lse"] - lse_expect).max() <= 1e-6 * v


def test_zero_weight_gives_ln_v():
    inp = si.make_flce_inputs(256, 128, 5000, 9, ignore_frac=0.1)
    inp.weight[:] = 0
    res = run_flce(inp, reduction="mean", use_bias=False)
    assert abs(res["loss"] - math.log(5000)) <= 1e-6 * math.log(5000)
    assert np.all(res["grad_hidden"] == 0.0)
    ref = _ref(inp, "mean", use_bias=False)
    assert_grad(res["grad_weight"], ref["grad_weight"], "grad_weight")


def test_all_targets_ignored():
    inp = si.make_flce_inputs(100, 64, 500, 2, ignore_frac=0.0)
    inp.target[:] = -100
    res = run_flce(inp, reduction="mean", use_bias=False)
    assert math.isnan(res["loss"]) and res["n_valid"] == 0
    assert np.all(res["grad_hidden"] == 0.0) and np.all(res["grad_weight"] == 0.0)
    res = run_flce(inp, reduction="sum", use_bias=False)
    assert res["loss"] == 0.0


def test_single_class_vocabulary():
    inp = si.make_flce_inputs(64, 16, 1, 3, ignore_frac=0.25)
    res = run_flce(inp, reduction="sum", use_bias=False)
    assert res["status"] == 0 and abs(res["loss"]) <= 1e-6
    assert np.abs(res["grad_weight"]).max() <= 1e-6


def test_empty_batch():
    import linear_cross_entropy_03_gb300 as flce
    h = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(100, 64, dtype=torch.bfloat16, device="cuda")
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    gw = torch.full((100, 64), 7.0, device="cuda")
    out = flce.fused_linear_cross_entropy(h, w, t, reduction="mean", grad_weight_out=gw)
    torch.cuda.synchronize()
    assert math.isnan(out["loss"].item())
    assert torch.all(gw == 0)
    out = flce.fused_linear_cross_entropy(h, w, t, reduction="sum")
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0


def test_ignore_index_inside_vocabulary():
    inp = si.make_flce_inputs(300, 64, 400, 4, ignore_frac=0.0)
    inp.target[::5] = 17
    ref = O.flce_reference(inp.hidden, inp.weight, None, inp.target, ignore_index=17, reduction="mean")
    res = run_flce(inp, reduction="mean", use_bias=False, ignore_index=17)
    assert res["n_valid"] == int((inp.target != 17).sum())
    assert_flce_parity(res, ref, "mean")


def test_out_of_range_target_sets_status_and_is_ignored():
    inp = si.make_flce_inputs(200, 64, 300, 8, ignore_frac=0.05)
    inp.target[3] = 300
    inp.target[50] = -7
    ref = O.flce_reference(inp.hidden, inp.weight, None, inp.target, reduction="mean")
    assert ref["status"] == "target_range"
    res = run_flce(inp, reduction="mean", use_bias=False)
    assert res["status"] & 0x1
    res["status"] = 0
    assert_flce_parity(res, ref, "mean")


def test_forward_only():
    inp = si.make_flce_inputs(500, 128, 2000, 12, ignore_frac=0.05)
    ref = _ref(inp, "none", use_bias=False)
    res = run_flce(inp, reduction="none", use_bias=False, grads=False)
    assert res["status"] == 0
    assert_loss(res["loss"], ref["loss"], "none")


def test_repeated_calls_are_deterministic():
    inp = si.make_flce_inputs(640, 128, 4000, 13, bias_std=0.1)
    a = run_flce(inp, reduction="mean", chunk=256)
    b = run_flce(inp, reduction="mean", chunk=256)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["grad_hidden"], b["grad_hidden"])
    assert np.array_equal(a["grad_weight"], b["grad_weight"])
    assert np.array_equal(a["grad_bias"], b["grad_bias"])  # fixed-order column sums, no atomics
