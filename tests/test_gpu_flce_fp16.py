"""GPU parity of the fused linear cross entropy with fp16 hidden / weight /
bias (flce_fwd_bwd_typed, FLCE_DTYPE_FP16) against the fp64 oracle, which
widens the same fp16 values exactly: every reduction, bias, ragged tails,
chunking, accumulation, small upstream gradients (the fp16 grad-logits are
stored relative to the rows' common scale) and a wider shape."""
import numpy as np
import pytest

import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_flce_parity, run_flce

pytestmark = pytest.mark.gpu


def _ref(inp, reduction, use_bias=True, **kw):
    return O.flce_reference(inp.hidden, inp.weight, inp.bias if use_bias else None, inp.target,
                            ignore_index=inp.ignore_index, reduction=reduction, **kw)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("shape,chunk", [((256, 128, 1024), 0), ((300, 136, 1000), 128),
                                         ((513, 264, 2049), 256)])
def test_fp16_ragged_with_bias(shape, chunk, reduction):
    n, h, v = shape
    inp = si.make_flce_inputs(n, h, v, 70 + n, w_std=0.05, bias_std=0.1, ignore_frac=0.1, dtype="fp16")
    go = si.make_grad_out(n, 9) if reduction == "none" else None
    ref = _ref(inp, reduction, grad_scale=0.5, grad_out=go)
    res = run_flce(inp, reduction=reduction, chunk=chunk, grad_scale=0.5, grad_out=go)
    assert res["status"] == 0
    assert_flce_parity(res, ref, reduction)


def test_fp16_small_upstream_gradients():
    # per-row upstream gradients of a mean taken outside (1/N): the stored
    # fp16 grad-logits are divided by the largest of them, so none underflow
    n, h, v = 1024, 128, 32768
    inp = si.make_flce_inputs(n, h, v, 81, ignore_frac=0.05, dtype="fp16")
    go = (si.make_grad_out(n, 3) / n).astype(np.float32)
    ref = _ref(inp, "none", use_bias=False, grad_out=go)
    res = run_flce(inp, reduction="none", use_bias=False, grad_out=go)
    assert_flce_parity(res, ref, "none")


def test_fp16_accumulate_and_chunks():
    inp = si.make_flce_inputs(200, 128, 3000, 85, bias_std=0.1, ignore_frac=0.05, dtype="fp16")
    gw0 = si.normal_f32(85, 11, (3000, 128), 0.01).astype(np.float64)
    gb0 = si.normal_f32(85, 12, (3000,), 0.01).astype(np.float64)
    ref = _ref(inp, "mean", grad_weight_init=gw0, grad_bias_init=gb0)
    res = run_flce(inp, reduction="mean", chunk=64, accumulate=True, grad_weight_init=gw0, grad_bias_init=gb0)
    assert_flce_parity(res, ref, "mean")


def test_fp16_wide_hidden():
    # H = 2048 (the Llama-3.2-1B width): several 512-column grad_H tiles and K blocks
    inp = si.make_flce_inputs(1024, 2048, 8192, 88, ignore_frac=0.05, dtype="fp16")
    ref = _ref(inp, "mean", use_bias=False)
    res = run_flce(inp, reduction="mean", use_bias=False, chunk=512)
    assert_flce_parity(res, ref, "mean")


def test_fp16_all_ignored_mean():
    inp = si.make_flce_inputs(64, 64, 500, 90, ignore_frac=1.0, dtype="fp16")
    res = run_flce(inp, reduction="mean", use_bias=False)
    assert res["n_valid"] == 0 and np.isnan(res["loss"])
    assert np.all(res["grad_hidden"] == 0.0) and np.all(res["grad_weight"] == 0.0)
