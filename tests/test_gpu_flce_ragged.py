"""GPU parity of flce_fwd_bwd (CTA-pair tensor-core kernels: 256 x 256 tiles,
grad_H in 256 x 512) against the fp64 oracle, on shapes with ragged tails in
every dimension, all three tile kinds and accumulation."""
import numpy as np
import pytest

import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_flce_parity, run_flce

pytestmark = pytest.mark.gpu


def _ref(inp, reduction, **kw):
    return O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, ignore_index=inp.ignore_index,
                            reduction=reduction, **kw)


def test_flce_tiny_config():
    inp = si.config_inputs("tiny")
    assert_flce_parity(run_flce(inp, reduction="mean"), _ref(inp, "mean"), "mean")


@pytest.mark.parametrize("shape,chunk", [((300, 136, 1000), 128), ((513, 264, 2049), 256),
                                         ((130, 8, 300), 0), ((1000, 520, 3000), 384)])
@pytest.mark.parametrize("reduction", ["none", "mean"])
def test_flce_ragged(shape, chunk, reduction):
    n, h, v = shape
    inp = si.make_flce_inputs(n, h, v, 70 + n, w_std=0.05, bias_std=0.1, ignore_frac=0.1)
    assert_flce_parity(run_flce(inp, reduction=reduction, chunk=chunk), _ref(inp, reduction), reduction)


def test_flce_small_tp_shard():
    inp = si.config_inputs("small_v32k")
    assert_flce_parity(run_flce(inp, reduction="sum"), _ref(inp, "sum"), "sum")


def test_flce_medium_long_k():
    inp = si.make_flce_inputs(1536, 1024, 9000, 99, ignore_frac=0.05)
    assert_flce_parity(run_flce(inp, reduction="mean", chunk=768), _ref(inp, "mean"), "mean")


def test_flce_accumulate():
    inp = si.make_flce_inputs(600, 192, 2600, 5, bias_std=0.1)
    gw0 = si.bf16_to_float32(si.normal_bf16(5, 11, (2600, 192), 0.01)).astype(np.float64)
    gb0 = si.bf16_to_float32(si.normal_bf16(5, 12, (2600,), 0.01)).astype(np.float64)
    ref = _ref(inp, "sum", grad_weight_init=gw0, grad_bias_init=gb0)
    res = run_flce(inp, reduction="sum", chunk=256, accumulate=True, grad_weight_init=gw0, grad_bias_init=gb0)
    assert_flce_parity(res, ref, "sum")
