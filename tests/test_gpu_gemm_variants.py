"""GPU parity of flce_fwd_bwd with each tensor-core kernel form -- CTA pairs
on 256 x 256 tiles (tcgen05 cta_group::2, the default) and one CTA per
128 x 256 tile -- against the fp64 oracle, on shapes with ragged tails in
every dimension, all three tile kinds and accumulation."""
import numpy as np
import pytest

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_flce_parity, run_flce

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[2, 1], ids=["cta_pair", "single_cta"])
def gemm_variant(request):
    assert flce.flce_set_gemm_variant(request.param) == request.param
    yield request.param
    flce.flce_set_gemm_variant(0)


def _ref(inp, reduction, **kw):
    return O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, ignore_index=inp.ignore_index,
                            reduction=reduction, **kw)


def test_variant_tiny_config():
    inp = si.config_inputs("tiny")
    assert_flce_parity(run_flce(inp, reduction="mean"), _ref(inp, "mean"), "mean")


@pytest.mark.parametrize("shape,chunk", [((300, 136, 1000), 128), ((513, 264, 2049), 256),
                                         ((130, 8, 300), 0), ((1000, 520, 3000), 384)])
@pytest.mark.parametrize("reduction", ["none", "mean"])
def test_variant_ragged(shape, chunk, reduction):
    n, h, v = shape
    inp = si.make_flce_inputs(n, h, v, 70 + n, w_std=0.05, bias_std=0.1, ignore_frac=0.1)
    assert_flce_parity(run_flce(inp, reduction=reduction, chunk=chunk), _ref(inp, reduction), reduction)


def test_variant_small_tp_shard():
    inp = si.config_inputs("small_v32k")
    assert_flce_parity(run_flce(inp, reduction="sum"), _ref(inp, "sum"), "sum")


def test_variant_medium_long_k():
    inp = si.make_flce_inputs(1536, 1024, 9000, 99, ignore_frac=0.05)
    assert_flce_parity(run_flce(inp, reduction="mean", chunk=768), _ref(inp, "mean"), "mean")


def test_variant_accumulate():
    inp = si.make_flce_inputs(600, 192, 2600, 5, bias_std=0.1)
    gw0 = si.bf16_to_float32(si.normal_bf16(5, 11, (2600, 192), 0.01)).astype(np.float64)
    gb0 = si.bf16_to_float32(si.normal_bf16(5, 12, (2600,), 0.01)).astype(np.float64)
    ref = _ref(inp, "sum", grad_weight_init=gw0, grad_bias_init=gb0)
    res = run_flce(inp, reduction="sum", chunk=256, accumulate=True, grad_weight_init=gw0, grad_bias_init=gb0)
    assert_flce_parity(res, ref, "sum")


def test_variant_matches_single_cta(gemm_variant):
    if gemm_variant != flce.GEMM_CTA_PAIR:
        pytest.skip("compares the two forms once")
    inp = si.make_flce_inputs(700, 256, 5000, 17, ignore_frac=0.05)
    pair = run_flce(inp, reduction="none", chunk=512)
    flce.flce_set_gemm_variant(flce.GEMM_SINGLE_CTA)
    try:
        single = run_flce(inp, reduction="none", chunk=512)
    finally:
        flce.flce_set_gemm_variant(flce.GEMM_CTA_PAIR)
    # the same products on both kernel forms: logits, LSE and losses agree to fp32 rounding
    assert np.abs(pair["lse"] - single["lse"]).max() <= 1e-5 * np.abs(single["lse"]).max()
    assert np.abs(pair["target_logit"] - single["target_logit"]).max() <= 1e-5 * np.abs(single["lse"]).max()
    assert np.abs(pair["grad_weight"] - single["grad_weight"]).max() <= 1e-3 * np.abs(single["grad_weight"]).max()
