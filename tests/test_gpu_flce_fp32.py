"""GPU checks of the fused linear cross entropy with fp32 hidden / weight /
bias (flce_fwd_bwd_typed).

FLCE_DTYPE_FP32 splits each operand into bf16 hi + lo planes and sums the
products hi.hi + hi.lo + lo.hi in fp32, keeps the chunk logits exactly and
forms their gradient in fp32: checked against the fp64 oracle on the fp32
values with the per-row LSE and target logit within 1e-5 of the largest
|LSE| (what fp32 accumulation allows), besides the method's tolerances.

FLCE_DTYPE_FP32_ROUNDED rounds the operands to bf16 (nearest, ties to even)
once: parity with the oracle within the method's tolerances (the rounding
moves each logit by about 2^-9 of its terms), and identity with the bf16
entry point run on the same inputs rounded on the host by the definition of
round-to-nearest-even, which pins the conversion kernel and the wiring of
the copies (loss, lse, grad_weight and grad_bias bit for bit, grad_hidden
after rounding its fp32 values the same way)."""
import numpy as np
import pytest

import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import LOSS_RTOL, assert_flce_parity, run_flce

pytestmark = pytest.mark.gpu


def _ref(inp, reduction, use_bias=True, **kw):
    return O.flce_reference(inp.hidden, inp.weight, inp.bias if use_bias else None, inp.target,
                            ignore_index=inp.ignore_index, reduction=reduction, **kw)


def _rne_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _with_ties(a: np.ndarray) -> np.ndarray:
    """Plant exact bf16 halfway values (both tie directions, both signs)."""
    a = a.copy()
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), -(1 + 3 * 2.0 ** -8),
                     0.5 + 2.0 ** -9, 2 + 2.0 ** -7], dtype=np.float32)
    flat = a.reshape(-1)
    flat[: ties.size] = ties
    flat[-ties.size:] = ties[::-1]
    return a


def test_rne_reference_rounds_ties_to_even():
    got = _rne_bf16_bits(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20], np.float32))
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even mantissa is 1 (0x3F80);
    # 1 + 3*2^-8 between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6 (0x3F82)
    assert got.tolist() == [0x3F80, 0x3F82, 0x3F81]


@pytest.mark.parametrize("mode,row_rtol", [("split", 1e-5), ("rounded", LOSS_RTOL)])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("shape,chunk", [((256, 128, 1024), 0), ((300, 136, 1000), 128)])
def test_fp32_parity_with_oracle(shape, chunk, reduction, mode, row_rtol):
    n, h, v = shape
    inp = si.make_flce_inputs(n, h, v, 170 + n, w_std=0.05, bias_std=0.1, ignore_frac=0.1, dtype="fp32")
    go = si.make_grad_out(n, 19) if reduction == "none" else None
    ref = _ref(inp, reduction, grad_scale=0.5, grad_out=go)
    res = run_flce(inp, reduction=reduction, chunk=chunk, grad_scale=0.5, grad_out=go, fp32_mode=mode)
    assert res["status"] == 0
    assert_flce_parity(res, ref, reduction, row_rtol=row_rtol)


def test_fp32_split_is_closer_than_rounded():
    # the split products leave the logits to fp32 accumulation: the per-row
    # LSE error is far below the rounded mode's
    n, h, v = 512, 1024, 4096
    inp = si.make_flce_inputs(n, h, v, 173, ignore_frac=0.05, dtype="fp32")
    ref = _ref(inp, "mean", use_bias=False)
    err = {}
    for mode in ("split", "rounded"):
        res = run_flce(inp, reduction="mean", use_bias=False, fp32_mode=mode)
        assert res["status"] == 0
        err[mode] = np.abs(res["lse"] - ref["lse"]).max()
    assert err["split"] <= 1e-5 * np.abs(ref["lse"]).max()
    assert err["split"] * 20 < err["rounded"], err


@pytest.mark.parametrize("reduction", ["none", "mean"])
def test_fp32_equals_bf16_path_on_rounded_inputs(reduction):
    n, h, v = 513, 264, 2049
    inp = si.make_flce_inputs(n, h, v, 177, w_std=0.05, bias_std=0.1, ignore_frac=0.1, dtype="fp32")
    inp = si.FlceInputs(_with_ties(inp.hidden), _with_ties(inp.weight), _with_ties(inp.bias), inp.target,
                        inp.ignore_index)
    rounded = si.FlceInputs(_rne_bf16_bits(inp.hidden), _rne_bf16_bits(inp.weight), _rne_bf16_bits(inp.bias),
                            inp.target, inp.ignore_index)
    a = run_flce(inp, reduction=reduction, chunk=256, keep_f32=True, fp32_mode="rounded")
    b = run_flce(rounded, reduction=reduction, chunk=256, keep_f32=True)
    assert a["status"] == 0 and b["status"] == 0 and a["n_valid"] == b["n_valid"]
    np.testing.assert_array_equal(a["loss"], b["loss"])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    np.testing.assert_array_equal(a["target_logit"], b["target_logit"])
    np.testing.assert_array_equal(a["grad_weight"], b["grad_weight"])
    np.testing.assert_array_equal(a["grad_bias"], b["grad_bias"])
    gh = _rne_bf16_bits(a["grad_hidden"].astype(np.float32))
    np.testing.assert_array_equal(gh, _rne_bf16_bits(b["grad_hidden"].astype(np.float32)))
    assert a["grad_hidden"].dtype == np.float32


@pytest.mark.parametrize("mode,row_rtol", [("split", 1e-5), ("rounded", LOSS_RTOL)])
def test_fp32_wide_hidden_accumulate(mode, row_rtol):
    # H = 2048: several 512-column grad_H tiles; grad_weight / grad_bias added to
    n, h, v = 1024, 2048, 8192
    inp = si.make_flce_inputs(n, h, v, 188, bias_std=0.1, ignore_frac=0.05, dtype="fp32")
    gw0 = si.normal_f32(188, 11, (v, h), 0.01).astype(np.float64)
    gb0 = si.normal_f32(188, 12, (v,), 0.01).astype(np.float64)
    ref = _ref(inp, "mean", grad_weight_init=gw0, grad_bias_init=gb0)
    res = run_flce(inp, reduction="mean", chunk=512, accumulate=True, grad_weight_init=gw0, grad_bias_init=gb0,
                   fp32_mode=mode)
    assert_flce_parity(res, ref, "mean", row_rtol=row_rtol)
