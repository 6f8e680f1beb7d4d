"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (default chunk unless a chunk is the point of the test).

The fp64 oracle computes: the LSE and target logit of every row (the full
projection, in row blocks) where that is affordable, from which the reduced
loss and grad_weight rows for sampled vocabulary ids follow exactly; and
grad_hidden rows for sampled tokens.  Sampled tokens cover chunk boundaries,
ignored rows, the first and last rows and seeded random rows; sampled
vocabulary ids cover the most frequent targets, never-targeted ids, tile
boundaries and seeded random ids.
"""
import numpy as np
import pytest
import torch

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import GRAD_RTOL, LOSS_RTOL, run_flce

pytestmark = pytest.mark.gpu


def sample_rows(n, chunk, seed, k=192):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, n - 1, n - 2}
    for c in range(chunk, n, chunk):
        fixed.update({c - 1, c, min(n - 1, c + 127), min(n - 1, c + 128)})
    rows = set(x for x in fixed if 0 <= x < n)
    rows.update(rng.choice(n, size=min(n, k), replace=False).tolist())
    return np.array(sorted(rows))


def sample_vocab(target, v, seed, k=64):
    rng = np.random.default_rng(seed)
    t = target[target >= 0]
    counts = np.bincount(t, minlength=v)
    top = np.argsort(-counts, kind="stable")[:k]
    never = np.nonzero(counts == 0)[0]
    never = never[rng.choice(never.size, size=min(k, never.size), replace=False)] if never.size else never
    edges = np.array([0, 1, 127, 128, 255, 256, v // 2, v - 257, v - 256, v - 129, v - 128, v - 2, v - 1])
    rand = rng.choice(v, size=k, replace=False)
    return np.unique(np.concatenate([top, never, edges[(edges >= 0) & (edges < v)], rand]))


def _check_rows(res, inp, rows, reduction, grad_out=None):
    ref = O.flce_rows(inp.hidden, inp.weight, inp.bias, inp.target, rows, reduction=reduction,
                      grad_out=grad_out)
    lse_scale = np.abs(ref["lse"]).max()
    assert np.abs(res["lse"][rows] - ref["lse"]).max() <= 1e-5 * lse_scale
    valid = ref["valid"]
    assert np.abs(res["target_logit"][rows][valid] - ref["target_logit"][valid]).max(initial=0.0) \
        <= 1e-5 * lse_scale
    assert np.all(res["target_logit"][rows][~valid] == 0.0)
    gh, gh_ref = res["grad_hidden"][rows], ref["grad_hidden"]
    assert np.abs(gh - gh_ref).max() <= GRAD_RTOL * np.abs(gh_ref).max(), "grad_hidden (sampled rows)"
    assert np.all(gh[~valid] == 0.0)
    return ref


def _check_weight_rows(res, inp, ids, lse_all, reduction):
    gw, gb = O.grad_weight_rows(inp.hidden, inp.weight, inp.bias, inp.target, ids, lse_all,
                                reduction=reduction)
    err = np.abs(res["grad_weight"][ids] - gw).max()
    assert err <= GRAD_RTOL * np.abs(gw).max(), f"grad_weight (sampled ids): {err}"
    if inp.bias is not None:
        assert np.abs(res["grad_bias"][ids] - gb).max() <= GRAD_RTOL * np.abs(gb).max()


@pytest.fixture(scope="module")
def llama32_1b():
    inp = si.config_inputs("llama32_1b")
    n = inp.hidden.shape[0]
    lse, zt = O.lse_rows(inp.hidden, inp.weight, None, np.arange(n), inp.target, row_block=512)
    return inp, lse, zt


@pytest.mark.parametrize("chunk", [1024, 2048, 4096])
def test_llama32_1b_chunk_sizes(llama32_1b, chunk):
    inp, lse, zt = llama32_1b
    n = inp.hidden.shape[0]
    valid = inp.target != inp.ignore_index
    loss_ref = float(np.where(valid, lse - zt, 0.0).sum() / valid.sum())
    res = run_flce(inp, reduction="mean", chunk=chunk, keep_f32=True)
    assert res["status"] == 0 and res["n_valid"] == int(valid.sum())
    assert abs(res["loss"] - loss_ref) <= LOSS_RTOL * abs(loss_ref)
    assert np.abs(res["lse"] - lse).max() <= 1e-5 * np.abs(lse).max()
    _check_rows(res, inp, sample_rows(n, chunk, 1), "mean")
    _check_weight_rows(res, inp, sample_vocab(inp.target, inp.weight.shape[0], 2), lse, "mean")


def test_llama3_8b_bench_configuration():
    inp = si.config_inputs("llama3_8b")
    n, v = inp.hidden.shape[0], inp.weight.shape[0]
    res = run_flce(inp, reduction="mean", chunk=0, keep_f32=True)
    chunk = flce.flce_default_chunk(n, inp.hidden.shape[1], v)
    lse, zt = O.lse_rows(inp.hidden, inp.weight, None, np.arange(n), inp.target, row_block=512)
    valid = inp.target != inp.ignore_index
    loss_ref = float(np.where(valid, lse - zt, 0.0).sum() / valid.sum())
    assert res["status"] == 0 and res["n_valid"] == int(valid.sum())
    assert abs(res["loss"] - loss_ref) <= LOSS_RTOL * abs(loss_ref)
    assert np.abs(res["lse"] - lse).max() <= 1e-5 * np.abs(lse).max()
    _check_rows(res, inp, sample_rows(n, chunk, 3), "mean")
    _check_weight_rows(res, inp, sample_vocab(inp.target, v, 4), lse, "mean")


def test_llama3_8b_with_bias():
    # the optional bias of the Llama-3-8B workload: the all-row oracle LSE
    # (with the bias), hence the reduced loss, grad_weight and grad_bias on
    # sampled vocabulary ids and grad_hidden on sampled rows
    inp = si.config_inputs("llama3_8b", with_bias=True)
    n, v = inp.hidden.shape[0], inp.weight.shape[0]
    res = run_flce(inp, reduction="mean", chunk=0, keep_f32=True)
    chunk = flce.flce_default_chunk(n, inp.hidden.shape[1], v)
    lse, zt = O.lse_rows(inp.hidden, inp.weight, inp.bias, np.arange(n), inp.target, row_block=512)
    valid = inp.target != inp.ignore_index
    loss_ref = float(np.where(valid, lse - zt, 0.0).sum() / valid.sum())
    assert res["status"] == 0 and res["n_valid"] == int(valid.sum())
    assert abs(res["loss"] - loss_ref) <= LOSS_RTOL * abs(loss_ref)
    assert np.abs(res["lse"] - lse).max() <= 1e-5 * np.abs(lse).max()
    assert np.abs(res["target_logit"][valid] - zt[valid]).max() <= 1e-5 * np.abs(lse).max()
    _check_rows(res, inp, sample_rows(n, chunk, 5, k=96), "mean")
    _check_weight_rows(res, inp, sample_vocab(inp.target, v, 6), lse, "mean")


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_llama32_1b_fp16_fp32_operands(dtype):
    # the fp16 and fp32 entry points at a full tensor-bound shape (K = 2048
    # for the forward, K = V = 128256 for grad_hidden): fp16 operands are
    # multiplied exactly as given, fp32 operands as bf16 hi + lo planes
    # (hi.hi + hi.lo + lo.hi); both leave the per-row LSE within 1e-5
    c = dict(si.CONFIGS["llama32_1b"])
    c.pop("reduction")
    inp = si.make_flce_inputs(**c, dtype=dtype)
    n, h, v = inp.hidden.shape[0], inp.hidden.shape[1], inp.weight.shape[0]
    res = run_flce(inp, reduction="mean", chunk=0, keep_f32=True)
    chunk = flce.flce_default_chunk(n, h, v)
    lse, zt = O.lse_rows(inp.hidden, inp.weight, None, np.arange(n), inp.target, row_block=512)
    valid = inp.target != inp.ignore_index
    loss_ref = float(np.where(valid, lse - zt, 0.0).sum() / valid.sum())
    assert res["status"] == 0 and res["n_valid"] == int(valid.sum())
    assert abs(res["loss"] - loss_ref) <= LOSS_RTOL * abs(loss_ref)
    assert np.abs(res["lse"] - lse).max() <= 1e-5 * np.abs(lse).max()
    assert np.abs(res["target_logit"][valid] - zt[valid]).max() <= 1e-5 * np.abs(lse).max()
    rows = sample_rows(n, chunk, 21, k=96)
    ref = O.flce_rows(inp.hidden, inp.weight, None, inp.target, rows, reduction="mean")
    gh = res["grad_hidden"][rows].astype(np.float64)
    assert np.abs(gh - ref["grad_hidden"]).max() <= GRAD_RTOL * np.abs(ref["grad_hidden"]).max()
    assert np.all(gh[~ref["valid"]] == 0.0)
    ids = sample_vocab(inp.target, v, 22)
    gw, _ = O.grad_weight_rows(inp.hidden, inp.weight, None, inp.target, ids, lse, reduction="mean")
    assert np.abs(res["grad_weight"][ids] - gw).max() <= GRAD_RTOL * np.abs(gw).max()


def test_stress_256k_vocab():
    # the large-vocabulary stress shape (Zipf targets, sum): the all-row
    # oracle LSE gives the summed loss and grad_weight / grad_hidden on samples
    inp = si.config_inputs("stress_256k")
    n, h, v = inp.hidden.shape[0], inp.hidden.shape[1], inp.weight.shape[0]
    res = run_flce(inp, reduction="sum", chunk=0, keep_f32=True)
    chunk = flce.flce_default_chunk(n, h, v)
    assert res["status"] == 0
    valid = inp.target != inp.ignore_index
    assert res["n_valid"] == int(valid.sum())
    lse, zt = O.lse_rows(inp.hidden, inp.weight, None, np.arange(n), inp.target, row_block=256)
    loss_ref = float(np.where(valid, lse - zt, 0.0).sum())
    assert abs(res["loss"] - loss_ref) <= LOSS_RTOL * abs(loss_ref)
    assert np.abs(res["lse"] - lse).max() <= 1e-5 * np.abs(lse).max()
    _check_rows(res, inp, sample_rows(n, chunk, 7, k=128), "sum")
    _check_weight_rows(res, inp, sample_vocab(inp.target, v, 8), lse, "sum")
    # every dZ row sums to zero, so the vocabulary rows of grad_W sum to zero
    colsum = res["grad_weight"].sum(axis=0, dtype=np.float64)
    assert np.abs(colsum).max() <= 1e-3 * np.abs(res["grad_weight"]).sum(axis=0, dtype=np.float64).max()
    # scratch stays bounded by the chunk's logits, far below the full logits
    ws = flce.flce_workspace_size(n, h, v, 0, "sum")
    assert ws <= chunk * v * 2 * 1.05 + 8 * n + (1 << 20)
    assert ws < n * v * 2 / 7
    torch.cuda.empty_cache()
