"""Checks that pin the oracle to facts other than itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError
when the oracle disagrees with a closed form, an invariant, brute-force
finite differences or the textbook library routine (PyTorch's
cross_entropy in float64).  test_oracle.py runs them on the real oracle;
test_oracle_mutations.py plants mistakes in the oracle and checks that at
least one pin fails for each.
"""
from __future__ import annotations

import math

import numpy as np

import synthetic_inputs as si

REDUCTIONS = ("none", "sum", "mean")


def _small_problem(n=37, h=16, v=50, seed=7, ignore_frac=0.2, bias=True):
    inp = si.make_flce_inputs(n, h, v, seed, w_std=0.3, bias_std=0.5 if bias else None,
                              ignore_frac=ignore_frac)
    return inp


def _scales(valid, reduction, g, go):
    n_valid = int(valid.sum())
    if reduction == "mean":
        s = np.full(valid.size, g / n_valid)
    elif reduction == "sum":
        s = np.full(valid.size, g)
    else:
        s = g * go
    return np.where(valid, s, 0.0)


def pin_zero_weight_closed_form(O):
    """W = 0, b = 0 => every logit is 0 => loss_n = ln V exactly, grad_H = 0,
    grad_W[v] = sum_valid s_n (1/V - [t_n = v]) H[n], grad_b[v] = sum_valid s_n (1/V - [t_n = v])."""
    n, h, v = 41, 24, 64
    inp = _small_problem(n, h, v, seed=11)
    hidden = si.bf16_to_float32(inp.hidden).astype(np.float64)
    w0 = np.zeros((v, h))
    b0 = np.zeros(v)
    go = si.make_grad_out(n, 3).astype(np.float64)
    g = 0.75
    t = inp.target
    valid = t != inp.ignore_index
    for red in REDUCTIONS:
        r = O.flce_reference(hidden, w0, b0, t, reduction=red, grad_scale=g,
                             grad_out=go if red == "none" else None)
        ln_v = math.log(v)
        rows = np.asarray(r["loss_rows"])
        assert np.all(rows[valid] == ln_v), "loss_n must be ln V exactly"
        assert np.all(rows[~valid] == 0.0), "ignored rows carry no loss"
        nv = int(valid.sum())
        if red == "mean":
            assert abs(r["loss"] - ln_v) <= 1e-14 * ln_v
        elif red == "sum":
            assert abs(r["loss"] - nv * ln_v) <= 1e-13 * nv * ln_v
        else:
            assert np.array_equal(np.asarray(r["loss"]), rows)
        assert np.all(r["grad_hidden"] == 0.0), "grad_H must vanish when W = 0"
        s = _scales(valid, red, g, go)
        gw = np.zeros((v, h))
        gb = np.zeros(v)
        for i in range(n):
            if not valid[i]:
                continue
            gw += s[i] / v * hidden[i][None, :]
            gw[t[i]] -= s[i] * hidden[i]
            gb += s[i] / v
            gb[t[i]] -= s[i]
        scale_w = max(1e-300, np.abs(gw).max())
        assert np.abs(r["grad_weight"] - gw).max() <= 1e-12 * scale_w, "grad_W closed form"
        assert np.abs(r["grad_bias"] - gb).max() <= 1e-12 * max(1e-300, np.abs(gb).max()), "grad_b closed form"


def pin_dlogit_rows(O):
    """Each valid dZ row sums to 0; ignored rows of dZ, loss and grad_H are exactly 0."""
    inp = _small_problem(seed=13)
    for red in REDUCTIONS:
        r = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction=red)
        valid = inp.target != inp.ignore_index
        dz = r["dz"]
        sums = dz.sum(axis=1)
        assert np.abs(sums[valid]).max() <= 1e-12 * max(1e-300, np.abs(dz).max()), "row sums"
        assert np.all(dz[~valid] == 0.0)
        assert np.all(np.asarray(r["loss_rows"])[~valid] == 0.0)
        assert np.all(r["grad_hidden"][~valid] == 0.0)
        # softmax part: dZ / s + onehot is a probability vector
        s = r["scale"][valid][:, None]
        p = dz[valid] / s
        p[np.arange(p.shape[0]), inp.target[valid]] += 1.0
        assert p.min() >= -1e-15 and np.abs(p.sum(axis=1) - 1).max() <= 1e-12


def pin_reduction_relations(O):
    """sum = sum of none; mean = sum / n_valid; the gradients follow the same weights."""
    inp = _small_problem(seed=17)
    valid = inp.target != inp.ignore_index
    nv = int(valid.sum())
    none = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction="none")
    sm = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction="sum")
    mn = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction="mean")
    assert abs(sm["loss"] - np.sum(none["loss"])) <= 1e-12 * abs(sm["loss"])
    assert abs(mn["loss"] - sm["loss"] / nv) <= 1e-12 * abs(mn["loss"])
    go = np.full(inp.target.size, 1.0 / nv)
    none_w = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction="none",
                              grad_out=go)
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        ref = mn[k]
        assert np.abs(none_w[k] - ref).max() <= 1e-12 * np.abs(ref).max(), k
        assert np.abs(sm[k] / nv - ref).max() <= 1e-12 * np.abs(ref).max(), k


def pin_shift_invariance(O):
    """Adding c to every bias, or the same vector u to every row of W, shifts each
    row's logits by a constant: loss, dZ, grad_W and grad_b are unchanged, and
    grad_H is unchanged because every dZ row sums to 0."""
    rng = np.random.default_rng(5)
    n, h, v = 9, 6, 11
    hid = rng.normal(size=(n, h))
    w = rng.normal(size=(v, h))
    b = rng.normal(size=v)
    t = rng.integers(0, v, n)
    t[2] = -100
    u = rng.normal(size=h)
    for red in REDUCTIONS:
        base = O.flce_reference(hid, w, b, t, reduction=red)
        for kw in (dict(weight=w, bias=b + 3.25), dict(weight=w + u[None, :], bias=b)):
            other = O.flce_reference(hid, kw["weight"], kw["bias"], t, reduction=red)
            assert np.allclose(np.asarray(base["loss"]), np.asarray(other["loss"]), rtol=1e-12, atol=1e-12)
            for k in ("dz", "grad_hidden", "grad_weight", "grad_bias"):
                assert np.abs(base[k] - other[k]).max() <= 1e-10 * max(1.0, np.abs(base[k]).max()), k


def _loss_scalar(O, hid, w, b, t, red, g, go):
    r = O.flce_reference(hid, w, b, t, reduction=red, grad_scale=g, grad_out=go)
    if red == "none":
        return float(np.sum(g * go * np.asarray(r["loss_rows"])))
    return g * float(r["loss"])


def pin_finite_differences(O):
    """Central differences of the (weighted) loss in fp64 on a tiny problem match
    grad_H, grad_W and grad_b for every reduction."""
    rng = np.random.default_rng(3)
    n, h, v = 3, 4, 5
    hid = rng.normal(size=(n, h))
    w = rng.normal(size=(v, h))
    b = rng.normal(size=v)
    t = np.array([4, -100, 1], dtype=np.int64)
    go = np.array([0.7, 1.3, 1.9])
    g = 1.5
    eps = 1e-6
    for red in REDUCTIONS:
        r = O.flce_reference(hid, w, b, t, reduction=red, grad_scale=g,
                             grad_out=go if red == "none" else None)
        for name, arr, grad in (("hidden", hid, r["grad_hidden"]), ("weight", w, r["grad_weight"]),
                                ("bias", b, r["grad_bias"])):
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                plus, minus = arr.copy(), arr.copy()
                plus[idx] += eps
                minus[idx] -= eps
                args_p = dict(hidden=hid, weight=w, bias=b)
                args_m = dict(hidden=hid, weight=w, bias=b)
                args_p[name], args_m[name] = plus, minus
                lp = g * _loss_scalar(O, args_p["hidden"], args_p["weight"], args_p["bias"], t, red, 1.0, go)
                lm = g * _loss_scalar(O, args_m["hidden"], args_m["weight"], args_m["bias"], t, red, 1.0, go)
                num[idx] = (lp - lm) / (2 * eps)
            err = np.abs(num - grad).max()
            assert err <= 1e-6 * max(1.0, np.abs(grad).max()), f"{red} {name}: {err}"


def pin_torch_cross_entropy(O):
    """Matches PyTorch's float64 cross_entropy + autograd (the routine the CE
    kernel's definition points to) for every reduction, with ignored rows."""
    import torch
    import torch.nn.functional as F
    inp = _small_problem(n=29, h=12, v=40, seed=19)
    hid = torch.tensor(si.bf16_to_float32(inp.hidden).astype(np.float64), requires_grad=True)
    w = torch.tensor(si.bf16_to_float32(inp.weight).astype(np.float64), requires_grad=True)
    b = torch.tensor(si.bf16_to_float32(inp.bias).astype(np.float64), requires_grad=True)
    t = torch.tensor(inp.target)
    go = si.make_grad_out(inp.target.size, 4).astype(np.float64)
    for red in REDUCTIONS:
        for p in (hid, w, b):
            p.grad = None
        z = hid @ w.T + b
        loss = F.cross_entropy(z, t, ignore_index=inp.ignore_index, reduction=red)
        upstream = torch.tensor(0.5 * go) if red == "none" else torch.tensor(0.5, dtype=torch.float64)
        loss.backward(upstream)
        r = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction=red,
                             grad_scale=0.5, grad_out=go if red == "none" else None)
        ref_loss = loss.detach().numpy()
        assert np.allclose(np.asarray(r["loss"]), ref_loss, rtol=1e-12, atol=1e-14), red
        for ours, theirs in ((r["grad_hidden"], hid.grad), (r["grad_weight"], w.grad), (r["grad_bias"], b.grad)):
            th = theirs.numpy()
            assert np.abs(ours - th).max() <= 1e-12 * max(1e-300, np.abs(th).max()), red


def pin_index_encoding(O):
    """H[n] = (1, 256, 0...), W[v] = (v mod 256, v div 256, 0...) gives z[n, v] = v
    exactly, so the gathered target logit equals the target id."""
    n, h, v = 64, 16, 70000
    hid = np.zeros((n, h))
    hid[:, 0] = 1.0
    hid[:, 1] = 256.0
    w = np.zeros((v, h))
    ids = np.arange(v)
    w[:, 0] = ids % 256
    w[:, 1] = ids // 256
    t = si.uniform_targets(1, 9, n, v)
    t[5] = -100
    rows = np.arange(n)
    r = O.flce_rows(hid, w, None, t, rows, reduction="sum")
    valid = t != -100
    assert np.array_equal(r["target_logit"][valid], t[valid].astype(np.float64))
    assert np.all(r["target_logit"][~valid] == 0.0)
    # the LSE of 0..V-1 in closed form: (V-1) + log(sum_k e^{-k}) = (V-1) + log(1/(1-e^-1)) (to fp64)
    expect = (v - 1) - math.log1p(-math.exp(-1.0))
    assert np.allclose(r["lse"], expect, rtol=1e-15, atol=1e-9)


def pin_ce_on_logits(O):
    """CE on materialised logits: constant logits give ln V; bf16 and fp32 logits
    match PyTorch float64 cross_entropy and its gradient."""
    import torch
    import torch.nn.functional as F
    n, v = 19, 33
    t = si.uniform_targets(2, 3, n, v)
    t[[1, 7]] = -100
    valid = t != -100
    r = O.ce_reference(np.zeros((n, v)), t, reduction="none")
    assert np.all(np.asarray(r["loss"])[valid] == math.log(v))
    r = O.ce_reference(np.full((n, v), 0.8125), t, reduction="none")
    assert np.abs(np.asarray(r["loss"])[valid] - math.log(v)).max() <= 4e-16 * 4
    for dtype in ("bf16", "fp16", "fp32"):
        logits, tt = si.make_ce_logits(n, v, 21, std=2.0, dtype=dtype, ignore_frac=0.15)
        z64 = si.bf16_to_float32(logits).astype(np.float64) if dtype == "bf16" else logits.astype(np.float64)
        for red in REDUCTIONS:
            zt = torch.tensor(z64, requires_grad=True)
            loss = F.cross_entropy(zt, torch.tensor(tt), ignore_index=-100, reduction=red)
            loss.backward(torch.ones_like(loss) * 2.0)
            r = O.ce_reference(logits, tt, reduction=red, grad_scale=2.0)
            assert np.allclose(np.asarray(r["loss"]), loss.detach().numpy(), rtol=1e-12, atol=1e-14)
            assert np.abs(r["dz"] - zt.grad.numpy()).max() <= 1e-13


def pin_edge_cases(O):
    """All targets ignored: mean is NaN (0/0), sum is 0, gradients are 0.
    V = 1: softmax is 1, so loss and gradients are 0.  An ignore_index inside
    [0, V) is ignored.  An out-of-range target is reported and ignored."""
    rng = np.random.default_rng(1)
    hid = rng.normal(size=(4, 3))
    w = rng.normal(size=(6, 3))
    t = np.full(4, -100, dtype=np.int64)
    r = O.flce_reference(hid, w, None, t, reduction="mean")
    assert math.isnan(r["loss"]) and np.all(r["grad_weight"] == 0) and np.all(r["grad_hidden"] == 0)
    assert O.flce_reference(hid, w, None, t, reduction="sum")["loss"] == 0.0
    r = O.flce_reference(hid, w[:1], None, np.zeros(4, dtype=np.int64), reduction="sum")
    assert abs(r["loss"]) <= 1e-15 and np.abs(r["grad_hidden"]).max() <= 1e-15
    t2 = np.array([2, 2, 5, 0], dtype=np.int64)
    r2 = O.flce_reference(hid, w, None, t2, ignore_index=2, reduction="none")
    assert np.all(np.asarray(r2["loss"])[:2] == 0.0) and r2["n_valid"] == 2
    t3 = np.array([1, 6, -7, 0], dtype=np.int64)
    r3 = O.flce_reference(hid, w, None, t3, reduction="none")
    assert r3["status"] == "target_range" and r3["n_valid"] == 2
    assert np.all(np.asarray(r3["loss"])[1:3] == 0.0)
    r4 = O.ce_reference(np.zeros((0, 5)), np.zeros(0, dtype=np.int64), reduction="sum")
    assert r4["loss"] == 0.0


def pin_sampled_forms(O):
    """The row-sampled helpers used at large shapes agree with the full form."""
    inp = _small_problem(n=50, h=16, v=70, seed=23)
    for red in REDUCTIONS:
        full = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction=red)
        rows = np.array([0, 3, 17, 49])
        part = O.flce_rows(inp.hidden, inp.weight, inp.bias, inp.target, rows, reduction=red)
        assert np.allclose(part["lse"], full["lse"][rows], rtol=1e-14)
        assert np.allclose(part["loss_rows"], np.asarray(full["loss_rows"])[rows], rtol=1e-13, atol=1e-15)
        assert np.abs(part["grad_hidden"] - full["grad_hidden"][rows]).max() <= 1e-13 * np.abs(full["grad_hidden"]).max()
        lse, zt = O.lse_rows(inp.hidden, inp.weight, inp.bias, np.arange(50), inp.target, row_block=7)
        assert np.allclose(lse, full["lse"], rtol=1e-14)
        ids = np.array([0, 5, 69])
        gw, gb = O.grad_weight_rows(inp.hidden, inp.weight, inp.bias, inp.target, ids, lse,
                                    reduction=red, row_block=8)
        assert np.abs(gw - full["grad_weight"][ids]).max() <= 1e-13 * np.abs(full["grad_weight"]).max()
        assert np.abs(gb - full["grad_bias"][ids]).max() <= 1e-13 * np.abs(full["grad_bias"]).max()


ALL_PINS = [pin_zero_weight_closed_form, pin_dlogit_rows, pin_reduction_relations,
            pin_shift_invariance, pin_finite_differences, pin_torch_cross_entropy,
            pin_index_encoding, pin_ce_on_logits, pin_edge_cases, pin_sampled_forms]
