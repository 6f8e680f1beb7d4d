"""Vocabulary-parallel building blocks on one GPU: the vocabulary is split
into uneven shards, each shard runs on its own slice, the per-row partials
are combined on the host exactly as a cross-shard all-reduce would (log-sum-
exp of the shard LSEs, sum of the shard target logits), and the shards'
gradients are formed from the combined values.  The assembled result is
compared with the fp64 oracle of the unsharded problem."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_grad, assert_loss, dev_bf16, host

pytestmark = pytest.mark.gpu


def combine_lse(parts):
    """log(sum_s exp(lse_s)) per row, max-shifted (what an all-reduce computes)."""
    a = np.stack(parts).astype(np.float64)
    m = a.max(axis=0)
    return m + np.log(np.exp(a - m).sum(axis=0))


def row_scales(target, reduction, ignore_index=-100, grad_scale=1.0):
    valid = target != ignore_index
    if reduction == "mean":
        s = grad_scale / max(1, int(valid.sum()))
    else:
        s = grad_scale
    return np.where(valid, s, 0.0).astype(np.float32), valid


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("cuts", [(0, 1000, 2200, 3000), (0, 8, 2992, 3000), (0, 1001, 3000), (0, 20004, 40008),
                                  (0, 80001, 160000)])
def test_ce_vocab_parallel(dtype, cuts):
    n, v = (300 if cuts[-1] <= 3000 else 64), cuts[-1]
    logits, t = si.make_ce_logits(n, v, 31, std=2.0, dtype=dtype, ignore_frac=0.1)
    ref = O.ce_reference(logits, t, reduction="mean")
    tt = torch.from_numpy(t).cuda()
    lses, zts, shards = [], [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = np.ascontiguousarray(logits[:, a:b])
        z = dev_bf16(part) if dtype == "bf16" else torch.from_numpy(part).cuda()  # fp32 / fp16
        lse = torch.empty(n, dtype=torch.float32, device="cuda")
        zt = torch.empty(n, dtype=torch.float32, device="cuda")
        assert flce.ce_vp_partials(z, dtype, tt, n, b - a, a, -100, lse, zt, None) == 0
        torch.cuda.synchronize()
        lses.append(lse.cpu().numpy())
        zts.append(zt.cpu().numpy())
        shards.append((a, b, z))
    lse_all = combine_lse(lses)
    zt_all = np.sum(np.stack(zts).astype(np.float64), axis=0)
    scale, valid = row_scales(t, "mean")
    loss = np.where(valid, lse_all - zt_all, 0.0).sum() / valid.sum()
    assert_loss(loss, ref["loss"], "mean")
    assert np.abs(lse_all - ref["lse"]).max() <= 1e-5 * np.abs(ref["lse"]).max()
    lse_d = torch.from_numpy(lse_all.astype(np.float32)).cuda()
    sc_d = torch.from_numpy(scale).cuda()
    grads = []
    for a, b, z in shards:
        g = torch.empty_like(z)
        assert flce.ce_vp_backward(z, dtype, g, tt, n, b - a, a, -100, lse_d, sc_d, None) == 0
        grads.append(g)
    torch.cuda.synchronize()
    grad = np.concatenate([host(g) for g in grads], axis=1)
    assert_grad(grad, ref["dz"], "grad_logits")
    assert np.all(grad[~valid] == 0.0)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_flce_vocab_parallel_two_chunks(reduction):
    n, h, v = 640, 192, 4000
    cuts = (0, 1500, 1508, 4000)          # uneven, including an 8-row shard
    chunk = 384                            # two chunks, the second ragged
    inp = si.make_flce_inputs(n, h, v, 57, w_std=0.05, bias_std=0.1, ignore_frac=0.1)
    ref = O.flce_reference(inp.hidden, inp.weight, inp.bias, inp.target, reduction=reduction)
    w_all = inp.weight
    shards = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        shards.append(dict(a=a, b=b, w=dev_bf16(np.ascontiguousarray(w_all[a:b])),
                           bias=dev_bf16(np.ascontiguousarray(inp.bias[a:b])),
                           gw=torch.empty(b - a, h, dtype=torch.float32, device="cuda"),
                           gb=torch.empty(b - a, dtype=torch.float32, device="cuda")))
    scale_all, valid_all = row_scales(inp.target, reduction)
    grad_hidden = np.zeros((n, h))
    loss_total = 0.0
    for ci, r0 in enumerate(range(0, n, chunk)):
        c = min(chunk, n - r0)
        hid = dev_bf16(np.ascontiguousarray(inp.hidden[r0:r0 + c]))
        tgt = torch.from_numpy(np.ascontiguousarray(inp.target[r0:r0 + c])).cuda()
        parts = []
        for s in shards:
            vs = s["b"] - s["a"]
            wsb = flce.flce_vp_workspace_size(c, h, vs)
            s["ws"] = torch.empty(wsb, dtype=torch.uint8, device="cuda")
            lse = torch.empty(c, device="cuda")
            lse16 = torch.empty(c, device="cuda")
            zt = torch.empty(c, device="cuda")
            st = flce.flce_vp_forward(hid, s["w"], s["bias"], tgt, c, h, vs, s["a"], -100, lse, lse16, zt,
                                      s["ws"], wsb, None)
            assert st == 0
            parts.append((lse, lse16, zt))
        torch.cuda.synchronize()
        lse_c = combine_lse([p[0].cpu().numpy() for p in parts])
        lse16_c = combine_lse([p[1].cpu().numpy() for p in parts])
        zt_c = np.sum(np.stack([p[2].cpu().numpy() for p in parts]).astype(np.float64), axis=0)
        valid = valid_all[r0:r0 + c]
        loss_total += float(np.where(valid, lse_c - zt_c, 0.0).sum())
        assert np.abs(lse_c - ref["lse"][r0:r0 + c]).max() <= 1e-5 * np.abs(ref["lse"]).max()
        lse16_d = torch.from_numpy(lse16_c.astype(np.float32)).cuda()
        sc_d = torch.from_numpy(scale_all[r0:r0 + c]).cuda()
        gh_sum = np.zeros((c, h))
        for s in shards:
            vs = s["b"] - s["a"]
            gh = torch.empty(c, h, dtype=torch.float32, device="cuda")
            st = flce.flce_vp_backward(hid, s["w"], tgt, c, h, vs, s["a"], -100, lse16_d, sc_d, gh, s["gw"],
                                       s["gb"], 1 if ci > 0 else 0, s["ws"], s["ws"].numel(), None)
            assert st == 0
            torch.cuda.synchronize()
            gh_sum += gh.cpu().numpy()
        grad_hidden[r0:r0 + c] = gh_sum
    loss = loss_total / valid_all.sum() if reduction == "mean" else loss_total
    assert_loss(loss, ref["loss"], reduction)
    assert_grad(grad_hidden, ref["grad_hidden"], "grad_hidden")
    gw = np.concatenate([host(s["gw"]) for s in shards], axis=0)
    gb = np.concatenate([host(s["gb"]) for s in shards], axis=0)
    assert_grad(gw, ref["grad_weight"], "grad_weight")
    assert_grad(gb, ref["grad_bias"], "grad_bias")
    assert np.all(grad_hidden[~valid_all] == 0.0)
