"""GPU parity of ce_fwd_bwd (cross entropy on materialised logits) against the
fp64 oracle: bf16, fp16 and fp32 logits, in place and out of place, loss
only, every reduction; the row-ring, half-row, streaming (two-pass) and
cluster forms, rows that are and are not whole 16-byte vectors."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from oracle import flce_oracle as O
from gpu_util import assert_grad, assert_loss, dev_bf16, host

pytestmark = pytest.mark.gpu


def _logits_dev(logits, dtype):
    if dtype == "bf16":
        return dev_bf16(logits)
    return torch.from_numpy(logits).cuda()  # float32 or float16


def _run(logits, t, dtype, reduction, *, in_place=False, want_grad=True, grad_scale=1.0, grad_out=None):
    z = _logits_dev(logits, dtype)
    keep = z.clone()
    go = torch.from_numpy(grad_out).cuda() if grad_out is not None else None
    out = flce.cross_entropy(z, torch.from_numpy(t).cuda(), reduction=reduction, in_place=in_place,
                             want_grad=want_grad, grad_scale=grad_scale, grad_out=go)
    torch.cuda.synchronize()
    if want_grad and not in_place:
        assert torch.equal(z.view(torch.int16) if dtype == "bf16" else z,
                           keep.view(torch.int16) if dtype == "bf16" else keep), "input logits changed"
    loss = host(out["loss"])
    grad = host(out["grad_logits"]) if want_grad else None
    return loss, grad, int(out["status"].item())


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("in_place", [False, True])
def test_ce_config_1024x32768(dtype, reduction, in_place):
    c = si.CE_CONFIG
    logits, t = si.make_ce_logits(c["n"], c["v"], c["seed"], std=c["std"], dtype=dtype,
                                  ignore_frac=c["ignore_frac"])
    go = si.make_grad_out(c["n"], 3) if reduction == "none" else None
    ref = O.ce_reference(logits, t, reduction=reduction, grad_scale=0.7, grad_out=go)
    loss, grad, status = _run(logits, t, dtype, reduction, in_place=in_place, grad_scale=0.7, grad_out=go)
    assert status == 0
    assert_loss(loss, ref["loss"], reduction)
    assert_grad(grad, ref["dz"], "grad_logits")
    assert np.all(grad[~ref["valid"]] == 0.0)
    if reduction == "none":
        assert np.all(loss[~ref["valid"]] == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("n,v", [(37, 1000), (64, 8192), (5, 8191), (9, 100003), (3, 1), (20, 70000),
                                 (16, 262144), (33, 20004), (33, 40008), (20000, 64), (1, 32768),
                                 (2000, 8), (16384, 72), (16385, 72), (400, 75000), (330, 80001)])
def test_ce_shapes(dtype, n, v):
    logits, t = si.make_ce_logits(n, v, 100 + n, std=2.0, dtype=dtype, ignore_frac=0.2)
    ref = O.ce_reference(logits, t, reduction="mean")
    loss, grad, status = _run(logits, t, dtype, "mean")
    assert status == 0
    assert_loss(loss, ref["loss"], "mean")
    if ref["n_valid"] > 0 and v > 1:
        assert_grad(grad, ref["dz"], "grad_logits")
    assert np.all(grad[~ref["valid"]] == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_ce_loss_only(dtype):
    logits, t = si.make_ce_logits(200, 5000, 4, dtype=dtype)
    ref = O.ce_reference(logits, t, reduction="sum")
    loss, _, status = _run(logits, t, dtype, "sum", want_grad=False)
    assert status == 0
    assert_loss(loss, ref["loss"], "sum")


@pytest.mark.parametrize("n", [1, 151, 152, 153, 1500])
def test_ce_one_launch_row_counts(n):
    # the single-launch form at grids below, at and above the SM count, and
    # with more rows than threads per CTA (the in-kernel count loops)
    logits, t = si.make_ce_logits(n, 4096, 300 + n, std=2.0, dtype="bf16", ignore_frac=0.3)
    for reduction in ("sum", "mean"):
        ref = O.ce_reference(logits, t, reduction=reduction)
        loss, grad, status = _run(logits, t, "bf16", reduction)
        assert status == 0
        assert_loss(loss, ref["loss"], reduction)
        if ref["n_valid"] > 0:
            assert_grad(grad, ref["dz"], "grad_logits")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("n,v", [(7, 17), (300, 1001), (153, 30001), (100, 9999), (64, 4097), (5, 18431),
                                 (40, 50257), (9, 36867), (20, 20001), (11, 32001)])
@pytest.mark.parametrize("in_place", [False, True])
def test_ce_rows_not_whole_vectors(dtype, n, v, in_place):
    # rows whose byte length is not a multiple of 16: the row-ring and
    # half-row kernels load each row's 16-byte-aligned covering range, mask the
    # neighbours' elements and store only their own (in place, a neighbour's
    # gradient must survive)
    logits, t = si.make_ce_logits(n, v, 400 + n + v, std=2.0, dtype=dtype, ignore_frac=0.1)
    for reduction in ("none", "mean"):
        go = si.make_grad_out(n, 5) if reduction == "none" else None
        ref = O.ce_reference(logits, t, reduction=reduction, grad_out=go)
        loss, grad, status = _run(logits, t, dtype, reduction, in_place=in_place, grad_out=go)
        assert status == 0
        assert_loss(loss, ref["loss"], reduction)
        assert_grad(grad, ref["dz"], "grad_logits")
        assert np.all(grad[~ref["valid"]] == 0.0)


def test_ce_out_of_range_target():
    logits, t = si.make_ce_logits(50, 300, 6)
    t[4] = 300
    ref = O.ce_reference(logits, t, reduction="mean")
    loss, grad, status = _run(logits, t, "bf16", "mean")
    assert status & 0x1
    assert_loss(loss, ref["loss"], "mean")
    assert np.all(grad[4] == 0.0)


def test_ce_empty():
    z = torch.empty(0, 100, dtype=torch.bfloat16, device="cuda")
    out = flce.cross_entropy(z, torch.empty(0, dtype=torch.int64, device="cuda"), reduction="sum")
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_ce_workspace_reused_and_dirty(reduction):
    # the single-launch form finds the CTA that adds the loss partials by
    # per-CTA flags set to the call's nonce: a workspace full of garbage, and
    # one left by an earlier call on other data, must not be mistaken for done
    n, v = 1024, 32768
    ws = torch.full((flce.ce_workspace_size(n, v, "bf16", reduction),), 0xFF, dtype=torch.uint8, device="cuda")
    for seed in (11, 12, 13):
        logits, t = si.make_ce_logits(n, v, seed, std=2.0, dtype="bf16", ignore_frac=0.05)
        ref = O.ce_reference(logits, t, reduction=reduction)
        out = flce.cross_entropy(dev_bf16(logits), torch.from_numpy(t).cuda(), reduction=reduction,
                                 workspace=ws)
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        assert_loss(host(out["loss"]), ref["loss"], reduction)
        assert_grad(host(out["grad_logits"]), ref["dz"], "grad_logits")


def test_ce_without_status_word():
    logits, t = si.make_ce_logits(300, 4000, 21, dtype="fp32")
    ref = O.ce_reference(logits, t, reduction="mean")
    z = torch.from_numpy(logits).cuda()
    loss = torch.empty(1, device="cuda")
    ws = torch.empty(flce.ce_workspace_size(300, 4000, "fp32", "mean"), dtype=torch.uint8, device="cuda")
    st = flce.ce_fwd_bwd(z, "fp32", z, torch.from_numpy(t).cuda(), 300, 4000, -100, "mean", 1.0, None, loss,
                         ws, ws.numel(), None, None)
    torch.cuda.synchronize()
    assert st == 0
    assert_loss(host(loss)[0], ref["loss"], "mean")
    assert_grad(host(z), ref["dz"], "grad_logits")


def test_ce_status_in_workspace_when_no_status_word():
    # status_dev NULL: the status lives in the workspace's first 4 bytes and
    # each call starts it from zero (the single-launch form clears it in CTA 0)
    n, v = 50, 300
    ws = torch.full((flce.ce_workspace_size(n, v, "bf16", "mean"),), 0x7F, dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    for bad in (True, False):
        logits, t = si.make_ce_logits(n, v, 6)
        if bad:
            t[4] = v
        z = dev_bf16(logits)
        st = flce.ce_fwd_bwd(z, "bf16", z, torch.from_numpy(t).cuda(), n, v, -100, "mean", 1.0, None, loss, ws,
                             ws.numel(), None, None)
        torch.cuda.synchronize()
        assert st == 0
        word = int(ws[:4].view(torch.int32).item())
        assert word == (0x1 if bad else 0), hex(word)


@pytest.mark.parametrize("n,v", [(1024, 32768), (600, 128256), (20000, 256)])
def test_ce_beside_kernels_holding_sms(n, v):
    # The single-launch form finds its last CTA with a counter that no CTA
    # waits on (a CTA that finds an older call's tag installs this call's
    # itself), so it must give the same result when another stream's kernels
    # hold part of the SMs while its CTAs start: a bounded bf16 matmul
    # launched just before, on a second stream.
    logits, t = si.make_ce_logits(n, v, 700 + n, std=2.0, dtype="bf16", ignore_frac=0.05)
    ref = O.ce_reference(logits, t, reduction="mean")
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    tt = torch.from_numpy(t).cuda()
    torch.cuda.synchronize()
    for _ in range(3):
        z = dev_bf16(logits)
        with torch.cuda.stream(side):
            for _ in range(4):
                a = (a @ a).clamp_(-1.0, 1.0)
        out = flce.cross_entropy(z, tt, reduction="mean", in_place=True)
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        assert_loss(host(out["loss"]), ref["loss"], "mean")
        assert_grad(host(out["grad_logits"]), ref["dz"], "grad_logits")
