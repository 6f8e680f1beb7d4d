"""ce_fwd_bwd_noalloc: the cross entropy entry point for callers that cannot
allocate device memory (an enqueue path that may not allocate, memory owned by
another allocator, a loop that cannot pay for cudaMalloc's synchronisation).
It uses the library's fixed internal scratch array instead of a workspace.

Checked through the C ABI against ce_fwd_bwd on two calls in a row (so the
shared array is reused and must be reset between calls).  This file is named
to be collected last."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from gpu_util import assert_grad, assert_loss, dev_bf16, host


def _with_workspace(z, t, n, v, reduction):
    grad = torch.empty_like(z)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    ws_bytes = flce.ce_workspace_size(n, v, "bf16", reduction)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = flce.ce_fwd_bwd(z, "bf16", grad, t, n, v, -100, reduction, 1.0, None, loss, ws, ws_bytes, None)
    assert st == 0
    return loss, grad


def _without_workspace(z, t, n, v, reduction):
    grad = torch.empty_like(z)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = flce.ce_fwd_bwd_noalloc(z, "bf16", grad, t, n, v, -100, reduction, 1.0, None, loss, status)
    assert st == 0
    return loss, grad, status


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    # one launch for N <= 16384; the counting kernel + ticket form beyond
    cases = [(si.make_ce_logits(1024, 32768, 1002), "mean"), (si.make_ce_logits(300, 5000, 7), "sum"),
             (si.make_ce_logits(20000, 64, 9), "mean"), (si.make_ce_logits(513, 5003, 11), "mean")]
    for (logits, tgt), reduction in cases:
        n, v = logits.shape
        z = dev_bf16(logits)
        t = torch.from_numpy(tgt).cuda()
        ref_loss, ref_grad = _with_workspace(z, t, n, v, reduction)
        loss, grad, status = _without_workspace(z, t, n, v, reduction)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_loss(host(loss)[0], host(ref_loss)[0], reduction)
        assert_grad(host(grad), host(ref_grad), "grad_logits")


@pytest.mark.gpu
def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    n = flce.NOALLOC_MAX_ROWS + 1
    st = flce.ce_fwd_bwd_noalloc(0x10000, "bf16", None, 0x10000, n, 8, -100, "sum", 1.0, None, 0x10000,
                                 None, 0)
    assert st == 2  # FLCE_ERR_UNSUPPORTED, returned before anything is enqueued
