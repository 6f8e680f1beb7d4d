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


def _dev(logits, dtype):
    return dev_bf16(logits) if dtype == "bf16" else torch.from_numpy(logits).cuda()


def _with_workspace(z, t, n, v, dtype, reduction, grad_out):
    grad = torch.empty_like(z)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    ws_bytes = flce.ce_workspace_size(n, v, dtype, reduction)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = flce.ce_fwd_bwd(z, dtype, grad, t, n, v, -100, reduction, 1.0, grad_out, loss, ws, ws_bytes, None)
    assert st == 0
    return loss, grad


def _without_workspace(z, t, n, v, dtype, reduction, grad_out, with_status):
    grad = torch.empty_like(z)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
    st = flce.ce_fwd_bwd_noalloc(z, dtype, grad, t, n, v, -100, reduction, 1.0, grad_out, loss, status)
    assert st == 0
    return loss, grad, status


# (n, v, seed, dtype, reduction, status word): one launch for N <= 16384 (row
# ring up to 72 KB rows, streaming form beyond); the counting kernel + ticket
# form for more rows, with both row forms
CASES = [(1024, 32768, 1002, "bf16", "mean", True), (300, 5000, 7, "bf16", "sum", True),
         (20000, 64, 9, "bf16", "mean", True), (513, 5003, 11, "bf16", "mean", True),
         (700, 3000, 13, "bf16", "none", True), (400, 8192, 15, "bf16", "mean", False),
         (256, 30000, 17, "fp32", "sum", True), (16400, 40000, 19, "bf16", "mean", True)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    for n, v, seed, dtype, reduction, with_status in CASES:
        logits, tgt = si.make_ce_logits(n, v, seed, dtype=dtype)
        z = _dev(logits, dtype)
        t = torch.from_numpy(tgt).cuda()
        go = torch.from_numpy(si.make_grad_out(n, seed)).cuda() if reduction == "none" else None
        ref_loss, ref_grad = _with_workspace(z, t, n, v, dtype, reduction, go)
        for _ in range(2):  # the second call finds the first call's contents in the shared array
            loss, grad, status = _without_workspace(z, t, n, v, dtype, reduction, go, with_status)
            torch.cuda.synchronize()
            if with_status:
                assert int(status.item()) == 0
            if reduction == "none":
                assert_loss(host(loss), host(ref_loss), reduction)
            else:
                assert_loss(host(loss)[0], host(ref_loss)[0], reduction)
            assert_grad(host(grad), host(ref_grad), "grad_logits")
        del z, ref_grad, grad
        torch.cuda.empty_cache()


@pytest.mark.gpu
def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    n = flce.NOALLOC_MAX_ROWS + 1
    st = flce.ce_fwd_bwd_noalloc(0x10000, "bf16", None, 0x10000, n, 8, -100, "sum", 1.0, None, 0x10000,
                                 None, 0)
    assert st == 2  # FLCE_ERR_UNSUPPORTED, returned before anything is enqueued


@pytest.mark.gpu
def test_noalloc_calls_leave_free_device_memory_unchanged():
    # every buffer is made first and every kernel form is loaded by a first
    # round of calls; later calls must not change the device's free memory
    forms = [(1024, 32768, 21, "bf16", "mean"), (64, 200000, 23, "bf16", "sum"), (20000, 64, 25, "bf16", "none")]
    bufs = []
    for n, v, seed, dtype, reduction in forms:
        logits, tgt = si.make_ce_logits(n, v, seed, dtype=dtype)
        z = _dev(logits, dtype)
        t = torch.from_numpy(tgt).cuda()
        go = torch.from_numpy(si.make_grad_out(n, seed)).cuda() if reduction == "none" else None
        loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        bufs.append((z, torch.empty_like(z), t, n, v, dtype, reduction, go, loss, status))

    def call_all():
        for z, grad, t, n, v, dtype, reduction, go, loss, status in bufs:
            assert flce.ce_fwd_bwd_noalloc(z, dtype, grad, t, n, v, -100, reduction, 1.0, go, loss, status) == 0
        torch.cuda.synchronize()

    call_all()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        call_all()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert all(int(b[-1].item()) == 0 for b in bufs)
