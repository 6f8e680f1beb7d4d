"""Failure detection on the GPU without faulting it: a pipeline wait that can
never be satisfied gives up after its limit and reports through the device
status word, and the context stays usable afterwards."""
import pytest
import torch

import linear_cross_entropy_03_gb300 as flce
import synthetic_inputs as si
from gpu_util import run_flce

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert flce.flce_selftest_wait_timeout(status, 20_000_000) == 0   # 20 ms
    torch.cuda.synchronize()
    assert int(status.item()) == flce.STATUS_BIT_TIMEOUT
    # the context still works
    inp = si.make_flce_inputs(64, 64, 256, 1)
    res = run_flce(inp, reduction="sum")
    assert res["status"] == 0


def test_status_word_is_caller_owned_and_accumulates():
    inp = si.make_flce_inputs(64, 64, 256, 2)
    inp.target[0] = 999
    h = torch.from_numpy(inp.hidden.view("int16")).view(torch.bfloat16).cuda()
    w = torch.from_numpy(inp.weight.view("int16")).view(torch.bfloat16).cuda()
    t = torch.from_numpy(inp.target).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flce.fused_linear_cross_entropy(h, w, t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & flce.STATUS_BIT_TARGET_RANGE
    t[0] = 1
    flce.fused_linear_cross_entropy(h, w, t, status=status)   # not cleared by the library
    torch.cuda.synchronize()
    assert int(status.item()) & flce.STATUS_BIT_TARGET_RANGE
