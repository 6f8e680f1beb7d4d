"""The C-ABI library on the CPU: it loads, exports every declared entry point,
rejects bad arguments before touching the GPU, and sizes its workspace by the
chunk, not by N * V."""
import ctypes
import json
import os
import re

import pytest

import linear_cross_entropy_03_gb300 as flce
from linear_cross_entropy_03_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")
FAKE = 0x10000  # 256-byte aligned, never dereferenced by the rejected calls


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return flce.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "flce_fwd_bwd" in names and "ce_fwd_bwd" in names and "flce_workspace_size" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/flce.h but not exported"
    assert flce.flce_version() >= 100


def test_status_strings(lib):
    for code in range(8):
        s = flce.flce_status_string(code)
        assert s.startswith("FLCE_")
    assert flce.flce_status_string(99) == "FLCE_UNKNOWN_STATUS"
    assert flce.flce_kernel_name(1) == "gemm_forward"


def _flce(**kw):
    args = dict(hidden=FAKE, weight=FAKE, bias=None, target=FAKE, N=16, H=64, V=100, ignore_index=-100,
                reduction=2, chunk=0, grad_scale=1.0, grad_out_none=None, loss=FAKE, grad_hidden=None,
                grad_weight=None, grad_bias=None, accumulate=0, n_valid_out=None, lse_out=None,
                target_logit_out=None, workspace=FAKE, workspace_bytes=1 << 40, status_dev=None, stream=0)
    args.update(kw)
    return flce.flce_fwd_bwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(N=-1), 1), (dict(V=0), 1), (dict(H=0), 1), (dict(H=60), 2), (dict(reduction=3), 1),
    (dict(chunk=-2), 1), (dict(loss=None), 1), (dict(weight=None), 1), (dict(hidden=None), 1),
    (dict(target=None), 1), (dict(grad_bias=FAKE), 1), (dict(grad_out_none=FAKE), 1),
    (dict(accumulate=2), 1), (dict(hidden=FAKE + 8), 7), (dict(weight=FAKE + 2), 7),
    (dict(grad_weight=FAKE + 4), 7), (dict(target=FAKE + 4), 7), (dict(workspace=None), 3),
    (dict(workspace=FAKE + 64), 3), (dict(workspace_bytes=100), 3),
])
def test_flce_rejects_bad_arguments(lib, kw, code):
    assert _flce(**kw) == code


def test_flce_typed_rejects_other_dtypes(lib):
    base = dict(hidden=FAKE, weight=FAKE, bias=None, target=FAKE, N=16, H=64, V=100, ignore_index=-100,
                reduction=2, chunk=0, grad_scale=1.0, grad_out_none=None, loss=FAKE, grad_hidden=None,
                grad_weight=None, grad_bias=None, accumulate=0, n_valid_out=None, lse_out=None,
                target_logit_out=None, workspace=FAKE, workspace_bytes=1 << 40, status_dev=None, stream=0)
    assert flce.flce_fwd_bwd_typed(7, **base) == 2
    assert flce.flce_fwd_bwd_typed(-1, **base) == 2
    for dt in ("fp16", "fp32"):
        assert flce.flce_fwd_bwd_typed(dt, **dict(base, N=-1)) == 1
        assert flce.flce_fwd_bwd_typed(dt, **dict(base, hidden=FAKE + 8)) == 7
        assert flce.flce_fwd_bwd_typed(dt, **dict(base, workspace_bytes=100)) == 3


def test_flce_typed_workspace_holds_fp32_copies(lib):
    n, h, v = 1000, 256, 5000
    base = flce.flce_workspace_size(n, h, v, 0, "mean")
    assert flce.flce_workspace_size_typed("bf16", n, h, v, 0, "mean") == base
    assert flce.flce_workspace_size_typed("fp16", n, h, v, 0, "mean") == base
    # rounded fp32 operands: one bf16 copy of hidden, weight and bias
    f32r = flce.flce_workspace_size_typed("fp32_rounded", n, h, v, 0, "mean")
    assert base + 2 * (n * h + v * h + v) <= f32r <= base + 2 * (n * h + v * h + v) + 3 * 256 + 2 * 64
    # split fp32 operands: bf16 hi + lo planes of hidden and weight, and a
    # second plane of chunk logits (the lower halves of their fp32 bits)
    f32 = flce.flce_workspace_size_typed("fp32", n, h, v, 0, "mean")
    chunk = flce.flce_default_chunk(n, h, v)
    vp = -(-v // 8) * 8
    extra = 4 * (n * h + v * h) + 2 * chunk * vp
    assert base + extra - 256 <= f32 <= base + extra + 4 * 256  # (256-byte rounding of each region)
    assert flce.flce_workspace_size_typed(7, n, h, v, 0, "mean") == 0
    assert flce.flce_workspace_size_typed("fp32", -1, h, v, 0, "mean") == 0


def _ce(**kw):
    args = dict(logits=FAKE, dtype=0, grad_logits=FAKE, target=FAKE, N=16, V=100, ignore_index=-100,
                reduction=2, grad_scale=1.0, grad_out_none=None, loss=FAKE, workspace=FAKE,
                workspace_bytes=1 << 40, status_dev=None, stream=0)
    args.update(kw)
    return flce.ce_fwd_bwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), 2), (dict(N=-3), 1), (dict(V=0), 1), (dict(reduction=7), 1), (dict(loss=None), 1),
    (dict(logits=None), 1), (dict(grad_out_none=FAKE), 1), (dict(logits=FAKE + 1), 7),
    (dict(grad_logits=FAKE + 100), 1), (dict(workspace_bytes=8), 3), (dict(workspace=None), 3),
])
def test_ce_rejects_bad_arguments(lib, kw, code):
    assert _ce(**kw) == code


def test_selftest_rejects_bad_arguments(lib):
    assert flce.flce_selftest_wait_timeout(None, 1000, 0) == 1
    assert flce.flce_selftest_wait_timeout(FAKE, 0, 0) == 1


def test_workspace_grows_with_chunk_not_n_times_v(lib):
    golden = json.load(open(os.path.join(ROOT, "tests", "golden", "page_figures.json")))
    e = golden["logits_example"]
    n, v, h = e["batch"] * e["seq_len"], e["vocab"], 4096
    full_logits = n * v * e["bytes_per_logit"]                      # the 16.8 GB of the page
    ws = flce.flce_workspace_size(n, h, v, 2048, "sum")
    # the chunk's bf16 logits, its per-row LSE partials (16 bytes per 256
    # columns at H = 4096, well under 1/16 of the logits' bytes), O(N) per-row terms and, with
    # 2048-token chunks, two K slices of grad_H partial sums (fp32 [2048, H] each)
    assert 2048 * v * 2 <= ws <= 2048 * v * 2 * (1 + 1 / 16 + 0.01) + 4 * n + 2 * 2048 * h * 4 + (1 << 20)
    assert ws < full_logits / 14
    ws2 = flce.flce_workspace_size(2 * n, h, v, 2048, "sum")
    assert ws2 - ws < 8 * n + 4096                                  # only O(N) per-row terms grow
    assert flce.flce_workspace_size(n, h, v, 4096, "sum") > 1.8 * ws
    assert flce.flce_workspace_size(n, h, v, 2048, "none") < ws    # no per-row loss buffer
    assert flce.flce_workspace_size(-1, h, v, 0, "sum") == 0
    c = flce.flce_default_chunk(16384, 4096, 128256)
    assert c == 8192 and c * 128256 * 2 <= (2 << 30)
    assert flce.flce_default_chunk(32768, 4096, 256000) == 4096
    assert flce.flce_default_chunk(100, 64, 1000) == 100
    assert flce.ce_workspace_size(1024, 32768, "bf16", "mean") < 16 * 1024
