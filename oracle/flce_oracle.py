"""Oracle for fused linear cross entropy (FLCE) and cross entropy on logits.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference arm may import this module.  It shares
no code, table or helper with the CUDA library and never imports it.

What it computes
----------------
The method makes no approximation: chunking over tokens changes where the
work happens, not what is computed ("liger-kernel 0.0.1 -> 0.1.1" PyPI diff,
README "Key Features", the "Exact" item).  So this oracle is the plain
definition, with no chunking:

* Flatten the hidden states to [N, H] and apply the lm_head,
  z = H W^T (+ b)  ("Peak Performance, Minimized Memory: Optimizing
  torchtune's performance with torch.compile & Liger Kernel", section
  "Introduction to Liger Kernel", Figure 1 "Fused Linear Cross Entropy",
  steps 1-2).
* Cross entropy as PyTorch's CrossEntropyLoss defines it, with ignore_index
  and reduction none / sum / mean (liger-kernel README, "Kernels",
  CrossEntropy item, which links that definition; DeepSpeed PR #8540
  "optional Liger vocab-parallel CE backend", "Changes" and "Real-device
  validation": FP32/FP16/BF16 logits, none/sum/mean, ignored targets).
* Its gradient with respect to the logits, dZ = scale * (softmax - onehot),
  formed in the forward pass (README "Kernels", CrossEntropy item: loss and
  gradient are computed together) and then the chunk gradients
  grad_H = dZ W and grad_W = dZ^T H (torchtune post, Figure 1, steps 3-4),
  plus grad_b = column sums of dZ when a bias is present.

Arithmetic: every input is widened exactly to float64 (bf16 and fp32 both
embed in fp64), every step runs in float64, numpy's matmul is the only
library primitive.  Nothing is rounded back to bf16.

Readings taken where the pages are silent (each is listed with the rest of
the design notes):
* mean divides by the number of valid targets over all N rows; 0 valid
  targets give loss NaN (0/0) and zero gradients;
* reduction none's gradient is that of sum_n g * grad_out[n] * loss_n
  (grad_out NULL means ones); g (grad_scale) multiplies every gradient;
* a target equal to ignore_index is ignored even if it lies in [0, V); a
  target outside [0, V) that is not ignore_index is reported (status
  "target_range") and the row is treated as ignored;
* no label smoothing, z-loss or soft-capping (none is on the pages).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

REDUCTIONS = ("none", "sum", "mean")


# ---------------------------------------------------------------- inputs

def widen(x) -> np.ndarray:
    """Exact float64 copy of a bf16 bit-pattern array (uint16/int16) or a float array."""
    a = np.asarray(x)
    if a.dtype in (np.uint16, np.int16):
        return (a.astype(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------- steps

def _logits(h: np.ndarray, w: np.ndarray, b: Optional[np.ndarray]) -> np.ndarray:
    """z[n, v] = sum_h H[n, h] W[v, h] (+ b[v]): the lm_head projection.

    torchtune post, Figure 1 "Fused Linear Cross Entropy", step 2 (apply the
    projection head to the flattened hidden states).
    """
    z = h @ w.T
    if b is not None:
        z = z + b[None, :]
    return z


def _log_sum_exp(z: np.ndarray) -> np.ndarray:
    """lse_n = m_n + log sum_v exp(z[n, v] - m_n), m_n = max_v z[n, v].

    The normaliser of the softmax in PyTorch's CrossEntropyLoss (README
    "Kernels", CrossEntropy item).
    """
    if z.shape[1] == 0:
        return np.full(z.shape[0], -np.inf)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def _validity(target: np.ndarray, ignore_index: int, vocab: int):
    """valid_n = target_n != ignore_index and 0 <= target_n < V.

    Ignored targets contribute neither loss nor gradient (DeepSpeed PR #8540,
    "Real-device validation": ignored targets).  Returns (valid, status).
    """
    t = np.asarray(target, dtype=np.int64)
    not_ignored = t != ignore_index
    in_range = (t >= 0) & (t < vocab)
    status = "target_range" if bool(np.any(not_ignored & ~in_range)) else "ok"
    return not_ignored & in_range, status


def _target_logits(z: np.ndarray, target: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """z[n, t_n] for valid rows, 0 elsewhere."""
    zt = np.zeros(z.shape[0])
    rows = np.nonzero(valid)[0]
    zt[rows] = z[rows, target[rows]]
    return zt


def _row_losses(lse: np.ndarray, zt: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """loss_n = lse_n - z[n, t_n] for valid rows, exactly 0 for ignored rows."""
    return np.where(valid, lse - zt, 0.0)


def _reduce(loss_rows: np.ndarray, valid: np.ndarray, reduction: str):
    """none -> the vector; sum -> its sum; mean -> sum / (number of valid rows)."""
    if reduction == "none":
        return loss_rows.copy()
    total = float(loss_rows.sum())
    if reduction == "sum":
        return total
    n_valid = int(valid.sum())
    return total / n_valid if n_valid > 0 else math.nan


def _row_scales(valid: np.ndarray, reduction: str, grad_scale: float,
                grad_out: Optional[np.ndarray]) -> np.ndarray:
    """d(reduced loss)/d(loss_n), times the upstream gradient g.

    mean: g / n_valid; sum: g; none: g * grad_out[n] (ones if absent).
    Ignored rows get 0.
    """
    n = valid.shape[0]
    if reduction == "mean":
        n_valid = int(valid.sum())
        s = np.full(n, grad_scale / n_valid if n_valid > 0 else 0.0)
    elif reduction == "sum":
        s = np.full(n, float(grad_scale))
    elif reduction == "none":
        go = np.ones(n) if grad_out is None else widen(grad_out)
        s = grad_scale * go
    else:
        raise ValueError(reduction)
    return np.where(valid, s, 0.0)


def _dlogits(z: np.ndarray, lse: np.ndarray, target: np.ndarray, valid: np.ndarray,
             scale: np.ndarray) -> np.ndarray:
    """dZ[n, v] = scale_n * (exp(z[n, v] - lse_n) - [v == t_n]); ignored rows are 0.

    The gradient the CE kernel writes in place of the logits (README
    "Kernels", CrossEntropy item; torchtune post, Figure 1, step 3).
    """
    p = np.exp(z - lse[:, None])
    rows = np.nonzero(valid)[0]
    p[rows, target[rows]] -= 1.0
    p *= scale[:, None]
    p[~valid] = 0.0
    return p


def _backprop(dz: np.ndarray, h: np.ndarray, w: np.ndarray):
    """grad_H = dZ W, grad_W = dZ^T H, grad_b[v] = sum_n dZ[n, v].

    torchtune post, Figure 1, step 4 (hidden-state gradients, and the
    projection-head gradients accumulated over chunks).
    """
    return dz @ w, dz.T @ h, dz.sum(axis=0)


# ---------------------------------------------------------------- API

def flce_reference(hidden, weight, bias, target, *, ignore_index: int = -100,
                   reduction: str = "mean", grad_scale: float = 1.0,
                   grad_out=None, grad_weight_init=None, grad_bias_init=None) -> dict:
    """Loss and gradients of cross_entropy(H W^T + b, target), all in fp64.

    ``hidden`` [N, H] and ``weight`` [V, H] (and ``bias`` [V]) are bf16 bit
    patterns or float arrays; ``target`` is int64 [N].  ``grad_weight_init``
    and ``grad_bias_init`` model accumulation into existing gradients.
    """
    if reduction not in REDUCTIONS:
        raise ValueError(reduction)
    h, w = widen(hidden), widen(weight)
    b = widen(bias) if bias is not None else None
    t = np.asarray(target, dtype=np.int64)
    z = _logits(h, w, b)
    out = _cross_entropy(z, t, ignore_index, reduction, grad_scale, grad_out)
    gh, gw, gb = _backprop(out["dz"], h, w)
    if grad_weight_init is not None:
        gw = gw + widen(grad_weight_init)
    if grad_bias_init is not None:
        gb = gb + widen(grad_bias_init)
    out.update(grad_hidden=gh, grad_weight=gw, grad_bias=gb if b is not None else None,
               logits=z)
    return out


def ce_reference(logits, target, *, ignore_index: int = -100, reduction: str = "mean",
                 grad_scale: float = 1.0, grad_out=None) -> dict:
    """Cross entropy and its logits gradient on materialised logits [N, V].

    The standalone CE kernel of the README "Kernels" list (CrossEntropy item):
    loss and grad_logits computed in one call.
    """
    if reduction not in REDUCTIONS:
        raise ValueError(reduction)
    z = widen(logits)
    return _cross_entropy(z, np.asarray(target, dtype=np.int64), ignore_index,
                          reduction, grad_scale, grad_out)


def _cross_entropy(z, t, ignore_index, reduction, grad_scale, grad_out) -> dict:
    n, v = z.shape
    valid, status = _validity(t, ignore_index, v)
    lse = _log_sum_exp(z)
    zt = _target_logits(z, t, valid)
    loss_rows = _row_losses(lse, zt, valid)
    loss = _reduce(loss_rows, valid, reduction)
    scale = _row_scales(valid, reduction, grad_scale, grad_out)
    dz = _dlogits(z, lse, t, valid, scale)
    return dict(loss=loss, loss_rows=loss_rows, lse=lse, target_logit=zt, dz=dz,
                valid=valid, n_valid=int(valid.sum()), scale=scale, status=status)


# ------------------------------------------- sampled forms for large shapes
#
# At the largest shapes the full fp64 product is ~1e13-1e14 flops.  These
# helpers compute the same definitions for chosen rows of the output (each
# row of z depends on one row of H only) or chosen vocabulary rows of grad_W
# (which need every row's LSE, passed in from ``lse_rows``).

def lse_rows(hidden, weight, bias, rows, target=None, *, row_block: int = 256):
    """lse_n and z[n, t_n] for the given rows, in blocks of ``row_block`` rows."""
    w = widen(weight)
    b = widen(bias) if bias is not None else None
    rows = np.asarray(rows, dtype=np.int64)
    lse = np.empty(rows.size)
    zt = np.zeros(rows.size)
    for s in range(0, rows.size, row_block):
        r = rows[s:s + row_block]
        z = _logits(widen(hidden[r]), w, b)
        lse[s:s + r.size] = _log_sum_exp(z)
        if target is not None:
            t = np.asarray(target, dtype=np.int64)[r]
            ok = (t >= 0) & (t < w.shape[0])
            zt[s:s + r.size][ok] = z[np.nonzero(ok)[0], t[ok]]
    return lse, zt


def flce_rows(hidden, weight, bias, target, rows, *, ignore_index: int = -100,
              reduction: str = "mean", grad_scale: float = 1.0, grad_out=None) -> dict:
    """Per-row loss, LSE and grad_H rows for the given rows only.

    n_valid (for mean) is counted over all N targets, as in the full form.
    """
    t_all = np.asarray(target, dtype=np.int64)
    w = widen(weight)
    b = widen(bias) if bias is not None else None
    valid_all, status = _validity(t_all, ignore_index, w.shape[0])
    scale_all = _row_scales(valid_all, reduction, grad_scale, grad_out)
    rows = np.asarray(rows, dtype=np.int64)
    z = _logits(widen(hidden[rows]), w, b)
    lse = _log_sum_exp(z)
    valid = valid_all[rows]
    t = t_all[rows]
    zt = _target_logits(z, t, valid)
    dz = _dlogits(z, lse, t, valid, scale_all[rows])
    return dict(lse=lse, target_logit=zt, loss_rows=_row_losses(lse, zt, valid),
                grad_hidden=dz @ w, valid=valid, status=status)


def grad_weight_rows(hidden, weight, bias, target, vocab_ids, lse_all, *,
                     ignore_index: int = -100, reduction: str = "mean",
                     grad_scale: float = 1.0, grad_out=None,
                     row_block: int = 4096):
    """grad_W[v, :] and grad_b[v] for the given vocabulary ids.

    dZ[:, v] needs every row's LSE, which the caller passes (``lse_all``,
    from ``lse_rows`` over all rows).
    """
    t = np.asarray(target, dtype=np.int64)
    w = widen(weight)
    ids = np.asarray(vocab_ids, dtype=np.int64)
    valid, _ = _validity(t, ignore_index, w.shape[0])
    scale = _row_scales(valid, reduction, grad_scale, grad_out)
    wv = w[ids]
    bv = widen(bias)[ids] if bias is not None else None
    gw = np.zeros((ids.size, w.shape[1]))
    gb = np.zeros(ids.size)
    for s in range(0, t.size, row_block):
        e = min(t.size, s + row_block)
        h = widen(hidden[s:e])
        z = _logits(h, wv, bv)                                   # [rows, ids]
        p = np.exp(z - lse_all[s:e, None])
        p -= ((t[s:e, None] == ids[None, :]) & valid[s:e, None]).astype(np.float64)
        p *= scale[s:e, None]
        p[~valid[s:e]] = 0.0
        gw += p.T @ h
        gb += p.sum(axis=0)
    return gw, gb


def full_logits_bytes(n_tokens: int, vocab: int, elem_bytes: int = 2) -> int:
    """Bytes of the [N, V] logits tensor that the fused method never builds."""
    return int(n_tokens) * int(vocab) * int(elem_bytes)
