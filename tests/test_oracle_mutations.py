"""Plants plausible mistakes in the oracle (on the CPU) and checks that the
pins catch every one of them: a dropped term, a wrong sign or index, a
wrong denominator, a missing mask, a transposed or permuted operand."""
import numpy as np
import pytest

import oracle.flce_oracle as O
from oracle_pins import ALL_PINS

_real = {k: getattr(O, k) for k in ("_logits", "_log_sum_exp", "_validity", "_target_logits",
                                     "_row_losses", "_reduce", "_row_scales", "_dlogits", "_backprop")}


def _dlogits_no_onehot(z, lse, target, valid, scale):
    p = np.exp(z - lse[:, None]) * scale[:, None]
    p[~valid] = 0.0
    return p


def _dlogits_flipped(z, lse, target, valid, scale):
    return -_real["_dlogits"](z, lse, target, valid, scale)


def _validity_range_only(target, ignore_index, vocab):
    t = np.asarray(target, dtype=np.int64)
    return (t >= 0) & (t < vocab), "ok"


def _dlogits_unmasked(z, lse, target, valid, scale):
    p = np.exp(z - lse[:, None])
    rows = np.nonzero(valid)[0]
    p[rows, target[rows]] -= 1.0
    return p * np.where(scale == 0, scale.max(), scale)[:, None]


def _reduce_mean_over_n(loss_rows, valid, reduction):
    if reduction == "mean":
        return float(loss_rows.sum()) / loss_rows.size
    return _real["_reduce"](loss_rows, valid, reduction)


def _row_scales_mean_over_n(valid, reduction, grad_scale, grad_out):
    if reduction == "mean":
        return np.where(valid, grad_scale / valid.size, 0.0)
    return _real["_row_scales"](valid, reduction, grad_scale, grad_out)


def _logits_no_bias(h, w, b):
    return h @ w.T


def _target_off_by_one(z, target, valid):
    return _real["_target_logits"](z, np.clip(target - 1, 0, None), valid)


def _lse_is_max(z):
    return z.max(axis=1) if z.shape[1] else np.full(z.shape[0], -np.inf)


def _lse_unshifted(z):
    if z.shape[1] == 0:
        return np.full(z.shape[0], -np.inf)
    m = z.max(axis=1)
    return m + np.log(np.exp(z).sum(axis=1))


def _backprop_permuted_w(dz, h, w):
    gh, gw, gb = _real["_backprop"](dz, h, w)
    return dz @ w[::-1], gw, gb


def _backprop_bias_wrong_axis(dz, h, w):
    gh, gw, gb = _real["_backprop"](dz, h, w)
    return gh, gw, dz.sum(axis=0) * 0 + dz.mean(axis=0)


def _row_scales_no_grad_out(valid, reduction, grad_scale, grad_out):
    return _real["_row_scales"](valid, reduction, grad_scale, None)


def _row_scales_no_g(valid, reduction, grad_scale, grad_out):
    return _real["_row_scales"](valid, reduction, 1.0, grad_out)


def _validity_no_range(target, ignore_index, vocab):
    t = np.asarray(target, dtype=np.int64)
    return t != ignore_index, "ok"


def _row_losses_signed(lse, zt, valid):
    return np.where(valid, zt - lse, 0.0)


MUTATIONS = {
    "dlogits_without_onehot": ("_dlogits", _dlogits_no_onehot),
    "dlogits_wrong_sign": ("_dlogits", _dlogits_flipped),
    "dlogits_ignored_rows_kept": ("_dlogits", _dlogits_unmasked),
    "ignore_index_inside_vocab_not_ignored": ("_validity", _validity_range_only),
    "mean_loss_over_all_rows": ("_reduce", _reduce_mean_over_n),
    "mean_grad_over_all_rows": ("_row_scales", _row_scales_mean_over_n),
    "bias_dropped": ("_logits", _logits_no_bias),
    "target_gather_off_by_one": ("_target_logits", _target_off_by_one),
    "lse_replaced_by_max": ("_log_sum_exp", _lse_is_max),
    "lse_missing_shift": ("_log_sum_exp", _lse_unshifted),
    "grad_hidden_permuted_weight": ("_backprop", _backprop_permuted_w),
    "grad_bias_mean_not_sum": ("_backprop", _backprop_bias_wrong_axis),
    "none_ignores_grad_out": ("_row_scales", _row_scales_no_grad_out),
    "grad_scale_dropped": ("_row_scales", _row_scales_no_g),
    "no_target_range_check": ("_validity", _validity_no_range),
    "loss_sign_flipped": ("_row_losses", _row_losses_signed),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(O)
        except Exception as e:  # noqa: BLE001 - any failure counts as detection
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin detects the planted mistake {name}"
