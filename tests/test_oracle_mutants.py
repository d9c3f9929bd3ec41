"""Plant plausible mistakes in the CPU oracle and check that its pins catch
each one: a dropped term, a wrong sign, a wrong index, a wrong normaliser, a
missing scale. CPU only; the mistakes live in monkeypatched copies of the
oracle's functions and are undone after each test."""
import numpy as np
import pytest

import oracle.flce_oracle as O
import oracle_pins as P

_orig = {k: getattr(O, k) for k in dir(O) if callable(getattr(O, k))}


def _token_losses_no_zloss(lse, z_target, sum_z, y, V, ignore_index,
                           label_smoothing=0.0, lse_square_scale=0.0):
    return _orig["token_losses_from_stats"](lse, z_target, sum_z, y, V, ignore_index,
                                            label_smoothing, 0.0)


def _token_losses_eps_not_over_v(lse, z_target, sum_z, y, V, ignore_index,
                                 label_smoothing=0.0, lse_square_scale=0.0):
    return _orig["token_losses_from_stats"](lse, z_target, sum_z, y, 1, ignore_index,
                                            label_smoothing, lse_square_scale)


def _dlogits_zloss_factor_one(z, lse, y, g, *, ignore_index=-100, label_smoothing=0.0,
                              lse_square_scale=0.0):
    return _orig["dlogits"](z, lse, y, g, ignore_index=ignore_index,
                            label_smoothing=label_smoothing,
                            lse_square_scale=lse_square_scale / 2)


def _dlogits_sign_eps(z, lse, y, g, *, ignore_index=-100, label_smoothing=0.0,
                      lse_square_scale=0.0):
    dz = _orig["dlogits"](z, lse, y, g, ignore_index=ignore_index,
                          label_smoothing=label_smoothing,
                          lse_square_scale=lse_square_scale)
    V = np.asarray(z).shape[1]
    valid = np.asarray(y) != ignore_index
    return dz + (2 * label_smoothing / V) * (np.asarray(g) * valid)[:, None]


def _dlogits_ignored_not_zeroed(z, lse, y, g, *, ignore_index=-100, label_smoothing=0.0,
                                lse_square_scale=0.0):
    y = np.asarray(y)
    yy = np.where(y == ignore_index, 0, y)
    g = np.where(y == ignore_index, 1.0, g)
    return _orig["dlogits"](z, lse, yy, g, ignore_index=ignore_index,
                            label_smoothing=label_smoothing,
                            lse_square_scale=lse_square_scale)


def _target_off_by_one(z, y, ignore_index):
    y = np.asarray(y)
    safe = np.where(y != ignore_index, (y + 1) % z.shape[1], 0)
    return z[np.arange(z.shape[0]), safe]


def _mean_over_n(dloss, y, ignore_index, reduction):
    g = _orig["row_grad_scale"](dloss, y, ignore_index, reduction)
    if reduction == "mean":
        t = max(_orig["total_count"](y, ignore_index), 1)
        g = g * t / np.asarray(y).size
    return g


def _lse_missing_max(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=1)
    return np.log(np.exp(z - m[:, None]).sum(axis=1))


def _logits_bias_unscaled(x, W, b=None, logit_scale=1.0):
    z = logit_scale * (np.asarray(x, np.float64) @ np.asarray(W, np.float64).T)
    if b is not None:
        z = z + np.asarray(b, np.float64)[None, :]
    return z


def _backward_no_scale(dloss, x, W, b, y, *, ignore_index=-100, label_smoothing=0.0,
                       lse_square_scale=0.0, logit_scale=1.0, reduction="mean"):
    dx, dW, db = _orig["backward"](dloss, x, W, b, y, ignore_index=ignore_index,
                                   label_smoothing=label_smoothing,
                                   lse_square_scale=lse_square_scale,
                                   logit_scale=logit_scale, reduction=reduction)
    f = 1.0 / logit_scale
    return dx * f, dW * f, (None if db is None else db * f)


def _backward_transposed_dx(dloss, x, W, b, y, **kw):
    dx, dW, db = _orig["backward"](dloss, x, W, b, y, **kw)
    return dx[::-1].copy(), dW, db


def _forward_lse_zero_for_ignored(x, W, b, y, **kw):
    loss, lse = _orig["forward"](x, W, b, y, **kw)
    return loss, np.where(np.asarray(y) != kw.get("ignore_index", -100), lse, 0.0)


def _token_losses_zloss_linear(lse, z_target, sum_z, y, V, ignore_index,
                               label_smoothing=0.0, lse_square_scale=0.0):
    base = _orig["token_losses_from_stats"](lse, z_target, sum_z, y, V, ignore_index,
                                            label_smoothing, 0.0)
    valid = np.asarray(y) != ignore_index
    return base + np.where(valid, float(lse_square_scale) * np.asarray(lse, np.float64), 0.0)


def _token_losses_eps_over_v_minus_1(lse, z_target, sum_z, y, V, ignore_index,
                                     label_smoothing=0.0, lse_square_scale=0.0):
    return _orig["token_losses_from_stats"](lse, z_target, sum_z, y, max(V - 1, 1),
                                            ignore_index, label_smoothing, lse_square_scale)


def _reduce_sum_mean_swapped(token_loss, y, ignore_index, reduction):
    r = {"sum": "mean", "mean": "sum"}.get(reduction, reduction)
    return _orig["reduce_losses"](token_loss, y, ignore_index, r)


def _grad_none_broadcasts_first(dloss, y, ignore_index, reduction):
    d = np.asarray(dloss, np.float64).reshape(-1)
    if reduction == "none":
        d = np.full(d.size, d[0])
    return _orig["row_grad_scale"](d, y, ignore_index, reduction)


def _dlogits_not_normalised(z, lse, y, g, *, ignore_index=-100, label_smoothing=0.0,
                            lse_square_scale=0.0):
    z64 = np.asarray(z, np.float64)
    dz = _orig["dlogits"](z, lse, y, g, ignore_index=ignore_index,
                          label_smoothing=label_smoothing, lse_square_scale=lse_square_scale)
    # softmax numerator exp(z - max) used as p: add the difference to p's term
    lse = np.asarray(lse, np.float64)
    m = z64.max(axis=1)
    fac = (1.0 + 2.0 * float(lse_square_scale) * lse)[:, None]
    extra = fac * (np.exp(z64 - m[:, None]) - np.exp(z64 - lse[:, None]))
    valid = np.asarray(y) != ignore_index
    return dz + extra * (np.asarray(g, np.float64) * valid)[:, None]


def _backward_dw_forgets_scale(dloss, x, W, b, y, **kw):
    dx, dW, db = _orig["backward"](dloss, x, W, b, y, **kw)
    return dx, dW / kw.get("logit_scale", 1.0), db


def _backward_db_forgets_scale(dloss, x, W, b, y, **kw):
    dx, dW, db = _orig["backward"](dloss, x, W, b, y, **kw)
    return dx, dW, (None if db is None else db / kw.get("logit_scale", 1.0))


MUTANTS = {
    "lse_zeroed_for_ignored_rows": {"forward": _forward_lse_zero_for_ignored},
    "zloss_linear_in_lse": {"token_losses_from_stats": _token_losses_zloss_linear},
    "smoothing_weight_eps_over_V_minus_1": {"token_losses_from_stats": _token_losses_eps_over_v_minus_1},
    "sum_and_mean_swapped": {"reduce_losses": _reduce_sum_mean_swapped},
    "none_reduction_uses_first_dloss": {"row_grad_scale": _grad_none_broadcasts_first},
    "softmax_not_normalised_in_grad": {"dlogits": _dlogits_not_normalised},
    "dW_forgets_logit_scale": {"backward": _backward_dw_forgets_scale},
    "db_forgets_logit_scale": {"backward": _backward_db_forgets_scale},
    "zloss_dropped_from_loss": {"token_losses_from_stats": _token_losses_no_zloss},
    "smoothing_weight_eps_not_eps_over_V": {"token_losses_from_stats": _token_losses_eps_not_over_v},
    "zloss_grad_factor_lam_not_2lam": {"dlogits": _dlogits_zloss_factor_one},
    "smoothing_grad_wrong_sign": {"dlogits": _dlogits_sign_eps},
    "ignored_rows_get_gradient": {"dlogits": _dlogits_ignored_not_zeroed},
    "target_index_off_by_one": {"_target_logits": _target_off_by_one},
    "mean_divides_by_N_not_total": {"row_grad_scale": _mean_over_n},
    "lse_drops_the_max": {"logsumexp_rows": _lse_missing_max},
    "bias_not_scaled": {"logits": _logits_bias_unscaled},
    "backward_forgets_logit_scale": {"backward": _backward_no_scale},
    "dx_rows_permuted": {"backward": _backward_transposed_dx},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    for attr, fn in MUTANTS[name].items():
        monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except AssertionError as e:
            caught.append((pin.__name__, (str(e).splitlines() or [""])[0]))
        except ImportError:
            pass
    assert caught, f"no pin caught the planted mistake {name}"
