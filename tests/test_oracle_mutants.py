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


MUTANTS = {
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
