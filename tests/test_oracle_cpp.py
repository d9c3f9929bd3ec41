"""The C++ fp64 reference (oracle/flce_oracle_ref.cpp), pinned on the CPU:
the hand-derived closed forms, agreement with the numpy oracle on random
problems with every option, an invariant of the gradient, and its argument
checks. (Two independent statements of one definition: a mistake in either
shows as a disagreement.)"""
import numpy as np
import pytest

import oracle_pins as P
from oracle import cpp as C
from oracle import flce_oracle as O


@pytest.fixture(scope="module", autouse=True)
def built():
    C.load()


@pytest.mark.parametrize("case", P.load_golden(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    x = np.array(P._ev(case["x"]))
    W = np.array(P._ev(case["W"]))
    b = None if case["b"] is None else np.array(P._ev(case["b"]))
    y = np.array(case["y"], dtype=np.int64)
    dloss = np.array(case["dloss"], dtype=np.float64)
    e = case["expect"]
    loss, lse = C.forward(x, W, b, y, **P._opts(case))
    P._close(lse, P._ev(e["lse"]), 1e-12, case["name"] + " lse")
    P._close(loss, P._ev(e["loss"]), 1e-12, case["name"] + " loss")
    dx, dW, db = C.backward(dloss, x, W, b, y, **P._opts(case))
    P._close(dx, P._ev(e["dx"]), 1e-12, case["name"] + " dx")
    P._close(dW, P._ev(e["dW"]), 1e-12, case["name"] + " dW")
    if "db" in e:
        P._close(db, P._ev(e["db"]), 1e-12, case["name"] + " db")


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_agrees_with_numpy_oracle(seed, reduction):
    r = np.random.default_rng(100 + seed)
    N, H, V = int(r.integers(1, 40)), int(r.integers(1, 24)), int(r.integers(1, 70))
    x = r.standard_normal((N, H)) * 2.0
    W = r.standard_normal((V, H)) * 0.7
    b = r.standard_normal(V) if seed != 2 else None
    ignore = [-100, 0, 3][seed - 1]
    y = r.integers(0, V, size=N)
    y[r.random(N) < 0.3] = ignore
    opts = dict(ignore_index=ignore, label_smoothing=[0.0, 0.1, 0.6][seed - 1],
                lse_square_scale=[0.0, 1e-2, 0.3][seed - 1], logit_scale=[1.0, -0.8, 1.7][seed - 1],
                reduction=reduction)
    dloss = r.standard_normal(N) if reduction == "none" else np.array([r.standard_normal()])
    loss_c, lse_c = C.forward(x, W, b, y, **opts)
    loss_n, lse_n = O.forward(x, W, b, y, **opts)
    P._close(lse_c, lse_n, 1e-12, "lse")
    P._close(loss_c, loss_n, 1e-12, "loss")
    for got, want, what in zip(C.backward(dloss, x, W, b, y, **opts),
                               O.backward(dloss, x, W, b, y, **opts), ("dx", "dW", "db")):
        if want is None:
            assert got is None
        else:
            P._close(got, want, 1e-12, what)


def test_db_sums_to_the_z_loss_term():
    # sum_v dz[n, v] = 2 lam g[n] lse[n], so sum_v db = s sum_n 2 lam g[n] lse[n].
    r = np.random.default_rng(5)
    N, H, V, s, lam = 12, 8, 33, 0.9, 0.05
    x, W, b = r.standard_normal((N, H)), r.standard_normal((V, H)), r.standard_normal(V)
    y = r.integers(0, V, size=N)
    y[4] = -100
    dloss = r.standard_normal(N)
    opts = dict(label_smoothing=0.2, lse_square_scale=lam, logit_scale=s, reduction="none")
    _, lse = C.forward(x, W, b, y, **opts)
    _, _, db = C.backward(dloss, x, W, b, y, **opts)
    g = np.where(y != -100, dloss, 0.0)
    assert abs(db.sum() - s * np.sum(2 * lam * g * lse)) <= 1e-12 * max(1.0, np.abs(db).sum())


def test_rejects_a_target_outside_the_vocabulary():
    x, W = np.ones((2, 8)), np.ones((5, 8))
    with pytest.raises(ValueError):
        C.forward(x, W, None, np.array([1, 5]))
    with pytest.raises(ValueError):
        C.backward(np.ones(1), x, W, None, np.array([-1, 2]))
    # the ignore index itself is fine, even when negative
    C.forward(x, W, None, np.array([-100, 2]))
