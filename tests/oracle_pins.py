"""Checks that pin the CPU oracle to things other than itself.

Each ``pin_*`` function raises AssertionError on a mismatch. They are run
as plain tests (tests/test_oracle_pins.py) and against oracles with planted
mistakes (tests/test_oracle_mutants.py), which must fail at least one pin.

Pins:
  * hand-derived closed forms (tests/golden/closed_form_cases.json);
  * an mpmath brute force of lse and the per-token loss at 50 digits;
  * torch.nn.functional.cross_entropy in float64 on the CPU, loss and
    autograd gradients (an independent library implementation);
  * scipy.special.logsumexp;
  * central finite differences of the oracle's forward against its backward;
  * invariants: dlogits rows sum to 2 lam g lse, ignored rows are zero,
    shift invariance of plain CE at lse around 200.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.flce_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")

_ENV = {"__builtins__": {}, "log": math.log, "exp": math.exp, "sqrt": math.sqrt}


def _ev(v):
    if isinstance(v, str):
        return float(eval(v, _ENV, {}))  # fixture expressions: numbers, + - * / **, log, exp
    if isinstance(v, list):
        return [_ev(e) for e in v]
    return None if v is None else float(v)


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _opts(c):
    return dict(ignore_index=c["ignore_index"], label_smoothing=c["label_smoothing"],
                lse_square_scale=c["lse_square_scale"], logit_scale=c["logit_scale"],
                reduction=c["reduction"])


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}\n got {a}\n want {b}"


def pin_golden_case(c, tol=1e-12):
    x = np.array(_ev(c["x"]))
    W = np.array(_ev(c["W"]))
    b = None if c["b"] is None else np.array(_ev(c["b"]))
    y = np.array(c["y"], dtype=np.int64)
    dloss = np.array(c["dloss"], dtype=np.float64)
    e = c["expect"]
    loss, lse = O.forward(x, W, b, y, **_opts(c))
    _close(lse, _ev(e["lse"]), tol, c["name"] + " lse")
    _close(loss, _ev(e["loss"]), tol, c["name"] + " loss")
    dx, dW, db = O.backward(dloss, x, W, b, y, **_opts(c))
    _close(dx, _ev(e["dx"]), tol, c["name"] + " dx")
    _close(dW, _ev(e["dW"]), tol, c["name"] + " dW")
    if "db" in e:
        _close(db, _ev(e["db"]), tol, c["name"] + " db")


def pin_golden_all():
    for c in load_golden():
        pin_golden_case(c)


def _rand_problem(seed, N=5, H=6, V=9, bias=True, scale=1.0, ignored=(1,), ignore_index=-100):
    r = np.random.default_rng(seed)
    x = r.standard_normal((N, H))
    W = r.standard_normal((V, H)) * scale
    b = r.standard_normal(V) * 0.5 if bias else None
    y = r.integers(0, V, size=N)
    for i in ignored:
        y[i] = ignore_index
    return x, W, b, y


def pin_mpmath_bruteforce(seed=7):
    """lse and per-token loss against 50-digit arithmetic on every term."""
    import mpmath
    mpmath.mp.dps = 50
    eps, lam, s = 0.15, 0.02, 0.7
    x, W, b, y = _rand_problem(seed)
    loss, lse = O.forward(x, W, b, y, label_smoothing=eps, lse_square_scale=lam,
                          logit_scale=s, reduction="none")
    V = W.shape[0]
    for n in range(x.shape[0]):
        z = [mpmath.mpf(s) * (mpmath.fsum(mpmath.mpf(x[n, h]) * mpmath.mpf(W[v, h])
                                          for h in range(x.shape[1])) + mpmath.mpf(b[v]))
             for v in range(V)]
        L = mpmath.log(mpmath.fsum(mpmath.exp(t) for t in z))
        assert abs(float(L) - lse[n]) <= 1e-13 * max(1.0, abs(float(L))), ("lse", n)
        if y[n] == -100:
            want = 0.0
        else:
            e = mpmath.mpf(eps)
            want = float((1 - e) * (L - z[y[n]]) + e * L - e / V * mpmath.fsum(z)
                         + mpmath.mpf(lam) * L * L)
        assert abs(want - loss[n]) <= 1e-12 * max(1.0, abs(want)), ("loss", n, want, loss[n])


def pin_torch_cross_entropy(seed=11):
    """Loss and gradients vs torch.nn.functional.cross_entropy (float64, CPU),
    plus lam * logsumexp^2 (torch.logsumexp) for the z-loss."""
    import torch
    import torch.nn.functional as F
    for red in ("mean", "sum", "none"):
        for eps, lam, s, ign in ((0.0, 0.0, 1.0, -100), (0.1, 0.0, 0.5, -100),
                                 (0.05, 1e-2, 1.3, 3)):
            x, W, b, y = _rand_problem(seed, N=7, H=5, V=11, ignored=(2, 5), ignore_index=ign)
            y[0] = (ign + 1) % 11 if ign >= 0 else 0  # make sure a valid row exists
            tx = torch.tensor(x, requires_grad=True)
            tW = torch.tensor(W, requires_grad=True)
            tb = torch.tensor(b, requires_grad=True)
            ty = torch.tensor(y)
            z = s * (tx @ tW.T + tb)
            ce = F.cross_entropy(z, ty, ignore_index=ign, label_smoothing=eps, reduction="none")
            valid = (ty != ign).double()
            zl = lam * torch.logsumexp(z, dim=1) ** 2 * valid
            per = ce + zl
            if red == "none":
                L = per
                up = torch.tensor(np.linspace(-1.0, 2.0, x.shape[0]))
            elif red == "sum":
                L = per.sum()
                up = torch.tensor(0.75, dtype=torch.float64)
            else:
                L = per.sum() / valid.sum()
                up = torch.tensor(1.25, dtype=torch.float64)
            (L * up).sum().backward()
            opts = dict(ignore_index=ign, label_smoothing=eps, lse_square_scale=lam,
                        logit_scale=s, reduction=red)
            loss, lse = O.forward(x, W, b, y, **opts)
            _close(loss, L.detach().numpy(), 1e-12, f"torch loss {red} {eps} {lam}")
            _close(lse, torch.logsumexp(z, 1).detach().numpy(), 1e-12, "torch lse")
            dx, dW, db = O.backward(up.numpy().reshape(-1), x, W, b, y, **opts)
            _close(dx, tx.grad.numpy(), 1e-11, f"torch dx {red}")
            _close(dW, tW.grad.numpy(), 1e-11, f"torch dW {red}")
            _close(db, tb.grad.numpy(), 1e-11, f"torch db {red}")


def pin_scipy_logsumexp(seed=3):
    from scipy.special import logsumexp
    r = np.random.default_rng(seed)
    z = r.standard_normal((64, 1000)) * 40.0 + 150.0
    _close(O.logsumexp_rows(z), logsumexp(z, axis=1), 1e-14, "scipy logsumexp")


def pin_finite_differences(seed=5):
    """Backward equals the central-difference derivative of the forward for
    J = sum_n dloss_n l_n (none) or dloss * loss (sum, mean)."""
    eps, lam, s = 0.1, 1e-2, 0.5
    for red in ("none", "sum", "mean"):
        x, W, b, y = _rand_problem(seed, N=4, H=8, V=16, ignored=(2,))
        dloss = np.array([0.3, -1.1, 0.7, 2.0]) if red == "none" else np.array([1.7])
        opts = dict(label_smoothing=eps, lse_square_scale=lam, logit_scale=s, reduction=red)

        def J(x_, W_, b_):
            loss, _ = O.forward(x_, W_, b_, y, **opts)
            return float(np.sum(np.asarray(loss) * dloss))

        dx, dW, db = O.backward(dloss, x, W, b, y, **opts)
        h = 1e-6
        for name, arr, grad in (("x", x, dx), ("W", W, dW), ("b", b, db)):
            num = np.zeros_like(arr)
            it = np.nditer(arr, flags=["multi_index"])
            for _ in it:
                i = it.multi_index
                p, m = arr.copy(), arr.copy()
                p[i] += h
                m[i] -= h
                args_p = {"x": (p, W, b), "W": (x, p, b), "b": (x, W, p)}[name]
                args_m = {"x": (m, W, b), "W": (x, m, b), "b": (x, W, m)}[name]
                num[i] = (J(*args_p) - J(*args_m)) / (2 * h)
            rel = np.linalg.norm(num - grad) / max(np.linalg.norm(num), 1e-30)
            assert rel <= 1e-6, f"FD {red} d{name}: rel {rel:.2e}"


def pin_invariants(seed=9):
    """Rows of dz sum to 2 lam g lse; ignored rows have zero dz and dx; the
    bias gradient sums to s * sum_n 2 lam g lse; plain CE loss is >= 0."""
    eps, lam, s = 0.2, 3e-2, 0.8
    x, W, b, y = _rand_problem(seed, N=6, H=4, V=10, ignored=(0, 4))
    g = O.row_grad_scale(np.array([1.5]), y, -100, "mean")
    z = O.logits(x, W, b, s)
    lse = O.logsumexp_rows(z)
    dz = O.dlogits(z, lse, y, g, label_smoothing=eps, lse_square_scale=lam)
    _close(dz.sum(axis=1), 2 * lam * g * lse, 1e-13, "dz row sums")
    assert np.all(dz[[0, 4]] == 0.0)
    dx, dW, db = O.backward(np.array([1.5]), x, W, b, y, label_smoothing=eps,
                            lse_square_scale=lam, logit_scale=s, reduction="mean")
    assert np.all(dx[[0, 4]] == 0.0)
    _close(db.sum(), s * np.sum(2 * lam * g * lse), 1e-12, "db sum")
    loss, _ = O.forward(x, W, b, y, reduction="none")
    assert np.all(loss >= 0.0)
    assert np.all(loss[[0, 4]] == 0.0)


def pin_shift_invariance(seed=13):
    """Adding c to every logit (through the bias) moves lse by c and leaves plain
    CE unchanged: checks cancellation at lse around 200 (large-logit regime)."""
    x, W, b, y = _rand_problem(seed, N=8, H=16, V=64, scale=1.0, ignored=())
    loss0, lse0 = O.forward(x, W, b, y, reduction="none")
    c = 200.0
    loss1, lse1 = O.forward(x, W, b + c, y, reduction="none")
    _close(lse1 - lse0, np.full(8, c), 1e-12, "lse shift")
    assert np.max(np.abs(loss1 - loss0)) <= 1e-10, "CE not shift invariant"


def pin_sampled_forms(seed=17):
    """row_stats / dx_rows / dW_db_rows (used at large sizes) agree with the full
    forward and backward (themselves pinned above)."""
    eps, lam, s = 0.1, 1e-3, 0.5
    x, W, b, y = _rand_problem(seed, N=9, H=5, V=13, ignored=(3, 7))
    for red, dl in (("mean", np.array([2.0])), ("sum", np.array([-0.5])),
                    ("none", np.linspace(-1, 1, 9))):
        opts = dict(label_smoothing=eps, lse_square_scale=lam, logit_scale=s, reduction=red)
        loss, lse = O.forward(x, W, b, y, **opts)
        dx, dW, db = O.backward(dl, x, W, b, y, **opts)
        rows = np.array([0, 3, 8])
        lse_r, zt, sz = O.row_stats(x, W, b, y, logit_scale=s, rows=rows, block=2)
        _close(lse_r, lse[rows], 1e-13, "row_stats lse")
        tl = O.token_losses_from_stats(lse_r, zt, sz, y[rows], 13, -100, eps, lam)
        full_tl, _ = O.forward(x, W, b, y, **dict(opts, reduction="none"))
        _close(tl, full_tl[rows], 1e-13, "token loss from stats")
        _close(O.dx_rows(rows, dl, x, W, b, y, **opts), dx[rows], 1e-13, "dx_rows")
        vr = np.array([1, 5, 12])
        lse_all, _, _ = O.row_stats(x, W, b, y, logit_scale=s)
        dWr, dbr = O.dW_db_rows(vr, lse_all, dl, x, W, b, y, **opts)
        _close(dWr, dW[vr], 1e-13, "dW rows")
        _close(dbr, db[vr], 1e-13, "db rows")


ALL_PINS = (pin_golden_all, pin_mpmath_bruteforce, pin_torch_cross_entropy,
            pin_scipy_logsumexp, pin_finite_differences, pin_invariants,
            pin_shift_invariance, pin_sampled_forms)
