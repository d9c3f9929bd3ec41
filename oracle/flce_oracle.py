"""CPU fp64 oracle for fused linear cross-entropy (FLCE).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline may import this module. The library never does, and shares no code
with it: this file restates the mathematics of the pages in plain numpy,
float64, over the same bf16- (or fp16-) rounded inputs the GPU sees, widened
exactly; also pinned against planted mistakes (tests/test_oracle_mutants.py).

What it computes (the plain definition; the GPU path reaches the same result
up to rounding order, by tiling and online softmax):

  z[n, v]  = s * (sum_h x[n, h] W[v, h] + b[v])                     (logits)
  lse[n]   = log sum_v exp(z[n, v])                                  (two-pass)
  l[n]     = (1 - eps)(lse[n] - z[n, y_n]) + eps*lse[n]
             - (eps / V) sum_v z[n, v] + lam * lse[n]^2                (0 if ignored)
  loss     = l (none) | sum_n l[n] (sum) | sum_n l[n] / total (mean)
  g[n]     = dloss (sum) | dloss / total (mean) | dloss[n] (none); 0 if ignored
  dz[n, v] = g[n] * ((1 + 2 lam lse[n]) p[n, v] - eps / V - (1 - eps) [v == y_n]),
             p = exp(z - lse)
  dx = s * dz W,   dW = s * dz^T x,   db = s * sum_n dz[n, :]

Sources, by page and section:
  * flash-linear-attention, fla/modules/fused_linear_cross_entropy.py:
    ``fused_linear_cross_entropy_forward`` (logits via F.linear, then the
    logit_scale, lse kept in fp32, ``total`` = non-ignored count) and
    ``cross_entropy_kernel`` (ignored rows: zero loss and gradient; loss =
    lse - z_y; label smoothing with eps/V; mean divides by ``total``).
  * Liger-Kernel PR #239 "Support Z Loss in CE", "Details": z_loss =
    lse_square_scale * lse^2 added per token, and the derivative
    (1 + 2 lse_square_scale lse) softmax - eps/K - (1 - eps) delta.
  * DeepSpeed PR #8792 "What": reduction "none" beside sum and mean; the
    logits are formed in fp32 or better (never rounded to bf16 first).

Parity status: every function below is pinned by the CPU tests
(tests/test_oracle_pins.py) against closed forms, an mpmath brute force,
torch.nn.functional.cross_entropy in float64, scipy.special.logsumexp and
central finite differences. No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

REDUCTIONS = ("none", "sum", "mean")


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


# --- forward ---------------------------------------------------------------

def logits(x, W, b=None, logit_scale=1.0):
    """z = s * (x W^T + b), dense float64 (fla fused_linear_cross_entropy_forward:
    F.linear then the logit_scale inside the lse and the loss kernel)."""
    x, W, b = _f64(x), _f64(W), _f64(b)
    z = x @ W.T
    if b is not None:
        z = z + b[None, :]
    return logit_scale * z


def logsumexp_rows(z):
    """lse[n] = log sum_v exp(z[n, v]), by the two-pass max-shifted definition."""
    z = _f64(z)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def valid_mask(y, ignore_index):
    return np.asarray(y) != ignore_index


def total_count(y, ignore_index):
    """Non-ignored token count (fla: ``total = target.ne(ignore_index).sum()``)."""
    return int(valid_mask(y, ignore_index).sum())


def token_losses_from_stats(lse, z_target, sum_z, y, V, ignore_index,
                            label_smoothing=0.0, lse_square_scale=0.0):
    """Per-token loss from the row statistics (lse, z at the target, sum of z).

    l = (1 - eps)(lse - z_y) + eps*lse - (eps/V) sum_v z_v + lam*lse^2,
    and 0 for ignored rows (fla cross_entropy_kernel: ignored rows return
    before any loss; label smoothing term; Liger PR #239 z_loss).
    """
    eps, lam = float(label_smoothing), float(lse_square_scale)
    lse, z_target, sum_z = _f64(lse), _f64(z_target), _f64(sum_z)
    loss = (1.0 - eps) * (lse - z_target) + eps * lse - (eps / V) * sum_z \
        + lam * lse * lse
    return np.where(valid_mask(y, ignore_index), loss, 0.0)


def reduce_losses(token_loss, y, ignore_index, reduction):
    """none -> per-token array; sum -> sum; mean -> sum / total, and 0 when
    every row is ignored (the fla kernel never divides an ignored row, and the
    loss buffer starts at zero)."""
    if reduction == "none":
        return _f64(token_loss)
    s = float(np.sum(token_loss))
    if reduction == "sum":
        return s
    if reduction == "mean":
        t = total_count(y, ignore_index)
        return s / t if t > 0 else 0.0
    raise ValueError(reduction)


def _target_logits(z, y, ignore_index):
    y = np.asarray(y)
    safe = np.where(valid_mask(y, ignore_index), y, 0)
    return z[np.arange(z.shape[0]), safe]


def forward(x, W, b, y, *, ignore_index=-100, label_smoothing=0.0,
            lse_square_scale=0.0, logit_scale=1.0, reduction="mean"):
    """Full forward: returns (loss, lse). lse is reported for every row,
    ignored ones included (fla computes it for the whole chunk)."""
    z = logits(x, W, b, logit_scale)
    lse = logsumexp_rows(z)
    tl = token_losses_from_stats(lse, _target_logits(z, y, ignore_index),
                                 z.sum(axis=1), y, z.shape[1], ignore_index,
                                 label_smoothing, lse_square_scale)
    return reduce_losses(tl, y, ignore_index, reduction), lse


def row_stats(x, W, b, y, *, ignore_index=-100, logit_scale=1.0, rows=None,
              block=64):
    """lse, z at the target and sum of z for each row in ``rows`` (all rows by
    default). Rows are independent; they are taken ``block`` at a time only to
    bound memory, and each row's reductions run over its whole vocabulary."""
    x = np.asarray(x)
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    y = np.asarray(y)
    W64 = _f64(W)
    b64 = _f64(b)
    lse = np.empty(rows.size)
    zt = np.empty(rows.size)
    sz = np.empty(rows.size)
    for i in range(0, rows.size, block):
        r = rows[i:i + block]
        z = logits(_f64(x[r]), W64, b64, logit_scale)
        lse[i:i + block] = logsumexp_rows(z)
        zt[i:i + block] = _target_logits(z, y[r], ignore_index)
        sz[i:i + block] = z.sum(axis=1)
    return lse, zt, sz


# --- backward --------------------------------------------------------------

def row_grad_scale(dloss, y, ignore_index, reduction):
    """g[n]: the upstream gradient each token's loss receives.

    sum -> dloss; mean -> dloss / total; none -> dloss[n]; 0 for ignored rows
    (fla cross_entropy_kernel divides by ``total`` under mean and zeroes
    ignored rows; fused_linear_cross_entropy_backward then multiplies by the
    upstream gradient)."""
    y = np.asarray(y)
    valid = valid_mask(y, ignore_index)
    d = _f64(dloss).reshape(-1)
    if reduction == "none":
        if d.size != y.size:
            raise ValueError("reduction none takes one upstream gradient per token")
        g = d.copy()
    elif reduction == "sum":
        g = np.full(y.size, d[0])
    elif reduction == "mean":
        t = total_count(y, ignore_index)
        g = np.full(y.size, d[0] / t if t > 0 else 0.0)
    else:
        raise ValueError(reduction)
    return np.where(valid, g, 0.0)


def dlogits(z, lse, y, g, *, ignore_index=-100, label_smoothing=0.0,
            lse_square_scale=0.0):
    """dL/dz = g * ((1 + 2 lam lse) softmax(z) - eps/V - (1 - eps) delta_y)
    (Liger PR #239 "Details", derivative of the total loss)."""
    z, lse, g = _f64(z), _f64(lse), _f64(g)
    eps, lam = float(label_smoothing), float(lse_square_scale)
    V = z.shape[1]
    p = np.exp(z - lse[:, None])
    dz = (1.0 + 2.0 * lam * lse)[:, None] * p - eps / V
    y = np.asarray(y)
    valid = valid_mask(y, ignore_index)
    idx = np.nonzero(valid)[0]
    dz[idx, y[idx]] -= (1.0 - eps)
    dz *= g[:, None]
    dz[~valid] = 0.0
    return dz


def backward(dloss, x, W, b, y, *, ignore_index=-100, label_smoothing=0.0,
             lse_square_scale=0.0, logit_scale=1.0, reduction="mean"):
    """Full backward: returns (dx, dW, db); db is None without a bias.

    dx = s dz W (fla: ``torch.mm(c_logits, weight)`` with the logit_scale
    folded into dz), dW = s dz^T x, db = s sum_n dz."""
    x64, W64 = _f64(x), _f64(W)
    z = logits(x64, W64, b, logit_scale)
    lse = logsumexp_rows(z)
    g = row_grad_scale(dloss, y, ignore_index, reduction)
    dz = dlogits(z, lse, y, g, ignore_index=ignore_index,
                 label_smoothing=label_smoothing, lse_square_scale=lse_square_scale)
    dL = logit_scale * dz
    dx = dL @ W64
    dW = dL.T @ x64
    db = dL.sum(axis=0) if b is not None else None
    return dx, dW, db


# --- sampled forms for large problems --------------------------------------

def dx_rows(rows, dloss, x, W, b, y, *, total=None, ignore_index=-100,
            label_smoothing=0.0, lse_square_scale=0.0, logit_scale=1.0,
            reduction="mean"):
    """dx for the given rows only (each needs just its own logits row).
    ``total`` is the non-ignored count of the whole batch (mean only)."""
    rows = np.asarray(rows)
    y = np.asarray(y)
    yr = y[rows]
    W64 = _f64(W)
    z = logits(_f64(np.asarray(x)[rows]), W64, b, logit_scale)
    lse = logsumexp_rows(z)
    if reduction == "none":
        g = row_grad_scale(_f64(dloss).reshape(-1)[rows], yr, ignore_index, "none")
    elif reduction == "mean":
        t = total_count(y, ignore_index) if total is None else total
        g = np.where(valid_mask(yr, ignore_index),
                     float(_f64(dloss).reshape(-1)[0]) / t if t > 0 else 0.0, 0.0)
    else:
        g = row_grad_scale(dloss, yr, ignore_index, reduction)
    dz = dlogits(z, lse, yr, g, ignore_index=ignore_index,
                 label_smoothing=label_smoothing, lse_square_scale=lse_square_scale)
    return (logit_scale * dz) @ W64


def dW_db_rows(vrows, lse_all, dloss, x, W, b, y, *, ignore_index=-100,
               label_smoothing=0.0, lse_square_scale=0.0, logit_scale=1.0,
               reduction="mean"):
    """dW[v, :] and db[v] for the given vocabulary rows. Needs every token's
    lse (``lse_all``, e.g. from ``row_stats``) because each vocab row of dW
    sums over all tokens: dW[v] = s sum_n dz[n, v] x[n]."""
    vrows = np.asarray(vrows)
    y = np.asarray(y)
    x64 = _f64(x)
    W64 = _f64(np.asarray(W)[vrows])
    bv = None if b is None else _f64(np.asarray(b)[vrows])
    eps, lam = float(label_smoothing), float(lse_square_scale)
    V = np.asarray(W).shape[0]
    zc = logits(x64, W64, bv, logit_scale)                # [N, |vrows|]
    lse_all = _f64(lse_all)
    g = row_grad_scale(dloss, y, ignore_index, reduction)
    p = np.exp(zc - lse_all[:, None])
    dz = (1.0 + 2.0 * lam * lse_all)[:, None] * p - eps / V
    dz -= (1.0 - eps) * (y[:, None] == vrows[None, :])
    dz *= g[:, None]
    dz[~valid_mask(y, ignore_index)] = 0.0
    dL = logit_scale * dz
    dW = dL.T @ x64
    db = dL.sum(axis=0)
    return dW, db
