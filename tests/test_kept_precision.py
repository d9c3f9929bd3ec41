"""The kept-probability representation, restated on the CPU (no GPU): each
logit is kept as q = 2^(z log2e - m_c) rounded to fp16, where m_c is the
row's running maximum of z log2e after the 32-column chunk that holds it, and
the backward rebuilds p = q 2^(m_c - lse log2e). This checks the precision
the design states for it against exact float64 softmax probabilities:
relative error <= 2^-11 where q is a normal fp16 value, absolute error
<= 2^-25 times the row's p-scale below that, and the running maximum never
lets q exceed 1 (so fp16 never overflows)."""
import numpy as np
import pytest

LOG2E = 1.4426950408889634


def kept_roundtrip(z, chunk=32):
    """(p rebuilt from the kept form, exact p, q, per-element 2^(m_c - lse2))."""
    t = z * LOG2E
    N, V = t.shape
    m_run = np.full(N, -np.inf)
    mc = np.empty_like(t)
    for c0 in range(0, V, chunk):
        m_run = np.maximum(m_run, t[:, c0:c0 + chunk].max(axis=1))
        mc[:, c0:c0 + chunk] = m_run[:, None]
    q = np.exp2(t - mc).astype(np.float16)
    lse2 = np.log2(np.exp2(t - t.max(axis=1, keepdims=True)).sum(axis=1)) + t.max(axis=1)
    factor = np.exp2(mc - lse2[:, None])
    p = q.astype(np.float64) * factor
    exact = np.exp2(t - lse2[:, None])
    return p, exact, q, factor


@pytest.mark.parametrize("std,V", [(1.28, 4096), (45.0, 3000), (0.02, 1000), (8.0, 257)])
def test_kept_probabilities_rebuild_softmax(std, V):
    r = np.random.default_rng(123)
    z = r.standard_normal((64, V)) * std
    p, exact, q, factor = kept_roundtrip(z)
    qf = q.astype(np.float64)
    assert np.all(qf <= 1.0) and np.all(np.isfinite(qf))
    normal = qf >= 2.0 ** -14
    rel = np.abs(p - exact)[normal] / exact[normal]
    assert rel.max() <= 2.0 ** -11 * (1 + 1e-9)
    # Subnormal or flushed q: the error is at most half an fp16 subnormal step
    # (2^-25) times the element's factor 2^(m_c - lse2) <= 1.
    sub = ~normal
    if sub.any():
        assert np.all(np.abs(p - exact)[sub] <= 2.0 ** -25 * factor[sub] * (1 + 1e-9))
    # Rows still sum to 1 to within the fp16 rounding.
    assert np.allclose(p.sum(axis=1), 1.0, atol=V * 2.0 ** -25 + 2.0 ** -10)


def test_running_maximum_is_what_bounds_q():
    # A row whose maximum sits in the last chunk: earlier chunks are stored
    # relative to their own (smaller) running maximum, so their q is large and
    # their factor small; the rebuilt p still matches.
    z = np.zeros((1, 96))
    z[0, :32] = -3.0
    z[0, 32:64] = 0.5
    z[0, 95] = 12.0
    p, exact, q, factor = kept_roundtrip(z)
    assert q[0, 0] == np.float16(1.0) and factor[0, 0] < factor[0, 95]
    assert np.allclose(p, exact, rtol=2.0 ** -11, atol=2.0 ** -25)
