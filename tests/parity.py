"""Helpers for GPU-vs-oracle parity: moving seeded inputs to the device,
running the C ABI through the binding, and the tolerances.

Tolerances (fixed for this method): loss and lse |got - ref| <= 1e-3 max(1,
|ref|); dx, dW, db compared as fp32 with relative Frobenius error <= 5e-3 and
max elementwise error <= 2^-7 max|ref|.
"""
from __future__ import annotations

import numpy as np
import torch

from linear_cross_entropy_gemm_gb300 import inputs as I

# Backward modes of the library (DeviceProblem.run).
MODE_NAMES = ("recompute", "stored", "kept", "budget")

LOSS_RTOL = 1e-3
GRAD_FROB = 5e-3
GRAD_MAX = 2.0 ** -7


def bf16_dev(bits: np.ndarray, dev, dtype: str = "bf16") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "fp16" else torch.bfloat16).to(dev)


def opts_of(wl: I.Workload) -> dict:
    return dict(ignore_index=wl.ignore_index, label_smoothing=wl.label_smoothing,
                lse_square_scale=wl.lse_square_scale, logit_scale=wl.logit_scale,
                reduction=wl.reduction)


class DeviceProblem:
    def __init__(self, inp: I.Inputs, dev="cuda:0"):
        self.inp = inp
        self.dev = torch.device(dev)
        dt = inp.wl.dtype
        self.x = bf16_dev(inp.x, self.dev, dt)
        self.W = bf16_dev(inp.W, self.dev, dt)
        self.b = None if inp.b is None else bf16_dev(inp.b, self.dev, dt)
        self.y = torch.from_numpy(inp.y).to(self.dev)
        self.dloss = torch.from_numpy(inp.dloss).to(self.dev)

    def run(self, *, dW_dtype=torch.float32, db_dtype=torch.float32, bwd_vocab_block=0,
            mode="recompute", keep_vocab=0, **over):
        """Forward + backward through the C ABI in one of the backward modes:
        "recompute" (every vocabulary block's logits recomputed), "stored"
        (every logit's probability kept by the forward, no recompute), "kept"
        (the probabilities of the kept block [0, keep_vocab) kept, by default
        one backward block, the other blocks recomputed) or "budget" (kept,
        as wide as flce_keep_vocab_within allows with its default extra)."""
        import linear_cross_entropy_gemm_gb300 as F
        assert mode in MODE_NAMES, mode
        opts = opts_of(self.inp.wl)
        opts.update(over)
        wl = self.inp.wl
        saved = kept = None
        if mode == "budget" and wl.N > 0:
            keep_vocab = F.flce_keep_vocab_within(wl.N, wl.H, wl.V, has_bias=wl.has_bias,
                                                  bwd_vocab_block=bwd_vocab_block,
                                                  input_fp16=wl.dtype == "fp16")
        if mode == "stored":
            n = F.flce_saved_size(wl.N, wl.H, wl.V, label_smoothing=opts["label_smoothing"],
                                  input_fp16=wl.dtype == "fp16")
            saved = torch.empty(max(n, 1), dtype=torch.uint8, device=self.dev)
        elif mode in ("kept", "budget") and wl.N > 0:
            n = F.flce_kept_size(wl.N, wl.H, wl.V, input_fp16=wl.dtype == "fp16",
                                 bwd_vocab_block=bwd_vocab_block, keep_vocab=keep_vocab)
            kept = torch.empty(max(n, 1), dtype=torch.uint8, device=self.dev)
        kv = keep_vocab if kept is not None else 0
        loss, lse = F.flce_forward(self.x, self.W, self.b, self.y, saved=saved, kept=kept,
                                   bwd_vocab_block=bwd_vocab_block, keep_vocab=kv, **opts)
        dx, dW, db = F.flce_backward(self.dloss, lse, self.x, self.W, self.b, self.y,
                                     dW_dtype=dW_dtype, db_dtype=db_dtype,
                                     bwd_vocab_block=bwd_vocab_block, saved=saved, kept=kept,
                                     keep_vocab=kv, **opts)
        torch.cuda.synchronize(self.dev)
        err = F.flce_read_device_error(self.dev)
        return dict(loss=loss, lse=lse, dx=dx, dW=dW, db=db, err=err)


def f64(inp: I.Inputs):
    dt = inp.wl.dtype
    return (I.bits_to_f64(inp.x, dt), I.bits_to_f64(inp.W, dt),
            None if inp.b is None else I.bits_to_f64(inp.b, dt))


def assert_loss_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    i = int(np.argmax(err)) if err.size else 0
    assert err.size == 0 or err[i] <= LOSS_RTOL, \
        f"{what}: |d|/max(1,|ref|) = {err[i]:.3e} at {i} (got {got[i]!r}, ref {ref[i]!r})"


def grad_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nref = np.linalg.norm(ref)
    frob = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got)
    mref = np.max(np.abs(ref)) if ref.size else 0.0
    mx = np.max(np.abs(got - ref)) if ref.size else 0.0
    return frob, mx, mref


def assert_grad_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    frob, mx, mref = grad_errors(got, ref)
    if mref == 0.0:
        assert mx == 0.0, f"{what}: expected exact zeros, max |got| {mx:.3e}"
        return
    assert frob <= GRAD_FROB and mx <= GRAD_MAX * mref, \
        f"{what}: rel-Frobenius {frob:.3e} (<= {GRAD_FROB}), max err {mx:.3e} " \
        f"(<= {GRAD_MAX * mref:.3e})"


def token_seams(N: int) -> list:
    """Token rows at the seams the kernels' tilings have at N tokens: the
    128-row tile, the 256-row CTA pair, the 4096-row band of the logits
    GEMMs' raster, and the last (possibly partial) tiles."""
    rows = {0, 1, N - 1, N - 2}
    for period in (128, 256, 4096):
        for k in range(period, N, period):
            if k in (period, 2 * period) or k >= N - 2 * period:
                rows.update((k - 1, k))
    if N > 256:
        rows.update((N - 257, N - 256, N - 129, N - 128))
        last = (N - 1) // 256 * 256
        rows.update((last - 1, last))
    return sorted(r for r in rows if 0 <= r < N)


def vocab_seams(V: int, block: int) -> list:
    """Vocabulary rows at the seams of the backward's vocabulary blocks (each
    block start -1, +0, +1), of the 256- and 512-column GEMM tiles near the
    start, and of the last tiles and block."""
    cols = {0, 1, 255, 256, 257, 511, 512, 513, V - 1, V - 2}
    for v0 in range(block, V, block):
        cols.update((v0 - 1, v0, v0 + 1))
    for period in (256, 512):
        last = (V - 1) // period * period
        cols.update((last - 1, last))
    last_block = (V - 1) // block * block
    cols.update((last_block, last_block + 1))
    return sorted(c for c in cols if 0 <= c < V)


def to_np(t):
    return None if t is None else t.detach().float().cpu().numpy()
