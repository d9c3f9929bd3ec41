"""flce_forward_noalloc: the forward pass for callers that cannot allocate
device memory (no workspace argument; the scratch is a fixed array inside
the library). Called through the C ABI and compared with flce_forward on the
same inputs, two calls in a row, so stale scratch from the first call must
not affect the second. Collected last on purpose: if it fails, a run that
stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import linear_cross_entropy_gemm_gb300 as F
from linear_cross_entropy_gemm_gb300 import _lib
from linear_cross_entropy_gemm_gb300 import inputs as I
from parity import DeviceProblem, assert_loss_close, opts_of, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024 * 1024


def _noalloc():
    lib = _lib.load()
    fn = lib.flce_forward_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(_lib.FlceParams), vp, vp, vp, vp, vp, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _run_noalloc(prob: DeviceProblem):
    wl = prob.inp.wl
    opts = opts_of(wl)
    p = _lib.params(wl.N, wl.H, wl.V, has_bias=prob.b is not None, **opts)
    loss = torch.full((wl.N if wl.reduction == "none" else 1,), float("nan"),
                      dtype=torch.float32, device=prob.dev)
    lse = torch.full((wl.N,), float("nan"), dtype=torch.float32, device=prob.dev)
    st = _noalloc()(p, prob.x.data_ptr(), prob.W.data_ptr(),
                    None if prob.b is None else prob.b.data_ptr(), prob.y.data_ptr(),
                    loss.data_ptr(), lse.data_ptr(), F.device_error_word(prob.dev).data_ptr(),
                    torch.cuda.current_stream(prob.dev).cuda_stream)
    assert st == 0, f"flce_forward_noalloc returned {_lib.STATUS_NAMES.get(st, st)}"
    torch.cuda.synchronize(prob.dev)
    assert F.flce_read_device_error(prob.dev) == 0
    return to_np(loss), to_np(lse)


def _run_reference(prob: DeviceProblem):
    loss, lse = F.flce_forward(prob.x, prob.W, prob.b, prob.y, **opts_of(prob.inp.wl))
    torch.cuda.synchronize(prob.dev)
    return to_np(loss), to_np(lse)


def test_noalloc_forward_matches_workspace_forward_twice():
    # Two different problems back to back: the second call reuses scratch the
    # first one filled with other shapes and values.
    first = DeviceProblem(I.make_inputs(I.WORKLOADS["medium"]))
    second = DeviceProblem(I.make_inputs(
        I.Workload("noalloc2", N=777, H=264, V=5000, seed=31, b_std=0.1, ignore_frac=0.1,
                   lse_square_scale=1e-3, logit_scale=0.8, reduction="none")))
    for prob in (first, second):
        got_loss, got_lse = _run_noalloc(prob)
        ref_loss, ref_lse = _run_reference(prob)
        assert_loss_close(got_loss, ref_loss, f"{prob.inp.wl.name} noalloc loss")
        assert_loss_close(got_lse, ref_lse, f"{prob.inp.wl.name} noalloc lse")
    again_loss, again_lse = _run_noalloc(first)
    ref_loss, ref_lse = _run_reference(first)
    assert_loss_close(again_loss, ref_loss, "medium noalloc loss, repeated")
    assert_loss_close(again_lse, ref_lse, "medium noalloc lse, repeated")


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    lib = _lib.load()
    p = _lib.params(32768, 64, 262144, label_smoothing=0.1)
    assert lib.flce_workspace_size(p, 0) > SCRATCH_BYTES
    f = ctypes.c_void_p(4096)  # rejected before any pointer is used
    st = _noalloc()(p, f, f, None, f, f, f, None, None)
    assert st == 3  # FLCE_ERR_WORKSPACE_TOO_SMALL
