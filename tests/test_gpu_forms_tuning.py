"""GPU parity of the GEMM kernel forms, selected per call through
flce_params_t.gemm_form (one CTA per 128 x 256 tile, a CTA pair per
256 x 256 tile, or a CTA pair per 256 x 512 tile with 8 or 16 epilogue
warps), and of configurations chosen by the autotuner."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_gemm_gb300 as F
from linear_cross_entropy_gemm_gb300 import inputs as I
from linear_cross_entropy_gemm_gb300 import tuning
from oracle import flce_oracle as O
from parity import assert_grad_close, assert_loss_close, bf16_dev, f64, opts_of, to_np
from test_gpu_parity import full_check

pytestmark = pytest.mark.gpu

FORMS = ["single", "pair", "wide"]

CASES = {
    "tiny": (I.WORKLOADS["tiny"], {}),
    # an odd number of 128-row tiles (a CTA pair's second half-tile is empty)
    # and a ragged vocabulary with a short last backward block
    "odd_tiles_ragged": (I.Workload("odd_tiles", N=300, H=264, V=1000, seed=31, b_std=0.5,
                                    ignore_frac=0.1, label_smoothing=0.1,
                                    lse_square_scale=1e-3, logit_scale=0.7, reduction="sum",
                                    dloss="normal_scalar"), {"bwd_vocab_block": 768}),
    "ragged_none": (I.Workload("ragged_none", N=129, H=72, V=257, seed=32, b_std=0.5,
                               ignore_frac=0.1, label_smoothing=0.2, reduction="none",
                               dloss="normal_per_token"), {"bwd_vocab_block": 256}),
    "fp16": (I.Workload("fp16_forms", N=640, H=512, V=3000, seed=33, b_std=0.1,
                        ignore_frac=0.05, label_smoothing=0.05, dtype="fp16"), {}),
}


@pytest.mark.parametrize("mode", ["recompute", "stored", "kept"])
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("form", FORMS)
def test_each_gemm_form_matches_the_oracle(form, case, mode):
    wl, kw = CASES[case]
    full_check(wl, mode=mode, gemm_form=form, **kw)


@pytest.mark.parametrize("warps", ["16", "8"])
def test_wide_epilogue_warp_counts_match_the_oracle(warps, monkeypatch):
    # The 256 x 512 kernel drains the forward and the bias-free recompute with
    # 16 epilogue warps, two per (lane quarter, N half) splitting the columns;
    # FLCE_WIDE_EPI_WARPS=8 gives every epilogue 8. V = 800: the second wide
    # tile's N half 1 has its first 32 columns in the vocabulary and its second
    # 128 wholly past V, so one warp of a split pair contributes nothing.
    if warps == "8":
        monkeypatch.setenv("FLCE_WIDE_EPI_WARPS", "8")
    else:
        monkeypatch.delenv("FLCE_WIDE_EPI_WARPS", raising=False)
    wl = I.Workload("wide_warps", N=300, H=264, V=800, seed=35, ignore_frac=0.1,
                    label_smoothing=0.1, lse_square_scale=1e-3, logit_scale=0.9)
    full_check(wl, gemm_form="wide", bwd_vocab_block=512)
    full_check(wl.with_(b_std=0.3, seed=36), gemm_form="wide")


def test_forms_compute_the_same_products():
    # Same inputs through both forms: every output within the parity bounds of
    # the other (they differ only in fp32 accumulation order inside a tile).
    wl = CASES["odd_tiles_ragged"][0]
    a = full_check(wl, gemm_form="single")
    for other in ("pair", "wide"):
        b = full_check(wl, gemm_form=other)
        for k in ("loss", "lse"):
            assert_loss_close(to_np(a[k]), to_np(b[k]), f"single vs {other} {k}")
        for k in ("dx", "dW", "db"):
            assert_grad_close(to_np(a[k]), to_np(b[k]).astype(np.float64),
                              f"single vs {other} {k}")


def test_invalid_gemm_form_is_rejected():
    wl = I.WORKLOADS["tiny"]
    inp = I.make_inputs(wl)
    x = bf16_dev(inp.x, "cuda:0")
    W = bf16_dev(inp.W, "cuda:0")
    y = torch.from_numpy(inp.y).cuda()
    with pytest.raises(F.FlceError):
        F.flce_forward(x, W, None, y, gemm_form=4)


def _device_inputs(wl):
    inp = I.make_inputs(wl)
    dt = wl.dtype
    x = bf16_dev(inp.x, "cuda:0", dt)
    W = bf16_dev(inp.W, "cuda:0", dt)
    b = None if inp.b is None else bf16_dev(inp.b, "cuda:0", dt)
    y = torch.from_numpy(inp.y).cuda()
    dloss = torch.from_numpy(inp.dloss).cuda()
    return inp, x, W, b, y, dloss


@pytest.mark.parametrize("mode", ["recompute", "kept"])
def test_autotune_picks_a_candidate_and_its_results_match_the_oracle(mode):
    wl = I.Workload("tune", N=1000, H=512, V=5000, seed=34, b_std=0.05, ignore_frac=0.05,
                    label_smoothing=0.1, lse_square_scale=1e-4)
    inp, x, W, b, y, dloss = _device_inputs(wl)
    opts = opts_of(wl)
    tuning.clear_cache()
    res = tuning.autotune(x, W, b, y, dloss=dloss, reps=2, mode=mode, **opts)
    blocks = tuning.vocab_block_candidates(wl.N, wl.V)
    assert set(res.forward_ms) == set(tuning.FORMS)
    assert set(res.backward_ms) == {(f, bv) for f in tuning.FORMS for bv in blocks}
    assert all(ms > 0 and np.isfinite(ms) for ms in res.forward_ms.values())
    cfg = res.config
    assert cfg.fwd_gemm_form in tuning.FORMS and cfg.bwd_gemm_form in tuning.FORMS
    assert cfg.bwd_vocab_block in blocks
    assert tuning.autotune(x, W, b, y, dloss=dloss, mode=mode, **opts) is res  # cached per key

    kept = None
    if mode == "kept":
        kept = torch.empty(F.flce_kept_size(wl.N, wl.H, wl.V,
                                            bwd_vocab_block=cfg.bwd_vocab_block),
                           dtype=torch.uint8, device=x.device)
    loss, lse = F.flce_forward(x, W, b, y, kept=kept, bwd_vocab_block=cfg.bwd_vocab_block,
                               **opts, **cfg.forward_kwargs())
    dx, dW, db = F.flce_backward(dloss, lse, x, W, b, y, kept=kept, **opts,
                                 **cfg.backward_kwargs())
    torch.cuda.synchronize()
    assert F.flce_read_device_error() == 0
    x64, W64, b64 = f64(inp)
    rl, rlse = O.forward(x64, W64, b64, inp.y, **opts)
    rdx, rdW, rdb = O.backward(inp.dloss.astype(np.float64), x64, W64, b64, inp.y, **opts)
    assert_loss_close(to_np(loss), rl, "tuned loss")
    assert_loss_close(to_np(lse), rlse, "tuned lse")
    assert_grad_close(to_np(dx), rdx, "tuned dx")
    assert_grad_close(to_np(dW), rdW, "tuned dW")
    assert_grad_close(to_np(db), rdb, "tuned db")


def test_autotuned_module_matches_the_default_module():
    wl = I.Workload("tune_module", N=384, H=256, V=2000, seed=35, b_std=0.05,
                    ignore_frac=0.1, label_smoothing=0.05, reduction="sum")
    inp, x, W, b, y, _ = _device_inputs(wl)
    outs = []
    for autotune in (False, True):
        tuning.clear_cache()
        xr = x.clone().requires_grad_(True)
        Wr = W.clone().requires_grad_(True)
        br = b.clone().requires_grad_(True)
        m = F.FusedLinearCrossEntropyLoss(label_smoothing=wl.label_smoothing, reduction="sum",
                                          autotune=autotune)
        loss = m(xr, y, Wr, br)
        loss.backward()
        torch.cuda.synchronize()
        outs.append([t.detach().float().cpu().numpy() for t in (loss, xr.grad, Wr.grad, br.grad)])
        if autotune:
            assert len(tuning.cached()) == 1
    (l0, dx0, dW0, db0), (l1, dx1, dW1, db1) = outs
    assert_loss_close(l1, l0, "autotuned module loss")
    for got, ref, what in ((dx1, dx0, "dx"), (dW1, dW0, "dW"), (db1, db0, "db")):
        assert_grad_close(got, ref.astype(np.float64), f"autotuned module {what}")
