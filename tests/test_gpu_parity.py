"""GPU parity: the sm_103a library (through its C ABI) against the CPU fp64
oracle on identical seeded inputs.

Small problems compare every output element; the full-size problems compare
every token's loss and lse, 256 sampled token rows of dx and 256 sampled
vocabulary rows of dW (and db). All tests need a GB300 (sm_103).
"""
import numpy as np
import pytest
import torch

import linear_cross_entropy_gemm_gb300 as F
from linear_cross_entropy_gemm_gb300 import inputs as I
from oracle import flce_oracle as O
from linear_cross_entropy_gemm_gb300 import tuning
from parity import (DeviceProblem, assert_grad_close, assert_loss_close, f64, opts_of, to_np,
                    token_seams, vocab_seams)

pytestmark = pytest.mark.gpu


MODES = ["recompute", "stored", "kept"]
# The full-size checks also run the kept block as wide as the method's memory
# budget allows (flce_keep_vocab_within): the whole vocabulary at the Llama-3
# head, one block at large_logit, half the vocabulary at vocab256k.
FULL_MODES = MODES + ["budget"]


def full_check(wl, *, bwd_vocab_block=0, dW_dtype=torch.float32, db_dtype=torch.float32,
               mode="recompute", gemm_form="default", keep_vocab=0):
    inp = I.make_inputs(wl)
    out = DeviceProblem(inp).run(bwd_vocab_block=bwd_vocab_block, dW_dtype=dW_dtype,
                                 db_dtype=db_dtype, mode=mode, gemm_form=gemm_form,
                                 keep_vocab=keep_vocab)
    assert out["err"] == 0, f"device error word {out['err']}"
    x64, W64, b64 = f64(inp)
    opts = opts_of(wl)
    rl, rlse = O.forward(x64, W64, b64, inp.y, **opts)
    rdx, rdW, rdb = O.backward(inp.dloss.astype(np.float64), x64, W64, b64, inp.y, **opts)
    assert_loss_close(to_np(out["loss"]), rl, f"{wl.name} loss")
    assert_loss_close(to_np(out["lse"]), rlse, f"{wl.name} lse")
    assert_grad_close(to_np(out["dx"]), rdx, f"{wl.name} dx")
    assert_grad_close(to_np(out["dW"]), rdW, f"{wl.name} dW")
    if wl.has_bias:
        assert_grad_close(to_np(out["db"]), rdb, f"{wl.name} db")
    return out


@pytest.mark.parametrize("mode", MODES)
def test_tiny_full(mode):
    full_check(I.WORKLOADS["tiny"], mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_medium_full_with_bias_smoothing_zloss(mode):
    full_check(I.WORKLOADS["medium"], mode=mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_ragged_tails_multi_block(reduction, mode):
    # N, H, V not multiples of the 128 x 256 x 64 tile; vocab blocks of 256
    # leave a 1-column last block.
    wl = I.Workload("ragged", N=129, H=72, V=257, seed=21, b_std=0.5, ignore_frac=0.1,
                    label_smoothing=0.2, lse_square_scale=1e-2, logit_scale=1.3,
                    reduction=reduction,
                    dloss="normal_per_token" if reduction == "none" else "normal_scalar")
    full_check(wl, bwd_vocab_block=256, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_degenerate_single_class_single_token(mode):
    wl = I.Workload("v1", N=1, H=8, V=1, seed=22, b_std=1.0, label_smoothing=0.3,
                    lse_square_scale=0.1, reduction="sum")
    full_check(wl, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_few_tokens_many_vocab_blocks(mode):
    wl = I.Workload("wide", N=5, H=64, V=5000, seed=23, x_std=2.0, w_std=0.1,
                    label_smoothing=0.05, reduction="mean")
    full_check(wl, bwd_vocab_block=1024, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_bf16_gradients_and_custom_ignore_index(mode):
    wl = I.Workload("bf16out", N=200, H=128, V=777, seed=24, b_std=0.1, ignore_frac=0.2,
                    ignore_index=5, reduction="mean")
    full_check(wl, dW_dtype=torch.bfloat16, db_dtype=torch.bfloat16, bwd_vocab_block=512,
               mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_negative_logit_scale_and_class_zero_ignored(mode):
    wl = I.Workload("negscale", N=257, H=136, V=999, seed=33, b_std=0.2, ignore_frac=0.0,
                    ignore_index=0, logit_scale=-0.75, label_smoothing=0.05,
                    lse_square_scale=2e-3, reduction="mean")
    full_check(wl, bwd_vocab_block=512, mode=mode)


def test_large_logits_small_shape_every_mode():
    # logit std ~45 (x, W, b ~ N(0, 1)): most tile probabilities underflow fp16
    # in the stored and kept modes; the ones that matter must survive.
    wl = I.WORKLOADS["large_logit"].with_(N=300, V=3000, H=2048)
    for mode in MODES:
        full_check(wl, bwd_vocab_block=1024, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_fp16_operands(mode):
    wl = I.WORKLOADS["medium"].with_(name="medium_fp16", dtype="fp16", N=1000, V=5000)
    full_check(wl, bwd_vocab_block=2048, mode=mode,
               dW_dtype=torch.float16, db_dtype=torch.float16)


@pytest.mark.parametrize("mode", MODES)
def test_fp16_loss_scaled_gradients_do_not_overflow(mode):
    # sum reduction with a 65536 loss scale: the target column's dlogit is
    # about -65536, beyond fp16's largest finite value, before the library's
    # power-of-two dL scaling; dx itself (~3e3) and dW (fp32) stay in range.
    wl = I.Workload("fp16_scaled", N=400, H=256, V=3000, seed=28, dtype="fp16", x_std=2.0,
                    w_std=0.05, reduction="sum", dloss_scale=65536.0)
    full_check(wl, bwd_vocab_block=1024, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_fp16_small_gradients_do_not_flush(mode):
    # mean over 4096 tokens of a 30000-way softmax: dlogits ~ 1e-9, below fp16's
    # smallest subnormal without the library's power-of-two dL scaling.
    wl = I.Workload("fp16_tiny_grads", N=4096, H=128, V=30000, seed=29, dtype="fp16",
                    reduction="mean")
    full_check(wl, mode=mode)


@pytest.mark.parametrize("keep_vocab", [512, 768, 1280, 1536])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_wider_kept_block_ragged(keep_vocab, reduction):
    # A kept block wider than one backward block: the forward keeps [0, K),
    # the backward converts it in place and recomputes [K, V) in 256-column
    # blocks staged at the start of the kept buffer. V = 1300: K = 512 leaves
    # 788 columns (256 + 256 + 256 + 20), K = 768 leaves 532, K = 1280 leaves
    # 20, K = 1536 keeps everything. Bias, smoothing and z-loss exercise the
    # kept-width db partials.
    wl = I.Workload("wide_kept", N=129, H=72, V=1300, seed=41, b_std=0.5, ignore_frac=0.1,
                    label_smoothing=0.2, lse_square_scale=1e-2, logit_scale=1.3,
                    reduction=reduction,
                    dloss="normal_per_token" if reduction == "none" else "normal_scalar")
    full_check(wl, bwd_vocab_block=256, mode="kept", keep_vocab=keep_vocab)


@pytest.mark.parametrize("gemm_form", ["default", "single", "pair", "wide"])
def test_wider_kept_block_many_tiles(gemm_form):
    # Several tiles in every direction: medium's options (bias, smoothing,
    # z-loss) at 1000 x 2048 x 32000 with 4096-column blocks and a 12288-wide
    # kept block (then 4 x 4096 recomputed and a 3328-column ragged block).
    wl = I.WORKLOADS["medium"].with_(N=1000)
    full_check(wl, bwd_vocab_block=4096, mode="kept", keep_vocab=12288, gemm_form=gemm_form)


def test_wider_kept_block_fp16():
    wl = I.WORKLOADS["medium"].with_(name="medium_fp16", dtype="fp16", N=1000, V=5000)
    full_check(wl, bwd_vocab_block=1024, mode="kept", keep_vocab=2560,
               dW_dtype=torch.float16, db_dtype=torch.float16)


def test_budget_mode_keeps_the_rule_width():
    # "budget": the width flce_keep_vocab_within picks. At this shape (bias,
    # 1024-column blocks) the method's fp32 dW allowance (4 V H bytes) buys
    # part of the vocabulary but not all of it.
    wl = I.WORKLOADS["medium"].with_(N=2000, H=256, V=6000)
    k = F.flce_keep_vocab_within(wl.N, wl.H, wl.V, has_bias=True, bwd_vocab_block=1024)
    assert 1024 < k < 6000
    full_check(wl, bwd_vocab_block=1024, mode="budget")


@pytest.mark.parametrize("mode", ["recompute", "kept"])
@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_against_the_cpp_reference(case, mode):
    # The same element-by-element bounds against the second statement of the
    # definition, the C++ fp64 reference (oracle/flce_oracle_ref.cpp).
    from oracle import cpp as C
    wl = I.WORKLOADS["tiny"] if case == "tiny" else I.Workload(
        "ragged_cpp", N=129, H=72, V=1300, seed=43, b_std=0.5, ignore_frac=0.1,
        label_smoothing=0.2, lse_square_scale=1e-2, logit_scale=1.3, reduction="none",
        dloss="normal_per_token")
    inp = I.make_inputs(wl)
    out = DeviceProblem(inp).run(bwd_vocab_block=256 if case == "ragged" else 0, mode=mode)
    assert out["err"] == 0
    x64, W64, b64 = f64(inp)
    opts = opts_of(wl)
    rl, rlse = C.forward(x64, W64, b64, inp.y, **opts)
    rdx, rdW, rdb = C.backward(inp.dloss.astype(np.float64), x64, W64, b64, inp.y, **opts)
    assert_loss_close(to_np(out["loss"]), rl, f"{wl.name} loss (C++ reference)")
    assert_loss_close(to_np(out["lse"]), rlse, f"{wl.name} lse (C++ reference)")
    assert_grad_close(to_np(out["dx"]), rdx, f"{wl.name} dx (C++ reference)")
    assert_grad_close(to_np(out["dW"]), rdW, f"{wl.name} dW (C++ reference)")
    if wl.has_bias:
        assert_grad_close(to_np(out["db"]), rdb, f"{wl.name} db (C++ reference)")


def test_fp16_product_beyond_fp16_range_before_bias():
    # x W^T ~ 7e4 (> 65504) with a cancelling bias: fp32 accumulation keeps the
    # logits finite (DeepSpeed PR #8792's fp32-output GEMM lesson).
    wl = I.Workload("fp16_bigdot", N=64, H=64, V=512, seed=30, dtype="fp16", reduction="mean")
    inp = I.make_inputs(wl)
    h16 = lambda v: np.full(1, v, np.float32).astype(np.float16).view(np.uint16)[0]
    inp.x[:] = h16(32.5)
    W = np.random.default_rng(3).standard_normal((wl.V, wl.H)).astype(np.float32)
    inp.W[:] = (32.5 + 0.05 * W).astype(np.float16).view(np.uint16)
    inp.b = np.full(wl.V, h16(-65504.0), dtype=np.uint16)
    wl2 = wl.with_(b_std=1.0)
    inp = I.Inputs(wl2, inp.x, inp.W, inp.b, inp.y, inp.dloss)
    out = DeviceProblem(inp).run()
    assert out["err"] == 0
    x64, W64, b64 = f64(inp)
    opts = opts_of(wl2)
    rl, rlse = O.forward(x64, W64, b64, inp.y, **opts)
    assert np.all(np.isfinite(to_np(out["lse"])))
    assert_loss_close(to_np(out["loss"]), rl, "fp16 big-dot loss")
    assert_loss_close(to_np(out["lse"]), rlse, "fp16 big-dot lse")
    # Gradients: finite. (Their values carry the ~0.03 absolute logit error
    # that fp32 accumulation of 7e4-sized dot products has in any GEMM, i.e.
    # a few percent in exp(z - lse); the oracle is exact, so no tight compare.)
    for k in ("dx", "dW", "db"):
        assert np.all(np.isfinite(to_np(out[k]))), k


def test_all_rows_ignored_mean_gives_zero():
    wl = I.Workload("allign", N=64, H=64, V=300, seed=25, ignore_frac=1.0, reduction="mean",
                    label_smoothing=0.1, lse_square_scale=1e-2)
    out = full_check(wl)
    assert float(out["loss"]) == 0.0
    assert torch.count_nonzero(out["dx"]).item() == 0
    assert torch.count_nonzero(out["dW"]).item() == 0


def test_empty_batch():
    dev = torch.device("cuda", 0)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    W = torch.randn(100, 64, device=dev).to(torch.bfloat16)
    y = torch.empty(0, dtype=torch.int64, device=dev)
    loss, lse = F.flce_forward(x, W, None, y, reduction="mean")
    dx, dW, _ = F.flce_backward(torch.ones(1, device=dev), lse, x, W, None, y)
    torch.cuda.synchronize()
    assert float(loss) == 0.0 and lse.numel() == 0 and dx.numel() == 0
    assert torch.count_nonzero(dW).item() == 0


def test_out_of_range_target_sets_device_error():
    wl = I.Workload("badtarget", N=40, H=64, V=100, seed=26)
    inp = I.make_inputs(wl)
    inp.y[3] = 100   # == V
    inp.y[7] = -5    # negative, not ignore_index
    out = DeviceProblem(inp).run()
    assert out["err"] & 1, "target error bit not raised"
    assert F.flce_read_device_error() == 0, "error word not cleared"


@pytest.mark.parametrize("mode", MODES)
def test_run_to_run_bitwise_determinism(mode):
    wl = I.WORKLOADS["medium"].with_(N=1000, V=3000)
    p = DeviceProblem(I.make_inputs(wl))
    a = p.run(bwd_vocab_block=1024, mode=mode)
    b = p.run(bwd_vocab_block=1024, mode=mode)
    for k in ("loss", "lse", "dx", "dW", "db"):
        assert torch.equal(a[k], b[k]), f"{k} differs between runs"


@pytest.mark.parametrize("mode", MODES + ["budget"])
def test_autograd_module_matches_c_abi(mode):
    wl = I.Workload("module", N=256, H=128, V=1000, seed=27, b_std=0.05, ignore_frac=0.05,
                    label_smoothing=0.1, lse_square_scale=1e-3, logit_scale=0.9)
    inp = I.make_inputs(wl)
    p = DeviceProblem(inp)
    ref = p.run(mode=mode)
    x = p.x.clone().requires_grad_(True)
    W = p.W.clone().requires_grad_(True)
    b = p.b.clone().requires_grad_(True)
    mod = F.FusedLinearCrossEntropyLoss(label_smoothing=0.1, lse_square_scale=1e-3,
                                        logit_scale=0.9, recompute=mode != "stored",
                                        keep_block=mode in ("kept", "budget"),
                                        keep_vocab="budget" if mode == "budget" else 0)
    loss = mod(x.view(2, 128, 128), p.y.view(2, 128), W, b)
    loss.backward()
    torch.cuda.synchronize()
    assert torch.equal(loss.detach().reshape(1), ref["loss"].reshape(1))
    assert torch.equal(x.grad, ref["dx"])
    assert torch.equal(W.grad, ref["dW"].to(torch.bfloat16))
    assert torch.equal(b.grad, ref["db"].to(torch.bfloat16))


# ------------------------------------------------------------ full sizes

_cache = {}


def _sampled(name, wl=None, modes=FULL_MODES):
    """GPU outputs plus the oracle on every token's statistics, 256 sampled
    dx rows and 256 sampled dW / db rows, for one full-size problem (a named
    workload, or `wl` under that name) in the given backward modes."""
    if name in _cache:
        return _cache[name]
    _cache.clear()
    wl = I.WORKLOADS[name] if wl is None else wl
    inp = I.make_inputs(wl)
    prob = DeviceProblem(inp)
    opts = opts_of(wl)
    x64, W64, b64 = f64(inp)
    lse, zt, sz = O.row_stats(x64, W64, b64, inp.y, ignore_index=wl.ignore_index,
                              logit_scale=wl.logit_scale, block=256)
    tl = O.token_losses_from_stats(lse, zt, sz, inp.y, wl.V, wl.ignore_index,
                                   wl.label_smoothing, wl.lse_square_scale)
    ref_loss = O.reduce_losses(tl, inp.y, wl.ignore_index, wl.reduction)
    # Forced samples: the seams of the tilings and of the backward vocabulary
    # block the library picks by default at this size (parity.token_seams,
    # parity.vocab_seams), ignored tokens, and the most frequent targets.
    ignored = np.nonzero(inp.y == wl.ignore_index)[0][:8]
    rows = I.sample_indices(wl.seed, wl.N, 256,
                            must_include=list(ignored) + token_seams(wl.N))
    valid_y = inp.y[inp.y != wl.ignore_index]
    top = np.argsort(-np.bincount(valid_y, minlength=wl.V))[:8] if valid_y.size else []
    block = tuning.library_default_block(wl.N, wl.V)
    vrows = I.sample_indices(wl.seed + 1, wl.V, 256,
                             must_include=list(top) + vocab_seams(wl.V, block))
    assert set(token_seams(wl.N)) <= set(rows.tolist())
    assert set(vocab_seams(wl.V, block)) <= set(vrows.tolist())
    dl = inp.dloss.astype(np.float64)
    rdx = O.dx_rows(rows, dl, x64, W64, b64, inp.y, **opts)
    rdW, rdb = O.dW_db_rows(vrows, lse, dl, x64, W64, b64, inp.y, **opts)
    got = {}
    for mode in modes:
        out = prob.run(mode=mode)
        assert out["err"] == 0, f"device error word {out['err']}"
        got[mode] = dict(loss=to_np(out["loss"]), lse=to_np(out["lse"]),
                          dx=to_np(out["dx"][torch.from_numpy(rows).to(out["dx"].device)]),
                          dW=to_np(out["dW"][torch.from_numpy(vrows).to(out["dW"].device)]),
                          db=None if out["db"] is None else to_np(out["db"])[vrows])
        del out
        torch.cuda.empty_cache()
    res = dict(wl=wl, got=got, ref=dict(loss=ref_loss, lse=lse, dx=rdx, dW=rdW, db=rdb))
    _cache[name] = res
    return res


@pytest.mark.parametrize("mode", FULL_MODES)
@pytest.mark.parametrize("name", ["llama3_head", "large_logit", "vocab256k"])
def test_full_size_sampled(name, mode):
    r = _sampled(name)
    g, ref, wl = r["got"][mode], r["ref"], r["wl"]
    assert_loss_close(g["loss"], ref["loss"], f"{name} loss")
    assert_loss_close(g["lse"], ref["lse"], f"{name} lse (all tokens)")
    assert_grad_close(g["dx"], ref["dx"], f"{name} dx (sampled rows)")
    assert_grad_close(g["dW"], ref["dW"], f"{name} dW (sampled vocab rows)")
    if wl.has_bias:
        assert_grad_close(g["db"], ref["db"], f"{name} db (sampled)")


@pytest.mark.parametrize("mode", ["kept", "recompute"])
def test_full_size_sampled_fp16_llama3_head(mode):
    # The headline shape with fp16 operands (the loss-scale-safe dL path). dx
    # is written in fp16: unscaled, the mean over 8192 tokens puts it near
    # 2e-6, in fp16's subnormals; as in fp16 training a loss scale (1024)
    # keeps it in range.
    wl = I.WORKLOADS["llama3_head"].with_(name="llama3_head_fp16", dtype="fp16",
                                          dloss_scale=1024.0)
    r = _sampled("llama3_head_fp16", wl, modes=["kept", "recompute"])
    g, ref = r["got"][mode], r["ref"]
    assert_loss_close(g["loss"], ref["loss"], "fp16 llama3_head loss")
    assert_loss_close(g["lse"], ref["lse"], "fp16 llama3_head lse (all tokens)")
    assert_grad_close(g["dx"], ref["dx"], "fp16 llama3_head dx (sampled rows)")
    assert_grad_close(g["dW"], ref["dW"], "fp16 llama3_head dW (sampled vocab rows)")


def test_bounded_wait_times_out_with_a_status_and_the_context_survives():
    # A wait on a barrier nothing arrives on gives up after ~1 ms of clocks,
    # sets the timeout bit, and the next FLCE call on the same context works.
    from linear_cross_entropy_gemm_gb300 import _lib
    dev = torch.device("cuda", 0)
    word = F.device_error_word(dev)
    st = _lib.load().flce_selftest_wait_timeout(word.data_ptr(), 2_000_000,
                                                torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0
    torch.cuda.synchronize(dev)
    assert F.flce_read_device_error(dev) == 2  # FLCE_DEVERR_TIMEOUT, then cleared
    full_check(I.WORKLOADS["tiny"])            # the context is still healthy


def test_non_contiguous_inputs_are_rejected():
    dev = torch.device("cuda", 0)
    x = torch.randn(64, 128, device=dev).to(torch.bfloat16)[:, ::2]
    W = torch.randn(100, 64, device=dev).to(torch.bfloat16)
    y = torch.zeros(64, dtype=torch.int64, device=dev)
    with pytest.raises(ValueError):
        F.flce_forward(x, W, None, y)


@pytest.mark.parametrize("mode,keep_vocab", [("recompute", 0), ("stored", 0), ("kept", 0),
                                             ("kept", 768)])
@pytest.mark.parametrize("N", [300, 129, 1])
def test_no_writes_outside_caller_buffers(N, mode, keep_vocab):
    # Every buffer the library writes gets a canary-filled guard region after
    # it (N = 300: an odd number of 128-row tiles, so a CTA pair's second half
    # is pure padding); the guards must be untouched after forward + backward.
    wl = I.Workload("guard", N=N, H=136, V=1300, seed=34, b_std=0.1, ignore_frac=0.1,
                    label_smoothing=0.1, lse_square_scale=1e-3)
    inp = I.make_inputs(wl)
    p = DeviceProblem(inp)
    opts = opts_of(wl)
    dev = p.dev
    G = 1 << 16  # guard bytes

    def guarded(nbytes):
        t = torch.full((nbytes + G,), 0xA5, dtype=torch.uint8, device=dev)
        return t

    def check(t, nbytes, what):
        tail = t[nbytes:]
        assert bool((tail == 0xA5).all()), f"{what}: write past the end"

    nf = F.flce_workspace_size(N, wl.H, wl.V, "forward", **opts)
    kind = {"kept": "backward_keep", "stored": "backward_store"}.get(mode, "backward")
    nb = F.flce_workspace_size(N, wl.H, wl.V, kind, bwd_vocab_block=512, keep_vocab=keep_vocab,
                               has_bias=wl.has_bias, **opts)
    # (the binding would allocate a workspace of its own if this one were
    # smaller than the call needs, and the guard would then check nothing)
    assert wl.has_bias
    wf, wb = guarded(nf), guarded(nb)
    state, ns, skw = None, 0, {}
    if mode == "stored":
        ns = F.flce_saved_size(N, wl.H, wl.V, **opts)
        state = guarded(ns)
        skw = dict(saved=state[:ns])
    elif mode == "kept":
        ns = F.flce_kept_size(N, wl.H, wl.V, bwd_vocab_block=512, keep_vocab=keep_vocab, **opts)
        state = guarded(ns)
        skw = dict(kept=state[:ns], keep_vocab=keep_vocab)
    lossb, lseb = guarded(4), guarded(4 * N)
    dxb, dWb, dbb = guarded(2 * N * wl.H), guarded(4 * wl.V * wl.H), guarded(4 * wl.V)
    loss = lossb[:4].view(torch.float32)
    lse = lseb[:4 * N].view(torch.float32)
    dx = dxb[:2 * N * wl.H].view(torch.bfloat16).view(N, wl.H)
    dW = dWb[:4 * wl.V * wl.H].view(torch.float32).view(wl.V, wl.H)
    db = dbb[:4 * wl.V].view(torch.float32)
    F.flce_forward(p.x, p.W, p.b, p.y, workspace=wf[:nf], out=(loss, lse),
                   bwd_vocab_block=512, **skw, **opts)
    F.flce_backward(p.dloss, lse, p.x, p.W, p.b, p.y, workspace=wb[:nb], out=(dx, dW, db),
                    bwd_vocab_block=512, **skw, **opts)
    torch.cuda.synchronize()
    assert F.flce_read_device_error(dev) == 0
    for t, n, what in ((wf, nf, "forward workspace"), (wb, nb, "backward workspace"),
                       (lossb, 4, "loss"), (lseb, 4 * N, "lse"), (dxb, 2 * N * wl.H, "dx"),
                       (dWb, 4 * wl.V * wl.H, "dW"), (dbb, 4 * wl.V, "db")):
        check(t, n, what)
    if state is not None:
        check(state, ns, f"{mode} state")
    ref = p.run(bwd_vocab_block=512, mode=mode, keep_vocab=keep_vocab)
    assert torch.equal(ref["dW"], dW) and torch.equal(ref["db"], db)
