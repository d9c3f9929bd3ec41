"""Vocabulary-parallel FLCE on one GPU: the vocabulary is cut into uneven
shards, each shard runs the library's shard kernels, the test stands in for
the collectives (elementwise max / sum over the shards' tensors), and the
result must match the CPU oracle on the whole vocabulary."""
import numpy as np
import pytest
import torch

from linear_cross_entropy_gemm_gb300 import inputs as I
from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
from oracle import flce_oracle as O
from parity import DeviceProblem, assert_grad_close, assert_loss_close, f64, opts_of, to_np

pytestmark = pytest.mark.gpu


def _sim_allreduce(tensors):
    """All-reduce over simulated ranks: returns a function per rank index that
    reduces in place across every rank's tensor of the same collective."""
    def run(op):
        stacked = torch.stack(tensors)
        red = stacked.max(0).values if op == "max" else stacked.sum(0)
        for t in tensors:
            t.copy_(red)
    return run


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode", ["recompute", "kept", "wider kept"])
@pytest.mark.parametrize("form", ["default", "single", "wide"])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_uneven_shards_match_whole_vocabulary(reduction, form, mode, dtype, monkeypatch):
    # The shard calls take no gemm_form of their own: the environment override
    # selects the kernel form for every call of the test (shard offsets in the
    # wide and single-CTA kernels as well as the default pairs).
    if form != "default":
        monkeypatch.setenv("FLCE_GEMM_FORM", form)
    # fp16: as in fp16 training, a loss scale keeps the fp16 dx above fp16's
    # subnormals.
    wl = I.Workload("vp", N=300, H=264, V=3001, seed=41, b_std=0.3, ignore_frac=0.1,
                    label_smoothing=0.1, lse_square_scale=1e-3, logit_scale=0.8,
                    reduction=reduction,
                    dloss="normal_per_token" if reduction == "none" else "normal_scalar",
                    dtype=dtype, dloss_scale=1024.0 if dtype == "fp16" else 1.0)
    inp = I.make_inputs(wl)
    prob = DeviceProblem(inp)
    opts = opts_of(wl)
    cuts = [0, 1000, 2256, 3001]
    shards = [(a, b - a) for a, b in zip(cuts[:-1], cuts[1:])]

    # Kept mode: each shard keeps its own first 512-column block (the shards
    # are 1000, 1256 and 745 columns wide); "wider kept": its first 768
    # columns (all of the third shard).
    bvb = 512
    kv = {"kept": 0, "wider kept": 768}.get(mode)
    sopts = dict(opts, keep_vocab=kv or 0)  # the shard calls' options
    kept = [VP.kept_size(wl.N, wl.H, n, vocab_start=a, vocab_total=wl.V, bwd_vocab_block=bvb,
                         keep_vocab=kv) for a, n in shards] if kv is not None else [0] * len(shards)
    kept = [torch.empty(k, dtype=torch.uint8, device=prob.dev) if k else None for k in kept]

    # forward: local stats, MAX of m, rescale, SUM of (d, z_y, sum z)
    stats = [VP.forward_shard(prob.x, prob.W[a:a + n].contiguous(), prob.b[a:a + n].contiguous(),
                              prob.y, vocab_start=a, vocab_total=wl.V, kept=k,
                              bwd_vocab_block=bvb, **sopts)
             for (a, n), k in zip(shards, kept)]
    gmax = [s[0].clone() for s in stats]
    _sim_allreduce(gmax)("max")
    for s, m in zip(stats, gmax):
        VP.rescale(s, m)
    _sim_allreduce([s[1:] for s in stats])("sum")
    loss, lse = VP.loss_from_stats(stats[0], prob.y, vocab_total=wl.V, H=wl.H, **opts)

    # backward: per-shard dW rows, db, fp32 dx partials summed then cast once
    parts = [VP.backward_shard(prob.dloss, lse, prob.x, prob.W[a:a + n].contiguous(),
                               prob.b[a:a + n].contiguous(), prob.y, vocab_start=a,
                               vocab_total=wl.V, kept=k, bwd_vocab_block=bvb, **sopts)
             for (a, n), k in zip(shards, kept)]
    dx32 = [p[0] for p in parts]
    _sim_allreduce(dx32)("sum")
    dx = VP.cast16(dx32[0], prob.x.dtype)
    dW = torch.cat([p[1] for p in parts])
    db = torch.cat([p[2] for p in parts])
    torch.cuda.synchronize()

    x64, W64, b64 = f64(inp)
    rl, rlse = O.forward(x64, W64, b64, inp.y, **opts)
    rdx, rdW, rdb = O.backward(inp.dloss.astype(np.float64), x64, W64, b64, inp.y, **opts)
    assert_loss_close(to_np(loss), rl, "sharded loss")
    assert_loss_close(to_np(lse), rlse, "sharded lse")
    assert_grad_close(to_np(dx), rdx, "sharded dx")
    assert_grad_close(to_np(dW), rdW, "sharded dW")
    assert_grad_close(to_np(db), rdb, "sharded db")

    # and the sharded path agrees with the whole-vocabulary call
    whole = prob.run()
    assert_loss_close(to_np(loss), to_np(whole["loss"]), "sharded vs whole loss")
    assert_grad_close(to_np(dW), to_np(whole["dW"]), "sharded vs whole dW")


def test_single_shard_covering_everything_equals_plain_call():
    wl = I.WORKLOADS["tiny"]
    inp = I.make_inputs(wl)
    prob = DeviceProblem(inp)
    opts = opts_of(wl)
    loss, lse = VP.vocab_parallel_forward(prob.x, prob.W, None, prob.y, vocab_start=0,
                                          vocab_total=wl.V, allreduce=lambda t, op: None, **opts)
    dx, dW, _ = VP.vocab_parallel_backward(prob.dloss, lse, prob.x, prob.W, None, prob.y,
                                           vocab_start=0, vocab_total=wl.V,
                                           allreduce=lambda t, op: None, **opts)
    whole = prob.run()
    assert torch.equal(lse, whole["lse"])
    assert_loss_close(to_np(loss), to_np(whole["loss"]), "one-shard loss")
    assert torch.equal(dW, whole["dW"])
    assert_grad_close(to_np(dx), to_np(whole["dx"]), "one-shard dx")
