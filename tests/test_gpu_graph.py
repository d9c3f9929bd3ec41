"""flce_forward + flce_backward captured into one CUDA graph, in the
recompute, kept-block and stored modes: the calls make no host synchronisation
or allocation of their own (the caller passes the workspace, the kept
buffer and the outputs), so a replay runs the same kernels on the captured
buffers. The library is run-to-run deterministic, so a replay must equal an
eager call bit for bit, also after the inputs are overwritten in place."""
import pytest
import torch

import linear_cross_entropy_gemm_gb300 as F
from linear_cross_entropy_gemm_gb300 import inputs as I
from parity import bf16_dev, opts_of

pytestmark = pytest.mark.gpu


def _problem(seed):
    wl = I.Workload("graph", N=640, H=256, V=3000, seed=seed, b_std=0.05, ignore_frac=0.05,
                    label_smoothing=0.1, lse_square_scale=1e-3, reduction="mean")
    inp = I.make_inputs(wl)
    return wl, inp


@pytest.mark.parametrize("mode", ["recompute", "kept", "wider kept", "stored"])
@pytest.mark.parametrize("form", ["single", "pair", "wide"])
def test_forward_backward_replay_in_a_cuda_graph_equals_eager(form, mode):
    wl, inp = _problem(41)
    dev = torch.device("cuda:0")
    x = bf16_dev(inp.x, dev)
    W = bf16_dev(inp.W, dev)
    b = bf16_dev(inp.b, dev)
    y = torch.from_numpy(inp.y).to(dev)
    dloss = torch.from_numpy(inp.dloss).to(dev)
    opts = opts_of(wl)
    N, H, V = wl.N, wl.H, wl.V
    fws = torch.empty(F.flce_workspace_size(N, H, V, "forward", has_bias=True, **opts),
                      dtype=torch.uint8, device=dev)
    # "wider kept": the kept block is [0, 1792), then 1024 + 184 columns
    # are recomputed.
    kv = 1792 if mode == "wider kept" else 0
    kind = {"kept": "backward_keep", "wider kept": "backward_keep",
            "stored": "backward_store"}.get(mode, "backward")
    bws = torch.empty(F.flce_workspace_size(N, H, V, kind, has_bias=True, bwd_vocab_block=1024,
                                            keep_vocab=kv, **opts), dtype=torch.uint8, device=dev)
    state = {}
    if mode in ("kept", "wider kept"):
        state = dict(kept=torch.empty(F.flce_kept_size(N, H, V, bwd_vocab_block=1024,
                                                       keep_vocab=kv),
                                      dtype=torch.uint8, device=dev), keep_vocab=kv)
    elif mode == "stored":
        state = dict(saved=torch.empty(F.flce_saved_size(N, H, V), dtype=torch.uint8,
                                       device=dev))
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dx = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    db = torch.empty(V, dtype=torch.float32, device=dev)

    def step():
        F.flce_forward(x, W, b, y, workspace=fws, out=(loss, lse), gemm_form=form,
                       bwd_vocab_block=1024, **state, **opts)
        F.flce_backward(dloss, lse, x, W, b, y, workspace=bws, out=(dx, dW, db),
                        gemm_form=form, bwd_vocab_block=1024, **state, **opts)

    def snapshot():
        torch.cuda.synchronize(dev)
        return [t.clone() for t in (loss, lse, dx, dW, db)]

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream(dev).wait_stream(side)
    eager = snapshot()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (loss, lse, dx, dW, db):
        t.zero_()
    g.replay()
    replayed = snapshot()
    for a, r in zip(eager, replayed):
        assert torch.equal(a, r)
    assert F.flce_read_device_error(dev) == 0

    # New inputs written into the captured buffers: the replay computes them.
    _, inp2 = _problem(42)
    x.copy_(bf16_dev(inp2.x, dev))
    y.copy_(torch.from_numpy(inp2.y).to(dev))
    g.replay()
    replayed2 = snapshot()
    step()
    eager2 = snapshot()
    for a, r in zip(eager2, replayed2):
        assert torch.equal(a, r)
    assert not torch.equal(eager[2], eager2[2])
