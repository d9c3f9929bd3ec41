"""Peak device memory of a forward + backward, measured, against the method's
budget: one [N, BVc] 16-bit block (the dL staging block, which in the
kept-block mode first holds the kept probabilities, plus their per-32-column
maxima), the fp32 dx accumulator, the db column partials (with a bias), the
forward's per-vocabulary-tile partials and per-token coefficients. No [V, H]
fp32 dW accumulator exists (dW is written once per block), and the library
allocates nothing itself: the device's free memory does not move during a
call. The budget mode (the kept block as wide as flce_keep_vocab_within
allows) may add the fp32 [V, H] allowance, 4 V H bytes."""
import pytest
import torch

import linear_cross_entropy_gemm_gb300 as F
from linear_cross_entropy_gemm_gb300 import inputs as I
from linear_cross_entropy_gemm_gb300 import tuning
from parity import DeviceProblem

pytestmark = pytest.mark.gpu


def scratch_bound(N, H, V, bv, has_bias):
    db_parts = 4 * -(-N // 128) * bv * 4 if has_bias else 0
    return (N * bv * 2 + N * (bv // 32) * 4 + N * H * 4 + db_parts + N * -(-V // 256) * 12
            + N * 32 + (1 << 20))


@pytest.mark.parametrize("mode", ["recompute", "kept", "budget"])
@pytest.mark.parametrize("name", ["tiny", "medium", "llama3_head", "large_logit", "vocab256k"])
def test_peak_memory_within_the_block_budget(name, mode):
    wl = I.WORKLOADS[name]
    N, H, V = wl.N, wl.H, wl.V
    dev = torch.device("cuda", 0)
    p = DeviceProblem(I.make_inputs(wl))
    p.run(mode=mode)  # first launches (module loading) outside the measurement
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    reserved0 = torch.cuda.memory_reserved(dev)
    out = p.run(mode=mode)
    torch.cuda.synchronize(dev)
    free1 = torch.cuda.mem_get_info(dev)[0]
    reserved1 = torch.cuda.memory_reserved(dev)
    assert out["err"] == 0
    peak = torch.cuda.max_memory_allocated(dev) - base
    outputs = sum(t.numel() * t.element_size()
                  for t in (out["loss"], out["lse"], out["dx"], out["dW"], out["db"])
                  if t is not None)
    bv = tuning.library_default_block(N, V)
    bound = scratch_bound(N, H, V, bv, wl.has_bias) + (4 * V * H if mode == "budget" else 0)
    assert peak - outputs <= bound, (peak - outputs, bound)
    # Everything the device gave away during the call went to torch's pool:
    # nothing was allocated behind the allocator's back.
    assert (free0 - free1) == (reserved1 - reserved0)
    # The kept-block mode takes no more memory than the recompute mode.
    if mode == "kept":
        kept = F.flce_kept_size(N, H, V)
        ws = F.flce_workspace_size(N, H, V, "backward_keep", has_bias=wl.has_bias,
                                   label_smoothing=wl.label_smoothing)
        ws_plain = F.flce_workspace_size(N, H, V, "backward", has_bias=wl.has_bias,
                                         label_smoothing=wl.label_smoothing)
        assert kept + ws <= ws_plain + N * (bv // 32) * 4 + (1 << 10)


@pytest.mark.parametrize("name", ["medium", "llama3_head"])
def test_autograd_module_peak_memory(name):
    # The user-facing module (default: one kept block): forward + backward
    # peaks at the library's scratch plus the gradients in the parameters'
    # own type (dW and db written as bf16 by the library; no fp32 [V, H]
    # temporary).
    wl = I.WORKLOADS[name]
    N, H, V = wl.N, wl.H, wl.V
    dev = torch.device("cuda", 0)
    p = DeviceProblem(I.make_inputs(wl))
    x = p.x.clone().requires_grad_(True)
    W = p.W.clone().requires_grad_(True)
    b = None if p.b is None else p.b.clone().requires_grad_(True)
    mod = F.FusedLinearCrossEntropyLoss(label_smoothing=wl.label_smoothing,
                                        lse_square_scale=wl.lse_square_scale,
                                        logit_scale=wl.logit_scale, reduction="mean")

    def step():
        loss = mod(x, p.y, W, b)
        loss.backward()
        return loss

    step()  # first launches (module loading) outside the measurement
    x.grad = W.grad = None
    if b is not None:
        b.grad = None
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step()
    torch.cuda.synchronize(dev)
    assert F.flce_read_device_error(dev) == 0
    assert W.grad.dtype == W.dtype and x.grad.dtype == x.dtype
    peak = torch.cuda.max_memory_allocated(dev) - base
    grads = (N * H + V * H + (V if b is not None else 0)) * 2
    bv = tuning.library_default_block(N, V)
    bound = scratch_bound(N, H, V, bv, wl.has_bias) + grads + (1 << 20)
    assert peak <= bound, (peak / 2**20, bound / 2**20)
