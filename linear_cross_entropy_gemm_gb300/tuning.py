"""Per-shape choice of the GEMM form and the backward vocabulary block.

The library defaults (wide CTA-pair GEMMs, 256 x 512 tiles; the widest
backward vocabulary block BVc whose [N, BVc] 16-bit dL staging buffer fits
1 GiB) are tuned for large heads. Other shapes can prefer the 256 x 256 pair
or single-CTA forms (more, smaller tiles fill the 152 SMs better) or another
BVc: the block count sets how many dW / dx GEMM launches a backward makes,
whether dx needs its fp32 accumulator (one block does not), and how ragged
the last block is.

``autotune`` times the candidates through the C ABI on the caller's own
tensors (CUDA events on the current stream, median of ``reps``) and keeps the
fastest per key. Only timing is done here; every candidate runs the same
kernels and computes the same results up to fp32 accumulation order.
"""
from __future__ import annotations

import dataclasses
import statistics
from typing import Callable, Dict, Optional, Sequence, Tuple

import torch

# The library's default staging budget and smallest default block (flce_api.cu).
DEFAULT_DL_BUDGET = 1 << 30
MIN_DEFAULT_BLOCK = 4096
# "default" is the library's own per-GEMM choice, so the tuner never does
# worse than a plain call (up to timing noise).
FORMS = ("default", "single", "pair", "wide")


@dataclasses.dataclass(frozen=True)
class FlceConfig:
    """Launch configuration of one problem key. "default" / 0 leave a choice
    to the library."""
    fwd_gemm_form: str = "default"
    bwd_gemm_form: str = "default"
    bwd_vocab_block: int = 0

    def forward_kwargs(self) -> dict:
        return {"gemm_form": self.fwd_gemm_form}

    def backward_kwargs(self) -> dict:
        return {"gemm_form": self.bwd_gemm_form, "bwd_vocab_block": self.bwd_vocab_block}


@dataclasses.dataclass(frozen=True)
class TuneResult:
    config: FlceConfig
    forward_ms: Dict[str, float]
    backward_ms: Dict[Tuple[str, int], float]
    key: tuple

    def as_dict(self) -> dict:
        return {"config": dataclasses.asdict(self.config),
                "forward_ms": dict(self.forward_ms),
                "backward_ms": {f"{f}/{bv}": ms for (f, bv), ms in self.backward_ms.items()}}


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def library_default_block(N: int, V: int, budget_bytes: int = DEFAULT_DL_BUDGET) -> int:
    """BVc the library picks for bwd_vocab_block = 0 (16-bit dL elements)."""
    bv = budget_bytes // (max(N, 1) * 2) // 256 * 256
    bv = max(bv, MIN_DEFAULT_BLOCK)
    return min(bv, round_up(V, 256))


def vocab_block_candidates(N: int, V: int, budget_bytes: int = DEFAULT_DL_BUDGET,
                           max_blocks: int = 8, min_block: int = 1024) -> list:
    """Backward vocabulary blocks to try, widest first: the library default and
    the splits of the vocabulary into k = 1..max_blocks nearly equal blocks
    (multiples of 256) whose dL buffer fits the budget and that are at least
    ``min_block`` wide (or the whole vocabulary, if that is narrower)."""
    vr = round_up(V, 256)
    out = {library_default_block(N, V, budget_bytes)}
    for k in range(1, max_blocks + 1):
        bv = round_up(-(-vr // k), 256)
        if N * bv * 2 <= budget_bytes and (bv >= min_block or bv == vr):
            out.add(bv)
    return sorted(out, reverse=True)


def select(forward_ms: Dict[str, float], backward_ms: Dict[Tuple[str, int], float]) -> FlceConfig:
    """Fastest forward form and fastest backward (form, block); ties go to the
    first candidate in the given order."""
    fwd = min(forward_ms, key=lambda k: forward_ms[k])
    bwd = min(backward_ms, key=lambda k: backward_ms[k])
    return FlceConfig(fwd_gemm_form=fwd, bwd_gemm_form=bwd[0], bwd_vocab_block=int(bwd[1]))


def problem_key(x, W, b, *, label_smoothing: float, dW_dtype, db_dtype,
                budget_bytes: int, mode: str = "recompute") -> tuple:
    """What the timings depend on: device, sizes, operand type, bias, the
    smoothing partial, the gradient output types, the staging budget and the
    backward mode."""
    return (torch.cuda.get_device_name(x.device), int(x.shape[0]), int(x.shape[1]),
            int(W.shape[0]), str(x.dtype), b is not None, float(label_smoothing) > 0.0,
            str(dW_dtype), str(db_dtype), int(budget_bytes), mode)


_CACHE: Dict[tuple, TuneResult] = {}


def cached() -> Dict[tuple, TuneResult]:
    return dict(_CACHE)


def clear_cache() -> None:
    _CACHE.clear()


def _event_timer(fn: Callable[[], None], reps: int, warmup: int) -> float:
    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def _interleaved(cands: Dict, timer: Callable[[Callable[[], None], int, int], float], reps: int,
                 warmup: int) -> Dict:
    """Median time per candidate, measured round-robin: every candidate is
    warmed up, then each repetition times every candidate once, so a drift of
    the GPU's clock (at the power cap it moves with temperature and the power
    history) falls on all candidates alike instead of on whichever ran last."""
    for fn in cands.values():
        timer(fn, 1, warmup)
    times = {k: [] for k in cands}
    for _ in range(reps):
        for k, fn in cands.items():
            times[k].append(timer(fn, 1, 0))
    return {k: statistics.median(v) for k, v in times.items()}


def autotune(x: torch.Tensor, W: torch.Tensor, b: Optional[torch.Tensor], y: torch.Tensor, *,
             dloss: Optional[torch.Tensor] = None, ignore_index: int = -100,
             label_smoothing: float = 0.0, lse_square_scale: float = 0.0,
             logit_scale: float = 1.0, reduction: str = "mean",
             dW_dtype: torch.dtype = torch.float32, db_dtype: torch.dtype = torch.float32,
             forms: Sequence[str] = FORMS, vocab_blocks: Optional[Sequence[int]] = None,
             budget_bytes: int = DEFAULT_DL_BUDGET, reps: int = 3, warmup: int = 1,
             use_cache: bool = True, mode: str = "recompute",
             timer: Callable[[Callable[[], None], int, int], float] = _event_timer) -> TuneResult:
    """Time flce_forward per GEMM form and the backward per (form, BVc) on
    these tensors, candidates interleaved round-robin (``_interleaved``), and
    return the fastest configuration (cached per ``problem_key``). mode "recompute" times flce_backward alone; mode "kept"
    times, per (form, BVc), the kept-block forward + backward pair (the kept
    block is BVc wide, so the pair is what the block choice changes), and
    backward_ms then holds those pair times. Allocates one set of outputs and
    the largest workspace (and kept buffer) the candidates need; synchronises
    the current stream."""
    from . import flce_backward, flce_forward, flce_kept_size, flce_workspace_size
    if mode not in ("recompute", "kept"):
        raise ValueError(f"autotune: mode must be 'recompute' or 'kept', got {mode!r}")
    key = problem_key(x, W, b, label_smoothing=label_smoothing, dW_dtype=dW_dtype,
                      db_dtype=db_dtype, budget_bytes=budget_bytes, mode=mode)
    if use_cache and key in _CACHE:
        return _CACHE[key]
    N, H = x.shape
    V = W.shape[0]
    dev = x.device
    opts = dict(ignore_index=ignore_index, label_smoothing=label_smoothing,
                lse_square_scale=lse_square_scale, logit_scale=logit_scale, reduction=reduction)
    size_opts = dict(opts, has_bias=b is not None, input_fp16=x.dtype == torch.float16)
    blocks = list(vocab_blocks) if vocab_blocks is not None else \
        vocab_block_candidates(N, V, budget_bytes)
    if dloss is None:
        dloss = torch.ones(N if reduction == "none" else 1, dtype=torch.float32, device=dev)

    ws_f = torch.empty(max(flce_workspace_size(N, H, V, "forward", **size_opts), 1),
                       dtype=torch.uint8, device=dev)
    kept = mode == "kept"
    need_b = max(flce_workspace_size(N, H, V, "backward_keep" if kept else "backward",
                                     bwd_vocab_block=bv, dW_fp32=dW_dtype == torch.float32,
                                     db_fp32=db_dtype == torch.float32, **size_opts)
                 for bv in blocks)
    ws_b = torch.empty(max(need_b, 1), dtype=torch.uint8, device=dev)
    kept_buf = None
    if kept:
        need_k = max(flce_kept_size(N, H, V, bwd_vocab_block=bv, **size_opts) for bv in blocks)
        kept_buf = torch.empty(max(need_k, 1), dtype=torch.uint8, device=dev)
    loss = torch.empty(N if reduction == "none" else 1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dx = torch.empty(N, H, dtype=x.dtype, device=dev)
    dW = torch.empty(V, H, dtype=dW_dtype, device=dev)
    db = torch.empty(V, dtype=db_dtype, device=dev) if b is not None else None

    forward_ms = _interleaved(
        {form: (lambda form=form: flce_forward(x, W, b, y, workspace=ws_f, out=(loss, lse),
                                               gemm_form=form, **opts)) for form in forms},
        timer, reps, warmup)
    flce_forward(x, W, b, y, workspace=ws_f, out=(loss, lse), **opts)
    def kept_pair(form, bv):
        flce_forward(x, W, b, y, workspace=ws_f, out=(loss, lse), gemm_form=form, kept=kept_buf,
                     bwd_vocab_block=bv, **opts)
        flce_backward(dloss, lse, x, W, b, y, dW_dtype=dW_dtype, db_dtype=db_dtype,
                      bwd_vocab_block=bv, workspace=ws_b, out=(dx, dW, db), gemm_form=form,
                      kept=kept_buf, **opts)

    cands = {}
    for form in forms:
        for bv in blocks:
            if kept:
                fn = lambda form=form, bv=int(bv): kept_pair(form, bv)
            else:
                fn = lambda form=form, bv=int(bv): flce_backward(
                    dloss, lse, x, W, b, y, dW_dtype=dW_dtype, db_dtype=db_dtype,
                    bwd_vocab_block=bv, workspace=ws_b, out=(dx, dW, db),
                    gemm_form=form, **opts)
            cands[(form, int(bv))] = fn
    backward_ms = _interleaved(cands, timer, reps, warmup)
    result = TuneResult(config=select(forward_ms, backward_ms), forward_ms=forward_ms,
                        backward_ms=backward_ms, key=key)
    if use_cache:
        _CACHE[key] = result
    return result
