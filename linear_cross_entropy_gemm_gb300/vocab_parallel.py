"""Vocabulary-parallel fused linear cross-entropy (DeepSpeed PR #8792).

Each rank holds the rows [vocab_start, vocab_start + V_local) of the LM head
(uneven shards allowed) and the same tokens and targets. Forward: every rank
folds its logits into per-token statistics (m, d, z_y, sum z) with the
library's kernels; one MAX all-reduce of m, a rescale of d to the common
max, and one SUM all-reduce of (d, z_y, sum z) give every rank the
whole-vocabulary lse and loss. Backward: each rank writes its own dW rows
and db and an fp32 partial dx; a SUM all-reduce of the fp32 partials comes
before the single cast to bf16, so partials that would overflow a narrower
type but cancel across shards stay finite.

The collectives are torch.distributed all-reduces on ``group`` (skipped when
there is a single rank); ``allreduce`` may replace them (a function
``allreduce(tensor, op)`` with op "max" or "sum", reducing in place).
All arithmetic runs in the library's CUDA kernels.

With ``kept`` (a uint8 CUDA tensor of ``kept_size`` bytes, the same on the
forward and the backward of a shard) the shard's forward also keeps the
probabilities of its own first backward vocabulary block, and its backward
converts them instead of recomputing that block (the kept-block mode of the
whole-vocabulary calls, per shard).
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import _lib
from . import _check_inputs, _ptr, _stream, device_error_word, params, FlceError

AllReduce = Callable[[torch.Tensor, str], None]


def _dist_allreduce(group) -> AllReduce:
    import torch.distributed as dist

    def f(t: torch.Tensor, op: str) -> None:
        if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
            return
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM, group=group)
    return f


def shard_range(vocab_total: int, world: int, rank: int) -> tuple:
    """The contiguous vocabulary rows [start, end) of rank `rank` when
    `vocab_total` rows are split over `world` ranks: shard boundaries at
    k * vocab_total / world rounded down to a multiple of 256 (the tile width),
    so the shards differ by at most 256 rows, plus the ragged end the last one
    takes. A vocabulary under 256 * world rows leaves some ranks empty."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"shard_range: rank {rank} of {world}")

    def bound(k):
        return vocab_total if k == world else (k * vocab_total // world) // 256 * 256
    return bound(rank), bound(rank + 1)


def _shard_params(N, H, V_local, vocab_start, vocab_total, has_bias, fp16, opts,
                  bwd_vocab_block=0):
    return params(N, H, V_local, has_bias=has_bias, vocab_start=vocab_start,
                  vocab_total=vocab_total, input_fp16=fp16, bwd_vocab_block=bwd_vocab_block,
                  **opts)


def kept_size(N, H, V_local, *, vocab_start, vocab_total, bwd_vocab_block=0,
              input_fp16=False, keep_vocab=0) -> int:
    """Bytes of a shard's kept state (flce_kept_size for the shard's rows;
    ``keep_vocab`` widens the kept block as in flce_forward, give it to
    forward_shard and backward_shard too)."""
    p = params(N, H, V_local, vocab_start=vocab_start, vocab_total=vocab_total,
               bwd_vocab_block=bwd_vocab_block, input_fp16=input_fp16, keep_vocab=keep_vocab)
    return int(_lib.load().flce_kept_size(p))


def _check_kept(kept, lib, p):
    if kept.dtype != torch.uint8 or not kept.is_cuda or not kept.is_contiguous():
        raise TypeError("flce: kept must be a contiguous uint8 CUDA tensor")
    if kept.numel() < lib.flce_kept_size(p):
        raise ValueError("flce: kept is smaller than the shard's flce_kept_size()")


def forward_shard(x, W, b, y, *, vocab_start, vocab_total, stream=None, kept=None,
                  bwd_vocab_block=0, **opts) -> torch.Tensor:
    """This shard's per-token statistics, a [4, N] fp32 tensor (m, d, z_y, sum z);
    with ``kept``, also the shard's kept block (for backward_shard(kept=))."""
    _check_inputs(x, W, b, y)
    lib = _lib.load()
    N, H = x.shape
    p = _shard_params(N, H, W.shape[0], vocab_start, vocab_total, b is not None,
                      x.dtype == torch.float16, opts, bwd_vocab_block)
    stats = torch.empty(4, N, dtype=torch.float32, device=x.device)
    ws = torch.empty(max(lib.flce_workspace_size(p, 0), 1), dtype=torch.uint8, device=x.device)
    if kept is not None:
        _check_kept(kept, lib, p)
        st = lib.flce_forward_shard_keep(p, _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(stats),
                                         _ptr(kept), kept.numel(), _ptr(ws), ws.numel(),
                                         _ptr(device_error_word(x.device)), _stream(stream))
    else:
        st = lib.flce_forward_shard(p, _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(stats),
                                    _ptr(ws), ws.numel(), _ptr(device_error_word(x.device)),
                                    _stream(stream))
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_forward_shard")
    return stats


def rescale(stats: torch.Tensor, global_max: torch.Tensor, stream=None) -> None:
    """d <- d 2^(m - M), m <- M (in place), M the all-shard max of m."""
    N = stats.shape[1]
    p = params(N, 8, 1)
    st = _lib.load().flce_shard_rescale(p, _ptr(stats), _ptr(global_max), _stream(stream))
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_shard_rescale")


def merge_stats(stats: torch.Tensor, allreduce: AllReduce,
                rescale_fn: Callable[[torch.Tensor, torch.Tensor], None] = rescale) -> torch.Tensor:
    """The exchange step: MAX all-reduce of m, rescale of d, SUM all-reduce of
    (d, z_y, sum z). After it every rank holds the whole-vocabulary stats."""
    gmax = stats[0].clone()
    allreduce(gmax, "max")
    rescale_fn(stats, gmax)
    rest = stats[1:]
    allreduce(rest, "sum")
    return stats


def loss_from_stats(stats, y, *, vocab_total, H, stream=None, **opts):
    """loss and lse from merged statistics (as flce_forward on the whole vocabulary)."""
    lib = _lib.load()
    N = stats.shape[1]
    p = params(N, H, vocab_total, **opts)
    red = opts.get("reduction", "mean")
    loss = torch.empty(N if red == "none" else 1, dtype=torch.float32, device=stats.device)
    lse = torch.empty(N, dtype=torch.float32, device=stats.device)
    ws = torch.empty(max(lib.flce_workspace_size(p, 0), 1), dtype=torch.uint8, device=stats.device)
    st = lib.flce_loss_from_stats(p, _ptr(stats), _ptr(y), _ptr(loss), _ptr(lse), _ptr(ws),
                                  ws.numel(), _ptr(device_error_word(stats.device)),
                                  _stream(stream))
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_loss_from_stats")
    return (loss if red == "none" else loss.view(())), lse


def backward_shard(dloss, lse, x, W, b, y, *, vocab_start, vocab_total, stream=None,
                   dW_dtype=torch.float32, db_dtype=torch.float32, bwd_vocab_block=0,
                   kept=None, **opts):
    """This shard's dW rows, db, and its fp32 partial dx [N, H]; with ``kept``
    (filled by forward_shard(kept=) with the same bwd_vocab_block), the kept
    block's dlogits come from the kept probabilities."""
    _check_inputs(x, W, b, y)
    lib = _lib.load()
    N, H = x.shape
    V = W.shape[0]
    p = params(N, H, V, has_bias=b is not None, vocab_start=vocab_start, vocab_total=vocab_total,
               dW_fp32=dW_dtype == torch.float32, db_fp32=db_dtype == torch.float32,
               bwd_vocab_block=bwd_vocab_block, input_fp16=x.dtype == torch.float16, **opts)
    dev = x.device
    dloss = dloss.reshape(-1).float().contiguous()
    dx = torch.empty(N, H, dtype=torch.float32, device=dev)
    dW = torch.empty(V, H, dtype=dW_dtype, device=dev)
    db = torch.empty(V, dtype=db_dtype, device=dev) if b is not None else None
    ws = torch.empty(max(lib.flce_workspace_size(p, 2 if kept is not None else 1), 1),
                     dtype=torch.uint8, device=dev)
    if kept is not None:
        _check_kept(kept, lib, p)
        st = lib.flce_backward_shard_keep(p, _ptr(dloss), _ptr(lse), _ptr(kept), kept.numel(),
                                          _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(dx), _ptr(dW),
                                          _ptr(db), _ptr(ws), ws.numel(),
                                          _ptr(device_error_word(dev)), _stream(stream))
    else:
        st = lib.flce_backward_shard(p, _ptr(dloss), _ptr(lse), _ptr(x), _ptr(W), _ptr(b),
                                     _ptr(y), _ptr(dx), _ptr(dW), _ptr(db), _ptr(ws), ws.numel(),
                                     _ptr(device_error_word(dev)), _stream(stream))
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_backward_shard")
    return dx, dW, db


def cast16(src: torch.Tensor, dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """fp32 -> bf16 / fp16 (round to nearest even) in the library's kernel."""
    dst = torch.empty(src.shape, dtype=dtype, device=src.device)
    st = _lib.load().flce_cast_f32(_ptr(src), _ptr(dst), src.numel(),
                                   1 if dtype == torch.float16 else 0, _stream(stream))
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_cast_f32")
    return dst


def vocab_parallel_forward(x, W_local, b_local, y, *, vocab_start: int, vocab_total: int,
                           group=None, allreduce: Optional[AllReduce] = None, kept=None,
                           bwd_vocab_block: int = 0, **opts):
    """Whole-vocabulary loss and lse on every rank from its vocabulary shard
    (``kept``: this shard's kept block, for vocab_parallel_backward)."""
    ar = allreduce or _dist_allreduce(group)
    stats = forward_shard(x, W_local, b_local, y, vocab_start=vocab_start,
                          vocab_total=vocab_total, kept=kept, bwd_vocab_block=bwd_vocab_block,
                          **opts)
    merge_stats(stats, ar)
    return loss_from_stats(stats, y, vocab_total=vocab_total, H=x.shape[1], **opts)


def vocab_parallel_backward(dloss, lse, x, W_local, b_local, y, *, vocab_start: int,
                            vocab_total: int, group=None, allreduce: Optional[AllReduce] = None,
                            **opts):
    """bf16 dx (summed over shards in fp32), this shard's dW rows and db
    (``kept`` and ``bwd_vocab_block`` as given to vocab_parallel_forward)."""
    ar = allreduce or _dist_allreduce(group)
    dx32, dW, db = backward_shard(dloss, lse, x, W_local, b_local, y, vocab_start=vocab_start,
                                  vocab_total=vocab_total, **opts)
    ar(dx32, "sum")
    return cast16(dx32, x.dtype), dW, db
