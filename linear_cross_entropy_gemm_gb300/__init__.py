"""GB300 (sm_103a) fused linear cross-entropy.

Python binding of the C ABI in ``include/flce.h``: the functions here only
check and marshal arguments (device pointers, sizes, the current CUDA
stream) and allocate outputs and workspace through PyTorch. Every step of the
computation runs in the library's CUDA kernels; if the library is missing,
calls raise instead of falling back to anything else.

    loss, lse = flce_forward(x, W, b, y, reduction="mean")
    dx, dW, db = flce_backward(dloss, lse, x, W, b, y, reduction="mean")

The loss follows the fla ``FusedLinearCrossEntropyLoss`` options
(ignore_index, label_smoothing, logit_scale, reduction) plus the z-loss
``lse_square_scale`` of Liger-Kernel PR #239 and reduction "none" of
DeepSpeed PR #8792.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import GEMM_FORMS, FlceError, params

__all__ = [
    "flce_forward", "flce_backward", "flce_workspace_size", "flce_read_device_error",
    "FusedLinearCrossEntropyFunction", "FusedLinearCrossEntropyLoss",
    "fused_linear_cross_entropy", "FlceError", "params", "KernelTrace", "flce_saved_size",
    "GEMM_FORMS", "resolved_gemm_form", "flce_kept_size", "flce_keep_vocab_within",
]

_err_words = {}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def device_error_word(device) -> torch.Tensor:
    """The int32 device word this binding passes as ``dev_err`` on ``device``."""
    d = torch.device(device)
    key = d.index if d.index is not None else torch.cuda.current_device()
    w = _err_words.get(key)
    if w is None:
        w = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda", key))
        _err_words[key] = w
    return w


_OPERAND_DTYPES = (torch.bfloat16, torch.float16)


def _check_inputs(x, W, b, y):
    if not (x.is_cuda and W.is_cuda and y.is_cuda):
        raise ValueError("flce: x, W and y must be CUDA tensors")
    if x.dtype not in _OPERAND_DTYPES or W.dtype != x.dtype:
        raise TypeError("flce: x and W must both be bf16 or both fp16")
    if b is not None and (b.dtype != x.dtype or not b.is_cuda):
        raise TypeError("flce: b must be a CUDA tensor of x's dtype")
    if y.dtype != torch.int64:
        raise TypeError("flce: y must be int64")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1] or y.shape != (x.shape[0],):
        raise ValueError(f"flce: bad shapes x{tuple(x.shape)} W{tuple(W.shape)} y{tuple(y.shape)}")
    if b is not None and b.shape != (W.shape[0],):
        raise ValueError("flce: b must have shape [V]")
    for t in (x, W, y) + ((b,) if b is not None else ()):
        if not t.is_contiguous():
            raise ValueError("flce: tensors must be contiguous")


class KernelTrace:
    """Caller-owned CUDA events for the traced entry points: after a traced
    call, ``launches()`` gives (kernel name, milliseconds) per launch, timed
    on the launching stream (flce_trace_t in include/flce.h)."""

    def __init__(self, capacity: int = 256):
        import ctypes
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.events:  # materialise the underlying cudaEvent_t
            e.record()
        self._handles = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.events])
        self._kinds = (ctypes.c_int32 * capacity)()
        self.struct = _lib.FlceTrace(ctypes.cast(self._handles, ctypes.POINTER(ctypes.c_void_p)),
                                     capacity, 0,
                                     ctypes.cast(self._kinds, ctypes.POINTER(ctypes.c_int32)))

    def launches(self):
        """Call after the stream has been synchronised."""
        n = self.struct.count
        return [(_lib.KERNEL_NAMES[self._kinds[i]], self.events[i].elapsed_time(self.events[i + 1]))
                for i in range(n - 1)]


def flce_workspace_size(N, H, V, which: str, **opts) -> int:
    """Workspace bytes of a call: which = "forward", "backward",
    "backward_keep" (the backward of a kept-block forward, which stages dL in
    the kept buffer and so needs no dL block of its own) or "backward_store"
    (the stored-probability backward)."""
    p = params(N, H, V, **opts)
    return int(_lib.load().flce_workspace_size(p, _lib.WORKSPACE_KIND[which]))


GEMMS = ("fwd_lse", "bwd_dlogits", "bwd_dw", "bwd_dx")


def resolved_gemm_form(N, H, V, gemm_form="default", gemm="fwd_lse", **opts) -> str:
    """The GEMM form ("single", "pair" or "wide") that calls with these
    parameters run for one GEMM (one of ``GEMMS``): ``gemm_form`` itself unless
    it is "default" (dx runs "wide" as "pair"), else the library's per-GEMM
    default (FLCE_GEMM_FORM in the environment overrides it)."""
    f = int(_lib.load().flce_resolved_gemm_form(params(N, H, V, gemm_form=gemm_form, **opts),
                                               GEMMS.index(gemm)))
    if f < 0:
        raise ValueError("flce: invalid parameters")
    return {v: k for k, v in GEMM_FORMS.items()}[f]


def flce_saved_size(N, H, V, **opts) -> int:
    """Bytes of the state flce_forward(..., saved=) keeps for the stored-
    probability backward: every logit's fp16 probability relative to its
    32-column chunk's running maximum, plus those maxima (~2.1 N V bytes)."""
    return int(_lib.load().flce_saved_size(params(N, H, V, **opts)))


def flce_kept_size(N, H, V, **opts) -> int:
    """Bytes of the state flce_forward(..., kept=) leaves for the backward: the
    kept block's fp16 probabilities [N, K] (K = ``keep_vocab``, by default one
    backward vocabulary block BVc) and the running maxima of its 32-column
    chunks. It doubles as the backward's dL staging block, so with one block a
    kept-block forward + backward takes the memory of the plain pair plus the
    chunk maxima."""
    return int(_lib.load().flce_kept_size(params(N, H, V, **opts)))


def flce_keep_vocab_within(N, H, V, extra_bytes: Optional[int] = None, **opts) -> int:
    """The widest kept block (``keep_vocab``) whose kept-mode memory (kept
    state + backward workspace) is at most the recompute backward's workspace
    plus ``extra_bytes``; at least one backward block. The default extra is
    4 V H bytes: the fp32 [V, H] dW accumulator that the method's memory budget
    allows for and this library never allocates."""
    extra = 4 * int(V) * int(H) if extra_bytes is None else int(extra_bytes)
    if extra < 0:
        raise ValueError("flce: extra_bytes must be >= 0")
    k = int(_lib.load().flce_keep_vocab_within(params(N, H, V, **opts), extra))
    if k <= 0:
        raise ValueError("flce: invalid parameters")
    return k


def flce_forward(x: torch.Tensor, W: torch.Tensor, b: Optional[torch.Tensor], y: torch.Tensor, *,
                 ignore_index: int = -100, label_smoothing: float = 0.0,
                 lse_square_scale: float = 0.0, logit_scale: float = 1.0,
                 reduction: str = "mean", workspace: Optional[torch.Tensor] = None,
                 out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                 stream=None, trace: Optional[KernelTrace] = None,
                 saved: Optional[torch.Tensor] = None,
                 gemm_form="default", kept: Optional[torch.Tensor] = None,
                 bwd_vocab_block: int = 0, keep_vocab: int = 0
                 ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Loss and per-token lse. loss is a 0-dim fp32 tensor (sum/mean) or [N]
    fp32 (none); lse is [N] fp32. Runs on the current stream, no sync.
    With ``saved`` (a uint8 CUDA tensor of flce_saved_size bytes) the forward
    also keeps the state the stored-probability backward needs.
    ``gemm_form``: "default", "single" (128 x 256 CTA tiles), "pair"
    (256 x 256 tiles on CTA pairs) or "wide" (256 x 512 tiles on CTA pairs);
    see ``tuning.autotune``. ``workspace``: a uint8 CUDA tensor of at least
    flce_workspace_size(..., "forward") bytes; when it is not given, or is
    smaller, a new one is allocated for the call.
    With ``kept`` (a uint8 CUDA tensor of flce_kept_size bytes; give the
    backward's ``bwd_vocab_block`` and ``keep_vocab`` here too) the forward
    also leaves the kept block's probabilities for flce_backward(..., kept=),
    which then skips that block's recompute. The kept block is the vocabulary
    columns [0, keep_vocab) (a multiple of 256; 0 = one backward block; see
    flce_keep_vocab_within)."""
    _check_inputs(x, W, b, y)
    lib = _lib.load()
    N, H = x.shape
    V = W.shape[0]
    if saved is not None and kept is not None:
        raise ValueError("flce: give saved= or kept=, not both")
    p = params(N, H, V, ignore_index=ignore_index, label_smoothing=label_smoothing,
               lse_square_scale=lse_square_scale, logit_scale=logit_scale,
               reduction=reduction, has_bias=b is not None,
               input_fp16=x.dtype == torch.float16, gemm_form=gemm_form,
               bwd_vocab_block=bwd_vocab_block, keep_vocab=keep_vocab)
    dev = x.device
    if out is not None:
        loss, lse = out
    else:
        loss = torch.empty(N if reduction == "none" else 1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    need = lib.flce_workspace_size(p, 0)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if saved is not None or kept is not None:
        state = saved if saved is not None else kept
        _check_state(state, lib, p, kept is not None)
        fn = lib.flce_forward_store if saved is not None else lib.flce_forward_keep
        st = fn(p, _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(loss), _ptr(lse), _ptr(state),
                state.numel(), _ptr(workspace), workspace.numel(), _ptr(device_error_word(dev)),
                _stream(stream), None if trace is None else trace.struct)
    else:
        args = (p, _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(loss), _ptr(lse), _ptr(workspace),
                workspace.numel(), _ptr(device_error_word(dev)), _stream(stream))
        st = lib.flce_forward(*args) if trace is None else lib.flce_forward_traced(*args, trace.struct)
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_forward")
    return (loss if reduction == "none" else loss.view(())), lse


def flce_backward(dloss: torch.Tensor, lse: torch.Tensor, x: torch.Tensor, W: torch.Tensor,
                  b: Optional[torch.Tensor], y: torch.Tensor, *, ignore_index: int = -100,
                  label_smoothing: float = 0.0, lse_square_scale: float = 0.0,
                  logit_scale: float = 1.0, reduction: str = "mean",
                  dW_dtype: torch.dtype = torch.float32, db_dtype: torch.dtype = torch.float32,
                  bwd_vocab_block: int = 0, workspace: Optional[torch.Tensor] = None,
                  out: Optional[Tuple] = None, stream=None, trace: Optional[KernelTrace] = None,
                  saved: Optional[torch.Tensor] = None, gemm_form="default",
                  kept: Optional[torch.Tensor] = None, keep_vocab: int = 0):
    """dx [N, H] bf16, dW [V, H] (dW_dtype fp32 or bf16), db [V] or None.
    With ``saved`` (filled by flce_forward(..., saved=)) the logits are not
    recomputed: dlogits come from the stored tile probabilities. With
    ``kept`` (filled by flce_forward(..., kept=) with the same options,
    ``bwd_vocab_block`` and ``keep_vocab``) the kept block's dlogits come
    from the kept probabilities and the buffer stages every block's dL; the
    call consumes it.
    ``bwd_vocab_block`` (0 = library default) and ``gemm_form`` select the
    vocabulary block and GEMM form; see ``tuning.autotune``. ``workspace``: as
    in flce_forward, with flce_workspace_size(..., "backward") bytes."""
    _check_inputs(x, W, b, y)
    lib = _lib.load()
    N, H = x.shape
    V = W.shape[0]
    dev = x.device
    dloss = dloss.reshape(-1)
    if dloss.dtype != torch.float32 or not dloss.is_cuda or not dloss.is_contiguous():
        raise TypeError("flce: dloss must be a contiguous fp32 CUDA tensor")
    if dloss.numel() != (N if reduction == "none" else 1):
        raise ValueError("flce: dloss must have N elements (none) or 1 (sum/mean)")
    if lse.dtype != torch.float32 or lse.shape != (N,):
        raise ValueError("flce: lse must be the forward's [N] fp32 output")
    if dW_dtype not in (torch.float32, x.dtype) or db_dtype not in (torch.float32, x.dtype):
        raise TypeError("flce: dW_dtype and db_dtype must be fp32 or x's dtype")
    p = params(N, H, V, ignore_index=ignore_index, label_smoothing=label_smoothing,
               lse_square_scale=lse_square_scale, logit_scale=logit_scale,
               reduction=reduction, has_bias=b is not None,
               dW_fp32=dW_dtype == torch.float32, db_fp32=db_dtype == torch.float32,
               bwd_vocab_block=bwd_vocab_block, input_fp16=x.dtype == torch.float16,
               gemm_form=gemm_form, keep_vocab=keep_vocab)
    if out is not None:
        dx, dW, db = out
    else:
        dx = torch.empty(N, H, dtype=x.dtype, device=dev)
        dW = torch.empty(V, H, dtype=dW_dtype, device=dev)
        db = torch.empty(V, dtype=db_dtype, device=dev) if b is not None else None
    if saved is not None and kept is not None:
        raise ValueError("flce: give saved= or kept=, not both")
    need = lib.flce_workspace_size(p, 2 if kept is not None else 3 if saved is not None else 1)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if saved is not None or kept is not None:
        state = saved if saved is not None else kept
        _check_state(state, lib, p, kept is not None)
        fn = lib.flce_backward_store if saved is not None else lib.flce_backward_keep
        st = fn(p, _ptr(dloss), _ptr(lse), _ptr(state), state.numel(), _ptr(x), _ptr(W), _ptr(b),
                _ptr(y), _ptr(dx), _ptr(dW), _ptr(db), _ptr(workspace), workspace.numel(),
                _ptr(device_error_word(dev)), _stream(stream),
                None if trace is None else trace.struct)
    else:
        args = (p, _ptr(dloss), _ptr(lse), _ptr(x), _ptr(W), _ptr(b), _ptr(y), _ptr(dx), _ptr(dW),
                _ptr(db), _ptr(workspace), workspace.numel(), _ptr(device_error_word(dev)),
                _stream(stream))
        st = lib.flce_backward(*args) if trace is None else lib.flce_backward_traced(*args, trace.struct)
    if st != _lib.FLCE_OK:
        raise FlceError(st, "flce_backward")
    return dx, dW, db


def _check_state(state, lib, p, kept: bool):
    what = "kept" if kept else "saved"
    if state.dtype != torch.uint8 or not state.is_cuda or not state.is_contiguous():
        raise TypeError(f"flce: {what} must be a contiguous uint8 CUDA tensor")
    need = lib.flce_kept_size(p) if kept else lib.flce_saved_size(p)
    if state.numel() < need:
        raise ValueError(f"flce: {what} is smaller than flce_{what}_size()")


def flce_read_device_error(device=None, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits
    (FLCE_DEVERR_TARGET = 1, FLCE_DEVERR_TIMEOUT = 2) raised by earlier calls."""
    import ctypes
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    h = ctypes.c_int32(0)
    st = _lib.load().flce_read_device_error(_ptr(device_error_word(dev)), _stream(stream),
                                           ctypes.byref(h))
    if st not in (_lib.FLCE_OK, 4, 6):
        raise FlceError(st, "flce_read_device_error")
    return int(h.value)


def _keep_width(keep_vocab, N, H, V, bias, x, bwd_vocab_block) -> int:
    """keep_vocab as the library takes it: 0 (one backward block), a column
    count rounded up to a multiple of 256, or "budget"
    (flce_keep_vocab_within with the method's fp32 dW accumulator allowance)."""
    if keep_vocab == "budget":
        return flce_keep_vocab_within(N, H, V, has_bias=bias is not None,
                                      input_fp16=x.dtype == torch.float16,
                                      bwd_vocab_block=bwd_vocab_block)
    if isinstance(keep_vocab, str) or int(keep_vocab) < 0:
        raise ValueError(f"keep_vocab: 0, a column count or 'budget', got {keep_vocab!r}")
    return (int(keep_vocab) + 255) // 256 * 256


class FusedLinearCrossEntropyFunction(torch.autograd.Function):
    """Autograd wrapper. By default the forward keeps lse and the first
    backward vocabulary block's probabilities (the buffer the backward stages
    dL in, so no extra memory but the chunk maxima) and the backward
    recomputes the other blocks' logits; keep_vocab widens the kept block
    (a column count, or "budget": the widest within the method's memory
    budget, see flce_keep_vocab_within); keep_block=False recomputes every
    block; recompute=False keeps every logit's probability (~2 N V bytes) and
    recomputes none."""

    @staticmethod
    def forward(ctx, x, target, weight, bias=None, ignore_index=-100, label_smoothing=0.0,
                lse_square_scale=0.0, logit_scale=1.0, reduction="mean", recompute=True,
                config=None, keep_block=True, keep_vocab=0):
        saved = kept = None
        N, H, V = x.shape[0], x.shape[1], weight.shape[0]
        bwd_kw = {} if config is None else config.backward_kwargs()
        bvb = bwd_kw.get("bwd_vocab_block", 0)
        kv = 0
        if not recompute:
            n = flce_saved_size(N, H, V, label_smoothing=label_smoothing,
                                input_fp16=x.dtype == torch.float16)
            saved = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
        elif keep_block and N > 0:
            kv = _keep_width(keep_vocab, N, H, V, bias, x, bvb)
            n = flce_kept_size(N, H, V, input_fp16=x.dtype == torch.float16,
                               bwd_vocab_block=bvb, keep_vocab=kv)
            kept = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
        ctx.config = config
        ctx.keep_vocab = kv
        loss, lse = flce_forward(x, weight, bias, target, ignore_index=ignore_index,
                                 label_smoothing=label_smoothing,
                                 lse_square_scale=lse_square_scale, logit_scale=logit_scale,
                                 reduction=reduction, saved=saved, kept=kept,
                                 bwd_vocab_block=bvb, keep_vocab=kv,
                                 **({} if config is None else config.forward_kwargs()))
        ctx.saved_state = saved
        ctx.kept_state = kept
        ctx.save_for_backward(x, target, weight, bias, lse)
        ctx.opts = dict(ignore_index=ignore_index, label_smoothing=label_smoothing,
                        lse_square_scale=lse_square_scale, logit_scale=logit_scale,
                        reduction=reduction)
        return loss

    @staticmethod
    def backward(ctx, dloss):
        x, target, weight, bias, lse = ctx.saved_tensors
        # dW and db are written in the parameters' own type by the library's
        # epilogues (fp32 sums rounded once to nearest even, as a cast of the
        # fp32 result would be), so no [V, H] fp32 temporary is allocated.
        dx, dW, db = flce_backward(dloss.float().contiguous(), lse, x, weight, bias, target,
                                   dW_dtype=weight.dtype,
                                   db_dtype=torch.float32 if bias is None else bias.dtype,
                                   saved=ctx.saved_state, kept=ctx.kept_state,
                                   keep_vocab=ctx.keep_vocab, **ctx.opts,
                                   **({} if ctx.config is None else ctx.config.backward_kwargs()))
        ctx.saved_state = ctx.kept_state = None
        return dx, None, dW, db, None, None, None, None, None, None, None, None, None


def fused_linear_cross_entropy(x, target, weight, bias=None, ignore_index=-100,
                               label_smoothing=0.0, lse_square_scale=0.0, logit_scale=1.0,
                               reduction="mean", recompute=True, config=None,
                               keep_block=True, keep_vocab=0):
    """Functional form; x [N, H] bf16, target [N] int64, weight [V, H] bf16.
    By default the forward keeps the first backward vocabulary block's
    probabilities in the buffer the backward stages dL in (no extra memory),
    so the backward recomputes the logits of the other blocks only;
    keep_vocab widens the kept block: a column count, or "budget" for the
    widest within the method's memory budget (flce_keep_vocab_within).
    keep_block=False recomputes all. recompute=False keeps fp16 tile
    probabilities of every logit (~2 N V bytes) so the backward skips the
    logits GEMM. ``config``: a ``tuning.FlceConfig`` (GEMM forms, backward
    vocabulary block), or None for the library defaults."""
    return FusedLinearCrossEntropyFunction.apply(x, target, weight, bias, ignore_index,
                                                 label_smoothing, lse_square_scale,
                                                 logit_scale, reduction, recompute, config,
                                                 keep_block, keep_vocab)


class FusedLinearCrossEntropyLoss(torch.nn.Module):
    """Module form: flattens x [..., H] and target [...] to [N, H] and [N]."""

    def __init__(self, ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0,
                 logit_scale=1.0, reduction="mean", recompute=True, autotune=False,
                 keep_block=True, keep_vocab=0):
        """autotune=True: the first call for each (shape, dtype, options) key
        times the GEMM forms and backward vocabulary blocks on the caller's
        tensors (tuning.autotune) and later calls reuse the fastest."""
        super().__init__()
        if reduction not in ("none", "sum", "mean"):
            raise ValueError(f"reduction: {reduction} is not supported")
        self.ignore_index = ignore_index
        self.label_smoothing = label_smoothing
        self.lse_square_scale = lse_square_scale
        self.logit_scale = logit_scale
        self.reduction = reduction
        self.recompute = recompute
        self.autotune = autotune
        self.keep_block = keep_block
        self.keep_vocab = keep_vocab

    def forward(self, x, target, weight, bias=None):
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        y2 = target.reshape(-1).contiguous()
        config = None
        if self.autotune:
            from . import tuning
            config = tuning.autotune(
                x2.detach(), weight.detach(), None if bias is None else bias.detach(), y2,
                ignore_index=self.ignore_index, label_smoothing=self.label_smoothing,
                lse_square_scale=self.lse_square_scale, logit_scale=self.logit_scale,
                reduction=self.reduction,
                mode="kept" if self.recompute and self.keep_block else "recompute").config
        return fused_linear_cross_entropy(
            x2, y2, weight, bias, self.ignore_index, self.label_smoothing,
            self.lse_square_scale, self.logit_scale, self.reduction, self.recompute, config,
            self.keep_block, self.keep_vocab)
