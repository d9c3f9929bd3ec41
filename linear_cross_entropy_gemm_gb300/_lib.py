"""ctypes view of the C ABI in include/flce.h (``libflce_gb300.so``).

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libflce_gb300.so")

REDUCTION = {"none": 0, "sum": 1, "mean": 2}

FLCE_OK = 0
STATUS_NAMES = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_ALIGNMENT",
    3: "FLCE_ERR_WORKSPACE_TOO_SMALL", 4: "FLCE_ERR_TARGET_OUT_OF_RANGE", 5: "FLCE_ERR_CUDA",
    6: "FLCE_ERR_TIMEOUT", 7: "FLCE_ERR_UNSUPPORTED",
}
# flce_gemm_form_t: "default" leaves the choice to the library.
GEMM_FORMS = {"default": 0, "single": 1, "pair": 2, "wide": 3}
DEVERR_TARGET = 1
DEVERR_TIMEOUT = 2


class FlceParams(ctypes.Structure):
    """Mirror of flce_params_t."""
    _fields_ = [
        ("N", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("V", ctypes.c_int64),
        ("ignore_index", ctypes.c_int64),
        ("label_smoothing", ctypes.c_float),
        ("lse_square_scale", ctypes.c_float),
        ("logit_scale", ctypes.c_float),
        ("reduction", ctypes.c_int32),
        ("has_bias", ctypes.c_int32),
        ("dW_fp32", ctypes.c_int32),
        ("db_fp32", ctypes.c_int32),
        ("bwd_vocab_block", ctypes.c_int64),
        ("vocab_start", ctypes.c_int64),
        ("vocab_total", ctypes.c_int64),
        ("input_fp16", ctypes.c_int32),
        ("gemm_form", ctypes.c_int32),
        ("keep_vocab", ctypes.c_int64),
    ]


class FlceTrace(ctypes.Structure):
    """Mirror of flce_trace_t."""
    _fields_ = [
        ("events", ctypes.POINTER(ctypes.c_void_p)),
        ("capacity", ctypes.c_int32),
        ("count", ctypes.c_int32),
        ("kinds", ctypes.POINTER(ctypes.c_int32)),
    ]


KERNEL_NAMES = ("fwd_lse", "fwd_merge", "fwd_finalize", "bwd_prep", "bwd_dlogits", "bwd_db",
                "bwd_dw", "bwd_dx", "bwd_convert")
# flce_workspace_size's `which`.
WORKSPACE_KIND = {"forward": 0, "backward": 1, "backward_keep": 2, "backward_store": 3}


class FlceError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({load().flce_status_string(status).decode()})")


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python linear_cross_entropy_gemm_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(FlceParams)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.flce_workspace_size.argtypes = [P, ctypes.c_int]
    lib.flce_workspace_size.restype = sz
    lib.flce_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.flce_forward.restype = ctypes.c_int
    lib.flce_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.flce_backward.restype = ctypes.c_int
    T = ctypes.POINTER(FlceTrace)
    lib.flce_forward_traced.argtypes = lib.flce_forward.argtypes + [T]
    lib.flce_forward_traced.restype = ctypes.c_int
    lib.flce_backward_traced.argtypes = lib.flce_backward.argtypes + [T]
    lib.flce_backward_traced.restype = ctypes.c_int
    lib.flce_saved_size.argtypes = [P]
    lib.flce_saved_size.restype = sz
    lib.flce_forward_store.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp, vp, T]
    lib.flce_forward_store.restype = ctypes.c_int
    lib.flce_backward_store.argtypes = [P, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                        vp, vp, T]
    lib.flce_backward_store.restype = ctypes.c_int
    lib.flce_kept_size.argtypes = [P]
    lib.flce_kept_size.restype = sz
    lib.flce_keep_vocab_within.argtypes = [P, sz]
    lib.flce_keep_vocab_within.restype = ctypes.c_int64
    lib.flce_forward_keep.argtypes = lib.flce_forward_store.argtypes
    lib.flce_forward_keep.restype = ctypes.c_int
    lib.flce_backward_keep.argtypes = lib.flce_backward_store.argtypes
    lib.flce_backward_keep.restype = ctypes.c_int
    lib.flce_forward_shard.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.flce_forward_shard.restype = ctypes.c_int
    lib.flce_forward_shard_keep.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp, vp]
    lib.flce_forward_shard_keep.restype = ctypes.c_int
    lib.flce_backward_shard_keep.argtypes = [P, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp,
                                             sz, vp, vp]
    lib.flce_backward_shard_keep.restype = ctypes.c_int
    lib.flce_shard_rescale.argtypes = [P, vp, vp, vp]
    lib.flce_shard_rescale.restype = ctypes.c_int
    lib.flce_loss_from_stats.argtypes = [P, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.flce_loss_from_stats.restype = ctypes.c_int
    lib.flce_backward_shard.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.flce_backward_shard.restype = ctypes.c_int
    lib.flce_cast_f32.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int32, vp]
    lib.flce_cast_f32.restype = ctypes.c_int
    lib.flce_selftest_wait_timeout.argtypes = [vp, ctypes.c_int64, vp]
    lib.flce_selftest_wait_timeout.restype = ctypes.c_int
    lib.flce_read_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.flce_read_device_error.restype = ctypes.c_int
    lib.flce_resolved_gemm_form.argtypes = [P, ctypes.c_int32]
    lib.flce_resolved_gemm_form.restype = ctypes.c_int32
    lib.flce_status_string.argtypes = [ctypes.c_int]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_version.argtypes = []
    lib.flce_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def params(N, H, V, *, ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0,
           logit_scale=1.0, reduction="mean", has_bias=False, dW_fp32=True, db_fp32=True,
           bwd_vocab_block=0, vocab_start=0, vocab_total=0, input_fp16=False,
           gemm_form="default", keep_vocab=0) -> FlceParams:
    if reduction not in REDUCTION:
        raise ValueError(f"reduction must be one of {sorted(REDUCTION)}, got {reduction!r}")
    form = GEMM_FORMS.get(gemm_form, gemm_form) if isinstance(gemm_form, str) else int(gemm_form)
    if isinstance(form, str):
        raise ValueError(f"gemm_form must be one of {sorted(GEMM_FORMS)}, got {gemm_form!r}")
    return FlceParams(int(N), int(H), int(V), int(ignore_index), float(label_smoothing),
                      float(lse_square_scale), float(logit_scale), REDUCTION[reduction],
                      int(bool(has_bias)), int(bool(dW_fp32)), int(bool(db_fp32)),
                      int(bwd_vocab_block), int(vocab_start), int(vocab_total),
                      int(bool(input_fp16)), form, int(keep_vocab))
