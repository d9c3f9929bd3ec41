"""ctypes view of the C++ fp64 reference (oracle/flce_oracle_ref.cpp).

TEST INFRASTRUCTURE. Only the tests use it. ``load()`` compiles the
reference with the host C++ compiler (g++ -O2, no architecture flags) when
the shared library is missing or older than its source, and loads it.
``forward`` / ``backward`` take and return numpy arrays with the same
meaning as oracle.flce_oracle.forward / backward.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "flce_oracle_ref.cpp")
LIB = os.path.join(HERE, "libflce_oracle_ref.so")
REDUCTION = {"none": 0, "sum": 1, "mean": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile the reference into oracle/libflce_oracle_ref.so; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler for the C++ reference")
    tmp = LIB + ".tmp"
    subprocess.run([cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", SRC, "-o", tmp],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        d, i64, vp = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
        lib.flce_ref_forward.argtypes = [i64, i64, i64, vp, vp, vp, vp, i64, d, d, d,
                                         ctypes.c_int, ctypes.c_int, vp, vp]
        lib.flce_ref_forward.restype = ctypes.c_int
        lib.flce_ref_backward.argtypes = [i64, i64, i64, vp, vp, vp, vp, i64, d, d, d,
                                          ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
        lib.flce_ref_backward.restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def forward(x, W, b, y, *, ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0,
            logit_scale=1.0, reduction="mean", threads=None):
    """(loss, lse): loss [N] for none, a 0-d array otherwise; lse [N]."""
    x, W, b, y = _c(x, np.float64), _c(W, np.float64), _c(b, np.float64), _c(y, np.int64)
    N, H = x.shape
    V = W.shape[0]
    loss = np.zeros(N if reduction == "none" else 1)
    lse = np.zeros(N)
    st = load().flce_ref_forward(N, H, V, _ptr(x), _ptr(W), _ptr(b), _ptr(y), int(ignore_index),
                                 float(label_smoothing), float(lse_square_scale),
                                 float(logit_scale), REDUCTION[reduction],
                                 threads or os.cpu_count() or 1, _ptr(loss), _ptr(lse))
    if st != 0:
        raise ValueError("flce_ref_forward: invalid arguments")
    return (loss if reduction == "none" else loss.reshape(())), lse


def backward(dloss, x, W, b, y, *, ignore_index=-100, label_smoothing=0.0,
             lse_square_scale=0.0, logit_scale=1.0, reduction="mean", threads=None):
    """(dx [N, H], dW [V, H], db [V] or None)."""
    x, W, b, y = _c(x, np.float64), _c(W, np.float64), _c(b, np.float64), _c(y, np.int64)
    dloss = np.ascontiguousarray(np.asarray(dloss, dtype=np.float64).reshape(-1))
    N, H = x.shape
    V = W.shape[0]
    dx = np.zeros((N, H))
    dW = np.zeros((V, H))
    db = np.zeros(V) if b is not None else None
    st = load().flce_ref_backward(N, H, V, _ptr(x), _ptr(W), _ptr(b), _ptr(y), int(ignore_index),
                                  float(label_smoothing), float(lse_square_scale),
                                  float(logit_scale), REDUCTION[reduction], _ptr(dloss),
                                  threads or os.cpu_count() or 1, _ptr(dx), _ptr(dW), _ptr(db))
    if st != 0:
        raise ValueError("flce_ref_backward: invalid arguments")
    return dx, dW, db
