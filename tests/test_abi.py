"""The C-ABI library builds, loads and exports every function include/flce.h
declares; host-side argument checks return the documented statuses. No
kernel is launched (these run without a GPU)."""
import ctypes
import os
import re

import pytest

from linear_cross_entropy_gemm_gb300 import _lib
from linear_cross_entropy_gemm_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("flce_forward", "flce_backward", "flce_workspace_size",
              "flce_read_device_error", "flce_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def _enum(prefix):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1): int(m.group(2))
            for m in re.finditer(prefix + r"([A-Z0-9_]+)\s*=\s*(\d+)", src)}


def test_binding_codes_match_the_header_enums():
    # Trace kinds (the binding's names index flce_kernel_t), GEMM forms and
    # reductions: the Python side must use the header's values.
    kinds = _enum("FLCE_KERNEL_")
    assert [k.lower() for k, _ in sorted(kinds.items(), key=lambda kv: kv[1])] == \
        list(_lib.KERNEL_NAMES)
    assert sorted(kinds.values()) == list(range(len(kinds)))
    forms = _enum("FLCE_GEMM_")
    assert {"default": forms["DEFAULT"], "single": forms["SINGLE_CTA"],
            "pair": forms["CTA_PAIR"], "wide": forms["WIDE_PAIR"]} == _lib.GEMM_FORMS
    red = _enum("FLCE_REDUCTION_")
    assert {k.lower(): v for k, v in red.items()} == _lib.REDUCTION


def test_params_struct_layout_matches_header():
    assert ctypes.sizeof(_lib.FlceParams) == 96
    assert _lib.FlceParams.bwd_vocab_block.offset == 64
    assert _lib.FlceParams.vocab_total.offset == 80
    assert _lib.FlceParams.input_fp16.offset == 88


def test_status_strings(lib):
    for s in range(8):
        assert lib.flce_status_string(s)
    assert lib.flce_version().decode().count(".") == 2


def test_workspace_sizes(lib):
    p = _lib.params(8192, 4096, 128256)
    fwd = lib.flce_workspace_size(p, 0)
    bwd = lib.flce_workspace_size(p, 1)
    nt = (128256 + 255) // 256
    assert fwd >= 2 * nt * 8192 * 4
    assert bwd >= 8192 * 16384 * 2 + 8192 * 4096 * 4
    ps = _lib.params(8192, 4096, 128256, label_smoothing=0.1)
    assert lib.flce_workspace_size(ps, 0) >= fwd + nt * 8192 * 4
    assert lib.flce_workspace_size(_lib.params(0, 64, 10), 0) == 0
    assert lib.flce_workspace_size(_lib.params(4, 12, 10), 0) == 0  # H % 8 != 0


@pytest.mark.parametrize("kw,status", [
    (dict(N=-1), 1), (dict(H=0), 1), (dict(V=0), 1), (dict(H=12), 2),
    (dict(label_smoothing=1.5), 1), (dict(lse_square_scale=-1.0), 1),
    (dict(bwd_vocab_block=100), 1), (dict(gemm_form=4), 1), (dict(gemm_form=-1), 1),
])
def test_invalid_params_rejected_on_host(lib, kw, status):
    base = dict(N=4, H=64, V=10)
    base.update(kw)
    N, H, V = base.pop("N"), base.pop("H"), base.pop("V")
    p = _lib.params(N, H, V, **base)
    fake = ctypes.c_void_p(4096)  # never dereferenced: rejected before any launch
    st = lib.flce_forward(p, fake, fake, None, fake, fake, fake, fake, 1 << 30, None, None)
    assert st == status


def test_null_and_misaligned_pointers_rejected(lib):
    p = _lib.params(4, 64, 10)
    f = ctypes.c_void_p(4096)
    assert lib.flce_forward(p, None, f, None, f, f, f, f, 1 << 30, None, None) == 1
    assert lib.flce_forward(p, ctypes.c_void_p(4098), f, None, f, f, f, f, 1 << 30, None,
                            None) == 2
    assert lib.flce_forward(p, f, f, None, f, f, f, f, 16, None, None) == 3
    pb = _lib.params(4, 64, 10, has_bias=True)
    assert lib.flce_forward(pb, f, f, None, f, f, f, f, 1 << 30, None, None) == 1
    assert lib.flce_backward(p, None, f, f, f, None, f, f, f, None, f, 1 << 30, None,
                             None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, lang, std):
    import shutil
    import subprocess
    cc = shutil.which("gcc") if lang == "c" else shutil.which("g++")
    if cc is None:
        pytest.skip("no host compiler")
    calls = "\n".join(f"  (void)&{n};" for n in declared_functions())
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "flce.h"\nint main(void) {\n  flce_params_t p = {0};\n'
                   '  (void)p;\n' + calls + "\n  return 0;\n}\n")
    r = subprocess.run([cc, std, "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_kept_and_stored_sizes(lib):
    # The kept state is one [N, BVc] fp16 block plus fp32 maxima per 32
    # columns; the kept backward's workspace is the plain backward's without
    # its dL block; the stored state is the kept state of a block spanning V.
    N, H, V = 8192, 4096, 128256
    p = _lib.params(N, H, V)
    bv = 65536  # the library default at N = 8192 (1 GiB of 16-bit dL)
    kept = lib.flce_kept_size(p)
    assert N * bv * 2 + N * (bv // 32) * 4 <= kept <= N * bv * 2 + N * (bv // 32) * 4 + 1024
    assert lib.flce_workspace_size(p, 1) - lib.flce_workspace_size(p, 2) >= N * bv * 2
    vr = (V + 255) // 256 * 256
    saved = lib.flce_saved_size(p)
    assert N * vr * 2 + N * (-(-V // 32)) * 4 <= saved <= N * vr * 2 + N * (-(-V // 32)) * 4 + 1024
    # one block over the vocabulary: no dx accumulator, no dL block
    assert lib.flce_workspace_size(p, 3) < lib.flce_workspace_size(p, 2)
    assert lib.flce_workspace_size(p, 4) == 0
    assert lib.flce_kept_size(_lib.params(0, 64, 10)) == 0
    # a vocabulary shard keeps its own first block; it has no stored mode
    shard = _lib.params(4, 64, 10, vocab_start=10, vocab_total=40)
    assert lib.flce_kept_size(shard) == lib.flce_kept_size(_lib.params(4, 64, 10)) > 0
    assert lib.flce_saved_size(shard) == 0


def test_kept_entry_points_reject_bad_arguments_on_host(lib):
    p = _lib.params(4, 64, 1000, bwd_vocab_block=256)
    f = ctypes.c_void_p(4096)  # never dereferenced: rejected before any launch
    need = lib.flce_kept_size(p)
    ws = 1 << 30
    # no kept buffer
    assert lib.flce_forward_keep(p, f, f, None, f, f, f, None, need, f, ws, None, None,
                                 None) == 1
    # too small, misaligned
    assert lib.flce_forward_keep(p, f, f, None, f, f, f, f, need - 1, f, ws, None, None,
                                 None) == 3
    assert lib.flce_forward_keep(p, f, f, None, f, f, f, ctypes.c_void_p(4104), need, f, ws,
                                 None, None, None) == 2
    assert lib.flce_backward_keep(p, f, f, f, need - 1, f, f, None, f, f, f, None, f, ws,
                                  None, None, None) == 3
    # the kept backward's workspace must hold its (dL-free) carving
    assert lib.flce_backward_keep(p, f, f, f, need, f, f, None, f, f, f, None, f, 16, None,
                                  None, None) == 3
    # stored mode: state too small
    ns = lib.flce_saved_size(p)
    assert lib.flce_forward_store(p, f, f, None, f, f, f, f, ns - 1, f, ws, None, None,
                                  None) == 3
    assert lib.flce_backward_store(p, f, f, f, ns - 1, f, f, None, f, f, f, None, f, ws, None,
                                   None, None) == 3
