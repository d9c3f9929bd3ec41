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


def test_params_struct_layout_matches_header(tmp_path):
    # The ctypes mirror against the C compiler's own layout of the header's
    # struct: every field's offset and the total size.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in _lib.FlceParams._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"flce.h\"\n"
                   "int main(void) {\n"
                   + "".join(f'  printf("%zu\\n", offsetof(flce_params_t, {f}));\n'
                             for f in fields)
                   + '  printf("%zu\\n", sizeof(flce_params_t));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    want = [getattr(_lib.FlceParams, f).offset for f in fields] + [ctypes.sizeof(_lib.FlceParams)]
    assert got == want, dict(zip(fields + ["sizeof"], zip(got, want)))
    assert ctypes.sizeof(_lib.FlceParams) == 104


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
    (dict(keep_vocab=100), 1), (dict(keep_vocab=-256), 1),
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


def test_wider_kept_block_sizes(lib):
    # keep_vocab = K keeps [N, K] fp16 plus maxima per 32 columns; below BVc
    # it keeps BVc, at or above the vocabulary it is the stored state.
    N, H, V = 8192, 4096, 128256
    bv = 65536
    vr = (V + 255) // 256 * 256

    def kept(k, **kw):
        return lib.flce_kept_size(_lib.params(N, H, V, keep_vocab=k, **kw))

    assert kept(0) == kept(256) == kept(bv)
    k = 98304
    assert N * k * 2 + N * (k // 32) * 4 <= kept(k) <= N * k * 2 + N * (k // 32) * 4 + 1024
    assert kept(vr) == kept(1 << 20) == lib.flce_saved_size(_lib.params(N, H, V))
    # the kept backward's workspace: a dx accumulator only while blocks remain
    # to recompute; db column partials as wide as the kept block
    ws = lambda k, **kw: lib.flce_workspace_size(_lib.params(N, H, V, keep_vocab=k, **kw), 2)
    assert ws(vr) == lib.flce_workspace_size(_lib.params(N, H, V), 3)
    assert ws(k) - ws(vr) >= N * H * 4
    rows = 4 * (N // 128)
    assert ws(k, has_bias=True) - ws(k) >= rows * k * 4
    assert ws(k, has_bias=True) - ws(k) - rows * k * 4 < 2048


def _kept_mode_bytes(lib, p):
    return lib.flce_kept_size(p) + lib.flce_workspace_size(p, 2)


@pytest.mark.parametrize("N,H,V,kw", [
    (8192, 4096, 128256, {}), (32768, 2048, 128000, dict(has_bias=True)),
    (16384, 4096, 262144, {}), (4096, 2048, 32000, dict(has_bias=True)),
    (512, 256, 4096, dict(bwd_vocab_block=1024)), (300, 64, 1000, dict(bwd_vocab_block=256)),
])
def test_keep_vocab_within_budget(lib, N, H, V, kw):
    # The rule: the widest of V, V - BVc, V - 2 BVc, ... (rounded up to 256,
    # at least BVc) whose kept-mode memory stays within the recompute
    # workspace plus the extra bytes; one block (BVc) when none fits.
    from linear_cross_entropy_gemm_gb300 import tuning
    p = _lib.params(N, H, V, **kw)
    base = lib.flce_workspace_size(p, 1)
    vr = (V + 255) // 256 * 256
    bvc = min(kw.get("bwd_vocab_block") or tuning.library_default_block(N, V), vr)
    cands = [min(vr, (V - j * bvc + 255) // 256 * 256) for j in range(V // bvc + 1)
             if V - j * bvc > bvc] or [vr]
    widths = []
    for extra in sorted((0, 1 << 20, 1 << 28, 4 * V * H, 1 << 34, 1 << 40)):
        k = lib.flce_keep_vocab_within(p, extra)
        fit = [c for c in cands
               if _kept_mode_bytes(lib, _lib.params(N, H, V, keep_vocab=c, **kw)) <= base + extra]
        assert k == (max(fit) if fit else bvc), (extra, k, fit)
        widths.append(k)
    assert widths == sorted(widths)  # more memory never keeps less
    assert widths[-1] == vr
    assert lib.flce_keep_vocab_within(_lib.params(0, H, V), 1 << 40) == 0


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


def test_budget_widths_at_the_five_workloads(lib):
    # The widths the budget rule (extra = 4 V H bytes) gives at the
    # workloads, as measured and documented: the whole vocabulary at tiny,
    # medium and the Llama-3 head, one 16384-column block at large_logit, half
    # of vocab256k's vocabulary.
    from linear_cross_entropy_gemm_gb300 import inputs as I
    want = {"tiny": 4096, "medium": 32000, "llama3_head": 128256, "large_logit": 16384,
            "vocab256k": 131072}
    for name, k in want.items():
        wl = I.WORKLOADS[name]
        p = _lib.params(wl.N, wl.H, wl.V, has_bias=wl.has_bias)
        got = lib.flce_keep_vocab_within(p, 4 * wl.V * wl.H)
        vr = (wl.V + 255) // 256 * 256
        assert min(got, vr) == min((k + 255) // 256 * 256, vr), (name, got)
