"""Host-side logic of the autotuner and the gemm_form parameter (no GPU)."""
import pytest

from linear_cross_entropy_gemm_gb300 import _lib
from linear_cross_entropy_gemm_gb300 import build as B
from linear_cross_entropy_gemm_gb300 import tuning


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


@pytest.mark.parametrize("N,V", [(8192, 128256), (16384, 262144), (512, 4096), (1, 7),
                                 (300, 1000), (32768, 128000), (1 << 20, 50000)])
def test_python_default_block_is_the_librarys(lib, N, V):
    # The workspace holds one [N, BVc] dL block: the library's default block
    # and the mirror's must give the same workspace size.
    p0 = _lib.params(N, 4096, V, bwd_vocab_block=0)
    bv = tuning.library_default_block(N, V)
    p1 = _lib.params(N, 4096, V, bwd_vocab_block=bv)
    assert lib.flce_workspace_size(p0, 1) == lib.flce_workspace_size(p1, 1)
    if bv > 256:  # a neighbouring block size changes it
        p2 = _lib.params(N, 4096, V, bwd_vocab_block=bv - 256)
        assert lib.flce_workspace_size(p2, 1) != lib.flce_workspace_size(p0, 1)


@pytest.mark.parametrize("N,V", [(8192, 128256), (16384, 262144), (512, 4096), (1, 7),
                                 (4096, 32000), (1 << 20, 50000)])
def test_vocab_block_candidates(N, V):
    c = tuning.vocab_block_candidates(N, V)
    vr = tuning.round_up(V, 256)
    assert c == sorted(set(c), reverse=True)
    assert tuning.library_default_block(N, V) in c
    for bv in c:
        assert bv % 256 == 0 and 256 <= bv <= vr
        assert N * bv * 2 <= tuning.DEFAULT_DL_BUDGET or bv == tuning.library_default_block(N, V)


def test_vocab_block_candidates_llama3_head():
    # two nearly equal blocks (64256 + 64000) beside the default 65536 + 62720
    c = tuning.vocab_block_candidates(8192, 128256)
    assert 65536 in c and 64256 in c and 128256 not in c


def test_small_vocab_gets_one_block():
    assert tuning.vocab_block_candidates(512, 4096)[0] == 4096


def test_select_takes_the_fastest_and_keeps_order_on_ties():
    cfg = tuning.select({"single": 2.0, "pair": 1.5},
                        {("single", 512): 3.0, ("pair", 512): 3.0, ("pair", 256): 4.0})
    assert cfg == tuning.FlceConfig("pair", "single", 512)
    assert cfg.forward_kwargs() == {"gemm_form": "pair"}
    assert cfg.backward_kwargs() == {"gemm_form": "single", "bwd_vocab_block": 512}


def test_gemm_form_parameter():
    assert _lib.params(4, 64, 10).gemm_form == 0
    assert _lib.params(4, 64, 10, gemm_form="single").gemm_form == 1
    assert _lib.params(4, 64, 10, gemm_form="pair").gemm_form == 2
    assert _lib.params(4, 64, 10, gemm_form="wide").gemm_form == 3
    assert _lib.params(4, 64, 10, gemm_form=2).gemm_form == 2
    with pytest.raises(ValueError):
        _lib.params(4, 64, 10, gemm_form="quad")


@pytest.mark.parametrize("N,H,V,expect", [
    # Llama-3 head: every GEMM long enough and large enough for 256 x 512 tiles
    (8192, 4096, 128256, dict(fwd_lse="wide", bwd_dlogits="wide", bwd_dw="wide")),
    # H = 2048: the logits GEMMs' K loop is too short; dW has too few wide tiles
    (32768, 2048, 128000, dict(fwd_lse="pair", bwd_dlogits="pair", bwd_dw="pair")),
    (4096, 2048, 32000, dict(fwd_lse="pair", bwd_dlogits="pair", bwd_dw="pair")),
    (16384, 4096, 262144, dict(fwd_lse="wide", bwd_dlogits="wide", bwd_dw="wide")),
    (512, 256, 4096, dict(fwd_lse="pair", bwd_dlogits="pair", bwd_dw="pair")),
])
def test_default_form_per_gemm(lib, monkeypatch, N, H, V, expect):
    import linear_cross_entropy_gemm_gb300 as F
    monkeypatch.delenv("FLCE_GEMM_FORM", raising=False)
    for gm, f in expect.items():
        assert F.resolved_gemm_form(N, H, V, gemm=gm) == f, gm
    assert F.resolved_gemm_form(N, H, V, gemm="bwd_dx") == "pair"


def test_explicit_and_environment_forms(lib, monkeypatch):
    import linear_cross_entropy_gemm_gb300 as F
    monkeypatch.delenv("FLCE_GEMM_FORM", raising=False)
    for f in ("single", "pair", "wide"):
        # an explicit form applies to every GEMM at any size (dx runs wide as pair)
        for gm in F.GEMMS:
            want = "pair" if (gm == "bwd_dx" and f == "wide") else f
            assert F.resolved_gemm_form(512, 256, 4096, gemm_form=f, gemm=gm) == want
        monkeypatch.setenv("FLCE_GEMM_FORM", f)
        assert F.resolved_gemm_form(512, 256, 4096) == f
        # the environment does not override an explicit form
        assert F.resolved_gemm_form(512, 256, 4096, gemm_form="single") == "single"
    assert lib.flce_resolved_gemm_form(None, 0) == -1
    assert lib.flce_resolved_gemm_form(_lib.params(4, 64, 10), 4) == -1
    assert lib.flce_resolved_gemm_form(_lib.params(4, 12, 10), 0) == -1  # invalid H


def test_tune_result_serialises():
    r = tuning.TuneResult(tuning.FlceConfig("pair", "pair", 65536), {"pair": 1.0},
                          {("pair", 65536): 2.0}, key=("dev",))
    d = r.as_dict()
    assert d["config"]["bwd_vocab_block"] == 65536 and d["backward_ms"] == {"pair/65536": 2.0}


@pytest.mark.parametrize("name", ["llama3_head", "large_logit", "vocab256k"])
def test_full_size_samples_cover_the_default_seams(name):
    # The full-size parity samples force the rows at every seam of the
    # default backward vocabulary block and of the tilings (host logic only).
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from parity import token_seams, vocab_seams
    from linear_cross_entropy_gemm_gb300 import inputs as I
    wl = I.WORKLOADS[name]
    bv = tuning.library_default_block(wl.N, wl.V)
    cols = set(vocab_seams(wl.V, bv))
    for v0 in range(bv, wl.V, bv):
        assert {v0 - 1, v0, v0 + 1} <= cols
    assert {511, 512, wl.V - 1} <= cols
    rows = set(token_seams(wl.N))
    assert {255, 256, 511, 512, 4095, 4096, wl.N - 256, wl.N - 1} <= rows
    rows_s = I.sample_indices(wl.seed, wl.N, 256, must_include=sorted(rows))
    cols_s = I.sample_indices(wl.seed + 1, wl.V, 256, must_include=sorted(cols))
    assert len(rows_s) == 256 and len(cols_s) == 256
    assert rows <= set(rows_s.tolist()) and cols <= set(cols_s.tolist())


def test_interleaved_timing_round_robins_the_candidates():
    # Every candidate is warmed up once, then timed once per repetition in a
    # fixed rotation; the result is each candidate's median.
    calls = []

    def timer(fn, reps, warmup):
        calls.append((fn(), reps, warmup))
        return {"a": [5.0, 1.0, 3.0], "b": [2.0, 2.0, 9.0]}[calls[-1][0]][
            sum(1 for c in calls[:-1] if c[0] == calls[-1][0] and c[1:] == (1, 0))]

    res = tuning._interleaved({"a": lambda: "a", "b": lambda: "b"}, timer, reps=3, warmup=2)
    assert [c for c in calls[:2]] == [("a", 1, 2), ("b", 1, 2)]
    assert [c[0] for c in calls[2:]] == ["a", "b", "a", "b", "a", "b"]
    assert res == {"a": 3.0, "b": 2.0}
