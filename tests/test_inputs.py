"""Seeded input generator: bf16 rounding, exact ignored counts, target laws,
determinism. CPU only."""
import numpy as np
import torch

from linear_cross_entropy_gemm_gb300 import inputs as I


def test_bf16_rounding_matches_torch_rne():
    r = np.random.default_rng(0)
    a = np.concatenate([r.standard_normal(100000).astype(np.float32) * 3,
                        np.array([1.00390625, 1.01171875, -2.0078125, 0.0, 65504.0], np.float32)])
    ours = I.f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = I.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(a).to(torch.bfloat16).double().numpy())


def test_workloads_are_deterministic_and_shaped():
    wl = I.WORKLOADS["tiny"]
    a, b = I.make_inputs(wl), I.make_inputs(wl)
    assert a.x.shape == (512, 256) and a.W.shape == (4096, 256) and a.b is None
    assert np.array_equal(a.x, b.x) and np.array_equal(a.W, b.W) and np.array_equal(a.y, b.y)
    assert int((a.y == -100).sum()) == round(0.05 * 512)
    valid = a.y[a.y != -100]
    assert valid.min() >= 0 and valid.max() < 4096
    xs = I.bf16_bits_to_f64(a.x)
    ws = I.bf16_bits_to_f64(a.W)
    assert abs(xs.std() - 1.0) < 0.02 and abs(ws.std() - 0.02) < 0.001


def test_streams_are_independent_of_other_sizes():
    w1 = I.WORKLOADS["tiny"]
    w2 = w1.with_(V=1000)
    assert np.array_equal(I.make_inputs(w1).x, I.make_inputs(w2).x)


def test_zipf_targets_follow_the_law():
    y = I.zipf_targets(5, 200000, 1000, 1.1)
    p = np.arange(1, 1001, dtype=np.float64) ** -1.1
    p /= p.sum()
    counts = np.bincount(y, minlength=1000) / y.size
    assert abs(counts[0] - p[0]) < 0.01 and abs(counts[9] - p[9]) < 0.005
    assert y.min() >= 0 and y.max() < 1000


def test_sample_indices_include_forced_and_are_sorted():
    s = I.sample_indices(3, 1000, 50, must_include=[7, 999, 7])
    assert s.size == 50 and 7 in s and 999 in s and np.all(np.diff(s) > 0)


def test_dloss_kinds():
    assert I.make_inputs(I.WORKLOADS["tiny"]).dloss.tolist() == [1.0]
    wl = I.WORKLOADS["tiny"].with_(reduction="none", dloss="normal_per_token")
    assert I.make_inputs(wl).dloss.shape == (512,)
