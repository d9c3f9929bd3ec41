"""bench.py prints one JSON line with the keys the benchmark contract needs.
The reference arm (the CPU oracle) runs here on a small shape; the GPU arm
is checked by a gpu-marked test on a small shape."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "2", "--warmup", "1", "--shape", "64,128,2048",
              "--sample-rows", "16"])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "cpu_baseline", "e2e", "config"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # The measured time of one sampled step, not an extrapolation to the workload.
    assert d["ms_per_step"] < 60_000 and d["extrapolated_ms_per_full_step"] >= d["ms_per_step"]
    assert d["config"]["workload"].startswith("llama3_head")


def test_reference_arm_other_workload_full_oracle():
    # The tiny workload's oracle runs on all its tokens (sample = N).
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny",
              "--sample-rows", "512", "--oracle-threads", "1"])
    assert d["config"]["workload"].startswith("tiny") and d["config"]["N"] == 512
    assert d["cpu_baseline"]["cores"] == 1
    assert abs(d["extrapolated_ms_per_full_step"] - d["ms_per_step"]) < 1e-6 * d["ms_per_step"]


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _run(["--steps", "3", "--warmup", "3", "--shape", "1024,256,8192", "--no-cpu-baseline"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "gpu_launches", "clocks", "modes", "memory"):
        assert k in d, k
    r = d["roofline"]
    assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5 and r["unit"] == "TFLOP/s"
    assert d["gpu_launches"] == 3 * (3 + 1 + 3)  # fwd, merge, finalize; prep; one block
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] == 4
    assert d["config"]["workload"].startswith("llama3_head")
    assert set(d["modes"]) == {"recompute", "stored"} and d["impl_config"]["mode"] == "kept"
    m = d["memory"]
    # The library allocates nothing; its scratch stays under the stated bound.
    assert m["device_free_drop_during_step_mib"] == 0
    assert m["scratch_mib"] <= m["scratch_bound_mib"]
    # Peak = scratch + outputs, up to the caching allocator's granularity (a
    # large block keeps a remainder under 1 MiB unsplit).
    assert 0 <= m["peak_extra_mib"] - m["scratch_mib"] - m["outputs_mib"] < 8.0
    # the same step with 16-bit dW and db: the same scratch, smaller outputs
    assert m["outputs_mib_16bit_grads"] < m["outputs_mib"]
    assert 0 <= m["peak_extra_mib_16bit_grads"] - m["scratch_mib"] - m["outputs_mib_16bit_grads"] < 8.0


@pytest.mark.gpu
def test_gpu_vocab_split_line_matches_the_replica_loss():
    # At one GPU the vocabulary split runs the shard calls on a single shard
    # (the whole vocabulary); its loss equals the plain path's.
    for mode in ("recompute", "kept"):
        common = ["--steps", "3", "--warmup", "3", "--shape", "1024,256,8192",
                  "--no-cpu-baseline", "--mode", mode, "--only-mode"]
        plain = _run(common)
        split = _run(common + ["--parallel", "vocab"])
        assert split["scaling"] == "strong" and split["impl_config"]["vocab_shard"] == [0, 8192]
        assert split["config"]["parallelism"].startswith("vocabulary split")
        assert split["roofline"]["bound"] == "tensor" and split["gpu_launches"] > 0
        assert abs(split["loss"] - plain["loss"]) <= 1e-6 * abs(plain["loss"])


@pytest.mark.gpu
def test_gpu_budget_mode_line():
    # The kept block as wide as the method's budget allows: at this shape and
    # block, part of the vocabulary (the rest is recomputed in 8192-column
    # blocks); the line reports the width and stays within its bound.
    import linear_cross_entropy_gemm_gb300 as F
    N, H, V, bv = 2048, 256, 65536, 8192
    k = F.flce_keep_vocab_within(N, H, V, bwd_vocab_block=bv)
    assert bv < k < V
    d = _run(["--steps", "3", "--warmup", "3", "--shape", f"{N},{H},{V}", "--no-cpu-baseline",
              "--mode", "budget", "--only-mode", "--bwd-vocab-block", str(bv)])
    assert d["impl_config"]["mode"] == "budget" and d["impl_config"]["keep_vocab"] == k
    nblk = 1 + -(-(V - k) // bv)
    assert d["gpu_launches"] == 3 * (4 + 3 * nblk)  # fwd, merge, finalize, prep; 3 per block
    m = d["memory"]
    assert m["device_free_drop_during_step_mib"] == 0
    assert m["scratch_mib"] <= m["scratch_bound_mib"]
    assert d["flops_executed_per_step"] == 8.0 * N * H * V - 2.0 * N * H * k
