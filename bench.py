"""Benchmark of the fused linear cross-entropy (FLCE) forward + backward.

One step = the forward and the backward (the whole hot path) over one batch
of a workload, by default the Llama-3-shaped head: N=8192 tokens, H=4096,
V=128256, bf16, mean reduction, no bias, dloss = 1. Prints ONE JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload tiny|medium|llama3_head|large_logit|vocab256k]
                  [--mode kept|recompute|stored|budget]

* value: tokens/s over all ranks, inputs resident in HBM, device time per
  step from CUDA events on the launching stream; L2 flushed (256 MiB write)
  between timed steps, outside the timed events.
* mode: the backward mode of the timed step. "kept" (the default, and the
  autograd module's): the forward keeps the first backward vocabulary
  block's probabilities in the buffer the backward stages dL in, and the
  backward recomputes the other blocks. "recompute": every block recomputed.
  "stored": every logit's probability kept (2 N V bytes more memory).
  "budget": the kept block as wide as the method's memory budget allows
  (flce_keep_vocab_within: kept-mode memory within the recompute mode's
  plus an fp32 [V, H] dW accumulator, which this library never allocates).
  The other modes are timed the same way and reported in "modes" ("budget"
  only where its kept block is neither one block nor the whole vocabulary).
* e2e: the same metric through the C ABI with the step's inputs (x, y,
  dloss) copied from pinned host memory and the loss read back every step;
  the next step's copy runs on a side stream during the current step. The
  gradients stay on the device, as in a training step.
* roofline: the dominant kernel (most device time), timed per launch with
  caller-owned CUDA events around each launch (flce_*_traced).
* memory: peak device memory above the live inputs across one step
  (torch's allocator; the library allocates nothing, which the device-level
  free memory confirms), split into the library's scratch and the outputs.
* cpu_baseline / --impl reference: the CPU fp64 oracle timed on this host's
  cores on the same bounded token sample of the workload (a slow reference
  implementation, not a target).
* --gpus N > 1 (torchrun): independent replicas, one per GPU, by default
  (weak scaling: every rank runs the whole workload); barrier + max over
  ranks. --parallel vocab splits the vocabulary instead (strong scaling):
  rank r holds its contiguous shard of W's rows and runs the library's
  vocabulary-shard calls, with the exchanges (a MAX and a SUM all-reduce of
  per-token statistics, a SUM all-reduce of the fp32 partial dx) done by
  NCCL all-reduces. Each shard keeps its own first block in the kept mode
  (recompute with --mode recompute; no stored mode for shards), and the
  shard calls are not traced per kernel, so that line's roofline is the
  whole step's. At N = 1 it runs the shard calls on one shard, the whole
  vocabulary.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time


def _oracle_threads_from_argv():
    """--oracle-threads T fixes the BLAS thread count of the CPU oracle; it
    must be in the environment before numpy loads its BLAS library."""
    for i, a in enumerate(sys.argv):
        if a == "--oracle-threads" and i + 1 < len(sys.argv):
            return sys.argv[i + 1]
        if a.startswith("--oracle-threads="):
            return a.split("=", 1)[1]
    return None


_T = _oracle_threads_from_argv()
if _T:
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = _T

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FLCE fwd+bwd ms, tokens/s, TFLOP/s (% bf16 TC peak) @ 8192×4096×128256"
HEADLINE = "llama3_head"
PAGES_MS = 19.897  # Liger-Kernel commit 95b01e9, B200, Llama-3 head shape (context)
L2_FLUSH_BYTES = 256 << 20
MODES = ("kept", "recompute", "stored", "budget")
# dram__bytes_read.sum + dram__bytes_write.sum per launch, averaged over a
# step's launches of each kernel, from one ncu capture of the Llama-3 head
# step in the kept-block mode (1-pass metrics, default GEMM forms and block,
# the committed build of these kernels). Not measured by this run; reported
# only for that exact configuration and labelled as such.
TRAFFIC_CAPTURE = {"fwd_lse": 5.027e9, "bwd_dlogits": 2.977e9, "bwd_dw": 4.465e9,
                   "bwd_dx": 6.483e9}
TRAFFIC_SOURCE = ("ncu capture of the kept-block Llama-3 head step on a GB300 "
                  "(dram__bytes_read.sum + dram__bytes_write.sum per launch); not measured "
                  "in this run")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while running (a
    20-step timed region of the Llama-3 head lasts about 0.4 s)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [t.strip() for t in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
                pw.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(value: float, ws: int, device) -> float:
    """Largest value over all ranks (one all-reduce MAX); the identity for a
    single process. Timing uses it so the slowest replica sets the number."""
    if ws <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def workload_of(args):
    from linear_cross_entropy_gemm_gb300 import inputs as I
    wl = I.WORKLOADS[args.workload]
    if args.shape:
        n_, h_, v_ = (int(t) for t in args.shape.split(","))
        wl = wl.with_(name=f"{wl.name}-shape", N=n_, H=h_, V=v_)
    if args.dtype != wl.dtype:
        wl = wl.with_(dtype=args.dtype)
    return wl


def config_of(wl, ws: int, vocab_split: bool = False) -> dict:
    """The workload's description, the same in both arms' JSON lines."""
    opts = [wl.reduction, "bias" if wl.has_bias else "no bias"]
    if wl.label_smoothing:
        opts.append(f"label_smoothing={wl.label_smoothing:g}")
    if wl.lse_square_scale:
        opts.append(f"lse_square_scale={wl.lse_square_scale:g}")
    if wl.logit_scale != 1.0:
        opts.append(f"logit_scale={wl.logit_scale:g}")
    if wl.ignore_frac:
        opts.append(f"{wl.n_ignored} ignored")
    opts.append(f"dloss={wl.dloss}")
    return {"workload": f"{wl.name}: N={wl.N} H={wl.H} V={wl.V} {wl.dtype}, " + ", ".join(opts),
            "N": wl.N, "H": wl.H, "V": wl.V, "dtype": wl.dtype,
            "parallelism": (f"vocabulary split over {ws} GPU(s)" if vocab_split else
                            "replicas" if ws > 1 else "single GPU"),
            "l2": "GPU arm: flushed (256 MiB write) before each timed step, outside the events"}


def options_of(wl) -> dict:
    return dict(ignore_index=wl.ignore_index, label_smoothing=wl.label_smoothing,
                lse_square_scale=wl.lse_square_scale, logit_scale=wl.logit_scale,
                reduction=wl.reduction)


# ----------------------------------------------------------- CPU oracle arm

class OracleSample:
    """The first `rows` tokens of the workload (all V, all H), widened to
    float64 once; run() times one oracle forward + backward over them."""

    def __init__(self, wl, rows: int):
        from linear_cross_entropy_gemm_gb300 import inputs as I
        inp = I.make_inputs(wl.with_(N=rows))
        self.x, self.W = I.bits_to_f64(inp.x, wl.dtype), I.bits_to_f64(inp.W, wl.dtype)
        self.b = None if inp.b is None else I.bits_to_f64(inp.b, wl.dtype)
        self.y, self.dloss = inp.y, inp.dloss.astype(np.float64)
        self.opts = options_of(wl)

    def run(self) -> float:
        from oracle import flce_oracle as O
        t0 = time.perf_counter()
        O.forward(self.x, self.W, self.b, self.y, **self.opts)
        O.backward(self.dloss, self.x, self.W, self.b, self.y, **self.opts)
        return time.perf_counter() - t0


def oracle_threads() -> int:
    t = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(t) if t else (os.cpu_count() or 1)


def sample_text(wl, rows: int, reps: int, secs: float) -> str:
    return (f"{rows} of {wl.N} tokens of {wl.name} per step (all V={wl.V}, H={wl.H}); "
            f"numpy float64 forward + backward, {reps} steps in {secs:.1f} s")


def cpu_baseline(wl, rows: int, min_seconds: float = 10.0):
    """The oracle over the sample, repeated until about min_seconds of work."""
    s = OracleSample(wl, rows)
    times = []
    while sum(times) < min_seconds or len(times) < 2:
        times.append(s.run())
    per_step = statistics.median(times)
    return {"value": rows / per_step, "unit": "tokens/s", "cores": oracle_threads(),
            "kind": "oracle", "sample": sample_text(wl, rows, len(times), sum(times)),
            "ms_per_sampled_step": per_step * 1e3,
            "extrapolated_ms_per_full_step": per_step / rows * wl.N * 1e3}


def run_reference(args):
    rank, _, ws = dist_env()
    if rank != 0:
        return
    wl = workload_of(args)
    rows = min(args.sample_rows, wl.N)
    sample = OracleSample(wl, rows)
    for _ in range(min(args.warmup, 1)):
        sample.run()
    times = [sample.run() for _ in range(args.steps)]
    per_step = sum(times) / len(times)
    value = rows / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, ws, args.parallel == "vocab"),
        "step": f"one oracle forward + backward over {rows} of the workload's {wl.N} tokens",
        "extrapolated_ms_per_full_step": per_step / rows * wl.N * 1e3,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_threads(),
                         "kind": "oracle", "sample": sample_text(wl, rows, len(times),
                                                                 sum(times))},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

class Problem:
    """Device inputs of one workload plus the buffers of one backward mode,
    and one forward + backward step through the binding (C ABI). With
    `shard` = (start, end) only W's rows [start, end) are on the device and a
    step runs the vocabulary-shard calls (vocab_parallel)."""

    def __init__(self, torch, F, wl, dev, tdt, fkw, bkw, shard=None, dw_dtype=None):
        from linear_cross_entropy_gemm_gb300 import inputs as I
        self.torch, self.F, self.wl, self.dev = torch, F, wl, dev
        self.fkw, self.bkw = fkw, bkw
        self.shard = shard
        inp = I.make_inputs(wl)
        r0, r1 = shard if shard is not None else (0, wl.V)
        self.host_x = torch.from_numpy(inp.x.view(np.int16)).view(tdt).pin_memory()
        self.host_y = torch.from_numpy(inp.y).pin_memory()
        self.host_dl = torch.from_numpy(inp.dloss).pin_memory()
        self.x = self.host_x.to(dev)
        self.W = torch.from_numpy(inp.W[r0:r1].view(np.int16)).view(tdt).to(dev)
        self.b = (None if inp.b is None else
                  torch.from_numpy(inp.b[r0:r1].view(np.int16)).view(tdt).to(dev))
        self.y = self.host_y.to(dev)
        self.dloss = self.host_dl.to(dev)
        self.opts = options_of(wl)
        self.tdt = tdt
        # dW (and db) output type: fp32, or the operands' 16-bit type.
        self.dw_dtype = torch.float32 if dw_dtype is None else dw_dtype
        self.bufs = None

    def keep_vocab(self, mode):
        """keep_vocab of a mode: the budget width for "budget", else 0."""
        if mode != "budget":
            return 0
        wl = self.wl
        return self.F.flce_keep_vocab_within(wl.N, wl.H, wl.V, has_bias=wl.has_bias,
                                             bwd_vocab_block=self.bkw.get("bwd_vocab_block", 0))

    def kept_cols(self, mode, bv):
        """Vocabulary columns whose logits the backward does not recompute."""
        V = self.wl.V
        return {"recompute": 0, "kept": min(bv, V), "stored": V,
                "budget": min(self.keep_vocab("budget"), V)}[mode]

    def allocate(self, mode):
        torch, F, wl = self.torch, self.F, self.wl
        N, H, V, dev = wl.N, wl.H, wl.V, self.dev
        if self.shard is not None:
            # The shard calls allocate their workspaces and outputs per call;
            # the kept block is the caller's.
            from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
            kept = None
            if mode == "kept":
                kept = torch.empty(VP.kept_size(
                    N, H, self.shard[1] - self.shard[0], vocab_start=self.shard[0],
                    vocab_total=V, bwd_vocab_block=self.bkw.get("bwd_vocab_block", 0),
                    input_fp16=self.tdt == torch.float16), dtype=torch.uint8, device=dev)
            self.bufs = {"mode": mode, "fws": None, "bws": None, "state": kept, "loss": None,
                         "lse": None, "dx": None, "dW": None, "db": None}
            return self.bufs
        bvb = self.bkw.get("bwd_vocab_block", 0)
        fp16 = self.tdt == torch.float16
        kv = self.keep_vocab(mode)
        b = {"mode": mode, "keep_vocab": kv}
        b["fws"] = torch.empty(F.flce_workspace_size(N, H, V, "forward", **self.opts),
                               dtype=torch.uint8, device=dev)
        kind = {"kept": "backward_keep", "budget": "backward_keep",
                "stored": "backward_store"}.get(mode, "backward")
        b["bws"] = torch.empty(F.flce_workspace_size(N, H, V, kind, bwd_vocab_block=bvb,
                                                     has_bias=wl.has_bias, keep_vocab=kv,
                                                     **self.opts),
                               dtype=torch.uint8, device=dev)
        b["state"] = None
        if mode == "stored":
            b["state"] = torch.empty(F.flce_saved_size(N, H, V, input_fp16=fp16, **self.opts),
                                     dtype=torch.uint8, device=dev)
        elif mode in ("kept", "budget"):
            b["state"] = torch.empty(F.flce_kept_size(N, H, V, input_fp16=fp16,
                                                      bwd_vocab_block=bvb, keep_vocab=kv),
                                     dtype=torch.uint8, device=dev)
        b["loss"] = torch.empty(N if wl.reduction == "none" else 1, dtype=torch.float32, device=dev)
        b["lse"] = torch.empty(N, dtype=torch.float32, device=dev)
        b["dx"] = torch.empty(N, H, dtype=self.tdt, device=dev)
        b["dW"] = torch.empty(V, H, dtype=self.dw_dtype, device=dev)
        b["db"] = torch.empty(V, dtype=self.dw_dtype, device=dev) if wl.has_bias else None
        self.bufs = b
        return b

    def release(self):
        self.bufs = None

    def scratch_bytes(self):
        b = self.bufs
        if self.shard is not None:
            return None  # allocated inside the shard calls: only the peak is known
        return sum(t.numel() for t in (b["fws"], b["bws"], b["state"]) if t is not None)

    def output_bytes(self):
        b = self.bufs
        return sum(t.numel() * t.element_size()
                   for t in (b["loss"], b["lse"], b["dx"], b["dW"], b["db"]) if t is not None)

    def step(self, ftr=None, btr=None, xb=None, yb=None, dlb=None):
        F, b = self.F, self.bufs
        xb = self.x if xb is None else xb
        yb = self.y if yb is None else yb
        dlb = self.dloss if dlb is None else dlb
        if self.shard is not None:
            from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
            sh = dict(vocab_start=self.shard[0], vocab_total=self.wl.V, kept=b["state"],
                      bwd_vocab_block=self.bkw.get("bwd_vocab_block", 0))
            b["loss"], b["lse"] = VP.vocab_parallel_forward(xb, self.W, self.b, yb, **sh,
                                                            **self.opts)
            b["dx"], b["dW"], b["db"] = VP.vocab_parallel_backward(
                dlb, b["lse"], xb, self.W, self.b, yb, dW_dtype=self.dw_dtype,
                db_dtype=self.dw_dtype, **sh, **self.opts)
            return
        st = {} if b["state"] is None else {("saved" if b["mode"] == "stored" else "kept"):
                                            b["state"]}
        if b["mode"] == "budget":
            st["keep_vocab"] = b["keep_vocab"]
        F.flce_forward(xb, self.W, self.b, yb, workspace=b["fws"], out=(b["loss"], b["lse"]),
                       trace=ftr, bwd_vocab_block=self.bkw.get("bwd_vocab_block", 0),
                       **st, **self.opts, **self.fkw)
        F.flce_backward(dlb, b["lse"], xb, self.W, self.b, yb, workspace=b["bws"],
                        out=(b["dx"], b["dW"], b["db"]), trace=btr, dW_dtype=self.dw_dtype,
                        db_dtype=self.dw_dtype, **st, **self.opts, **self.bkw)


def end_to_end(torch, stream, prob, steps, barrier):
    """Milliseconds per step of `steps` steps, each fed from the host: copy the
    step's inputs (pinned x, y, dloss) into one of two device buffer sets on a
    copy stream, run the step on `stream` once they have landed, and read the
    loss back. The copy of step i+1 waits only for step i-1 (the last user of
    its buffer set)."""
    dev = prob.x.device
    host_in = (prob.host_x, prob.host_y, prob.host_dl)
    bufs = [(prob.x, prob.y, prob.dloss),
            (torch.empty_like(prob.x), torch.empty_like(prob.y), torch.empty_like(prob.dloss))]
    host_loss = torch.empty(prob.wl.N if prob.wl.reduction == "none" else 1,
                            dtype=torch.float32).pin_memory()
    copy_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    free = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(i):
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(free[i % 2])
            for d, h in zip(bufs[i % 2], host_in):
                d.copy_(h, non_blocking=True)
            ready[i % 2].record(copy_stream)

    def run(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(ready[i % 2])
            xb, yb, dlb = bufs[i % 2]
            prob.step(xb=xb, yb=yb, dlb=dlb)
            free[i % 2].record(stream)
            host_loss.copy_(prob.bufs["loss"].reshape(-1), non_blocking=True)

    run(2)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    h2d_bytes = sum(t.numel() * t.element_size() for t in host_in)
    return e0.elapsed_time(e1) / steps, h2d_bytes, host_loss.numel() * 4


def kernel_flops(name, wl, kept_cols):
    """Algorithmic flops per step of each GEMM kernel when the backward
    recomputes all but `kept_cols` vocabulary columns."""
    N, H, V = wl.N, wl.H, wl.V
    f = {"fwd_lse": 2.0 * N * H * V, "bwd_dw": 2.0 * N * H * V, "bwd_dx": 2.0 * N * H * V}
    if kept_cols < V:
        f["bwd_dlogits"] = 2.0 * N * H * (V - kept_cols)
    return f.get(name)


def timed_steps(torch, prob, args, stream, flush, barrier, clocks=None):
    """K device-timed steps (L2 flushed before each, outside the events) with
    per-launch events; returns (ms per step, {kernel: [ms per launch]}, launches)."""
    F = prob.F
    ftr, btr = F.KernelTrace(16), F.KernelTrace(256)
    for _ in range(args.warmup):
        prob.step()
    barrier()
    if clocks:
        clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    per_kernel, launches = {}, 0
    barrier()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        prob.step(ftr=ftr, btr=btr)
        ev[i][1].record(stream)
        torch.cuda.synchronize(prob.dev)
        for name, ms in ftr.launches() + btr.launches():
            per_kernel.setdefault(name, []).append(ms)
            launches += 1
    barrier()
    clk = clocks.stop() if clocks else None
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    return ms, per_kernel, launches, clk


def run_ours(args):
    import torch
    import torch.distributed as dist

    import linear_cross_entropy_gemm_gb300 as F
    from linear_cross_entropy_gemm_gb300 import tuning

    rank, local, ws = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workload_of(args)
    tdt = torch.float16 if wl.dtype == "fp16" else torch.bfloat16
    pk = peaks()
    N, H, V = wl.N, wl.H, wl.V
    fkw, bkw = {}, {"bwd_vocab_block": args.bwd_vocab_block}
    tune = None
    vocab_split = args.parallel == "vocab"
    shard = None
    if vocab_split:
        from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
        if args.autotune or V < 256 * ws or args.mode in ("stored", "budget"):
            raise SystemExit("--parallel vocab: kept or recompute mode, no autotuning, and "
                             "V >= 256 per rank")
        args.only_mode = True
        shard = VP.shard_range(V, ws, rank)
    prob = Problem(torch, F, wl, dev, tdt, fkw, bkw, shard=shard,
                   dw_dtype=tdt if args.dw_dtype == "16bit" else torch.float32)
    if args.autotune:
        res = tuning.autotune(prob.x, prob.W, prob.b, prob.y, dloss=prob.dloss, reps=3,
                              mode="kept" if args.mode in ("kept", "budget") else "recompute",
                              **prob.opts)
        fkw.update(res.config.forward_kwargs())
        bkw.update(res.config.backward_kwargs())
        tune = res.as_dict()
    bvb = bkw["bwd_vocab_block"]
    bv_used = bvb or tuning.library_default_block(N, V)
    forms_used = {gm: F.resolved_gemm_form(N, H, V, (fkw if gm == "fwd_lse" else bkw).get(
        "gemm_form", "default"), gemm=gm, bwd_vocab_block=bvb) for gm in F.GEMMS}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    bv_default = bvb or tuning.library_default_block(N, V)
    distinct = {"budget": prob.kept_cols("budget", bv_default)
                not in (min(bv_default, V), V)}
    modes = [args.mode] + ([] if args.only_mode else
                           [m for m in MODES if m != args.mode and distinct.get(m, True)])
    results = {}
    for mode in modes:
        # Memory: everything allocated above the live inputs across one step.
        barrier()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        prob.allocate(mode)
        prob.step()
        barrier()
        free0 = torch.cuda.mem_get_info(dev)[0]
        prob.step()
        barrier()
        free1 = torch.cuda.mem_get_info(dev)[0]
        scratch = prob.scratch_bytes()
        mem = {"peak_extra_mib": (torch.cuda.max_memory_allocated(dev) - base) / 2**20,
               "scratch_mib": None if scratch is None else scratch / 2**20,
               "outputs_mib": None if scratch is None else prob.output_bytes() / 2**20,
               "device_free_drop_during_step_mib": (free0 - free1) / 2**20}
        clocks = ClockSampler(local) if mode == args.mode else None
        ms, per_kernel, launches, clk = timed_steps(torch, prob, args, stream, flush, barrier,
                                                    clocks)
        ms = max_over_ranks(ms, ws, dev)
        e2e = None
        if mode == args.mode:
            e2e = end_to_end(torch, stream, prob, args.steps, barrier)
            e2e = (max_over_ranks(e2e[0], ws, dev), e2e[1], e2e[2])
        loss_value = float(prob.bufs["loss"].double().sum())
        results[mode] = dict(ms=ms, per_kernel=per_kernel, launches=launches, clk=clk, mem=mem,
                             e2e=e2e, loss=loss_value)
        prob.release()

    if shard is None and prob.dw_dtype == torch.float32:
        # The same step's peak with dW and db in the operands' 16-bit type
        # (what the autograd module returns): one untimed step.
        barrier()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        prob.dw_dtype = tdt
        prob.allocate(args.mode)
        prob.step()
        barrier()
        results[args.mode]["mem"]["peak_extra_mib_16bit_grads"] = (
            torch.cuda.max_memory_allocated(dev) - base) / 2**20
        results[args.mode]["mem"]["outputs_mib_16bit_grads"] = prob.output_bytes() / 2**20
        prob.release()
        prob.dw_dtype = torch.float32

    head = results[args.mode]
    ms, per_kernel = head["ms"], head["per_kernel"]
    steps_ = args.steps
    totals = {k: sum(v) for k, v in per_kernel.items()}
    kern = {k: {"launches_per_step": len(v) // steps_, "ms_per_step": sum(v) / steps_,
                "share": sum(v) / sum(totals.values())} for k, v in sorted(per_kernel.items())}
    dom = max(totals, key=totals.get) if totals else None
    dom_ms = totals[dom] / steps_ if totals else None
    kept_cols = prob.kept_cols(args.mode, bv_used) if shard is None else None
    dom_flops = kernel_flops(dom, wl, kept_cols) if totals else None
    v_local = V if shard is None else shard[1] - shard[0]
    if vocab_split:
        # The shard calls are not traced per kernel: the roofline is the whole
        # step's, one rank's executed flops over its step time.
        kept_cols = min(tuning.library_default_block(N, v_local) if not bvb else bvb, v_local)
        step_flops = 8.0 * N * H * v_local - (2.0 * N * H * kept_cols if args.mode == "kept"
                                               else 0)
        achieved = step_flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "whole step (vocabulary shard)",
                "achieved": achieved, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_sus"], "frac_of_burst_peak": achieved / pk["bf16"],
                "peak_kind": f"bf16 sustained ({pk['src']})",
                "algorithmic_flops_per_step": step_flops, "traffic": None}
        nblk = -(-v_local // tuning.library_default_block(N, v_local))
        # forward GEMM + shard statistics, rescale, merge (+ finalize), prep,
        # per block dlogits (+ db) + dW + dx, the fp32 -> 16-bit dx cast
        head["launches"] = steps_ * (2 + 1 + (1 if wl.reduction == "none" else 2) + 1
                                     + nblk * (3 + (1 if wl.has_bias else 0)) + 1)
    elif dom_flops is not None:
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12
        default_cfg = ((N, H, V) == (8192, 4096, 128256) and wl.dtype == "bf16"
                       and bv_used == tuning.library_default_block(N, V)
                       and forms_used == {"fwd_lse": "wide", "bwd_dlogits": "wide",
                                          "bwd_dw": "wide", "bwd_dx": "pair"}
                       and os.environ.get("FLCE_RASTER", "1") != "0"
                       and args.mode == "kept")
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": pk["bf16_sus"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_sus"],
                "peak_kind": f"bf16 sustained ({pk['src']}); the kernel is timed inside a long step",
                "frac_of_burst_peak": achieved / pk["bf16"],
                "launches_per_step": len(per_kernel[dom]) // steps_, "ms_per_step": dom_ms,
                "algorithmic_flops_per_step": dom_flops,
                "traffic": TRAFFIC_CAPTURE[dom] if default_cfg else None,
                "traffic_unit": "bytes per launch",
                "traffic_source": TRAFFIC_SOURCE if default_cfg else None}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": pk["hbm"],
                "unit": "GB/s", "frac": None, "traffic": None}
    flops_8 = 8.0 * N * H * V
    if vocab_split:
        kept_cols = min(tuning.library_default_block(N, v_local) if not bvb else bvb, v_local)
        executed = 8.0 * N * H * v_local - (2.0 * N * H * kept_cols if args.mode == "kept" else 0)
    else:
        executed = sum(kernel_flops(k, wl, kept_cols) or 0.0 for k in totals)
    tflops = flops_8 / (ms * 1e-3) / 1e12
    # Replicas: every rank runs the whole workload. Vocabulary split: the
    # ranks run one workload together.
    value = (1 if vocab_split else ws) * N / (ms * 1e-3)
    e2e_ms, h2d, d2h = head["e2e"]
    other = {}
    for m, r in results.items():
        if m == args.mode:
            continue
        other[m] = {"ms_per_step": r["ms"], "value": ws * N / (r["ms"] * 1e-3),
                    "keep_vocab": prob.keep_vocab(m) or None,
                    "unit": "tokens/s", "tflops_8nhv_equivalent": flops_8 / (r["ms"] * 1e-3) / 1e12,
                    "memory": r["mem"], "loss": r["loss"],
                    "kernels": {k: {"launches_per_step": len(v) // steps_,
                                    "ms_per_step": sum(v) / steps_}
                                for k, v in sorted(r["per_kernel"].items())}}
    budget = {
        # The library's scratch bound: one [N, BVc] 16-bit block (dL staging,
        # or the kept probabilities) and the kept block's per-32-column maxima,
        # the fp32 dx accumulator, the db column partials (with a bias), the
        # forward's per-tile partials and the per-token coefficients; in the
        # budget mode plus the fp32 [V, H] allowance its kept block may use.
        "scratch_bound_mib": (N * bv_used * 2 + N * (bv_used // 32) * 4 + N * H * 4
                              + (4 * -(-N // 128) * bv_used * 4 if wl.has_bias else 0)
                              + N * -(-V // 256) * 12 + N * 32
                              + (V * H * 4 if args.mode == "budget" else 0)) / 2**20 + 1,
        # The method's memory budget, one [N, BV] block set plus an fp32
        # [V, H] dW accumulator, with BV the backward vocabulary block.
        "method_budget_mib": (N * bv_used * 2 + V * H * 4) / 2**20,
    }
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong" if vocab_split else "weak",
        "vs_baseline": (value / ((1 if vocab_split else ws) * N / (PAGES_MS * 1e-3))
                        if wl.dtype == "bf16" and (N, H, V) == (8192, 4096, 128256) else None),
        "dtype": wl.dtype, "data": "synthetic",
        "config": config_of(wl, ws, vocab_split),
        "impl_config": {"mode": args.mode, "bwd_vocab_block": bv_used,
                        "dW_dtype": "fp32" if args.dw_dtype == "fp32" else wl.dtype,
                        "keep_vocab": (prob.keep_vocab(args.mode) if shard is None else 0) or None,
                        "gemm_form": forms_used,
                        **({"vocab_shard": list(shard)} if vocab_split else {})},
        "loss": head["loss"],
        "tflops_8nhv": tflops, "frac_bf16_peak_8nhv": tflops / pk["bf16_sus"],
        "frac_bf16_burst_8nhv": tflops / pk["bf16"],
        "tflops_executed": executed / (ms * 1e-3) / 1e12,
        "flops_executed_per_step": executed,
        "tflops_6nhv_useful": tflops * 0.75,
        "roofline": roof,
        "kernels": kern if not vocab_split else None,
        "gpu_launches": head["launches"],
        "memory": dict(head["mem"], **budget),
        "e2e": {"value": ws * N / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "x, y, dloss copied in and the loss read back every step; dx, dW "
                        "(and db) stay on the device, as in a training step"},
        "clocks": head["clk"],
        "modes": other,
    }
    if tune is not None:
        line["autotune"] = tune
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, min(args.sample_rows, N))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    from linear_cross_entropy_gemm_gb300 import inputs as I
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(I.WORKLOADS))
    ap.add_argument("--mode", default="kept", choices=MODES,
                    help="backward mode of the timed step (the others are timed beside it)")
    ap.add_argument("--only-mode", action="store_true", help="time --mode only")
    ap.add_argument("--parallel", default="replicas", choices=["replicas", "vocab"],
                    help="ranks under torchrun: independent replicas (default) or one "
                         "vocabulary split")
    ap.add_argument("--sample-rows", type=int, default=256,
                    help="tokens per oracle step (reference arm and cpu_baseline)")
    ap.add_argument("--oracle-threads", default=None,
                    help="BLAS threads of the CPU oracle (default: all cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="", help="N,H,V override (profiling captures only)")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"],
                    help="operand type (the headline workload is bf16; fp16 is a side measurement)")
    ap.add_argument("--autotune", action="store_true",
                    help="time the GEMM forms and backward vocabulary blocks first and run the "
                         "fastest (tuning.autotune); the table goes into the JSON line")
    ap.add_argument("--dw-dtype", default="fp32", choices=["fp32", "16bit"],
                    help="dW and db output type: fp32, or the operands' type (what the "
                         "autograd module returns)")
    ap.add_argument("--bwd-vocab-block", type=int, default=0,
                    help="backward vocabulary block (multiple of 256); 0 = library default")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
