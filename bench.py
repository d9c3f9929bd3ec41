"""Benchmark of the fused linear cross-entropy (FLCE) forward + backward.

One step = flce_forward + flce_backward (the whole hot path) over one batch
of the Llama-3-shaped head: N=8192 tokens, H=4096, V=128256, bf16, mean
reduction, no bias, dloss = 1. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

* value: tokens/s over all ranks, inputs resident in HBM, device time per
  step from CUDA events on the launching stream; L2 flushed (256 MiB write)
  between timed steps, outside the timed events.
* e2e: the same metric through the C ABI with the step's inputs (x, y,
  dloss) copied from pinned host memory and the loss read back every step;
  the next step's copy runs on a side stream during the current step.
* roofline: the dominant kernel (most device time), timed per launch with
  caller-owned CUDA events around each launch (flce_*_traced).
* cpu_baseline / --impl reference: the CPU fp64 oracle timed on this host's
  cores on a bounded sample of the same workload (a slow reference
  implementation, not a target).
* --gpus N > 1 (torchrun): independent replicas, one per GPU ("replicas
  only": the path is not sharded across GPUs); barrier + max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3_head"
METRIC = "FLCE fwd+bwd ms, tokens/s, TFLOP/s (% bf16 TC peak) @ 8192×4096×128256"
PAGES_MS = 19.897  # Liger-Kernel commit 95b01e9, B200, same shape (context)
L2_FLUSH_BYTES = 256 << 20
# dram__bytes_read.sum + dram__bytes_write.sum per launch (average over the
# step's launches of that kernel) from one ncu capture of this workload's full
# step (1-pass metrics; profiles/dram_traffic_llama3_head.md). Must be
# re-measured (or removed) whenever one of these kernels or its raster changes.
TRAFFIC_PER_LAUNCH = {"fwd_lse": 2.986e9, "bwd_dlogits": 3.138e9, "bwd_dw": 4.212e9,
                      "bwd_dx": 5.979e9}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
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
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [t.strip() for t in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
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


# ----------------------------------------------------------- CPU oracle arm

class OracleSample:
    """The first `rows` tokens of the workload (all V, all H), widened to
    float64 once; run() times one oracle forward + backward over them."""

    def __init__(self, wl, rows: int):
        from linear_cross_entropy_gemm_gb300 import inputs as I
        inp = I.make_inputs(wl.with_(N=rows))
        self.x, self.W = I.bf16_bits_to_f64(inp.x), I.bf16_bits_to_f64(inp.W)
        self.b = None if inp.b is None else I.bf16_bits_to_f64(inp.b)
        self.y, self.dloss = inp.y, inp.dloss.astype(np.float64)
        self.opts = dict(ignore_index=wl.ignore_index, label_smoothing=wl.label_smoothing,
                         lse_square_scale=wl.lse_square_scale, logit_scale=wl.logit_scale,
                         reduction=wl.reduction)

    def run(self) -> float:
        from oracle import flce_oracle as O
        t0 = time.perf_counter()
        O.forward(self.x, self.W, self.b, self.y, **self.opts)
        O.backward(self.dloss, self.x, self.W, self.b, self.y, **self.opts)
        return time.perf_counter() - t0


def cpu_baseline(wl, rows: int):
    secs, cores = OracleSample(wl, rows).run(), os.cpu_count()
    return {"value": rows / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} of {wl.N} tokens of {wl.name} (all V={wl.V}, H={wl.H}); "
                      f"numpy float64 forward + backward, {secs:.1f} s"}


def run_reference(args):
    rank, _, ws = dist_env()
    if rank != 0:
        return
    from linear_cross_entropy_gemm_gb300 import inputs as I
    wl = I.WORKLOADS[WORKLOAD]
    if args.shape:
        n_, h_, v_ = (int(t) for t in args.shape.split(","))
        wl = wl.with_(name=f"{wl.name}-shape", N=n_, H=h_, V=v_)
    rows = min(args.ref_rows, wl.N)
    sample = OracleSample(wl, rows)
    for _ in range(min(args.warmup, 1)):
        sample.run()
    times = [sample.run() for _ in range(args.steps)]
    cores = os.cpu_count()
    per_tok = sum(times) / (rows * len(times))
    value = 1.0 / per_tok
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_tok * wl.N * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name} N={wl.N} H={wl.H} V={wl.V} bf16 inputs, mean",
                   "sample_tokens_per_step": rows, "extrapolated": "ms_per_step = per-token time x N"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} tokens per step of {wl.N}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def end_to_end(torch, stream, step, dev_in, host_in, loss, host_loss, steps, barrier):
    """Milliseconds per step of `steps` steps, each fed from the host: copy the
    step's inputs (host_in, pinned) into one of two device buffer sets on a
    copy stream, run step(xb, yb, dlb) on `stream` once they have landed, and
    read the loss back. The copy of step i+1 waits only for step i-1 (the last
    user of its buffer set)."""
    dev = dev_in[0].device
    bufs = [dev_in, tuple(torch.empty_like(t) for t in dev_in)]
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
            step(xb=xb, yb=yb, dlb=dlb)
            free[i % 2].record(stream)
            host_loss.copy_(loss, non_blocking=True)

    run(2)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def run_ours(args):
    import torch
    import torch.distributed as dist

    import linear_cross_entropy_gemm_gb300 as F
    from linear_cross_entropy_gemm_gb300 import inputs as I

    rank, local, ws = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[WORKLOAD]
    if args.shape:
        n_, h_, v_ = (int(t) for t in args.shape.split(","))
        wl = wl.with_(name=f"{wl.name}-shape", N=n_, H=h_, V=v_)
    if args.dtype != wl.dtype:
        wl = wl.with_(dtype=args.dtype)
    tdt = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    pk = peaks()

    inp = I.make_inputs(wl)
    host_x = torch.from_numpy(inp.x.view(np.int16)).view(tdt).pin_memory()
    host_y = torch.from_numpy(inp.y).pin_memory()
    host_dl = torch.from_numpy(inp.dloss).pin_memory()
    x = host_x.to(dev)
    W = torch.from_numpy(inp.W.view(np.int16)).view(tdt).to(dev)
    y = host_y.to(dev)
    dloss = host_dl.to(dev)
    opts = dict(ignore_index=wl.ignore_index, label_smoothing=wl.label_smoothing,
                lse_square_scale=wl.lse_square_scale, logit_scale=wl.logit_scale,
                reduction=wl.reduction)
    N, H, V = wl.N, wl.H, wl.V
    from linear_cross_entropy_gemm_gb300 import tuning
    tune = None
    fkw, bkw = {}, {"bwd_vocab_block": args.bwd_vocab_block}
    if args.autotune:
        res = tuning.autotune(x, W, None, y, dloss=dloss, reps=3, **opts)
        fkw, bkw = res.config.forward_kwargs(), res.config.backward_kwargs()
        tune = res.as_dict()
    bvb = bkw["bwd_vocab_block"]
    bv_used = bvb or tuning.library_default_block(N, V)
    forms_used = {gm: F.resolved_gemm_form(N, H, V, (fkw if gm == "fwd_lse" else bkw).get(
        "gemm_form", "default"), gemm=gm, bwd_vocab_block=bvb) for gm in F.GEMMS}
    fws = torch.empty(F.flce_workspace_size(N, H, V, "forward", **opts), dtype=torch.uint8, device=dev)
    bws = torch.empty(F.flce_workspace_size(N, H, V, "backward", bwd_vocab_block=bvb,
                                            **opts), dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dx = torch.empty(N, H, dtype=tdt, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ftr, btr = F.KernelTrace(8), F.KernelTrace(256)
    host_loss = torch.empty(1, dtype=torch.float32).pin_memory()

    def step(trace=False, xb=x, yb=y, dlb=dloss):
        F.flce_forward(xb, W, None, yb, workspace=fws, out=(loss, lse),
                       trace=ftr if trace else None, **opts, **fkw)
        F.flce_backward(dlb, lse, xb, W, None, yb, workspace=bws, out=(dx, dW, None),
                        trace=btr if trace else None, **opts, **bkw)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()

    # ---- device-timed steps (inputs resident), L2 flushed between steps
    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    per_kernel = {}
    launches = 0
    barrier()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step(trace=True)
        ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        for name, ms in ftr.launches() + btr.launches():
            per_kernel.setdefault(name, []).append(ms)
            launches += 1
    barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), ws, dev)

    # ---- stored-probability backward (no logits recompute), same timing rules
    stored = None
    if not args.no_stored_mode:
        saved = torch.empty(F.flce_saved_size(N, H, V, input_fp16=args.dtype == "fp16", **opts),
                            dtype=torch.uint8, device=dev)

        def step_stored(trace=False):
            F.flce_forward(x, W, None, y, workspace=fws, out=(loss, lse), saved=saved,
                           trace=ftr if trace else None, **opts, **fkw)
            F.flce_backward(dloss, lse, x, W, None, y, workspace=bws, out=(dx, dW, None),
                            saved=saved, trace=btr if trace else None, **opts, **bkw)

        for _ in range(args.warmup):
            step_stored()
        barrier()
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        sk = {}
        for i in range(args.steps):
            flush.zero_()
            sev[i][0].record(stream)
            step_stored(trace=True)
            sev[i][1].record(stream)
            torch.cuda.synchronize(dev)
            for name, kms in ftr.launches() + btr.launches():
                sk.setdefault(name, []).append(kms)
        barrier()
        sms = max_over_ranks(sum(a.elapsed_time(b) for a, b in sev) / args.steps, ws, dev)
        stored = {"ms_per_step": sms, "value": ws * N / (sms * 1e-3), "unit": "tokens/s",
                  "tflops_6nhv": 6.0 * N * H * V / (sms * 1e-3) / 1e12,
                  "saved_bytes": saved.numel(),
                  "kernels": {("bwd_convert" if k == "bwd_dlogits" else
                               "fwd_lse_store" if k == "fwd_lse" else k):
                              {"launches_per_step": len(v) // args.steps,
                               "ms_per_step": sum(v) / args.steps} for k, v in sorted(sk.items())},
                  "note": "flce_forward_store/flce_backward_store: fp16 tile probabilities "
                          "kept from the forward, no logits recompute (6NHV flops)"}
        del saved

    # ---- end to end through the C ABI with host buffers. Every step's inputs
    # are copied from pinned host memory and its loss read back inside the
    # timed region; step i+1's copy runs on a side stream while step i
    # computes (two device input buffers), so the copies overlap the kernels.
    e2e_ms = end_to_end(torch, stream, step, (x, y, dloss), (host_x, host_y, host_dl), loss,
                        host_loss, args.steps, barrier)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)

    # ---- roofline of the dominant kernel
    flops_per = {"fwd_lse": 2.0 * N * H * V, "bwd_dlogits": 2.0 * N * H * V,
                 "bwd_dw": 2.0 * N * H * V, "bwd_dx": 2.0 * N * H * V}
    totals = {k: sum(v) for k, v in per_kernel.items()}
    dom = max(totals, key=totals.get)
    steps_ = args.steps
    dom_ms_per_step = totals[dom] / steps_
    tensor_dom = dom in flops_per
    if tensor_dom:
        achieved = flops_per[dom] / (dom_ms_per_step * 1e-3) / 1e12
        peak = pk["bf16_sus"]
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": f"bf16 sustained, {pk['src']}",
                "launches_per_step": len(per_kernel[dom]) // steps_,
                "ms_per_step": dom_ms_per_step,
                "algorithmic_flops_per_step": flops_per[dom],
                "traffic": (TRAFFIC_PER_LAUNCH.get(dom) if (N, H, V) == (8192, 4096, 128256)
                            and args.dtype == "bf16"
                            and bv_used == tuning.library_default_block(N, V)
                            and forms_used == {"fwd_lse": "wide", "bwd_dlogits": "wide",
                                               "bwd_dw": "wide", "bwd_dx": "pair"}
                            and os.environ.get("FLCE_RASTER", "1") != "0" else None),
                "traffic_unit": "bytes per launch (ncu dram read + write)"}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": pk["hbm"],
                "unit": "GB/s", "frac": None, "traffic": None}
    tflops = 8.0 * N * H * V / (ms * 1e-3) / 1e12
    value = ws * N / (ms * 1e-3)
    kern = {k: {"launches_per_step": len(v) // steps_, "ms_per_step": sum(v) / steps_,
                "share": sum(v) / sum(totals.values())} for k, v in sorted(per_kernel.items())}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / (ws * N / (PAGES_MS * 1e-3)) if args.dtype == "bf16" and
                        (N, H, V) == (8192, 4096, 128256) else None),
        "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": f"{wl.name}: N={N} H={H} V={V} {args.dtype}, mean, no bias, dloss=1",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "flushed (256 MiB write) before each timed step, outside the events",
                   "bwd_vocab_block": bv_used, "dW_dtype": "fp32",
                   "gemm_form": forms_used,
                   "N": N, "H": H, "V": V},
        "tflops_8nhv": tflops, "frac_bf16_peak_8nhv": tflops / pk["bf16_sus"],
        "tflops_6nhv_useful": tflops * 0.75,
        "roofline": roof,
        "kernels": kern,
        "gpu_launches": launches,
        "e2e": {"value": ws * N / (e2e_ms * 1e-3), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": host_x.numel() * 2 + host_y.numel() * 8 + host_dl.numel() * 4,
                "d2h_bytes_per_step": 4},
        "clocks": clk,
        "wall_s_timed": wall,
        "stored_mode": stored,
    }
    if tune is not None:
        line["autotune"] = tune
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="", help="N,H,V override (profiling captures only)")
    ap.add_argument("--no-stored-mode", action="store_true")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"],
                    help="operand type (the headline workload is bf16; fp16 is a side measurement)")
    ap.add_argument("--autotune", action="store_true",
                    help="time the GEMM forms and backward vocabulary blocks first and run the "
                         "fastest (tuning.autotune); the table goes into the JSON line")
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
