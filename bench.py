"""Throughput of the W4A16 group-quantized matmul on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

Default workload: one-row decode through one feed-forward block's weights,
i.e. one step = the gate+up GEMV (M=1, K=5120, N=34816, group 128, z=8) and the
down GEMV (M=1, K=17408, N=5120), each on its own seeded synthetic input.
Metric: effective HBM GB/s = algorithmic bytes of the step (packed codes +
bf16 scales + zero points + x + y) / device time. Prompt workloads report
TFLOP/s (2*M*K*N) instead.

L2 is defeated by rotating over enough weight copies that one rotation moves
more than four times the 129 MB L2 (decode) ; the prompt GEMM is compute-bound
and runs on one copy.

Prints ONE JSON line (rank 0). Under torchrun with N > 1 every rank runs the
same workload on its own GPU (replicas: the matmul shards with no exchange);
value = all ranks' bytes / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.workloads import WORKLOADS, algorithmic_bytes, gateup_bytes, gemm_flops  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_hash() -> str:
    """Hash of the CUDA sources: a stored ncu traffic figure is only reported
    while the kernels it was measured on are unchanged."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_w4a16_group_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*"))):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(f, "rb") as fh:
                h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def stored_traffic(name: str):
    """DRAM bytes (read + write) per launch measured by ncu for `name`, or None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("bytes_per_launch", {}).get(name)
DEFAULT = "decode_ffn_m1"  # gate+up GEMV followed by the down GEMV


def parse_shape(spec: str) -> dict:
    """'M,N,K,G,sym|asym' -> an ad-hoc workload (profiling cases)."""
    m, n, k, g, s = spec.split(",")
    return dict(kind="gemm", M=int(m), N=int(n), K=int(k), group=int(g), sym=(s == "sym"), affine=(s == "affine"),
                scale_range=(0.005, 0.02), x_scale=1.0)


def step_parts(workload: str):
    """[(name, params)] of the calls one step makes."""
    if workload.startswith("shape:"):
        return [(workload, parse_shape(workload[len("shape:"):]))]
    if workload == DEFAULT:
        return [("decode_gateup_m1_k5120_n34816", WORKLOADS["decode_gateup_m1_k5120_n34816"]),
                ("decode_down_m1_k17408_n5120", WORKLOADS["decode_down_m1_k17408_n5120"])]
    return [(workload, WORKLOADS[workload])]


def part_units(w):
    """(units per call, metric unit, is_flops): FLOPs for the prompt regime
    (M > 32, tensor-bound), algorithmic bytes for decode (M <= 32, HBM-bound)."""
    aff = w.get("affine", False)
    if w["kind"] == "gateup":
        if w["M"] > 32:
            return gemm_flops(w["M"], 2 * w["N"], w["K"]), "TFLOP/s", True
        return gateup_bytes(w["M"], w["N"], w["K"], w["group"], w["sym"], aff), "GB/s", False
    if w["M"] > 32:
        return gemm_flops(w["M"], w["N"], w["K"]), "TFLOP/s", True
    return algorithmic_bytes(w["M"], w["N"], w["K"], w["group"], w["sym"], aff), "GB/s", False


def metric_name(workload):
    parts = step_parts(workload)
    if part_units(parts[0][1])[2]:
        if parts[0][1]["kind"] == "gateup":
            return "W4A16 fused gate/up GEMM TFLOP/s (M=4096, K=5120, 2x17408)"
        return "W4A16 GEMM TFLOP/s (M>32)"
    return "W4A16 GEMM eff. HBM GB/s (M=1..16)"


def new_problem(w):
    return synth.make_problem(w["M"], w["N"], w["K"], w["group"], w["sym"], scale_range=w["scale_range"],
                              x_scale=w["x_scale"], seed=0, gateup=w["kind"] == "gateup",
                              affine=w.get("affine", False))


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 - 0.3 <= t <= t1 + 0.3] or [r for _, r in self.rows[-5:]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: one process per GPU, no data exchange)
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (every rank calls this); x itself on one
    process. The timed region's length is the slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_step: float, steps: int, world: int, ms: float, scale: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (ms), in the metric's unit (scale 1e-9 for GB/s, 1e-12 for TFLOP/s)."""
    return world * units_per_step * steps / (ms * 1e-3) * scale


# ---------------------------------------------------------------------------
# CUDA arm
# ---------------------------------------------------------------------------
SPEC_HBM_GBS = 7900.0  # nominal HBM3e bandwidth of one GB300 (context beside the measured copy peak)


def quantiles(v):
    a = np.asarray(v, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90))}


class Workload:
    """One workload's device buffers (weights rotated over enough copies that
    L2 never holds the next call's weights) and the library calls of a step."""

    def __init__(self, name, args, dev, mode="y", topk_k=8, max_copies=None):
        import torch
        import gemm_w4a16_group_gb300 as w4
        self.torch, self.w4, self.args, self.mode, self.topk_k = torch, w4, args, mode, topk_k

        def up(a):
            a = np.ascontiguousarray(a)
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

        parts = []
        for pname, w in step_parts(name):
            p = new_problem(w)
            units, unit, is_flops = part_units(w)
            if mode == "argmax" and not is_flops:
                units -= 2 * w["M"] * w["N"]  # no logits written
            wbytes = algorithmic_bytes(1, w["N"], w["K"], w["group"], w["sym"], w.get("affine", False)) * \
                (2 if w["kind"] == "gateup" else 1)
            parts.append(dict(name=pname, w=w, p=p, units=units, unit=unit, is_flops=is_flops, wbytes=wbytes))
        total_w = sum(pt["wbytes"] for pt in parts)
        copies = 1 if parts[0]["is_flops"] else max(2, math.ceil(4 * L2_BYTES / total_w) + 1)
        if max_copies:
            copies = min(copies, max_copies)
        for pt in parts:
            p, w = pt["p"], pt["w"]
            zd = None if p["zeros"] is None else up(p["zeros"])
            if p["affine"] and w["kind"] == "gateup":
                packed = w4.repack_affine_gateup(up(p["qweight"]), up(p["scales"]), up(p["biases"]),
                                                 up(p["qweight_up"]), up(p["scales_up"]), up(p["biases_up"]), w["N"],
                                                 w["K"], w["group"])
            elif p["affine"]:
                packed = w4.repack_affine(up(p["qweight"]), up(p["scales"]), up(p["biases"]), w["N"], w["K"],
                                          w["group"])
            elif w["kind"] == "gateup":
                packed = w4.repack_gateup(up(p["qweight"]), up(p["scales"]), zd, up(p["qweight_up"]),
                                          up(p["scales_up"]), None if p["zeros_up"] is None else up(p["zeros_up"]),
                                          w["N"], w["K"], w["group"], w["sym"])
            else:
                packed = w4.repack(up(p["qweight"]), up(p["scales"]), zd, w["N"], w["K"], w["group"], w["sym"])
            pt["packed"] = [packed] + [packed.clone() for _ in range(copies - 1)]
            pt["x"] = up(p["x"])
            pt["y"] = torch.empty((w["M"], w["N"]), dtype=torch.bfloat16, device=dev)
            # affine form on the tcgen05 GEMM: the group sums of x, formed every call
            pt["xs"] = (torch.empty(w4.xsum_bytes(w["M"], w["K"], w["group"]) // 2, dtype=torch.bfloat16, device=dev)
                        if p["affine"] and (w["M"] > 32 or args.kernel == "tc") else None)
            pt["idx"] = torch.empty(w["M"], dtype=torch.int64, device=dev)
            pt["tk_idx"] = torch.empty((w["M"], topk_k), dtype=torch.int64, device=dev)
            pt["tk_val"] = torch.empty((w["M"], topk_k), dtype=torch.bfloat16, device=dev)
            pt["idx_host"] = torch.empty(w["M"], dtype=torch.int64).pin_memory()
            pt["x_host"] = torch.from_numpy(p["x"].view(np.int16)).pin_memory()
            pt["y_host"] = torch.empty((w["M"], w["N"]), dtype=torch.int16).pin_memory()
            del pt["p"]
        self.parts, self.copies, self.total_w = parts, copies, total_w

    def call(self, pt, c, s, x=None, y=None):
        w4, w, args = self.w4, pt["w"], self.args
        xin = pt["x"] if x is None else x
        if self.mode == "argmax" and w["kind"] != "gateup":
            # the greedy pick only: the logits are not stored
            w4.gemm_argmax(xin, pt["packed"][c], w["N"], w["K"], w["group"], w["sym"], stream=s,
                           index_out=pt["idx"])
            return
        if self.mode == "gemm_topk":
            w4.gemm_topk(xin, pt["packed"][c], w["N"], w["K"], w["group"], w["sym"], self.topk_k,
                         out=pt["y"] if y is None else y, index_out=pt["tk_idx"], values_out=pt["tk_val"], stream=s)
            return
        if self.mode == "topk":  # the selection alone, over logits already in pt["y"]
            w4.topk(pt["y"], self.topk_k, index_out=pt["tk_idx"], values_out=pt["tk_val"], stream=s)
            return
        if w.get("affine", False) and args.noalloc:
            w4.gemm_affine_noalloc(xin, pt["packed"][c], w["N"], w["K"], w["group"], out=pt["y"] if y is None else y,
                                   stream=s)
            return
        if w.get("affine", False):
            xs = None
            if pt["xs"] is not None:
                xs = w4.xsum(xin, w["K"], w["group"], out=pt["xs"], stream=s)
            fn = w4.gateup_silu_affine if w["kind"] == "gateup" else w4.gemm_affine
            fn(xin, pt["packed"][c], w["N"], w["K"], w["group"], xs, out=pt["y"] if y is None else y, stream=s)
            return
        fn = w4.gateup_silu if w["kind"] == "gateup" else w4.gemm
        fn(xin, pt["packed"][c], w["N"], w["K"], w["group"], w["sym"], out=pt["y"] if y is None else y, stream=s)

    def launches_per_call(self, pt):
        if self.mode == "argmax" and pt["w"]["kind"] != "gateup":
            return 3  # zero the keys, the GEMM, keys to indices
        if self.mode == "gemm_topk":
            return 2
        return 2 if pt["xs"] is not None else 1  # the affine tcgen05 GEMM's group-sum pre-pass

    def steps(self, first, n, s, only=None):
        for i in range(n):
            for j, pt in enumerate(self.parts):
                if only is None or j == only:
                    self.call(pt, (first + i) % self.copies, s)

    def capture(self, first, n, s, only=None):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=s):
            self.steps(first, n, s, only)
        return g


def timed(fn, s, world):
    """Milliseconds of fn()'s device work on stream s, CUDA events on s, a
    barrier and a synchronize on both sides."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    a.record(s)
    fn()
    b.record(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    return a.elapsed_time(b)


def measure(wl, nsteps, nwarm, s, world, eager=False, stats_ms=200.0, max_replays=400):
    """Exactly nsteps timed steps (one graph replay, or an eager loop) after
    nwarm untimed ones; per-call times from graphs of the same launches of
    each call alone; then the same graphs replayed again until each has run
    for stats_ms, for the median and the 10th / 90th percentiles."""
    import torch
    with torch.cuda.stream(s):
        wl.steps(0, nwarm, s)
    torch.cuda.synchronize()
    if eager:
        run_all = lambda: wl.steps(nwarm, nsteps, s)  # noqa: E731
        run_part = [lambda j=j: wl.steps(nwarm, nsteps, s, j) for j in range(len(wl.parts))]
    else:
        g_all = wl.capture(nwarm, nsteps, s)
        g_part = [wl.capture(nwarm, nsteps, s, j) for j in range(len(wl.parts))]
        for g in [g_all] + g_part:  # upload and run each graph once, untimed
            with torch.cuda.stream(s):
                g.replay()
        run_all = g_all.replay
        run_part = [g.replay for g in g_part]
    with torch.cuda.stream(s):
        ms = timed(run_all, s, world)
        per_call = [timed(run_part[j], s, world) / nsteps for j in range(len(wl.parts))]
        step_samples, call_samples = [], [[] for _ in wl.parts]
        while sum(step_samples) < stats_ms and len(step_samples) < max_replays:
            step_samples.append(timed(run_all, s, world) / nsteps)
        for j in range(len(wl.parts)):
            acc = 0.0
            while acc < stats_ms and len(call_samples[j]) < max_replays:
                t = timed(run_part[j], s, world)
                acc += t
                call_samples[j].append(t / nsteps)
    return {"ms": ms, "per_call_ms": per_call,
            "stats": {"replays": len(step_samples), "calls_per_replay": nsteps,
                      "ms_per_step": quantiles(step_samples),
                      "per_call_ms": [quantiles(c) for c in call_samples],
                      "replays_per_call": [len(c) for c in call_samples]}}


def secondary_block(args, dev, s, peaks):
    """The other headline numbers in the same run: the 4,096-row fused prompt
    GEMM (TFLOP/s against the bf16 burst peak), the 248,320-row head at 1 and
    5 rows (GB/s), the head's top-k, and the cuBLAS bf16 GEMM of the prompt's
    shape as a yardstick. Each: its per-call median and 10th / 90th
    percentiles over >= 200 ms of graph replays."""
    import torch
    out = {}

    def entry(wl, name, steps):
        m = measure(wl, steps, 3, s, 1)
        pt = wl.parts[0]
        q = m["stats"]["per_call_ms"][0]
        scale = 1e-12 if pt["is_flops"] else 1e-9
        val = pt["units"] / (q["median"] * 1e-3) * scale
        peak = peaks["bf16_tflops"] if pt["is_flops"] else peaks["hbm_gbs"]
        e = {"workload": name, "unit": pt["unit"], "value": round(val, 2), "per_call_ms": q,
             "calls_timed": sum(m["stats"]["replays_per_call"]) * steps,
             "roofline": {"bound": "tensor" if pt["is_flops"] else "hbm", "achieved": round(val, 2), "peak": peak,
                          "frac": round(val / peak, 4), "peak_src": peaks["src"] + (" bf16 burst" if pt["is_flops"]
                                                                                   else " copy")},
             "l2": (f"rotating {wl.copies} weight copies" if wl.copies > 1 else "compute-bound; one weight copy")}
        if not pt["is_flops"]:
            e["roofline"]["frac_of_spec"] = round(val / SPEC_HBM_GBS, 4)
        return e

    wl = Workload("prompt_gateup_m4096_k5120_n17408", args, dev)
    out["prompt_gateup_m4096_k5120_n17408"] = entry(wl, "prompt_gateup_m4096_k5120_n17408", 10)
    del wl
    for M in (1, 5):
        name = f"lm_head_m{M}_k5120_n248320"
        wl = Workload(name, args, dev)
        out[name] = entry(wl, name, 20)
        if M == 1:
            # the top-8 of the head's logits: the selection alone, and the GEMM with it
            wl.mode = "topk"
            m = measure(wl, 20, 3, s, 1)
            out["topk_k8_m1_n248320"] = {"unit": "us per call", "per_call_us": {
                k: round(v * 1e3, 3) for k, v in m["stats"]["per_call_ms"][0].items()}}
            wl.mode = "gemm_topk"
            m = measure(wl, 20, 3, s, 1)
            out["lm_head_topk8_m1_k5120_n248320"] = {"unit": "us per call", "per_call_us": {
                k: round(v * 1e3, 3) for k, v in m["stats"]["per_call_ms"][0].items()}}
        del wl
    torch.cuda.empty_cache()
    # yardstick: cuBLAS bf16 GEMM of the prompt's shape (a library call, not the path)
    Mp, Kp, Np = 4096, 5120, 2 * 17408
    a = torch.randn(Mp, Kp, device=dev, dtype=torch.bfloat16)
    b = torch.randn(Np, Kp, device=dev, dtype=torch.bfloat16)
    c = torch.empty(Mp, Np, device=dev, dtype=torch.bfloat16)
    with torch.cuda.stream(s):
        for _ in range(3):
            torch.matmul(a, b.t(), out=c)
        samples = []
        while sum(samples) < 200.0 and len(samples) < 400:
            samples.append(timed(lambda: torch.matmul(a, b.t(), out=c), s, 1))
    q = quantiles(samples)
    tf = 2.0 * Mp * Kp * Np / (q["median"] * 1e-3) * 1e-12
    out["cublas_bf16_m4096_k5120_n34816"] = {
        "unit": "TFLOP/s", "value": round(tf, 2), "per_call_ms": q, "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
        "note": "torch.matmul on bf16 operands (cuBLAS); a yardstick, not the W4A16 path"}
    del a, b, c
    torch.cuda.empty_cache()
    return out


def workload_config(args, world):
    """What the step computes (the same dict on both arms of a run)."""
    return {"workload": args.workload, "calls_per_step": [name for name, _ in step_parts(args.workload)],
            "kernel": args.kernel, "parallelism": f"replicas x{world}",
            "output": "argmax" if args.argmax else (f"y and top-{args.topk}" if args.topk else "y"),
            "entry": "w4a16_gemm_affine_noalloc" if args.noalloc else "default"}


def run_cuda(args, rank, world):
    import torch
    import gemm_w4a16_group_gb300 as w4

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w4.lib()
    w4.set_kernel_override({"auto": 0, "gemv": 1, "smallm": 2, "tc": 3, "xstaged": 4, "decode_tc": 5}[args.kernel])
    # decode calls stream their (read-only, already complete) weights while
    # the previous kernel finishes; x and y wait for it
    w4.set_programmatic_overlap(not args.no_overlap)
    peaks = load_peaks()

    if args.argmax and any(w.get("affine", False) for _, w in step_parts(args.workload)):
        raise SystemExit("--argmax takes the zero-point forms only")
    if args.noalloc and any(not w.get("affine", False) or w["kind"] != "gemm" for _, w in step_parts(args.workload)):
        raise SystemExit("--noalloc takes the affine plain-GEMM workloads only")
    if args.topk and any(w["kind"] == "gateup" or w.get("affine", False) for _, w in step_parts(args.workload)):
        raise SystemExit("--topk takes the zero-point GEMM workloads only")
    mode = "argmax" if args.argmax else ("gemm_topk" if args.topk else "y")
    wl = Workload(args.workload, args, dev, mode=mode, topk_k=args.topk or 8)
    parts = wl.parts
    torch.cuda.synchronize()

    # Device time comes from CUDA-graph replays: a decode server launches its
    # steps from graphs, and an eager Python loop would time the host's launch
    # path instead of the kernels (a decode call is ~10-30 us of device work).
    s = torch.cuda.Stream(device=dev) if not args.eager else torch.cuda.current_stream()
    nsteps, nwarm = args.steps, args.warmup
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    t_begin = time.time()
    m = measure(wl, nsteps, nwarm, s, world, eager=args.eager)
    t_end = time.time()
    ms, per_call_ms = m["ms"], m["per_call_ms"]
    copies = wl.copies
    launches_per_step = sum(wl.launches_per_call(pt) for pt in parts)
    if w4.kernel_status() != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the timed region")
    ms = max_over_ranks(ms, world)
    if world > 1:
        torch.distributed.barrier()

    # end to end, eager through the public API: pinned host x -> device, the
    # calls, device y -> pinned host, every step
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    xd = [torch.empty_like(pt["x"]) for pt in parts]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        e_start.record(s)
        for i in range(nsteps):
            for j, pt in enumerate(parts):
                xd[j].copy_(pt["x_host"].view(pt["x"].dtype), non_blocking=True)
                wl.call(pt, (nwarm + nsteps + i) % wl.copies, s, x=xd[j])
                if args.argmax and pt["w"]["kind"] != "gateup":
                    pt["idx_host"].copy_(pt["idx"], non_blocking=True)
                else:
                    pt["y_host"].copy_(pt["y"].view(torch.int16), non_blocking=True)
        e_stop.record(s)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop)
    e2e_ms = max_over_ranks(e2e_ms, world)

    secondary = None
    if rank == 0 and not args.no_secondary and args.workload == DEFAULT and world == 1:
        secondary = secondary_block(args, dev, s, peaks)
        if w4.kernel_status() != 0:
            raise RuntimeError("a kernel's bounded wait gave up during the secondary measurements")
    sampler.stop()
    if rank != 0:
        return None

    units_step = sum(pt["units"] for pt in parts)
    is_flops = parts[0]["is_flops"]
    scale = 1e-12 if is_flops else 1e-9
    value = job_value(units_step, nsteps, world, ms, scale)
    e2e = job_value(units_step, nsteps, world, e2e_ms, scale)
    dom = max(range(len(parts)), key=lambda j: parts[j]["units"])
    d = parts[dom]
    achieved = d["units"] / (per_call_ms[dom] * 1e-3) * scale
    peak = peaks["bf16_tflops"] if is_flops else peaks["hbm_gbs"]
    clocks = sampler.summary(t_begin, t_end)
    h2d = sum(pt["x"].numel() * 2 for pt in parts)
    d2h = sum(pt["idx"].numel() * 8 if args.argmax and pt["w"]["kind"] != "gateup" else pt["y"].numel() * 2
              for pt in parts)
    roof = {"bound": "tensor" if is_flops else "hbm", "kernel": d["name"],
            "achieved": round(achieved, 2), "peak": peak, "unit": d["unit"],
            "frac": round(achieved / peak, 4), "traffic": stored_traffic(d["name"]),
            "peak_src": peaks["src"] + (" bf16 burst" if is_flops else " copy")}
    if not is_flops:
        # the same figure against the nominal HBM3e bandwidth (the copy peak above is the denominator)
        roof["spec_peak"] = SPEC_HBM_GBS
        roof["frac_of_spec"] = round(achieved / SPEC_HBM_GBS, 4)
    line = {
        "metric": metric_name(args.workload), "value": round(value, 2), "unit": parts[0]["unit"],
        "n_gpus": world, "steps": nsteps, "warmup": nwarm, "ms_per_step": ms / nsteps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; shapes and distributions of the workload table)",
        "config": workload_config(args, world),
        "timing": {"l2": (f"rotating {copies} weight copies ({copies * wl.total_w / 1e6:.0f} MB > 4x L2)"
                          if copies > 1 else "compute-bound; one weight copy"),
                   "launch": ("eager" if args.eager else "cuda graph")
                   + ("" if args.no_overlap else ", programmatic overlap"),
                   "per_call_ms": [round(v, 5) for v in per_call_ms],
                   "repeats": ("value and ms_per_step: exactly --steps steps in one timed region; stats: the "
                               "same step graph (and each call's graph) replayed again until >= 200 ms each")},
        "roofline": roof,
        "stats": m["stats"],
        "e2e": {"value": round(e2e, 2), "unit": parts[0]["unit"], "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # kernels of this library per timed step
        "gpu_launches": nsteps * launches_per_step,
        "clocks": clocks,
    }
    if secondary is not None:
        line["secondary"] = secondary
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds, single_s=args.cpu_single_seconds)
    return line


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def _oracle_problems(workload):
    parts = step_parts(workload)
    return [(name, w, new_problem(w)) for name, w in parts], part_units(parts[0][1])[2]


def _oracle_step(probs, is_flops, frac=1.0, nthreads=0):
    """One step of the float64 oracle over every part of the workload: M rows
    (at most 16 for gate/up and where the unit is FLOP/s) by all output
    columns, or with `frac` < 1 that share of the columns, evenly spaced,
    through the oracle's sampled-output functions. Returns (seconds, units,
    description)."""
    import oracle
    seconds, units, descs, whole = 0.0, 0.0, [], True
    for name, w, p in probs:
        gate = w["kind"] == "gateup"
        M, N, K, G = w["M"], w["N"], w["K"], w["group"]
        rows = min(16, M) if (gate or is_flops) else M
        ncols = N if frac >= 1.0 else max(1, min(N, int(round(N * frac))))
        cols = np.arange(N, dtype=np.int64) if ncols == N else (np.arange(ncols, dtype=np.int64) * N) // ncols
        mi, ni = np.repeat(np.arange(rows, dtype=np.int64), ncols), np.tile(cols, rows)
        t0 = time.perf_counter()
        if gate and p["affine"]:
            oracle.gateup_silu_affine_at(p["x"], p["qweight"], p["scales"], p["biases"], p["qweight_up"],
                                         p["scales_up"], p["biases_up"], M, N, K, G, mi, ni, nthreads)
        elif gate:
            oracle.gateup_silu_at(p["x"], p["qweight"], p["scales"], p["zeros"], p["qweight_up"], p["scales_up"],
                                  p["zeros_up"], M, N, K, G, w["sym"], mi, ni, nthreads)
        elif ncols == N and p["affine"]:
            oracle.gemm_affine(p["x"][:rows], p["qweight"], p["scales"], p["biases"], rows, N, K, G, nthreads)
        elif ncols == N:
            oracle.gemm(p["x"][:rows], p["qweight"], p["scales"], p["zeros"], rows, N, K, G, w["sym"], nthreads)
        elif p["affine"]:
            oracle.gemm_affine_at(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, G, mi, ni, nthreads)
        else:
            oracle.gemm_at(p["x"], p["qweight"], p["scales"], p["zeros"], M, N, K, G, w["sym"], mi, ni, nthreads)
        seconds += time.perf_counter() - t0
        if is_flops:
            units += gemm_flops(rows, (2 if gate else 1) * ncols, K)
        elif gate:
            units += gateup_bytes(rows, ncols, K, G, w["sym"], p["affine"])
        else:
            units += algorithmic_bytes(rows, ncols, K, G, w["sym"], p["affine"])
        whole = whole and rows == M and ncols == N
        what = "gate/up column pairs" if gate else "columns"
        descs.append(f"{name}: {rows} of {M} rows x {ncols} of {N} {what}")
    return seconds, units, "whole step" if whole else "; ".join(descs)


def _oracle_result(units, seconds, reps, desc, is_flops):
    import oracle
    scale = 1e-12 if is_flops else 1e-9
    return {"value": units / seconds * scale, "unit": "TFLOP/s" if is_flops else "GB/s",
            "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{desc}, {reps} repetition(s), {seconds:.1f} s", "seconds": seconds, "reps": reps}


def cpu_baseline(workload, budget_s=10.0, single_s=5.0):
    """The float64 oracle as it stands, on every host core, over whole steps
    of the workload's bounded sample until `budget_s` seconds of oracle work;
    returns value in the workload's unit. `single_thread`: the same oracle on
    one thread, over an evenly spaced share of the output columns sized so
    that about `single_s` seconds of work run."""
    probs, is_flops = _oracle_problems(workload)
    seconds, units, reps = 0.0, 0.0, 0
    while True:  # at least one step
        s, u, desc = _oracle_step(probs, is_flops)
        seconds, units, reps = seconds + s, units + u, reps + 1
        if seconds >= budget_s:
            break
    res = _oracle_result(units, seconds, reps, desc, is_flops)
    if single_s > 0:
        probe, _, _ = _oracle_step(probs, is_flops, 0.01, nthreads=1)
        frac = min(1.0, max(1e-4, 0.01 * (single_s / 3.0) / max(probe, 1e-6)))
        s1, u1, r1 = 0.0, 0.0, 0
        while True:
            s, u, desc1 = _oracle_step(probs, is_flops, frac, nthreads=1)
            s1, u1, r1 = s1 + s, u1 + u, r1 + 1
            if s1 >= single_s:
                break
        one = _oracle_result(u1, s1, r1, desc1, is_flops)
        res["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1, "sample": one["sample"]}
    return res


REFERENCE_BUDGET_S = 120.0  # the reference arm's warm-up and timed steps together


def run_reference(args, rank, world):
    """The reference arm: the oracle on rank 0's host cores (the other ranks
    do no work), exactly --warmup untimed and --steps timed steps. When that
    many whole steps of the bounded sample would take more than two minutes,
    every step samples the same smaller share of the output columns."""
    if rank != 0:
        return None
    probs, is_flops = _oracle_problems(args.workload)
    probe, _, _ = _oracle_step(probs, is_flops)
    est = (args.warmup + args.steps) * probe
    frac = 1.0 if est <= REFERENCE_BUDGET_S else REFERENCE_BUDGET_S / est
    for _ in range(args.warmup):
        _oracle_step(probs, is_flops, frac)
    seconds, units, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        s, u, desc = _oracle_step(probs, is_flops, frac)
        seconds, units = seconds + s, units + u
    cb = _oracle_result(units, seconds, args.steps, desc, is_flops)
    return {"impl": "reference", "metric": metric_name(args.workload), "value": cb["value"],
            "unit": cb["unit"], "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cb["seconds"] * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, world),
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": cb["value"], "unit": cb["unit"], "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default=DEFAULT,
                    help=f"{DEFAULT} (default), one of {sorted(WORKLOADS)}, or shape:M,N,K,G,sym|asym")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps from Python instead of a CUDA graph")
    ap.add_argument("--no-overlap", action="store_true", help="no programmatic overlap between decode calls")
    ap.add_argument("--argmax", action="store_true",
                    help="time the fused argmax (w4a16_gemm_argmax, no logits stored) instead of the GEMM")
    ap.add_argument("--topk", type=int, default=0,
                    help="time w4a16_gemm_topk with this k (the GEMM, then the top-k of its logits)")
    ap.add_argument("--noalloc", action="store_true",
                    help="affine plain GEMM through w4a16_gemm_affine_noalloc (group sums in the library's array)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-single-seconds", type=float, default=5.0,
                    help="budget of the single-threaded oracle figure in cpu_baseline")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the prompt GEMM, LM head, top-k and cuBLAS figures of the default line")
    ap.add_argument("--print-source-hash", action="store_true", help="print the kernel source hash and exit")
    ap.add_argument("--kernel", default="auto", choices=["auto", "gemv", "smallm", "tc", "xstaged", "decode_tc"],
                    help="kernel override for A/B measurement (default: automatic choice)")
    args = ap.parse_args()
    if args.print_source_hash:
        print(kernel_source_hash())
        return
    args.warmup = max(3, args.warmup)
    if args.steps < 1:
        ap.error("--steps must be at least 1")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl")
        line = run_cuda(args, rank, world)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
