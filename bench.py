#!/usr/bin/env python
"""Benchmark: quantized GEMV weight GB/s of a Qwen3-4B-shaped Q8_0 decode step on one GB300.

One step is one decode pass over the projections of a Qwen3-4B-shaped dense model in Q8_0:
36 layers x (attn_q 4096x2560, attn_k 1024x2560, attn_v 1024x2560, attn_output 2560x4096,
ffn_gate 9728x2560, ffn_up 9728x2560, ffn_down 2560x9728) plus the tied output head
151936x2560: 4.27 GB of distinct raw GGUF blocks per step (far larger than the 129 MB L2, so
every step streams its weights from HBM).  Every layer holds its own copy of the synthetic
weight bytes at its own address.  Projections that read the same input share one launch
(qgemv_multi: q, k, v; gate, up), so a step is 36 x 4 + 1 = 145 GEMV launches.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--tokens T] [--sections main|all]
    python bench.py --impl reference ...   # the CPU oracle, timed on the host cores

Prints ONE JSON line (rank 0).  ``value`` is weight bytes / device time with everything
resident in HBM; ``e2e`` is the same metric through the public binding with the step's input
activations copied from pinned host memory and the head's logits copied back, every step.
The step is captured once in a CUDA graph and replayed.
With ``--sections all`` a ``detail`` object adds T = 4 / 16, per-projection times, the
K-quant and Q4_0 shapes, the MoE layer and the T = 512 prefill GEMM.  Multi-GPU: replicas only (each rank runs the
same step on its own GPU; no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gguf_synth as gs  # noqa: E402

LAYERS = 36
PROJ = [n for n in gs.QWEN3_4B_PROJ if n != "output_tied"]
HEAD = "output_tied"
METRIC = "quantized GEMV weight GB/s, Qwen3-4B-shaped Q8_0 decode step (36 layers + tied head)"
UNIT = "GB/s"
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--tokens", type=int, default=1, help="token columns T of the headline step (1..16)")
    p.add_argument("--layers", type=int, default=LAYERS)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--weights", choices=["static", "ordered"], default="static",
                   help="static: the weights are immutable parameters, so each GEMV may start streaming "
                        "them before its predecessor ends (qg_set_static_weights); ordered: every launch "
                        "waits for its predecessor before it reads anything")
    p.add_argument("--sections", choices=["main", "all", "gemm", "moe", "moe1", "moe8", "moe512", "kquant", "proj", "head"], default="all",
                   help="main: the headline line only; all: plus the detail object; gemm / moe / kquant / "
                        "proj: only that detail section, printed as its own JSON line (for profiling runs)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "of measured"
    return 6800.0, 1900.0, "of fallback"


def workload_config(args, layers=None):
    layers = args.layers if layers is None else layers
    return {
        "workload": f"qwen3-4b-shaped Q8_0 decode projections, {layers} layers x 7 + tied head 151936x2560, "
                    f"T={args.tokens}",
        "weights": "Q8_0 raw GGUF blocks (d = f16(|N(0,1)|*0.02), codes uniform [-127,127])",
        "activations": "f32 N(0,1), token-major [T][N]",
        "tokens": args.tokens,
        "layers": layers,
        "launches_per_step": 4 * layers + 1,
        "weight_bytes_per_step": step_weight_bytes(layers),
        "l2": "inputs larger than L2: every step streams its own 4.27 GB of distinct weights",
        "parallelism": f"replicas x{args.gpus}",
        "weights_mode": getattr(args, "weights", "static"),
    }


def step_weight_bytes(layers):
    per_layer = sum(gs.tensor_bytes(gs.Q8_0, *gs.QWEN3_4B_PROJ[n]) for n in PROJ)
    return layers * per_layer + gs.tensor_bytes(gs.Q8_0, *gs.QWEN3_4B_PROJ[HEAD])


def step_act_bytes(layers, T):
    per_layer = sum(T * (m + n) * 4 for (m, n) in (gs.QWEN3_4B_PROJ[p] for p in PROJ))
    m, n = gs.QWEN3_4B_PROJ[HEAD]
    return layers * per_layer + T * (m + n) * 4


# ---- CPU oracle (baseline leg and the reference arm) ------------------------------------------

def oracle_sample():
    """A bounded sample of the step for the oracle: every projection of one layer with its own
    weights, plus the first 1/8 of the tied head's rows (T = 1)."""
    items = []
    for i, name in enumerate(PROJ + [HEAD]):
        M, N = gs.QWEN3_4B_PROJ[name]
        if name == HEAD:
            M = M // 8
        w = gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=100 + i)
        items.append((M, N, w))
    xs = {N: gs.activations(1, N, seed=0) for N in {it[1] for it in items}}
    return items, xs


def time_oracle(items, xs, threads, min_seconds):
    import oracle

    nbytes = sum(it[2].nbytes for it in items)
    done, t0 = 0, time.perf_counter()
    while True:
        for M, N, w in items:
            oracle.gemv(gs.Q8_0, w, M, N, xs[N], threads=threads)
        done += nbytes
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return done / el / 1e9, el, done


def cpu_threads():
    return os.cpu_count() or 1


def sample_text():
    return ("oracle (plain C, f64 accumulation) over one layer's 7 Q8_0 projections + the first 18992 rows "
            "of the tied head, T=1, repeated for >= 10 s; OpenMP rows over all host cores")


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    items, xs = oracle_sample()
    threads = cpu_threads()
    nbytes = sum(it[2].nbytes for it in items)
    for _ in range(args.warmup):
        for M, N, w in items:
            oracle.gemv(gs.Q8_0, w, M, N, xs[N], threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for M, N, w in items:
            oracle.gemv(gs.Q8_0, w, M, N, xs[N], threads=threads)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    cfg = workload_config(args)
    cfg["sample"] = sample_text().replace(", repeated for >= 10 s", "")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": cfg["sample"]},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- clocks -----------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.rows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            self.rows.append(parts)

    def summary(self, t0, t1):
        """Samples whose timestamps fall in [t0, t1] (host wall clock); all samples if none do."""
        def ts(r):
            whole, _, frac = r[0].partition(".")
            try:
                return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
            except ValueError:
                return 0.0
        rows = [r for r in self.rows if t0 - 0.15 <= ts(r) <= t1 + 0.15]
        window = "timed"
        if not rows:
            rows, window = self.rows, "whole run"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        pw = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "window": window,
                "power_w_median": statistics.median(pw) if pw else None}


# ---- GPU arm ----------------------------------------------------------------------------------

def profiled_traffic():
    """DRAM bytes per launch of the headline kernel from the committed ncu summary, when that
    summary was taken on the current sources of that kernel (same hash); else None."""
    path = os.path.join(ROOT, "profiles", "qgemv_q8_0_qwen3_4b_decode_t1.md")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    traffic, sha = None, None
    for line in open(path):
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1])
        if line.startswith("kernel_sources_sha256:"):
            sha = line.split(":", 1)[1].strip()
    return traffic if (sha == want and traffic) else None


def kernel_source_hash():
    """Hash of the headline kernel's sources: its translation unit and the headers it includes."""
    csrc = os.path.join(ROOT, "gguf_block_dequant_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in ("qg_gemv1.cu", "qg_gemv.cu", "qg_decode.cuh", "qg_common.cuh", "qg_pipe.cuh",
                                              "qg_host.h")]
    files.append(os.path.join(ROOT, "include", "ggufdq.h"))
    h = hashlib.sha256()
    for path in files:
        h.update(os.path.basename(path).encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


class Decode:
    """Device-resident weights and buffers of the decode step."""

    def __init__(self, torch, qg, layers, T, dev):
        self.torch, self.qg, self.T, self.layers = torch, qg, T, layers
        self.w = {}
        for i, name in enumerate(PROJ):
            M, N = gs.QWEN3_4B_PROJ[name]
            host = torch.from_numpy(gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=100 + i))
            base = host.to(dev)
            self.w[name] = [base] + [base.clone() for _ in range(layers - 1)]
            del host
        M, N = gs.QWEN3_4B_PROJ[HEAD]
        self.w[HEAD] = [torch.from_numpy(gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=107)).to(dev)]
        self.Ns = sorted({n for (_, n) in gs.QWEN3_4B_PROJ.values()})
        self.x = {N: torch.from_numpy(gs.activations(16, N, seed=0)).to(dev) for N in self.Ns}
        self.y = {name: torch.empty((16, gs.QWEN3_4B_PROJ[name][0]), dtype=torch.float32, device=dev)
                  for name in gs.QWEN3_4B_PROJ}

    def gemv(self, name, wt, T):
        M, N = gs.QWEN3_4B_PROJ[name]
        if T == 1:
            self.qg.qgemv(gs.Q8_0, wt, self.x[N], M, N, self.y[name])
        else:
            self.qg.qgemv_t(gs.Q8_0, wt, self.x[N], self.y[name], M, N, T)

    def multi(self, names, l, T):
        N = gs.QWEN3_4B_PROJ[names[0]][1]
        self.qg.qgemv_multi(gs.Q8_0, [self.w[n][l] for n in names], [self.y[n] for n in names], self.x[N], N, T)

    def step(self, T=None):
        T = self.T if T is None else T
        for l in range(self.layers):
            self.multi(("attn_q", "attn_k", "attn_v"), l, T)
            self.gemv("attn_output", self.w["attn_output"][l], T)
            self.multi(("ffn_gate", "ffn_up"), l, T)
            self.gemv("ffn_down", self.w["ffn_down"][l], T)
        self.gemv(HEAD, self.w[HEAD][0], T)


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        fn()  # first call outside capture: per-device setup (attributes, driver entry points)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    stream.synchronize()
    return g


def time_graph(torch, g, stream, steps, warmup):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def run_section(args):
    """One detail section alone (no headline measurement), for short profiling runs."""
    import torch

    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build as qbuild

    torch.cuda.set_device(0)
    qbuild.build()
    qg.load()
    hbm, _, _ = peaks()
    stream = torch.cuda.Stream()
    qg.set_static_weights(args.weights == "static", stream)
    if args.sections == "gemm":
        res = run_gemm(torch, qg, stream, reps=args.steps, warmup=args.warmup)
    elif args.sections == "moe":
        res = run_moe(torch, qg, stream, hbm, reps=args.steps, warmup=args.warmup)
    elif args.sections == "moe1":  # one expert pool, one token: a small case for profiling
        res = run_moe(torch, qg, stream, hbm, layers=1, reps=args.steps, warmup=args.warmup, Ts=(1,))
    elif args.sections == "moe8":  # one expert pool, eight tokens: a small case for profiling
        res = run_moe(torch, qg, stream, hbm, layers=1, reps=args.steps, warmup=args.warmup, Ts=(8,))
    elif args.sections == "moe512":  # one expert pool, 512 tokens: a small case for profiling
        res = run_moe(torch, qg, stream, hbm, layers=1, reps=args.steps, warmup=args.warmup, Ts=(512,))
    elif args.sections == "kquant":
        res = run_kquant(torch, qg, stream, hbm, reps=args.steps, warmup=args.warmup)
    elif args.sections == "head":
        D = Decode(torch, qg, 1, 1, torch.device("cuda", 0))
        res = run_head_steps(torch, qg, D, stream, hbm, reps=args.steps, warmup=args.warmup)
    else:
        D = Decode(torch, qg, args.layers, args.tokens, torch.device("cuda", 0))
        res = run_projections(torch, D, stream, hbm, reps=args.steps, warmup=args.warmup)
    print(json.dumps({"section": args.sections, "result": res}), flush=True)
    return 0


def max_over_ranks(torch, dist, el, device):
    """The job's time: every rank contributes its own elapsed seconds and gets the slowest."""
    t = torch.tensor([el], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_rank_step, world, steps, el):
    """Whole-job throughput: the bytes every rank streamed over the slowest rank's time."""
    return bytes_per_rank_step * world * steps / el / 1e9


def run_ours(args):
    import torch

    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build as qbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0 or world == 1:
        qbuild.build()
    if world > 1:
        dist.barrier()
    qg.load()
    hbm, bf16, peak_src = peaks()
    T = args.tokens
    D = Decode(torch, qg, args.layers, T, dev)
    stream = torch.cuda.Stream(device=dev)
    wbytes = step_weight_bytes(args.layers)
    abytes = step_act_bytes(args.layers, T)
    launches = 4 * args.layers + 1

    qg.set_static_weights(args.weights == "static", stream)
    g = capture(torch, lambda: D.step(T), stream)
    if qg.device_status() != 0:
        raise RuntimeError("device status set after the first step")

    def timed():
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        smi_id = vis.split(",")[torch.cuda.current_device()] if vis else str(torch.cuda.current_device())
        sampler = ClockSampler(smi_id)
        time_graph(torch, g, stream, 0, args.warmup)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        h0 = time.time()
        el = time_graph(torch, g, stream, args.steps, 0)
        torch.cuda.synchronize()
        h1 = time.time()
        sampler.stop()
        return el, sampler.summary(h0, h1)

    el, clocks = timed()
    if any(r in BAD_REASONS for r in clocks.get("reasons", [])):
        el, clocks = timed()  # measured once more, as the timing rules ask
        clocks["remeasured"] = True
    if world > 1:
        el = max_over_ranks(torch, dist, el, dev)
    value = job_gbps(wbytes, world, args.steps, el)
    achieved = (wbytes + abytes) / (el / args.steps) / 1e9  # every launch in the step is this kernel

    # end to end: pinned host activations in, head logits out, every step
    hx = {N: D.x[N][:T].cpu().pin_memory() for N in D.Ns}
    hy = torch.empty((T, gs.QWEN3_4B_PROJ[HEAD][0]), dtype=torch.float32).pin_memory()

    def e2e_step():
        for N in D.Ns:
            D.x[N][:T].copy_(hx[N], non_blocking=True)
        g.replay()
        hy.copy_(D.y[HEAD][:T], non_blocking=True)

    e2e_steps = max(10, args.steps // 4)
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
    el_e2e = e0.elapsed_time(e1) / 1e3
    h2d = sum(T * N * 4 for N in D.Ns)
    d2h = T * gs.QWEN3_4B_PROJ[HEAD][0] * 4
    if qg.device_status() != 0:
        raise RuntimeError("device status set during the benchmark")

    detail = None
    if args.sections == "all" and rank == 0:
        detail = run_detail(torch, qg, D, stream, args, hbm)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        items, xs = oracle_sample()
        v, secs, done = time_oracle(items, xs, cpu_threads(), 10.0)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": sample_text(), "seconds": round(secs, 2), "bytes": done}

    if rank == 0:
        traffic = profiled_traffic()
        cfg = workload_config(args)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "kernel": ("qgemv1_kernel<Q8_0> (one token)" if T == 1 else "qgemv_kernel<Q8_0,T=%d>" % T), "achieved": round(achieved, 2),
                         "peak": hbm, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": traffic,
                         "algorithmic_bytes_per_launch": round((wbytes + abytes) / launches, 1)},
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": {"value": round(wbytes * e2e_steps / el_e2e / 1e9, 2), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(el_e2e / e2e_steps * 1e3, 4)},
            "gpu_launches": launches * args.steps,
        }
        if detail is not None:
            line["detail"] = detail
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_detail(torch, qg, D, stream, args, hbm):
    """Secondary numbers: T = 4 / 8 / 16 steps, per-projection T = 1 times, K-quant shapes, MoE."""
    out = {}
    wbytes = step_weight_bytes(args.layers)
    other = "ordered" if args.weights == "static" else "static"
    prev = qg.set_static_weights(other == "static", stream)
    g = capture(torch, lambda: D.step(args.tokens), stream)
    qg.set_static_weights(prev, stream)
    steps = max(20, args.steps // 4)
    el = time_graph(torch, g, stream, steps, 3)
    gbs = wbytes * steps / el / 1e9
    out[f"decode_step_T{args.tokens}_{other}_weights"] = {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                                                         "us_per_step": round(el / steps * 1e6, 1)}
    del g
    for T in (4, 8, 16):
        if T == args.tokens:
            continue
        g = capture(torch, lambda T=T: D.step(T), stream)
        steps = max(20, args.steps // 8)
        el = time_graph(torch, g, stream, steps, 3)
        gbs = wbytes * steps / el / 1e9
        out[f"decode_step_T{T}"] = {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                                    "us_per_step": round(el / steps * 1e6, 1),
                                    "tokens_per_s": round(T * steps / el, 1)}
        del g
    out["q8_0_T1_per_projection"] = run_projections(torch, D, stream, hbm)
    out["kquant"] = run_kquant(torch, qg, stream, hbm)
    out["head_steps"] = run_head_steps(torch, qg, D, stream, hbm)
    out["moe_layer"] = run_moe(torch, qg, stream, hbm)
    out["prefill_gemm"] = run_gemm(torch, qg, stream)
    return out


def run_gemm(torch, qg, stream, reps=10, warmup=3):
    """Prefill dequant-GEMM, Q8_0, T = 512: 9728x2560 and 2560x9728 (tcgen05, bf16 operands,
    f32 accumulation), each call = X f32 -> bf16 conversion + the GEMM kernel, rotating over
    weight copies that exceed 3x L2."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _, bf16_peak, src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    T = 512
    for M, N in ((9728, 2560), (2560, 9728)):
        b = gs.tensor_bytes(gs.Q8_0, M, N)
        R = max(2, -(-3 * l2 // b))
        base = torch.from_numpy(gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=500)).to(dev)
        ws_w = [base] + [base.clone() for _ in range(R - 1)]
        x = torch.from_numpy(gs.activations(T, N, seed=0, stream=501)).to(dev)
        y = torch.empty((T, M), dtype=torch.float32, device=dev)
        ws = torch.empty(qg.qgemm_workspace_size(gs.Q8_0, M, N, T), dtype=torch.uint8, device=dev)

        def calls():
            for w in ws_w:
                qg.qgemm(gs.Q8_0, w, x, y, M, N, T, ws)
        g = capture(torch, calls, stream)
        el = time_graph(torch, g, stream, reps, warmup)
        n = reps * R
        us = el / n * 1e6
        flop = 2.0 * M * N * T
        tf = flop / (us * 1e-6) / 1e12
        res[f"q8_0_{M}x{N}_T{T}"] = {"us": round(us, 2), "TFLOP/s": round(tf, 1),
                                     "frac_bf16_peak": round(tf / bf16_peak, 4), "peak_source": src,
                                     "weight_GB/s": round(b / (us * 1e-6) / 1e9, 1),
                                     # X -> bf16, the GEMM, and (when tiles are split over CTAs) the part sums
                                     "launches_per_call": 2 if (M // 128) * ((T + 255) // 256) % 152 == 0 else 3}
        del g
    if qg.device_status() != 0:
        raise RuntimeError("device status set in the GEMM benchmark")
    return res


def run_moe(torch, qg, stream, hbm, layers=8, reps=50, warmup=3, Ts=(1, 8, 512)):
    """Qwen3-30B-A3B-shaped MoE layer in Q8_0 (H 2048, F 768, 128 experts, top-8): one
    moe_layer call per layer, each layer with its own expert pool and its own input tokens,
    rotating over `layers` pools (8 x 641 MB, far above L2)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    H, F, E, k = gs.MOE_H, gs.MOE_F, gs.MOE_E, gs.MOE_K
    go, uo, do, stride = gs.moe_expert_record_layout(H, F, gs.Q8_0)
    base = torch.from_numpy(gs.moe_experts(E, H, F, gs.Q8_0, seed=0).reshape(-1)).to(dev)
    pools = [base] + [base.clone() for _ in range(layers - 1)]
    wr = [torch.from_numpy(gs.router_weights(E, H, seed=l)).to(dev) for l in range(layers)]
    res = {}
    for T in Ts:
        xn = [torch.from_numpy(gs.activations(T, H, seed=l, stream=40)).to(dev) for l in range(layers)]
        x = torch.from_numpy(gs.activations(T, H, seed=0, stream=41)).to(dev)
        ids = torch.zeros((layers, T, k), dtype=torch.int32, device=dev)
        wts = torch.zeros((layers, T, k), dtype=torch.float32, device=dev)
        act = torch.zeros((T * k, F), dtype=torch.float32, device=dev)
        ws = torch.zeros(qg.moe_workspace_size(T, k, E, H, F), dtype=torch.uint8, device=dev)

        def calls():
            for l in range(layers):
                p = pools[l]
                qg.moe_layer(gs.Q8_0, xn[l], wr[l], p[go:], p[uo:], p[do:], stride, None, E, T, H, F, E, k,
                             ids[l], wts[l], act, x, ws)
        g = capture(torch, calls, stream)
        r = max(3, reps // 10) if T > 16 else reps
        el = time_graph(torch, g, stream, r, warmup)
        n = r * layers
        us = el / n * 1e6
        uniq = [len(np.unique(ids[l].cpu().numpy())) for l in range(layers)]
        U = float(np.mean(uniq))
        nbytes = U * stride + E * H * 4 + T * H * 4 * 3 + 2 * T * k * 4
        roof_us = nbytes / (hbm * 1e9) * 1e6
        res[f"T{T}"] = {"us_per_layer": round(us, 2), "unique_experts": round(U, 2),
                        "bytes_per_layer": int(nbytes), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                        "roofline_us": round(roof_us, 2), "frac_of_roofline": round(roof_us / us, 4),
                        "launches_per_layer": 1 if T == 1 else 4 if T <= 16 else 6,
                        "tokens_per_s": round(T / (us * 1e-6), 1),
                        "path": ("one cooperative launch: router, top-k, gate/up, down + combine" if T == 1 else
                                 "CUDA cores, grouped per expert" if T <= 16 else "tcgen05 grouped per expert (bf16)")}
        del g
        if qg.device_status() != 0:
            raise RuntimeError("device status set in the MoE benchmark")
    return res


def run_projections(torch, D, stream, hbm, reps=20, warmup=3):
    """One projection at a time (T = 1), rotating over its layer copies."""
    per = {}
    for name in PROJ + [HEAD]:
        M, N = gs.QWEN3_4B_PROJ[name]
        copies = D.w[name]
        g = capture(torch, lambda name=name, copies=copies: [D.gemv(name, c, 1) for c in copies], stream)
        el = time_graph(torch, g, stream, reps, warmup)
        n = reps * len(copies)
        b = gs.tensor_bytes(gs.Q8_0, M, N)
        per[name] = {"us": round(el / n * 1e6, 2), "GB/s": round(b * n / el / 1e9, 1),
                     "frac_hbm": round(b * n / el / 1e9 / hbm, 4)}
        del g
    return per


def run_kquant(torch, qg, stream, hbm, reps=10, warmup=3):
    """Q4_K / Q6_K 17408x5120 and 5120x17408, Q4_0 2112x2816, Q8_0 1024x1024 at T in {1, 8},
    each rotating over enough weight copies to exceed 3x L2."""
    dev = torch.device("cuda", torch.cuda.current_device())
    res = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cases = [(gs.Q4_K, 17408, 5120), (gs.Q4_K, 5120, 17408), (gs.Q6_K, 17408, 5120), (gs.Q6_K, 5120, 17408),
             (gs.Q4_0, 2112, 2816), (gs.Q8_0, 1024, 1024)]
    for qt, M, N in cases:
        b = gs.tensor_bytes(qt, M, N)
        R = max(2, -(-3 * l2 // b))
        base = torch.from_numpy(gs.quant_blocks(qt, M, N, seed=0, stream=200 + qt)).to(dev)
        ws = [base] + [base.clone() for _ in range(R - 1)]
        x = torch.from_numpy(gs.activations(8, N, seed=0)).to(dev)
        y = torch.empty((8, M), dtype=torch.float32, device=dev)
        for T in (1, 8):
            def calls(T=T):
                for w in ws:
                    if T == 1:
                        qg.qgemv(qt, w, x, M, N, y)
                    else:
                        qg.qgemv_t(qt, w, x, y, M, N, T)
            g = capture(torch, calls, stream)
            el = time_graph(torch, g, stream, reps, warmup)
            n = reps * R
            key = f"{gs.TYPE_NAME[qt]}_{M}x{N}_T{T}"
            res[key] = {"us": round(el / n * 1e6, 2), "GB/s": round(b * n / el / 1e9, 1),
                        "frac_hbm": round(b * n / el / 1e9 / hbm, 4), "copies": R}
            del g
        del ws, base
    res["Q8_0_1024x1024_T1_batched"] = run_batched(torch, qg, stream, hbm, l2, reps, warmup, gs.Q8_0, 1024, 1024, 208)
    res["Q4_0_2112x2816_T1_batched"] = run_batched(torch, qg, stream, hbm, l2, reps, warmup, gs.Q4_0, 2112, 2816, 209)
    return res


def run_head_steps(torch, qg, D, stream, hbm, reps=10, warmup=3):
    """The steps on either side of the GEMV chain: the Gemma-shaped Q6_K tied head 262144 x 2816
    (606 MB, above L2) alone and with its argmax, the Qwen3 Q8_0 head with its argmax, a
    16-token embedding gather from the Qwen3 table and the RMSNorm of one token."""
    dev = torch.device("cuda", torch.cuda.current_device())
    res = {}

    def timed(fn, n_calls):
        g = capture(torch, fn, stream)
        el = time_graph(torch, g, stream, reps, warmup)
        del g
        return el / (reps * n_calls)

    V6, N6 = 262144, 2816
    w6 = torch.from_numpy(gs.quant_blocks(gs.Q6_K, V6, N6, seed=0, stream=214)).to(dev)
    b6 = gs.tensor_bytes(gs.Q6_K, V6, N6)
    x6 = torch.from_numpy(gs.activations(1, N6, seed=0)).to(dev)
    lg6 = torch.empty((1, V6), dtype=torch.float32, device=dev)
    ids = torch.empty(16, dtype=torch.int32, device=dev)
    t = timed(lambda: [qg.qgemv(gs.Q6_K, w6, x6, V6, N6, lg6) for _ in range(2)], 2)
    res["q6_k_head_262144x2816_T1"] = {"us": round(t * 1e6, 2), "GB/s": round(b6 / t / 1e9, 1),
                                       "frac_hbm": round(b6 / t / 1e9 / hbm, 4)}
    t = timed(lambda: [qg.head_argmax(gs.Q6_K, w6, x6, V6, N6, 1, lg6, ids) for _ in range(2)], 2)
    res["q6_k_head_argmax_262144x2816_T1"] = {"us": round(t * 1e6, 2), "GB/s": round(b6 / t / 1e9, 1),
                                              "frac_hbm": round(b6 / t / 1e9 / hbm, 4), "d2h_bytes": 4}
    del w6
    M, N = gs.QWEN3_4B_PROJ[HEAD]
    wh = D.w[HEAD][0]
    bh = gs.tensor_bytes(gs.Q8_0, M, N)
    xh = D.x[N]
    lg = torch.empty((1, M), dtype=torch.float32, device=dev)
    t = timed(lambda: [qg.head_argmax(gs.Q8_0, wh, xh, M, N, 1, lg, ids) for _ in range(2)], 2)
    res["q8_0_head_argmax_151936x2560_T1"] = {"us": round(t * 1e6, 2), "GB/s": round(bh / t / 1e9, 1),
                                              "frac_hbm": round(bh / t / 1e9 / hbm, 4), "d2h_bytes": 4,
                                              "logits_d2h_bytes_saved": M * 4}
    tok = torch.from_numpy(np.random.default_rng(0).integers(0, M, 16).astype(np.int32)).to(dev)
    emb = torch.empty((16, N), dtype=torch.float32, device=dev)
    t = timed(lambda: [qg.embed_rows(gs.Q8_0, wh, M, N, tok, emb) for _ in range(8)], 8)
    res["q8_0_embed_16_rows_of_151936x2560"] = {"us": round(t * 1e6, 2), "bytes_read": 16 * gs.row_bytes(gs.Q8_0, N)}
    wn = torch.ones(N, dtype=torch.float32, device=dev)
    yn = torch.empty((1, N), dtype=torch.float32, device=dev)
    t = timed(lambda: [qg.rmsnorm(xh[:1], wn, 1e-6, yn) for _ in range(8)], 8)
    res["rmsnorm_1x2560"] = {"us": round(t * 1e6, 2)}
    return res


def run_batched(torch, qg, stream, hbm, l2, reps, warmup, qt, M, N, sid):
    """Small matrices (the 1.1 MB Q8_0 1024x1024, the 3.3 MB Q4_0 2112x2816) are below what one
    launch needs to fill HBM: a launch costs about as much as the edges around it.  Independent
    matrices over the same input in one qgemv_multi launch (4 per launch) show the rate the
    kernel reaches once the launch edges are shared."""
    dev = torch.device("cuda", torch.cuda.current_device())
    b = gs.tensor_bytes(qt, M, N)
    R = max(8, -(-3 * l2 // b))
    R -= R % 4
    base = torch.from_numpy(gs.quant_blocks(qt, M, N, seed=0, stream=sid)).to(dev)
    ws = [base] + [base.clone() for _ in range(R - 1)]
    x = torch.from_numpy(gs.activations(1, N, seed=0)).to(dev)
    ys = [torch.empty((1, M), dtype=torch.float32, device=dev) for _ in range(4)]

    def calls():
        for i in range(0, R, 4):
            qg.qgemv_multi(qt, ws[i:i + 4], ys, x, N, 1)
    g = capture(torch, calls, stream)
    el = time_graph(torch, g, stream, reps, warmup)
    n = reps * R
    del g
    return {"matrices_per_launch": 4, "us_per_matrix": round(el / n * 1e6, 3), "GB/s": round(b * n / el / 1e9, 1),
            "frac_hbm": round(b * n / el / 1e9 / hbm, 4), "copies": R}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.sections not in ("main", "all"):
        return run_section(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
