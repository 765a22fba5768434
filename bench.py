"""Benchmark of the sparse MoE FFN layer (one step = one whole moe_forward:
routing, grouping, grouped gate/up + SiLU, grouped down + weight, combine),
with the model's bf16 weights.

    python bench.py [--config decode] [--steps K] [--warmup W] [--gpus N]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed

Prints ONE JSON line (rank 0).  Under torchrun every rank runs an independent
replica of the same per-GPU workload (the layer has no cross-GPU step), and
the value is the tokens of all ranks over the slowest rank's time; with
--gpus N > 1 and no torchrun environment, bench.py starts the N ranks itself
through torch.distributed.run.  The decode line also carries a "prefill"
record: the prefill workload timed in the same run (its grouped GEMMs are
the tensor-bound half of the metric), through moe_forward and through
moe_forward_prepared (fp16 down weights made once at load).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_moe_ffn_gb300.inputs import CONFIGS, MoEShape, make_inputs, to_device  # noqa: E402

METRIC = "MoE-layer tokens/s & TFLOPS (decode: % HBM roofline; prefill: % bf16 peak)"
UNIT = "tokens/s"
WORKLOADS = {
    "tiny": "tiny MoE layer: N=16, H=64, E=6, top-2, I=128, norm_topk_prob=True",
    "decode": "Qwen3-30B-A3B-shaped MoE decode: N=64, H=2048, E=128, top-8, I=768, "
              "norm_topk_prob=True",
    "prefill": "Qwen3-30B-A3B-shaped MoE prefill: N=8192, H=2048, E=128, top-8, I=768, "
               "norm_topk_prob=True",
    "talker": "talker-style MoE with shared expert: N=2048, H=2048, E=64, top-6, I=768, "
              "I_s=2048, norm_topk_prob=False",
    "skewed": "skewed-routing stress: N=16384, H=2048, E=128, top-8, I=768, 8 hot experts",
}
BOUND = {"tiny": "hbm", "decode": "hbm", "talker": "hbm", "prefill": "tensor", "skewed": "tensor"}
STAGES = ("route", "align", "gather", "gate_up", "down", "shared", "combine")
# kernel sources behind each stage (the GEMM stages run the one-CTA, the
# sparse-block or the CTA-pair kernel depending on the batch)
GEMM_SOURCES = ("grouped_gemm.cu", "sparse_gemm.cu", "pair_gemm.cu", "gemm_common.cuh", "pair_rows.cuh")
SOURCES = {"route": ("router.cu",), "align": ("align.cu",), "gather": ("grouped_gemm.cu",),
           "gate_up": GEMM_SOURCES, "down": GEMM_SOURCES, "shared": GEMM_SOURCES,
           "combine": ("combine.cu", "pair_rows.cuh")}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ------------------------------------------------------------------ helpers


def check_status(ws, what):
    """A run whose kernels recorded a device-side failure reports no number."""
    from sparse_moe_ffn_gb300 import binding
    status = binding.moe_read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after the {what}: "
                           f"{binding.moe_status_string(status)}")

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"])}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(stage):
    h = hashlib.sha256()
    for f in sorted({*SOURCES[stage], "ptx.cuh", "kernels.cuh"}):
        with open(os.path.join(ROOT, "sparse_moe_ffn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(stage, config):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{config}/{stage}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != source_hash(stage):
        return None
    return rec.get("bytes_per_launch")


def algorithmic_work(shape: MoEShape, touched: int):
    """Per-stage algorithmic bytes and FLOPs of one layer call (padding rows,
    re-reads and the act/ypair intermediates are overheads, not work).  The
    shared expert runs inside the gate/up and down launches (its chunks are
    virtual experts), so its work is counted there; the shared stage has no
    launches of its own."""
    N, H, E, k, I, Is = shape.N, shape.H, shape.E, shape.k, shape.I, shape.I_s
    P = N * k
    b = {
        "route": E * H * 2 + N * H * 2 + P * 8,
        "align": P * 4 + P * 4,
        "gather": 0,  # x rows copied into expert order: an intermediate, not work
        "gate_up": touched * 2 * I * H * 2 + N * H * 2 + P * I * 2 + 2 * Is * H * 2 + N * Is * 2,
        "down": (touched * H * I * 2 + P * I * 2 + P * H * 2 + P * 4
                 + ((Is * H * 2 + N * Is * 2 + N * H * 2) if Is else 0)),
        "shared": 0,
        "combine": P * H * 2 + N * H * 2 + (N * H * 2 if Is else 0),
    }
    f = {
        "route": 2 * N * H * (E + (1 if Is else 0)),
        "align": 0,
        "gather": 0,
        "gate_up": 4 * H * I * P + 4 * H * Is * N,
        "down": 2 * H * I * P + 2 * H * Is * N,
        "shared": 0,
        "combine": 0,
    }
    layer_flops = 2 * N * H * E + 6 * H * I * P + (N * (6 * H * Is + 2 * H) if Is else 0)
    layer_bytes = (touched * 3 * H * I * 2 + E * H * 2 + ((3 * H * Is * 2 + 2 * H) if Is else 0)
                   + 2 * N * H * 2 + P * 8)
    return b, f, layer_flops, layer_bytes


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons (read only)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.4)  # nvidia-smi start-up
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(", ") for ln in self.file if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        import datetime
        def ts(s):
            try:
                return datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        parsed = []
        for r in rows:
            if len(r) < 10:
                continue
            t = ts(r[0])
            try:
                sm, smax = float(r[2]), float(r[3])
            except ValueError:
                continue
            parsed.append((t, sm, smax, r[6:10]))
        if not parsed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [p for p in parsed if p[0] is not None and t0 - 0.03 <= p[0] <= t1 + 0.03]
        use = inside or parsed
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in use for i, v in enumerate(p[3])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(p[1] for p in use),
                "sm_max_mhz": max(p[2] for p in use), "reasons": reasons,
                "samples": len(use), "window": "timed region" if inside else "around the run"}


# --------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- CPU oracle leg

def oracle_bits(cpu_inputs):
    import oracle
    return {n: oracle.bf16_bits(t.to(torch.bfloat16)) for n, t in cpu_inputs.items()}


def time_oracle(shape, bits, target_s: float):
    """Tokens/s of the fp64 oracle on a bounded sample of the workload: whole
    passes over the first min(N, 64) tokens until target_s has elapsed."""
    import numpy as np
    import oracle
    rows = np.arange(min(shape.N, 64), dtype=np.int64)
    threads = oracle.hardware_threads()
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_forward(bits, shape.k, shape.norm_topk_prob, rows=rows, nthreads=threads)
        done += len(rows)
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return done / el, threads, done, el


# ----------------------------------------------------------------- our arm

def time_prefill(args, device, peaks):
    """The prefill workload (N=8192) timed on this GPU through both forms of
    the down weights: layer ms per call (median of five rounds that
    alternate the two forms, so that a clock or thermal drift hits both
    alike), and the grouped GEMMs (gate/up and down, from the start of
    gate/up to the end of down, with no event between them so that their
    hand-off overlap is kept) against the bf16 tensor peak."""
    from sparse_moe_ffn_gb300 import binding

    shape = CONFIGS["prefill"]
    cpu = make_inputs(shape, seed=args.seed)
    d_bf16 = to_device(cpu, device)
    del cpu
    forms = {"bf16_down": d_bf16, "f16_down_prepared": binding.prepare_weights(d_bf16)}
    ws = binding.alloc_workspace(shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s, device)
    out = torch.empty((shape.N, shape.H), dtype=torch.bfloat16, device=device)
    steps, warm, rounds = args.prefill_steps, 5, 5
    _, sflops, layer_flops, _ = algorithmic_work(shape, shape.E)
    gemm_flops = sflops["gate_up"] + sflops["down"]
    rec = {"workload": WORKLOADS["prefill"], "steps": steps, "warmup": warm, "rounds": rounds}

    def step(d):
        binding.moe_forward(d["x"], d["router"], d["w_gate"], d["w_up"], d["w_down"], shape.k,
                            shape.norm_topk_prob, None, out=out, workspace=ws)

    for form, d in forms.items():
        for _ in range(warm):
            step(d)
    torch.cuda.synchronize()
    check_status(ws, "prefill warm-up")
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    t0 = time.time()
    times = {form: [] for form in forms}
    for _ in range(rounds):
        for form, d in forms.items():
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(steps):
                step(d)
            s1.record()
            torch.cuda.synchronize()
            times[form].append(s0.elapsed_time(s1) / steps)
    t1 = time.time()
    check_status(ws, "prefill timed steps")
    for form, d in forms.items():
        ms = statistics.median(times[form])
        # grouped GEMMs: events before gate/up and after down only
        evs = []
        for _ in range(steps):
            e = [None] * (len(STAGES) + 1)
            e[STAGES.index("gate_up")] = torch.cuda.Event(enable_timing=True)
            e[STAGES.index("shared")] = torch.cuda.Event(enable_timing=True)
            evs.append(e)
            binding.set_stage_events(e)
            step(d)
        binding.set_stage_events(None)
        torch.cuda.synchronize()
        gemm_ms = statistics.mean(e[STAGES.index("gate_up")].elapsed_time(e[STAGES.index("shared")])
                                  for e in evs)
        achieved = gemm_flops / (gemm_ms / 1e3) / 1e12
        rec[form] = {
            "entry": "moe_forward_prepared" if form.startswith("f16") else "moe_forward",
            "ms_per_step": round(ms, 5), "ms_per_round": [round(t, 5) for t in times[form]],
            "tokens_per_s": round(shape.N / (ms / 1e3), 1),
            "tflops": round(layer_flops / (ms / 1e3) / 1e12, 2),
            "layer_frac_of_bf16_peak": round(layer_flops / (ms / 1e3) / 1e12
                                             / peaks["bf16_tflops"], 4),
            "roofline": {"bound": "tensor", "kernel": "gate_up+down", "achieved":
                         round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "kernel_ms": round(gemm_ms, 5), "algorithmic_per_launch": gemm_flops,
                         "window": "CUDA events before the gate/up launch and after the down "
                                   "launch, a separate pass of the same steps"},
        }
    check_status(ws, "prefill GEMM pass")
    rec["clocks"] = ClockSampler.summarize(sampler.stop(), t0, t1)
    del forms, d_bf16, ws, out
    torch.cuda.empty_cache()
    return rec


def run_ours(args, world, rank, local):
    from sparse_moe_ffn_gb300 import binding

    shape = CONFIGS[args.config]
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cpu = make_inputs(shape, seed=args.seed)
    # model load: the model's bf16 weights to the device (moe_forward takes
    # them as they are)
    d = to_device(cpu, device)
    if args.down_weights == "f16":  # informational runs of moe_forward_prepared
        d = binding.prepare_weights(d)
    shared = {n: d[n] for n in binding.SHARED_KEYS} if shape.I_s else None
    ws = binding.alloc_workspace(shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s, device)
    out = torch.empty((shape.N, shape.H), dtype=torch.bfloat16, device=device)

    def step():
        binding.moe_forward(d["x"], d["router"], d["w_gate"], d["w_up"], d["w_down"], shape.k,
                            shape.norm_topk_prob, shared, out=out, workspace=ws)

    # warm-up; the last warm-up step records every stage boundary to find the
    # dominant kernel.  The timed region runs the K steps with no stage events:
    # an event recorded between two launches removes the programmatic
    # dependent-launch overlap of the kernels around it (~15 us per decode
    # step).  A second pass of K steps then brackets the dominant kernel's
    # launches with events for the roofline; its duration there is an upper
    # bound (the launch no longer overlaps its predecessor).
    nst = len(STAGES) + 1
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(nst)]
    for i in range(args.warmup):
        if i == args.warmup - 1:
            binding.set_stage_events(probe)
        step()
    binding.set_stage_events(None)
    torch.cuda.synchronize()
    check_status(ws, "warm-up")
    probe_ms = {s: probe[j].elapsed_time(probe[j + 1]) for j, s in enumerate(STAGES)}
    dom = max(("route", "gate_up", "down", "shared", "combine"), key=lambda s: probe_ms[s])
    j_dom = STAGES.index(dom)

    ev = [[None] * nst for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][j_dom] = torch.cuda.Event(enable_timing=True)
        ev[i][j_dom + 1] = torch.cuda.Event(enable_timing=True)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    launches0 = binding.moe_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for i in range(args.steps):
        step()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    launches = binding.moe_kernel_launch_count() - launches0
    clocks = ClockSampler.summarize(sampler.stop(), t0, t1)
    check_status(ws, "timed region")
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, world, device)
    # roofline pass: the same K steps, the dominant kernel bracketed by events
    for i in range(args.steps):
        binding.set_stage_events(ev[i])
        step()
    binding.set_stage_events(None)
    torch.cuda.synchronize()
    dom_ms = statistics.mean(ev[i][j_dom].elapsed_time(ev[i][j_dom + 1])
                             for i in range(args.steps))

    # routed experts that received rows (the shared expert's chunks follow them)
    touched = int((binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k,
                                           shape.I_s)["counts"][:shape.E] > 0).sum().item())
    sbytes, sflops, layer_flops, layer_bytes = algorithmic_work(shape, touched)
    ms_step = ms_max / args.steps
    value = shape.N * args.steps * world / (ms_max / 1e3)
    tflops = layer_flops * args.steps * world / (ms_max / 1e3) / 1e12

    # roofline of the dominant kernel (largest share of the step)
    peaks, peak_src = load_peaks()
    bound = BOUND[args.config]
    if bound == "tensor" and sflops[dom] == 0:
        bound = "hbm"
    if bound == "hbm":
        achieved = sbytes[dom] / (dom_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        achieved = sflops[dom] / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof.update(frac=round(achieved / roof["peak"], 4), traffic=measured_traffic(dom, args.config),
                kernel=dom, kernel_ms=round(dom_ms, 5), peak_source=f"{peak_src} (MEASURED_PEAKS.json)" if peak_src ==
                "measured" else "fallback", algorithmic_per_launch=(
                    sbytes[dom] if roof["bound"] == "hbm" else sflops[dom]),
                window=f"second pass of {args.steps} steps after the timed region, CUDA events "
                       "around the kernel's launch on its stream (the event removes the launch "
                       "overlap with the previous kernel, so kernel_ms is an upper bound)")

    # end to end through the public call with host buffers
    x_host = cpu["x"].to(torch.bfloat16).pin_memory()
    out_host = torch.empty((shape.N, shape.H), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(d["x"])
    weights = {n: t for n, t in d.items() if n != "x"}

    def e2e_step():
        binding.moe_forward_from_host(x_host, out_host, x_dev, out, weights, shape.k,
                                      shape.norm_topk_prob, ws)

    for _ in range(args.warmup):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(args.steps):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    barrier(world)
    check_status(ws, "end-to-end steps")
    e2e_ms = max_over_ranks(s2.elapsed_time(e2), world, device)
    e2e = {"value": round(shape.N * args.steps * world / (e2e_ms / 1e3), 1), "unit": UNIT,
           "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
           "d2h_bytes_per_step": out_host.numel() * out_host.element_size()}

    # the same steps through moe_forward_prepared (fp16 down weights made
    # once at load; information next to the bf16 headline)
    d16 = binding.prepare_weights(d)
    shared16 = {n: d16[n] for n in binding.SHARED_KEYS} if shape.I_s else None
    for _ in range(args.warmup):
        binding.moe_forward(d16["x"], d16["router"], d16["w_gate"], d16["w_up"], d16["w_down"],
                            shape.k, shape.norm_topk_prob, shared16, out=out, workspace=ws)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    for _ in range(args.steps):
        binding.moe_forward(d16["x"], d16["router"], d16["w_gate"], d16["w_up"], d16["w_down"],
                            shape.k, shape.norm_topk_prob, shared16, out=out, workspace=ws)
    p1.record()
    torch.cuda.synchronize()
    check_status(ws, "prepared-weight steps")
    prep_ms = p0.elapsed_time(p1) / args.steps
    prepared_rec = {"entry": "moe_forward_prepared", "ms_per_step": round(prep_ms, 5),
                    "tokens_per_s": round(shape.N / (prep_ms / 1e3), 1)}
    del d16, shared16

    # the decode loop under CUDA-graph replay (buckets 1, 2, 4, ... 128; this
    # workload's batch replays its own bucket), the step's activations copied
    # into the captured input each step
    graph_rec = None
    if shape.N <= binding.DECODE_BUCKETS[-1]:
        graphs = binding.ForwardGraphSet({n: t for n, t in d.items() if n != "x"}, shape.k,
                                         shape.norm_topk_prob)
        for _ in range(args.warmup):
            graphs(d["x"])
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            graphs(d["x"])
        g1.record()
        torch.cuda.synchronize()
        if graphs.read_device_status() != 0:
            raise RuntimeError("device status after the graph-replay steps")
        gms = g0.elapsed_time(g1) / args.steps
        graph_rec = {"us_per_step": round(gms * 1e3, 2),
                     "tokens_per_s": round(shape.N / (gms / 1e3), 1),
                     "bucket": graphs.bucket_of(shape.N), "buckets": list(graphs.buckets)}
        del graphs

    prefill_rec = None
    if rank == 0 and args.config == "decode" and not args.no_prefill:
        prefill_rec = time_prefill(args, device, peaks)

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, threads, rows, el = time_oracle(shape, oracle_bits(cpu), args.cpu_seconds)
        cpu_base = {"value": round(tps, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": f"fp64 C oracle, {rows} token rows (repeated passes over the "
                              f"first {min(shape.N, 64)} tokens of the same inputs), "
                              f"{el:.1f} s wall on {threads} threads"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, random init)",
        "config": workload_config(args, shape, world),
        "tflops": round(tflops, 2),
        "entry": ("moe_forward (bf16 weights, as the layer is defined)" if args.down_weights ==
                  "bf16" else "moe_forward_prepared (fp16 down weights made once at load)"),
        "prepared_down_weights": prepared_rec,
        "graph_replay": graph_rec,
        "stage_ms_warmup_probe": {s: round(v, 5) for s, v in probe_ms.items()},
        "experts_touched": touched,
        "roofline": roof,
        "cpu_baseline": cpu_base,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if prefill_rec is not None:
        line["prefill"] = prefill_rec
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ reference arm

def workload_config(args, shape, world) -> dict:
    """The `config` object of both arms' JSON lines (the same workload)."""
    return {"workload": WORKLOADS[args.config], "N": shape.N, "H": shape.H, "E": shape.E,
            "k": shape.k, "I": shape.I, "I_s": shape.I_s,
            "norm_topk_prob": shape.norm_topk_prob, "seed": args.seed,
            "l2": "inputs larger than L2 (expert weights "
                  f"{3 * shape.E * shape.H * shape.I * 2 / 1e9:.2f} GB > 129 MB)"
                  if shape.E * shape.H * shape.I * 6 > 129e6 else
                  "inputs smaller than L2 (not flushed: latency-bound case)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, world, rank):
    """The fp64 CPU oracle as the reference arm (host cores, bounded samples)."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    shape = CONFIGS[args.config]
    bits = oracle_bits(make_inputs(shape, seed=args.seed))
    threads = oracle.hardware_threads()
    # size each step's sample so that W + K steps take about two minutes
    probe = np.arange(min(shape.N, threads), dtype=np.int64)
    t = time.perf_counter()
    oracle.moe_forward(bits, shape.k, shape.norm_topk_prob, rows=probe, nthreads=threads)
    per_row = (time.perf_counter() - t) / len(probe)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(max(1, min(shape.N, budget / max(per_row, 1e-9))))
    rows = np.arange(n_rows, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.moe_forward(bits, shape.k, shape.norm_topk_prob, rows=rows, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.moe_forward(bits, shape.k, shape.norm_topk_prob, rows=rows, nthreads=threads)
    el = time.perf_counter() - t0
    value = n_rows * args.steps / el
    sample = (f"each step: the first {n_rows} of the {shape.N} tokens of the workload, fp64 C "
              f"oracle on {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, shape, world),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def spawn_ranks(n: int) -> int:
    """Runs this script under torch.distributed.run with n local ranks (the
    same arguments), and returns its exit code."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-steps", type=int, default=50)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--down-weights", default="bf16", choices=["bf16", "f16"],
                    help="form of the down weights of the timed steps: the model's bf16 "
                         "(moe_forward) or fp16 copies made at load (moe_forward_prepared)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # start the N ranks (one process per GPU) ourselves
        sys.exit(spawn_ranks(args.gpus))
    if args.gpus != int(os.environ.get("WORLD_SIZE", "1")):
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={os.environ.get('WORLD_SIZE', '1')}")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        from sparse_moe_ffn_gb300 import build as lib_build
        lib_build.build()
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
