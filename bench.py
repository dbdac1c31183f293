"""Batch-1 NVFP4 decode-GEMV bench: weight-stream GB/s on the 4096x14336 MLP set.

One step = the three projections of one decoder MLP in NVFP4 at batch 1
(gate 14336x4096, up 14336x4096, down 4096x14336): gate and up read the same
x and are independent, so they run as one q4_gemv_grouped launch; down (whose
input a real MLP computes from gate and up) is its own q4_gemv launch after
it, chained by programmatic dependent launch.  The weights come from the seeded synthetic
recipe (W ~ N(0,0.02) with U(0.5,2) row scales, NVFP4 per 16, bf16 x).

L2 policy: inputs larger than L2 -- the step rotates through distinct copies
of the weight set totalling >= max(1 GiB, 4 x L2), so no step finds its
weights in the 129 MB L2.  The timed loop is one CUDA graph per rotation.

Output: one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.  Under torchrun (N > 1) every
rank runs its own replica (the path has no exchange step: replicas only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-stream GB/s and % of GB300 HBM peak for batch-1 4-bit dequant-GEMV"
WORKLOAD = "nvfp4_gemv_m1_mlp_4096x14336_set"
SET = [("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
CONFIG_ID = 5          # seed block of this workload's synthetic draws
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
DOMINANT = "gemv_tma_fp4<MT=1, NVFP4> group of 2 (gate and up, 2 x 14336x4096 in one launch)"
PROFILE = "gemv_tma_nvfp4_pair_2x14336x4096.md"
PROFILED_SOURCES = ("bit_block_quantized_gb300/csrc/gemv_tma.cu", "bit_block_quantized_gb300/csrc/q4_internal.cuh",
                    "bit_block_quantized_gb300/csrc/tma_map.cuh")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", action="store_true",
                    help="small profiling case: 4 grouped gate+up launches (2 x 14336x4096, 66 MB) on "
                         "one weight copy, no timing, no JSON line")
    ap.add_argument("--ncu-lanes-case", action="store_true",
                    help="small profiling case: one launch of each kernel of the next rows and of the FP4 "
                         "tensor-core path")
    ap.add_argument("--ncu-rows-case", action="store_true",
                    help="small profiling case: one launch of each remaining row's kernel on its own shape")
    ap.add_argument("--ncu-gemm-case", default=None, metavar="FMT:M",
                    help="small profiling case of the tensor-core small-batch GEMM: 3 launches of "
                         "FMT (nvfp4|q4k) at batch M on one 14336x4096 weight copy")
    ap.add_argument("--no-small-m", action="store_true",
                    help="skip the small-batch tensor-core GEMM measurements")
    ap.add_argument("--kernel-reps", type=int, default=0,
                    help="replays of each per-launch graph (~400 launches) for the roofline timing (0: 3)")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the per-row measurements of the other formats, dequant and repack")
    ap.add_argument("--fp4-slices", default="", choices=["", "gate_up", "all"],
                    help="run those launches of the step on the FP4 tensor-core kernel (Q4_FLAG_FP4_SLICES)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the Llama-7B layer-set sweep over every format at batch 1, 4 and 8")
    return ap.parse_args()


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha():
    h = hashlib.sha256()
    for rel in PROFILED_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, only if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", PROFILE)
    try:
        text = open(p).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != source_sha():
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 200 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"q4_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm

def build_workload(torch, q4, synth, copies=None, distinct=False):
    """Host NVFP4 tensors of the set + device copies rotating past L2.

    ``copies`` None sizes the rotation to max(1 GiB, 4 x L2); ``distinct``
    draws every copy from its own seeds (the parity test of the step uses it
    to tell the copies apart; the bench's copies hold the same weights)."""
    def draw(copy):
        out = []
        for i, (name, N, K) in enumerate(SET):
            layer = synth.make_layer("nvfp4", N, K, config=CONFIG_ID, matrix=i + 10 * copy, row_scale=True)
            xbits, _ = synth.draw_x(1, K, config=CONFIG_ID, matrix=0 if name in ("gate", "up") else i)
            out.append((name, N, K, layer, xbits))
        return out
    host = draw(0)
    set_bytes = sum(q4.q4_packed_bytes("nvfp4", N, K) for _, N, K in SET)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    if copies is None:
        copies = int(np.ceil(max(1 << 30, 4 * l2) / set_bytes))
    hosts = [host] + [draw(c) if distinct else host for c in range(1, copies)]
    dev = []
    for c in range(copies):
        mats = []
        for name, N, K, layer, xbits in hosts[c]:
            w = torch.from_numpy(layer["w"]).cuda()
            s = torch.from_numpy(layer["scales"]).cuda()
            mats.append((name, N, K, w, s, layer["scale2"]))
        dev.append(mats)
    xs = [torch.from_numpy(h[4].view(np.int16)).cuda().view(torch.bfloat16) for h in host]
    xs[1] = xs[0]                                   # gate and up read the same activations
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in SET]
    return hosts, dev, xs, ys, set_bytes, copies, l2


def mlp_auxes(q4, dev, fp4_slices=""):
    """One q4_aux per matrix of every copy (each carries its copy's scale2).
    ``fp4_slices``: "gate_up" or "all" sets Q4_FLAG_FP4_SLICES on those
    matrices (the FP4 tensor-core kernel instead of the TMA-fed one)."""
    def flags(i):
        on = fp4_slices == "all" or (fp4_slices == "gate_up" and i < 2)
        return q4.Q4_FLAG_FP4_SLICES if on else 0
    return [[q4.make_aux(scale2=m[5], fmt="nvfp4", flags=flags(i)) for i, m in enumerate(mats)] for mats in dev]


def mlp_step_fns(q4, dev, auxes, xs, ys):
    """The step's two calls on weight copy ``c``: q4_gemv_grouped(gate, up)
    with the shared x, then q4_gemv(down), both on stream ``s``.  ``auxes``
    is :func:`mlp_auxes` of ``dev``."""
    def gate_up(c, s):
        (_, N0, K0, w0, s0, _), (_, N1, K1, w1, s1, _) = dev[c][0], dev[c][1]
        q4.q4_gemv_grouped([("nvfp4", w0, s0, auxes[c][0], xs[0], ys[0], N0, K0),
                            ("nvfp4", w1, s1, auxes[c][1], xs[1], ys[1], N1, K1)], 1, stream=s)

    def down(c, s):
        _, N, K, w, sc, _ = dev[c][2]
        q4.q4_gemv("nvfp4", w, sc, auxes[c][2], xs[2], ys[2], 1, N, K, stream=s)

    def step(c, s):
        gate_up(c, s)
        down(c, s)
    return gate_up, down, step


MAX_STEPS_PER_GRAPH = 2048


SPIN_CYCLES = 100_000         # device spin before the timed region's start event (~50 us at 2 GHz)


def timed_graphs(torch, step, stream, steps, copies, cap=MAX_STEPS_PER_GRAPH):
    """CUDA graphs that together run exactly ``steps`` steps, step i on copy
    i % copies: one graph of all of them when steps <= cap (the usual case:
    no graph boundary inside the timed region, so programmatic dependent
    launch chains every launch to the next); otherwise a graph of a whole
    number of rotations, replayed, plus one graph for the remainder.
    Returns [(graph, replays)]."""
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i % copies, stream)
        return g
    if steps <= cap:
        return [(capture(steps), 1)]
    chunk = copies * max(1, cap // copies)
    plan = [(capture(chunk), steps // chunk)]
    if steps % chunk:
        plan.append((capture(steps % chunk), 1))
    return plan


def replay(plan):
    for g, n in plan:
        for _ in range(n):
            g.replay()


def run_ours(args, rank, world):
    import torch

    import bit_block_quantized_gb300 as q4
    import synth
    from bit_block_quantized_gb300 import build as q4build

    q4build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    hosts, dev, xs, ys, set_bytes, copies, l2 = build_workload(torch, q4, synth)
    host = hosts[0]
    auxes = mlp_auxes(q4, dev, args.fp4_slices)
    stream = torch.cuda.Stream()
    gate_up, down, step = mlp_step_fns(q4, dev, auxes, xs, ys)

    with torch.cuda.stream(stream):
        for c in range(copies):
            step(c, stream)
        gate_up(0, stream)
        path_gate_up = q4.q4_last_gemv_path()
        down(0, stream)
        path_down = q4.q4_last_gemv_path()
        torch.cuda.synchronize()
        warm = timed_graphs(torch, step, stream, max(args.warmup, 1), copies)
        timed = timed_graphs(torch, step, stream, args.steps, copies)
        # per-launch graphs for the roofline of each launch
        # ~400 launches per graph: like the timed steps, no graph boundary among the launches timed
        kern_rounds = max(1, 400 // copies)
        g_kern = []
        for fn in (gate_up, down):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(kern_rounds):
                    for c in range(copies):
                        fn(c, stream)
            g_kern.append(g)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # The clock sampler starts before the warm-up: its start-up (a process and a short sleep) left the
        # GPU idle just before the timed steps when it started after the barrier, and a 20-step region
        # (~0.5 ms) then began at lowered clocks (+1.5-2 us per step, measured).
        with ClockSampler(torch.cuda.current_device()) as clk:
            replay(warm)
            for g, _ in timed:           # uploads the timed graphs (untimed; their steps are extra warm-up)
                g.replay()
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            # A ~50 us device-side spin ahead of the start event: the host submits the timed graph while
            # it runs, so the region starts with the graph's first kernel already queued instead of
            # counting the host's graph-launch latency (~10-15 us, a whole step's worth at 20 steps).
            torch.cuda._sleep(SPIN_CYCLES)
            start.record(stream)
            replay(timed)
            end.record(stream)
            torch.cuda.synchronize()
        barrier()
        ms = start.elapsed_time(end)
        # per-kernel average launch duration (same stream, inputs > L2)
        kern_ms = []
        reps = args.kernel_reps if args.kernel_reps > 0 else 3
        for j in range(len(g_kern)):
            g_kern[j].replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g_kern[j].replay()
            b.record(stream)
            torch.cuda.synchronize()
            kern_ms.append(a.elapsed_time(b) / (reps * kern_rounds * copies))

    ms = max_over_ranks(ms, world, "cuda")

    # end to end through the public API: pinned host x in, y out, every step
    e2e = run_e2e(args, torch, q4, dev, auxes, host, stream)

    if rank != 0:
        return None
    peak, peak_kind = measured_hbm_peak()
    value = whole_job_gbps(world, set_bytes, args.steps, ms)
    gate_up_bytes = 2 * q4.q4_packed_bytes("nvfp4", 14336, 4096)
    down_bytes = q4.q4_packed_bytes("nvfp4", 4096, 14336)
    achieved = gate_up_bytes / (kern_ms[0] * 1e-3) / 1e9
    per_kernel = {"gate+up (one grouped launch)": {"us_per_launch": round(kern_ms[0] * 1e3, 3),
                                                   "GBps": round(gate_up_bytes / (kern_ms[0] * 1e-3) / 1e9, 1),
                                                   "path": path_gate_up},
                  "down": {"us_per_launch": round(kern_ms[1] * 1e3, 3),
                           "GBps": round(down_bytes / (kern_ms[1] * 1e-3) / 1e9, 1), "path": path_down}}
    x_bytes = 4096 * 2 + 14336 * 2
    y_bytes = sum(N * 4 for _, N, _ in SET)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded W ~ N(0,0.02) x U(0.5,2) rows, NVFP4 per 16; x ~ N(0,1) bf16)",
        "config": {"workload": WORKLOAD, "batch": 1, "fp4_slices": args.fp4_slices or "off",
                   "matrices": [f"{n} {N}x{K}" for n, N, K in SET],
                   "weight_bytes_per_step": set_bytes, "x_bytes_per_step": x_bytes,
                   "y_bytes_per_step": y_bytes,
                   "l2": f"inputs larger than L2: {copies} rotating copies of the set = "
                         f"{copies * set_bytes / 1e9:.2f} GB (L2 {l2 / 1e6:.0f} MB)",
                   "launch": "2 launches per step: q4_gemv_grouped(gate, up) (shared x) then q4_gemv(down), "
                             "chained by programmatic dependent launch; the timed steps are one CUDA graph "
                             f"(up to {MAX_STEPS_PER_GRAPH} steps per graph), step i on weight copy i % copies",
                   "warmup": "clock sampling starts, then the --warmup steps as a graph and one untimed replay of the timed graph "
                             "(its upload); a ~50 us device spin precedes the start event, so the host's submission of "
                             "the timed graph is not inside the region",
                   "parallelism": f"replicas x{world}"},
        "pct_of_hbm_peak": {"measured": round(value / world / peak, 4),
                            "nominal_7900": round(value / world / NOMINAL_HBM_GBS, 4)},
        "per_kernel": per_kernel,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "kernel": DOMINANT, "algorithmic_bytes_per_launch": gate_up_bytes,
                     "timing": "average launch duration: CUDA events on the launching stream around graphs of "
                               "~400 launches of this kernel over the rotating weight copies (no graph boundary "
                               "among them, as in the timed steps), after the timed region"},
        "tokens_equivalent_per_s": {"value": round(tokens_equivalent(ms / args.steps, world), 1),
                                    "layers": LAYERS,
                                    "note": "batch-1 decode of a model whose every layer is this MLP set, "
                                            "weight streaming only"},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_small_m:
        line["small_m_gemm"] = small_m_gemm(torch, q4, synth, peak)
    if not args.no_rows:
        line["other_rows"] = other_rows(torch, q4, synth, peak)
    if not args.no_sweep:
        line["layer_set_sweep"] = layer_set_sweep(torch, q4, peak)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, host)
        if not args.no_rows:
            line["cpu_baseline"]["rows"] = cpu_baseline_rows()
    return line


def max_over_ranks(value, world, device):
    """The largest of every rank's value: the job's time is its slowest rank's."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


LAYERS = 32   # decoder layers of the model whose every layer is this MLP set (the tokens-equivalent rate)


def tokens_equivalent(ms_per_step, world, layers=LAYERS):
    """Whole-job batch-1 tokens per second if every one of `layers` layers
    streamed this set once per token: world / (layers x step time)."""
    return world * 1000.0 / (layers * ms_per_step)


def whole_job_gbps(world, bytes_per_step, steps, ms):
    """Whole-job throughput: every rank streams the set `steps` times within
    the slowest rank's `ms` (replicas: per-rank work fixed as N grows)."""
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


def run_e2e(args, torch, q4, dev, auxes, host, stream):
    """Same metric through the public API with host buffers: every step copies
    the two activation vectors from pinned host memory (one copy), runs the
    grouped gate+up call and the down call, reads the three outputs back (one
    copy) and waits for them on the host.  The step is replayed as a CUDA
    graph of exactly those operations, as a decode loop would; the same step
    issued eagerly from Python is timed beside it."""
    K_gu, K_dn = SET[0][2], SET[2][2]
    x_h = torch.empty(K_gu + K_dn, dtype=torch.bfloat16).pin_memory()
    x_h[:K_gu].copy_(torch.from_numpy(host[0][4].view(np.int16)).view(torch.bfloat16).reshape(-1))
    x_h[K_gu:].copy_(torch.from_numpy(host[2][4].view(np.int16)).view(torch.bfloat16).reshape(-1))
    x_d = torch.empty_like(x_h, device="cuda")
    xd_gu, xd_dn = x_d[:K_gu].view(1, K_gu), x_d[K_gu:].view(1, K_dn)
    n_out = sum(N for _, N, _ in SET)
    y_h = torch.empty(n_out, dtype=torch.float32).pin_memory()
    y_d = torch.empty(n_out, dtype=torch.float32, device="cuda")
    offs = np.cumsum([0] + [N for _, N, _ in SET])
    ys_d = [y_d[offs[j]:offs[j + 1]].view(1, -1) for j in range(3)]
    copies = len(dev)
    n = args.e2e_steps

    def one(c):
        x_d.copy_(x_h, non_blocking=True)
        (_, N0, K0, w0, s0, _), (_, N1, K1, w1, s1, _), (_, N2, K2, w2, s2, _) = dev[c]
        q4.q4_gemv_grouped([("nvfp4", w0, s0, auxes[c][0], xd_gu, ys_d[0], N0, K0),
                            ("nvfp4", w1, s1, auxes[c][1], xd_gu, ys_d[1], N1, K1)], 1, stream=stream)
        q4.q4_gemv("nvfp4", w2, s2, auxes[c][2], xd_dn, ys_d[2], 1, N2, K2, stream=stream)
        y_h.copy_(y_d, non_blocking=True)

    with torch.cuda.stream(stream):
        for c in range(min(copies, 20)):
            one(c % copies)
            stream.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            one(i % copies)
            stream.synchronize()
        dt_eager = time.perf_counter() - t0
        graphs = []
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                one(c)
            graphs.append(g)
        for c in range(copies):
            graphs[c].replay()
            stream.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            graphs[i % copies].replay()
            stream.synchronize()
        dt = time.perf_counter() - t0
    set_bytes = sum(q4.q4_packed_bytes("nvfp4", N, K) for _, N, K in SET)
    return {"value": round(set_bytes * n / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": x_h.numel() * 2,
            "d2h_bytes_per_step": n_out * 4,
            "steps": n, "ms_per_step": dt * 1e3 / n,
            "eager": {"value": round(set_bytes * n / dt_eager / 1e9, 1), "ms_per_step": dt_eager * 1e3 / n},
            "note": "per step: one pinned H2D copy of both x vectors, q4_gemv_grouped(gate, up) + q4_gemv(down), "
                    "one D2H copy of the three y, host waits; replayed as one CUDA graph per weight copy "
                    "(eager: the same calls issued from Python each step)"}


# --------------------------------------------------------- oracle on host

def cpu_baseline(seconds, host=None, sample_rows=None):
    """The CPU oracle as it stands (single thread, f64 accumulation), timed on
    a bounded row sample of the same three matrices."""
    import oracle
    import synth
    oracle.build()
    if host is None:
        host = []
        for i, (name, N, K) in enumerate(SET):
            layer = synth.make_layer("nvfp4", N, K, config=CONFIG_ID, matrix=i, row_scale=True)
            xbits, _ = synth.draw_x(1, K, config=CONFIG_ID, matrix=0 if name in ("gate", "up") else i)
            host.append((name, N, K, layer, xbits))
    # calibrate: rows per second on a small probe, then size the sample
    name, N, K, layer, xbits = host[0]
    T = oracle.Tensor("nvfp4", N, K, layer["w"], layer["scales"], scale2=layer["scale2"])
    xf = oracle.bf16_bits_to_f32(xbits)
    t0 = time.perf_counter()
    oracle.gemv(T, xf, rows=np.arange(64))
    per_row_4096 = (time.perf_counter() - t0) / 64
    if sample_rows is None:
        frac = min(1.0, seconds / (per_row_4096 * (14336 + 14336 + 4096 * 3.5)))
    else:
        frac = sample_rows
    bytes_done, t_total, t_all, rows_done = 0, 0.0, 0.0, 0
    cores = os.cpu_count() or 1
    for name, N, K, layer, xbits in host:
        rows = np.arange(max(1, int(N * frac)))
        T = oracle.Tensor("nvfp4", N, K, layer["w"], layer["scales"], scale2=layer["scale2"])
        xf = oracle.bf16_bits_to_f32(xbits)
        t0 = time.perf_counter()
        oracle.gemv(T, xf, rows=rows)
        t_total += time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle_rows_all_cores(oracle, T, xf, rows, cores)
        t_all += time.perf_counter() - t0
        bytes_done += rows.size * (K // 2 + K // 16)
        rows_done += rows.size
    return {"value": round(bytes_done / t_total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows_done} rows ({frac:.3%}) of each of the 3 set matrices, batch 1, "
                      f"{t_total:.1f} s", "cpu": _cpu_name(),
            "all_cores": {"value": round(bytes_done / t_all / 1e9, 4), "unit": "GB/s", "cores": cores,
                          "kind": "oracle", "sample": f"the same rows split over {cores} host threads, {t_all:.1f} s",
                          "nproc": cores}}


def oracle_rows_all_cores(oracle, T, xf, rows, cores):
    """The oracle GEMV over ``rows``, split into chunks that run on ``cores``
    host threads (the C oracle releases the interpreter lock; each row's
    arithmetic is the oracle's own)."""
    from concurrent.futures import ThreadPoolExecutor
    chunks = np.array_split(np.asarray(rows), max(1, min(len(rows), cores * 4)))
    with ThreadPoolExecutor(cores) as ex:
        return list(ex.map(lambda r: oracle.gemv(T, xf, rows=r), chunks))


A16Q8_ROW = "f2 NVFP4 A16-Q8 GEMV (integer-exact)"

# The other rows' shapes and synthetic recipes (see other_rows), for the oracle beside each.
ORACLE_ROWS = [("a1 NVFP4 GEMV", "nvfp4", 14336, 4096, 4, 5, dict(row_scale=True), "bf16"),
               ("a2 Q4_K GEMV", "q4k", 4096, 4096, 1, 1, dict(), "f32"),
               ("a3 MXFP4 GEMV", "mxfp4", 4096, 11008, 1, 2, dict(outliers=True), "bf16"),
               ("a4 Q4_0 GEMV", "q40", 4096, 11008, 1, 2, dict(outliers=True), "f32"),
               ("a5 GPTQ GEMV", "gptq", 4096, 11008, 1, 2, dict(outliers=True), "f32"),
               ("a5 AWQ GEMV", "awq", 4096, 11008, 1, 2, dict(outliers=True), "f32")]


def cpu_baseline_rows(rows_per_matrix=1024):
    """The CPU oracle as it stands (single thread, f64 accumulation) beside
    each other row: a GEMV over a bounded sample of rows of the row's K,
    format and synthetic recipe (the oracle's cost per row does not depend
    on N), and the NVFP4 dequant of the same rows; GB/s over the sampled
    rows' packed bytes (plus the f32 output for dequant)."""
    import oracle
    import synth
    oracle.build()
    out = []
    for tag, fmt, N, K, M, config, kw, xd in ORACLE_ROWS:
        layer = synth.make_layer(fmt, rows_per_matrix, K, config=config, matrix=0, **kw)
        T = oracle.Tensor(layer["fmt"], rows_per_matrix, K, layer["w"], layer["scales"], layer["zeros"],
                          layer["g_idx"], layer["group"], layer["scale2"])
        xb, xf = synth.draw_x(M, K, config=config, matrix=5, dtype=xd)
        rows = np.arange(rows_per_matrix)
        t0 = time.perf_counter()
        if tag.startswith("a1"):
            oracle.dequant(T, rows=rows)
            dq = time.perf_counter() - t0
            t0 = time.perf_counter()
        oracle.gemv(T, xf, rows=rows)
        dt = time.perf_counter() - t0
        row_bytes = q4_packed_row_bytes(fmt, K)
        out.append({"row": tag, "shape": f"{N}x{K}", "M": M, "sample": f"{rows.size} rows of K = {K}",
                    "GBps": round(rows.size * row_bytes / dt / 1e9, 4), "seconds": round(dt, 3)})
        if tag.startswith("a1"):
            out.append({"row": "a6 dequant NVFP4 -> f32", "shape": f"{N}x{K}", "sample": f"{rows.size} rows of K = {K}",
                        "GBps": round(rows.size * (row_bytes + 4 * K) / dq / 1e9, 4), "seconds": round(dq, 3)})
    layer = synth.make_layer("nvfp4", rows_per_matrix, 4096, config=5, matrix=0, row_scale=True)
    T = oracle.Tensor("nvfp4", rows_per_matrix, 4096, layer["w"], layer["scales"], scale2=layer["scale2"])
    _, xf = synth.draw_x(1, 4096, config=5, matrix=5, dtype="bf16")
    t0 = time.perf_counter()
    oracle.gemv_a16q8(T, xf)
    dt = time.perf_counter() - t0
    out.append({"row": A16Q8_ROW, "shape": "14336x4096", "M": 1, "sample": f"{rows_per_matrix} rows of K = 4096",
                "GBps": round(rows_per_matrix * q4_packed_row_bytes("nvfp4", 4096) / dt / 1e9, 4),
                "seconds": round(dt, 3)})
    isi = float(np.float32(2688.0) / np.float32(np.abs(xf).max()))
    t0 = time.perf_counter()
    oracle.gemv_w4a4(T, xf, isi)
    dt = time.perf_counter() - t0
    out.append({"row": "f1 W4A4 GEMV, integer-exact contract", "shape": "14336x4096", "M": 1,
                "sample": f"{rows_per_matrix} rows of K = 4096",
                "GBps": round(rows_per_matrix * q4_packed_row_bytes("nvfp4", 4096) / dt / 1e9, 4),
                "seconds": round(dt, 3)})
    ql = synth.make_layer("q4k", rows_per_matrix, 4096, config=1, matrix=0)
    _, qxf = synth.draw_x(1, 4096, config=1, matrix=5, dtype="f32")
    t0 = time.perf_counter()
    oracle.gemv_q4k_q8(oracle.Tensor("q4k", rows_per_matrix, 4096, ql["w"]), qxf)
    dt = time.perf_counter() - t0
    out.append({"row": "f2 Q4_K x Q8 (W4A8) GEMV, integer sub-block sums", "shape": "4096x4096", "M": 1,
                "sample": f"{rows_per_matrix} rows of K = 4096",
                "GBps": round(rows_per_matrix * q4_packed_row_bytes("q4k", 4096) / dt / 1e9, 4),
                "seconds": round(dt, 3)})
    return out


def q4_packed_row_bytes(fmt, K):
    """Packed bytes of one weight row, payload + scales (+ zeros), group 128."""
    return {"nvfp4": K // 2 + K // 16, "mxfp4": K // 2 + K // 32, "q4k": K // 256 * 144, "q40": K // 32 * 18,
            "gptq": K // 2 + K // 128 * 2 + K // 128 // 2, "awq": K // 2 + K // 128 * 2 + K // 128 // 2}[fmt]


def _cpu_name():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores, each step a bounded
    sample of the same workload (rank 0 only)."""
    if rank != 0:
        return None
    import synth
    import oracle
    oracle.build()
    host = []
    for i, (name, N, K) in enumerate(SET):
        layer = synth.make_layer("nvfp4", N, K, config=CONFIG_ID, matrix=i, row_scale=True)
        xbits, _ = synth.draw_x(1, K, config=CONFIG_ID, matrix=0 if name in ("gate", "up") else i)
        host.append((name, N, K, layer, xbits))
    # size each step's sample so that the whole run stays near a minute
    rows_per_matrix = int(max(1, min(64, 60.0 / (max(args.steps, 1) * 0.65e-3))))
    tensors = [(oracle.Tensor("nvfp4", N, K, l["w"], l["scales"], scale2=l["scale2"]),
                oracle.bf16_bits_to_f32(xb), K) for _, N, K, l, xb in host]

    def step():
        b = 0
        for T, xf, K in tensors:
            oracle.gemv(T, xf, rows=np.arange(rows_per_matrix))
            b += rows_per_matrix * (K // 2 + K // 16)
        return b
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    total = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": 1,
                       "sample_per_step": f"{rows_per_matrix} rows of each of the 3 set matrices"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{rows_per_matrix} rows per matrix per step", "cpu": _cpu_name()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


GEMM_SHAPE = (14336, 4096)
GEMM_BATCHES = (16, 64, 128)


def small_m_gemm(torch, q4, synth, peak_hbm):
    """The small-batch tensor-core GEMM, Y[M][N] = X . W^T for M in 16/64/128
    on the 14336 x 4096 layer, NVFP4 and Q4_K weights drawn like the 1024 x
    4096 NVFP4 case (W ~ N(0, 0.02)), x ~ N(0, 1) bf16, f32 y.  Each launch
    reads a different one of 6 weight copies (> L2); CUDA events on the
    launching stream.  Reported per (format, M): microseconds per launch,
    bytes moved (weights + x + y) per second, bf16 tensor TFLOP/s, and the
    fractions of the measured HBM and bf16 peaks."""
    N, K = GEMM_SHAPE
    tflops_peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tflops_peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        tflops_peak = 1900.0
    out = []
    stream = torch.cuda.Stream()
    for fmt in ("nvfp4", "q4k"):
        layer = synth.make_layer(fmt, N, K, config=4, matrix=0)
        base = {k: (None if layer[k] is None else torch.from_numpy(
            np.ascontiguousarray(layer[k]).view(np.int16) if layer[k].dtype == np.uint16
            else np.ascontiguousarray(layer[k])).cuda()) for k in ("w", "scales")}
        copies = [base] + [{k: (None if v is None else v.clone()) for k, v in base.items()} for _ in range(5)]
        wbytes = q4.q4_packed_bytes(fmt, N, K)
        aux = q4.make_aux(scale2=layer["scale2"], x_dtype=q4.Q4_DT_BF16, fmt=fmt)
        for M in GEMM_BATCHES:
            xb, _ = synth.draw_x(M, K, config=4, matrix=7)
            x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            with torch.cuda.stream(stream):
                def launch(i):
                    c = copies[i % len(copies)]
                    q4.q4_gemv(fmt, c["w"], c["scales"], aux, x, y, M, N, K, stream=stream)
                for i in range(12):
                    launch(i)
                torch.cuda.synchronize()
                reps = 120
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for i in range(reps):
                    launch(i)
                b.record(stream)
                torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / reps
            moved = wbytes + M * K * 2 + M * N * 4
            gbs = moved / us / 1e3
            tf = 2.0 * M * N * K / us / 1e6
            out.append({"fmt": fmt, "M": M, "us_per_launch": round(us, 2), "GBps": round(gbs, 1),
                         "TFLOPs": round(tf, 1), "frac_hbm": round(gbs / peak_hbm, 4),
                         "frac_bf16": round(tf / tflops_peak, 4), "path": q4.q4_last_gemv_path()})
        del copies, base
        torch.cuda.empty_cache()
    return {"workload": f"small-batch GEMM M x {N} x {K}, NVFP4 and Q4_K (bf16 x, f32 y)",
            "kernel": "gemm_tc_kernel (tcgen05.mma, A decoded into TMEM, x by TMA)",
            "l2": "6 rotating weight copies, 198 MB > L2",
            "peaks": {"hbm_GBps": peak_hbm, "bf16_TFLOPs": tflops_peak},
            "entries": out}


def _dev_layer(torch, layer):
    out = {}
    for k in ("w", "scales", "zeros", "g_idx"):
        a = layer[k]
        if a is None:
            out[k] = None
            continue
        a = np.ascontiguousarray(a)
        out[k] = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    return out


def _time_launches(torch, stream, launch, reps=200, warm=10):
    with torch.cuda.stream(stream):
        for i in range(warm):
            launch(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            launch(i)
        b.record(stream)
        torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def _time_graph(torch, stream, launch, reps=200, warm=10, cells=5):
    """Device time per launch with the `reps` launches captured into one CUDA
    graph, replayed `cells` times, each replay between its own two events (on
    `stream`), so no host launch gap enters the time: how the headline step is
    timed.  For the GEMV rows, whose calls allocate nothing and never
    synchronize.  If the capture fails the launches are issued one by one
    instead.  Returns (median us per launch over the cells, "graph" or
    "eager", coefficient of variation over the cells or None)."""
    with torch.cuda.stream(stream):
        for i in range(warm):
            launch(i)
        torch.cuda.synchronize()
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    launch(i)
        except Exception:
            torch.cuda.synchronize()
            return _time_launches(torch, stream, launch, reps, warm), "eager", None
        g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(cells)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 / reps for a, b in ev]
    return statistics.median(us), "graph", statistics.pstdev(us) / statistics.mean(us)


def _cv(v):
    return None if v is None else round(v, 4)


def other_rows(torch, q4, synth, peak_hbm):
    """Each remaining hot-path row on its own configuration's shape: the GEMV
    of every format at batch 1 (NVFP4 also at batch 4 and 8), dequant and
    repack.  Every launch reads a different weight copy (working set > L2);
    CUDA events on the launching stream, the GEMV rows' launches replayed as
    one CUDA graph.  Bytes are the row's algorithmic
    bytes: packed weights (q4_packed_bytes) + x + y for a GEMV, packed +
    f32 output for dequant, packed in + packed out for repack."""
    stream = torch.cuda.Stream()
    target = 256 * 1024 * 1024
    rows = []

    def copies_of(d, nbytes):
        n = max(2, -(-target // nbytes))
        return [d] + [{k: (None if v is None else v.clone()) for k, v in d.items()} for _ in range(n - 1)]

    def gemv_row(tag, fmt, N, K, M, config, kw, xdtype):
        layer = synth.make_layer(fmt, N, K, config=config, matrix=0, **kw)
        packed = q4.q4_packed_bytes(fmt, N, K)
        cps = copies_of(_dev_layer(torch, layer), packed)
        xb, _ = synth.draw_x(M, K, config=config, matrix=5, dtype="bf16" if xdtype == q4.Q4_DT_BF16 else "f32")
        xa = np.ascontiguousarray(xb)
        x = (torch.from_numpy(xa.view(np.int16)).cuda().view(torch.bfloat16) if xdtype == q4.Q4_DT_BF16
             else torch.from_numpy(xa.astype(np.float32)).cuda())
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        auxes = [q4.make_aux(scale2=layer["scale2"], zeros=c["zeros"], g_idx=c["g_idx"], group=layer["group"],
                             x_dtype=xdtype, fmt=fmt) for c in cps]

        def launch(i):
            c = cps[i % len(cps)]
            q4.q4_gemv(fmt, c["w"], c["scales"], auxes[i % len(cps)], x, y, M, N, K, stream=stream)
        us, how, cv = _time_graph(torch, stream, launch)
        moved = packed + x.numel() * x.element_size() + y.numel() * 4
        rows.append({"row": tag, "shape": f"{N}x{K}", "M": M, "us_per_launch": round(us, 2),
                     "GBps": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4),
                     "path": q4.q4_last_gemv_path(), "timing": how, "cv": _cv(cv)})

    gemv_row("a1 NVFP4 GEMV", "nvfp4", 14336, 4096, 4, 5, dict(row_scale=True), q4.Q4_DT_BF16)
    gemv_row("a1 NVFP4 GEMV", "nvfp4", 14336, 4096, 8, 5, dict(row_scale=True), q4.Q4_DT_BF16)
    gemv_row("a2 Q4_K GEMV", "q4k", 4096, 4096, 1, 1, dict(), q4.Q4_DT_F32)
    gemv_row("a3 MXFP4 GEMV", "mxfp4", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_BF16)
    gemv_row("a4 Q4_0 GEMV", "q40", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32)
    gemv_row("a5 GPTQ GEMV", "gptq", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32)
    gemv_row("a5 AWQ GEMV", "awq", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32)
    torch.cuda.empty_cache()

    # the integer-exact A16-Q8 lane on the 14336x4096 NVFP4 layer at batch 1
    N, K, M = 14336, 4096, 1
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    packed = q4.q4_packed_bytes("nvfp4", N, K)
    cps = copies_of(_dev_layer(torch, layer), packed)
    xb, _ = synth.draw_x(M, K, config=5, matrix=5, dtype="bf16")
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], x_dtype=q4.Q4_DT_BF16, fmt="nvfp4")
    us, how, cv = _time_graph(torch, stream, lambda i: q4.q4_gemv_a16q8(cps[i % len(cps)]["w"],
                                                                    cps[i % len(cps)]["scales"], aux, x, y, M, N, K,
                                                                    stream=stream))
    moved = packed + x.numel() * 2 + y.numel() * 4
    rows.append({"row": A16Q8_ROW, "shape": f"{N}x{K}", "M": M, "us_per_launch": round(us, 2),
                 "GBps": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4),
                 "path": q4.q4_last_gemv_path(), "timing": how, "cv": _cv(cv)})
    del cps
    torch.cuda.empty_cache()

    # the next rows' lanes on the 14336x4096 layer at batch 1 (and W4A8 on its Q4_K layer)
    N, K, M = 14336, 4096, 1
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    packed = q4.q4_packed_bytes("nvfp4", N, K)
    cps = copies_of(_dev_layer(torch, layer), packed)
    xb, xf = synth.draw_x(M, K, config=5, matrix=5, dtype="bf16")
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], x_dtype=q4.Q4_DT_BF16, fmt="nvfp4")
    isi = float(np.float32(2688.0) / np.float32(np.abs(xf).max()))
    G = float(np.float32(1.0) / np.float32(isi))
    moved = packed + x.numel() * 2 + y.numel() * 4

    def lane_row(tag, fn, nbytes=moved, path=True):
        us, how, cv = _time_graph(torch, stream, fn)
        row = {"row": tag, "shape": f"{N}x{K}", "M": M, "us_per_launch": round(us, 2),
               "GBps": round(nbytes / us / 1e3, 1), "frac_hbm": round(nbytes / us / 1e3 / peak_hbm, 4),
               "timing": how, "cv": _cv(cv)}
        if path:
            row["path"] = q4.q4_last_gemv_path()
        rows.append(row)
    auxf = q4.make_aux(scale2=layer["scale2"], x_dtype=q4.Q4_DT_BF16, fmt="nvfp4", flags=q4.Q4_FLAG_FP4_SLICES)
    lane_row("a1 NVFP4 GEMV, FP4 tensor cores with exact x slices (opt-in)",
             lambda i: q4.q4_gemv("nvfp4", cps[i % len(cps)]["w"], cps[i % len(cps)]["scales"], auxf, x, y, M, N, K,
                                  stream=stream))
    lane_row("f1 W4A4 GEMV, integer-exact contract", lambda i: q4.q4_gemv_w4a4(
        cps[i % len(cps)]["w"], cps[i % len(cps)]["scales"], aux, isi, x, y, M, N, K, stream=stream))
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    xsc = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    q4.q4_quantize_nvfp4_scaled(x, q4.Q4_DT_BF16, G, xq, xsc, M, K, stream=stream)
    lane_row("f1 W4A4 GEMV on the FP4 tensor cores (activations already NVFP4)", lambda i: q4.q4_gemv_w4a4_tc(
        cps[i % len(cps)]["w"], cps[i % len(cps)]["scales"], aux, xq, xsc, G, y, M, N, K, stream=stream),
        nbytes=packed + xq.numel() + xsc.numel() + y.numel() * 4)
    del cps
    torch.cuda.empty_cache()
    qlayer = synth.make_layer("q4k", 4096, 4096, config=1, matrix=0)
    qpacked = q4.q4_packed_bytes("q4k", 4096, 4096)
    qcps = copies_of(_dev_layer(torch, qlayer), qpacked)
    _, qxf = synth.draw_x(1, 4096, config=1, matrix=5, dtype="f32")
    qx = torch.from_numpy(np.ascontiguousarray(qxf, np.float32)).cuda()
    qy = torch.empty((1, 4096), dtype=torch.float32, device="cuda")
    us, how, cv = _time_graph(torch, stream, lambda i: q4.q4_gemv_q4k_q8(qcps[i % len(qcps)]["w"], None, qx, qy, 1,
                                                                      4096, 4096, stream=stream))
    qmoved = qpacked + qx.numel() * 4 + qy.numel() * 4
    rows.append({"row": "f2 Q4_K x Q8 (W4A8) GEMV, integer sub-block sums", "shape": "4096x4096", "M": 1,
                 "us_per_launch": round(us, 2), "GBps": round(qmoved / us / 1e3, 1),
                 "frac_hbm": round(qmoved / us / 1e3 / peak_hbm, 4), "path": q4.q4_last_gemv_path(),
                 "timing": how, "cv": _cv(cv)})
    del qcps
    torch.cuda.empty_cache()
    # f3: the GPU quantizers on the 14336x4096 layer (f32 W in, packed out)
    Wd = torch.from_numpy(synth.draw_weights(N, K, config=5, matrix=0, row_scale=True)).cuda()
    pay = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scl = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(4, dtype=torch.float32, device="cuda")
    qb = torch.empty((N, K // 256, 144), dtype=torch.uint8, device="cuda")
    us = _time_launches(torch, stream, lambda i: q4.q4_quantize_nvfp4(Wd, q4.Q4_DT_F32, pay, scl, s2, N, K,
                                                                      stream=stream), reps=40)
    qbytes = N * K * 4 + packed
    rows.append({"row": "f3 NVFP4 quantizer (f32 W -> payload, scales, scale2; four launches)", "shape": f"{N}x{K}",
                 "us_per_call": round(us, 2), "GBps": round(qbytes / us / 1e3, 1),
                 "frac_hbm": round(qbytes / us / 1e3 / peak_hbm, 4),
                 "note": "W is read twice (tensor maximum, then the groups): bytes count it once"})
    us = _time_launches(torch, stream, lambda i: q4.q4_quantize_q4k(Wd, q4.Q4_DT_F32, qb, N, K, stream=stream), reps=40)
    qbytes = N * K * 4 + q4.q4_packed_bytes("q4k", N, K)
    rows.append({"row": "f3 Q4_K fit (f32 W -> 144-byte super-blocks)", "shape": f"{N}x{K}",
                 "us_per_launch": round(us, 2), "GBps": round(qbytes / us / 1e3, 1),
                 "frac_hbm": round(qbytes / us / 1e3 / peak_hbm, 4)})
    del Wd, pay, scl, qb
    torch.cuda.empty_cache()
    # f4: 3-bit stream packing of 64 Mi codes (u8 in, words out); four input/output pairs (352 MB) rotate
    # so that no launch finds its codes in L2
    n = 64 << 20
    pairs = [(torch.randint(0, 8, (n,), dtype=torch.uint8, device="cuda"),
              torch.empty(n * 3 // 32, dtype=torch.int32, device="cuda")) for _ in range(4)]
    us = _time_launches(torch, stream, lambda i: q4.q4_pack_bits(pairs[i % 4][0], n, 3, pairs[i % 4][1],
                                                                 stream=stream), reps=40)
    pbytes = n + pairs[0][1].numel() * 4
    rows.append({"row": "f4 3-bit stream packer (u8 codes -> words)", "shape": f"{n} codes",
                 "us_per_launch": round(us, 2), "GBps": round(pbytes / us / 1e3, 1),
                 "frac_hbm": round(pbytes / us / 1e3 / peak_hbm, 4), "l2": "4 rotating input/output pairs, 352 MB"})
    del pairs
    torch.cuda.empty_cache()

    # a6: dequant NVFP4 14336x4096 to f32 (write-bound)
    N, K = 14336, 4096
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    packed = q4.q4_packed_bytes("nvfp4", N, K)
    cps = copies_of(_dev_layer(torch, layer), packed)[:6]
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], fmt="nvfp4")
    us = _time_launches(torch, stream, lambda i: q4.q4_dequant("nvfp4", cps[i % len(cps)]["w"],
                                                               cps[i % len(cps)]["scales"], aux, out, N, K,
                                                               stream=stream), reps=60)
    moved = packed + N * K * 4
    rows.append({"row": "a6 dequant NVFP4 -> f32", "shape": f"{N}x{K}", "us_per_launch": round(us, 2),
                 "GBps": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4)})
    del cps, out
    torch.cuda.empty_cache()

    # a6: dequant Q4_K 14336x4096 to f32 (same output, 144-byte super-blocks in)
    layer = synth.make_layer("q4k", N, K, config=4, matrix=0)
    packed = q4.q4_packed_bytes("q4k", N, K)
    cps = copies_of(_dev_layer(torch, layer), packed)[:6]
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    us = _time_launches(torch, stream, lambda i: q4.q4_dequant("q4k", cps[i % len(cps)]["w"], None, None, out, N, K,
                                                               stream=stream), reps=60)
    moved = packed + N * K * 4
    rows.append({"row": "a6 dequant Q4_K -> f32", "shape": f"{N}x{K}", "us_per_launch": round(us, 2),
                 "GBps": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4)})
    del cps, out
    torch.cuda.empty_cache()

    # a7: repack GPTQ -> AWQ 4096x11008 (read once, write once)
    N, K = 4096, 11008
    layer = synth.make_layer("gptq", N, K, config=2, matrix=0, outliers=True)
    packed = q4.q4_packed_bytes("gptq", N, K)
    cps = copies_of(_dev_layer(torch, layer), packed)
    w = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((K // 128, N), dtype=torch.int16, device="cuda")
    z = torch.empty((K // 128, N // 8), dtype=torch.int32, device="cuda")
    auxes = [q4.make_aux(zeros=c["zeros"], group=128, fmt="gptq") for c in cps]
    us = _time_launches(torch, stream, lambda i: q4.q4_repack("gptq", cps[i % len(cps)]["w"],
                                                              cps[i % len(cps)]["scales"], auxes[i % len(cps)],
                                                              "awq", w, sc, z, None, N, K, stream=stream))
    moved = 2 * packed
    rows.append({"row": "a7 repack GPTQ -> AWQ", "shape": f"{N}x{K}", "us_per_launch": round(us, 2),
                 "GBps": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4)})
    del cps
    torch.cuda.empty_cache()
    return {"l2": "each launch reads a different weight copy; working set >= 256 MB per row",
            "timing": "CUDA events around 200 launches: for the GEMV rows one CUDA graph of the 200 launches "
                      "replayed 5 times, each between its own events, the median reported with the coefficient "
                      "of variation 'cv' (no host launch gaps, as the headline step; a row's 'timing' says 'eager' "
                      "if its calls could not be captured), for the others launch by launch",
            "peak_hbm_GBps": peak_hbm, "entries": rows}


LLAMA7B_SET = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
               ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)]
SWEEP_FORMATS = ("nvfp4", "mxfp4", "q4k", "q40", "gptq", "awq")
SWEEP_BATCHES = (1, 4, 8)


def _device_layer(torch, q4, fmt, N, K, gen):
    """One seeded synthetic tensor of ``fmt`` built on the device.  NVFP4 and
    Q4_K: W ~ N(0, 0.02) x U(0.5, 2) per row, quantized by the library's GPU
    quantizers.  The other formats: seeded random codes with valid scales of
    the same magnitude (their decode cost does not depend on the values)."""
    dev = "cuda"
    d = {"scales": None, "zeros": None, "scale2": 1.0}
    if fmt in ("nvfp4", "q4k"):
        W = torch.randn((N, K), generator=gen, device=dev) * 0.02
        W *= torch.rand((N, 1), generator=gen, device=dev) * 1.5 + 0.5
        if fmt == "nvfp4":
            d["w"] = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
            d["scales"] = torch.empty((N, K // 16), dtype=torch.uint8, device=dev)
            s2 = torch.empty(4, dtype=torch.float32, device=dev)
            q4.q4_quantize_nvfp4(W, q4.Q4_DT_F32, d["w"], d["scales"], s2, N, K)
            d["scale2"] = float(s2[0].item())
        else:
            d["w"] = torch.empty((N, K // 256, 144), dtype=torch.uint8, device=dev)
            q4.q4_quantize_q4k(W, q4.Q4_DT_F32, d["w"], N, K)
        del W
        return d
    rnd = lambda shape, hi: torch.randint(0, hi, shape, generator=gen, device=dev)  # noqa: E731
    if fmt == "mxfp4":
        d["w"] = rnd((N, K // 2), 256).to(torch.uint8)
        d["scales"] = (rnd((N, K // 32), 3) + 120).to(torch.uint8)            # 2^-7 .. 2^-5
    elif fmt == "q40":
        blk = rnd((N, K // 32, 18), 256).to(torch.uint8)
        blk[:, :, 0:2] = torch.tensor([0x20, 0x1A], dtype=torch.uint8, device=dev)   # fp16 d = 0.0025
        d["w"] = blk
    else:
        G = K // 128
        words = (N, K // 8) if fmt == "gptq" else (K, N // 8)
        w = rnd(words, 1 << 16) | (rnd(words, 1 << 16) << 16)
        d["w"] = (w.t().contiguous() if fmt == "gptq" else w).to(torch.int32)
        d["scales"] = torch.full((G, N), 0x1A20, dtype=torch.int16, device=dev)
        z = torch.zeros((G, N // 8), dtype=torch.int64, device=dev)
        for j in range(8):
            z |= rnd((G, N // 8), 15) << (4 * j)                             # stored zeros 0..14
        d["zeros"] = z.to(torch.int32)
    return d


def layer_set_sweep(torch, q4, peak_hbm, batches=SWEEP_BATCHES, formats=SWEEP_FORMATS):
    """The Llama-7B-shaped decoder layer set (q/k/v/o 4096x4096, gate/up
    11008x4096, down 4096x11008) in every format at batch 1, 4 and 8: one
    pass = the seven GEMVs of one layer as four calls (q4_gemv_grouped of
    q, k, v and of gate, up, which read the same x; o and down alone),
    captured as one CUDA graph over rotating weight copies (> 4 x L2).  Reported per
    (format, batch): microseconds per layer, weight bytes per second, the
    fraction of the measured HBM peak, the tokens-equivalent rate of a
    32-layer model (weight streaming only) and the kernel paths."""
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda")
    out = []
    for fi, fmt in enumerate(formats):
        gen.manual_seed(3000 + fi)
        base = [_device_layer(torch, q4, fmt, N, K, gen) for _, N, K in LLAMA7B_SET]
        layer_bytes = sum(q4.q4_packed_bytes(fmt, N, K) for _, N, K in LLAMA7B_SET)
        ncopies = max(2, -(-4 * l2 // layer_bytes))
        copies = [base] + [[{k: (v.clone() if torch.is_tensor(v) else v) for k, v in m.items()} for m in base]
                           for _ in range(ncopies - 1)]
        for M in batches:
            xdt = torch.bfloat16                     # the layer-set configuration's activations, every format
            xs = {K: torch.randn((M, K), generator=gen, device="cuda").to(xdt) for K in (4096, 11008)}
            ys = [torch.empty((M, N), device="cuda") for _, N, _ in LLAMA7B_SET]
            auxes = [[q4.make_aux(scale2=m["scale2"], zeros=m["zeros"], group=128, x_dtype=xdt, fmt=fmt) for m in c]
                     for c in copies]
            paths = []

            def layer(c, s, record=False):
                # q, k, v read one x and gate, up another: one grouped call each; o and down alone
                for grp in ((0, 1, 2), (3,), (4, 5), (6,)):
                    q4.q4_gemv_grouped([(fmt, copies[c][i]["w"], copies[c][i]["scales"], auxes[c][i],
                                         xs[LLAMA7B_SET[i][2]], ys[i], LLAMA7B_SET[i][1], LLAMA7B_SET[i][2])
                                        for i in grp], M, stream=s)
                    if record:
                        paths.append(q4.q4_last_gemv_path())
            with torch.cuda.stream(stream):
                layer(0, stream, record=True)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for c in range(ncopies):
                        layer(c, stream)
                for _ in range(3):
                    g.replay()
                torch.cuda.synchronize()
                # five cells of two back-to-back replays each, every cell between its own events
                reps, cells = 2, 5
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(cells)]
                for a, b in ev:
                    a.record(stream)
                    for _ in range(reps):
                        g.replay()
                    b.record(stream)
                torch.cuda.synchronize()
            cell_us = [a.elapsed_time(b) * 1e3 / (reps * ncopies) for a, b in ev]
            us = statistics.median(cell_us)
            gbs = layer_bytes / us / 1e3
            out.append({"fmt": fmt, "M": M, "us_per_layer": round(us, 2), "GBps": round(gbs, 1),
                        "frac_hbm": round(gbs / peak_hbm, 4),
                        "cv": round(statistics.pstdev(cell_us) / statistics.mean(cell_us), 4),
                        "tokens_equivalent_per_s": round(1e6 / (LAYERS * us), 1),
                        "paths": sorted(set(paths))})
            del xs, ys
        del copies, base
        torch.cuda.empty_cache()
    return {"workload": "Llama-7B layer set: q, k, v, o 4096x4096; gate, up 11008x4096; down 4096x11008",
            "formats": list(formats), "batches": list(batches),
            "data": "seeded on the device: NVFP4 and Q4_K quantized from W ~ N(0,0.02) x U(0.5,2) rows by the "
                    "library's GPU quantizers; MXFP4, Q4_0, GPTQ, AWQ as seeded random codes with valid scales; "
                    "x ~ N(0,1) bf16 for every format",
            "l2": "each layer pass reads a different weight copy (copies > 4 x L2)",
            "launch": "per layer: q4_gemv_grouped(q, k, v), q4_gemv(o), q4_gemv_grouped(gate, up), q4_gemv(down); "
                      "one CUDA graph over the copies",
            "timing": "per cell the median over 5 timed repetitions (each two replays of the graph between its own "
                      "CUDA events), with the coefficient of variation over the 5",
            "peak_hbm_GBps": peak_hbm, "entries": out}


def ncu_gemm_case(spec):
    """3 launches of the small-batch GEMM on one weight copy, for ncu."""
    import torch

    import bit_block_quantized_gb300 as q4
    import synth
    from bit_block_quantized_gb300 import build as q4build
    q4build.build()
    fmt, M = spec.split(":")
    M = int(M)
    N, K = GEMM_SHAPE
    layer = synth.make_layer(fmt, N, K, config=4, matrix=0)
    dev = {k: (None if layer[k] is None else torch.from_numpy(
        np.ascontiguousarray(layer[k]).view(np.int16) if layer[k].dtype == np.uint16
        else np.ascontiguousarray(layer[k])).cuda()) for k in ("w", "scales")}
    xb, _ = synth.draw_x(M, K, config=4, matrix=7)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], x_dtype=q4.Q4_DT_BF16, fmt=fmt)
    for _ in range(3):
        q4.q4_gemv(fmt, dev["w"], dev["scales"], aux, x, y, M, N, K)
    torch.cuda.synchronize()
    print("ncu gemm case done:", q4.q4_last_gemv_path(), "last_error", q4.q4_last_error())


def ncu_case():
    """A few launches of the dominant kernel (gate and up as one grouped
    launch, 66 MB) on one weight copy, for ncu captures sized well under a
    few GB of device memory."""
    import torch

    import bit_block_quantized_gb300 as q4
    import synth
    from bit_block_quantized_gb300 import build as q4build
    q4build.build()
    mats = []
    for i in (0, 1):
        name, N, K = SET[i]
        layer = synth.make_layer("nvfp4", N, K, config=CONFIG_ID, matrix=i, row_scale=True)
        mats.append((N, K, torch.from_numpy(layer["w"]).cuda(), torch.from_numpy(layer["scales"]).cuda(),
                     q4.make_aux(scale2=layer["scale2"], fmt="nvfp4")))
    xbits, _ = synth.draw_x(1, SET[0][2], config=CONFIG_ID, matrix=0)
    x = torch.from_numpy(xbits.view(np.int16)).cuda().view(torch.bfloat16)
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for N, *_ in mats]
    for _ in range(4):
        q4.q4_gemv_grouped([("nvfp4", w, s, aux, x, y, N, K) for (N, K, w, s, aux), y in zip(mats, ys)], 1)
    torch.cuda.synchronize()
    print("ncu case done, last_error", q4.q4_last_error())


def ncu_rows_case():
    """One launch of each remaining row's kernel on its own shape (one weight
    copy, a few hundred MB of device memory at most), for a single-pass ncu
    launch list with DRAM bytes.  Prints each row's algorithmic bytes."""
    import torch

    import bit_block_quantized_gb300 as q4
    import synth
    from bit_block_quantized_gb300 import build as q4build
    q4build.build()
    stream = torch.cuda.Stream()
    for tag, fmt, N, K, M, config, kw, xdt in (
            ("a1 NVFP4 M=4", "nvfp4", 14336, 4096, 4, 5, dict(row_scale=True), q4.Q4_DT_BF16),
            ("a1 NVFP4 M=8", "nvfp4", 14336, 4096, 8, 5, dict(row_scale=True), q4.Q4_DT_BF16),
            ("a2 Q4_K", "q4k", 4096, 4096, 1, 1, dict(), q4.Q4_DT_F32),
            ("a3 MXFP4", "mxfp4", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_BF16),
            ("a4 Q4_0", "q40", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32),
            ("a5 GPTQ", "gptq", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32),
            ("a5 AWQ", "awq", 4096, 11008, 1, 2, dict(outliers=True), q4.Q4_DT_F32)):
        layer = synth.make_layer(fmt, N, K, config=config, matrix=0, **kw)
        d = _dev_layer(torch, layer)
        xb, _ = synth.draw_x(M, K, config=config, matrix=5, dtype="bf16" if xdt == q4.Q4_DT_BF16 else "f32")
        xa = np.ascontiguousarray(xb)
        x = (torch.from_numpy(xa.view(np.int16)).cuda().view(torch.bfloat16) if xdt == q4.Q4_DT_BF16
             else torch.from_numpy(xa.astype(np.float32)).cuda())
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        aux = q4.make_aux(scale2=layer["scale2"], zeros=d["zeros"], g_idx=d["g_idx"], group=layer["group"],
                          x_dtype=xdt, fmt=fmt)
        q4.q4_gemv(fmt, d["w"], d["scales"], aux, x, y, M, N, K, stream=stream)
        torch.cuda.synchronize()
        moved = q4.q4_packed_bytes(fmt, N, K) + x.numel() * x.element_size() + y.numel() * 4
        print(f"{tag}: {N}x{K} path {q4.q4_last_gemv_path()} algorithmic bytes {moved}")
    N, K = 14336, 4096
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    d = _dev_layer(torch, layer)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q4.q4_dequant("nvfp4", d["w"], d["scales"], q4.make_aux(scale2=layer["scale2"], fmt="nvfp4"), out, N, K,
                  stream=stream)
    torch.cuda.synchronize()
    print(f"a6 dequant NVFP4 -> f32: {N}x{K} algorithmic bytes {q4.q4_packed_bytes('nvfp4', N, K) + N * K * 4}")
    del out
    N, K = 4096, 11008
    layer = synth.make_layer("gptq", N, K, config=2, matrix=0, outliers=True)
    d = _dev_layer(torch, layer)
    w = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((K // 128, N), dtype=torch.int16, device="cuda")
    z = torch.empty((K // 128, N // 8), dtype=torch.int32, device="cuda")
    q4.q4_repack("gptq", d["w"], d["scales"], q4.make_aux(zeros=d["zeros"], group=128, fmt="gptq"), "awq", w, sc, z,
                 None, N, K, stream=stream)
    print(f"a7 repack GPTQ -> AWQ: {N}x{K} algorithmic bytes {2 * q4.q4_packed_bytes('gptq', N, K)}")
    N, K = 14336, 4096
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    d = _dev_layer(torch, layer)
    xb, _ = synth.draw_x(1, K, config=5, matrix=5, dtype="bf16")
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    q4.q4_gemv_a16q8(d["w"], d["scales"], q4.make_aux(scale2=layer["scale2"], fmt="nvfp4"), x, y, 1, N, K,
                     stream=stream)
    torch.cuda.synchronize()
    print(f"{A16Q8_ROW}: {N}x{K} algorithmic bytes {q4.q4_packed_bytes('nvfp4', N, K) + K * 2 + N * 4}")
    print("ncu rows case done, last_error", q4.q4_last_error())


def ncu_lanes_case():
    """One launch of each kernel added for the next rows and of the FP4
    tensor-core path, on one weight copy (a few hundred MB of device memory at
    most), for single-kernel ncu captures.  Prints each launch's algorithmic
    bytes."""
    import torch

    import bit_block_quantized_gb300 as q4
    import synth
    from bit_block_quantized_gb300 import build as q4build
    q4build.build()
    stream = torch.cuda.Stream()
    mats = []
    for i in (0, 1):
        name, N, K = SET[i]
        layer = synth.make_layer("nvfp4", N, K, config=CONFIG_ID, matrix=i, row_scale=True)
        d = _dev_layer(torch, layer)
        mats.append((N, K, d, q4.make_aux(scale2=layer["scale2"], fmt="nvfp4", flags=q4.Q4_FLAG_FP4_SLICES)))
    xb, xf = synth.draw_x(1, 4096, config=CONFIG_ID, matrix=0)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for N, *_ in mats]
    q4.q4_gemv_grouped([("nvfp4", d["w"], d["scales"], aux, x, y, N, K) for (N, K, d, aux), y in zip(mats, ys)], 1,
                       stream=stream)
    torch.cuda.synchronize()
    print(f"gemv_fp4tc (slices) gate+up: {q4.q4_last_gemv_path()} algorithmic bytes "
          f"{2 * q4.q4_packed_bytes('nvfp4', 14336, 4096) + 4096 * 2 + 2 * 14336 * 4}")
    N, K, d, aux = mats[0]
    isi = float(np.float32(2688.0) / np.float32(np.abs(xf).max()))
    G = float(np.float32(1.0) / np.float32(isi))
    xq = torch.empty((1, K // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((1, K // 16), dtype=torch.uint8, device="cuda")
    q4.q4_quantize_nvfp4_scaled(x, q4.Q4_DT_BF16, G, xq, xs, 1, K, stream=stream)
    q4.q4_gemv_w4a4_tc(d["w"], d["scales"], aux, xq, xs, G, ys[0], 1, N, K, stream=stream)
    torch.cuda.synchronize()
    print(f"gemv_fp4tc (W4A4) {N}x{K}: algorithmic bytes {q4.q4_packed_bytes('nvfp4', N, K) + K // 2 + K // 16 + N * 4}")
    q4.q4_gemv_w4a4(d["w"], d["scales"], aux, isi, x, ys[0], 1, N, K, stream=stream)
    torch.cuda.synchronize()
    print(f"gemv_w4a4 {N}x{K}: algorithmic bytes {q4.q4_packed_bytes('nvfp4', N, K) + K * 2 + N * 4}")
    ql = synth.make_layer("q4k", 4096, 4096, config=1, matrix=0)
    dq = _dev_layer(torch, ql)
    _, qxf = synth.draw_x(1, 4096, config=1, matrix=5, dtype="f32")
    qx = torch.from_numpy(np.ascontiguousarray(qxf, np.float32)).cuda()
    qy = torch.empty((1, 4096), dtype=torch.float32, device="cuda")
    q4.q4_gemv_q4k_q8(dq["w"], None, qx, qy, 1, 4096, 4096, stream=stream)
    torch.cuda.synchronize()
    print(f"gemv_q4k_q8 4096x4096: algorithmic bytes {q4.q4_packed_bytes('q4k', 4096, 4096) + 4096 * 8}")
    W = torch.from_numpy(synth.draw_weights(N, K, config=5, matrix=0, row_scale=True)).cuda()
    pay = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scl = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(4, dtype=torch.float32, device="cuda")
    qb = torch.empty((N, K // 256, 144), dtype=torch.uint8, device="cuda")
    q4.q4_quantize_nvfp4(W, q4.Q4_DT_F32, pay, scl, s2, N, K, stream=stream)
    q4.q4_quantize_q4k(W, q4.Q4_DT_F32, qb, N, K, stream=stream)
    torch.cuda.synchronize()
    print(f"quantize {N}x{K}: f32 in {N * K * 4}, NVFP4 out {q4.q4_packed_bytes('nvfp4', N, K)}, "
          f"Q4_K out {q4.q4_packed_bytes('q4k', N, K)}")
    n = 64 << 20
    codes = torch.randint(0, 8, (n,), dtype=torch.uint8, device="cuda")
    words = torch.empty(n * 3 // 32, dtype=torch.int32, device="cuda")
    q4.q4_pack_bits(codes, n, 3, words, stream=stream)
    torch.cuda.synchronize()
    print(f"pack_bits 3-bit: {n} codes, bytes {n + words.numel() * 4}")
    al = synth.make_layer("awq", 4096, 11008, config=2, matrix=0, outliers=True)
    da = _dev_layer(torch, al)
    axb, _ = synth.draw_x(1, 11008, config=2, matrix=5)
    ax = torch.from_numpy(axb.view(np.int16)).cuda().view(torch.bfloat16)
    ay = torch.empty((1, 4096), dtype=torch.float32, device="cuda")
    aaux = q4.make_aux(zeros=da["zeros"], group=128, x_dtype=torch.bfloat16, fmt="awq")
    q4.q4_gemv("awq", da["w"], da["scales"], aaux, ax, ay, 1, 4096, 11008, stream=stream)
    torch.cuda.synchronize()
    print(f"{q4.q4_last_gemv_path()} AWQ 4096x11008: algorithmic bytes "
          f"{q4.q4_packed_bytes('awq', 4096, 11008) + 11008 * 2 + 4096 * 4}")
    print("ncu lanes case done, last_error", q4.q4_last_error())


def main():
    args = parse()
    if args.ncu_rows_case:
        ncu_rows_case()
        return
    if args.ncu_lanes_case:
        ncu_lanes_case()
        return
    if args.ncu_case:
        ncu_case()
        return
    if args.ncu_gemm_case:
        ncu_gemm_case(args.ncu_gemm_case)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        line = run_ours(args, rank, world)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
