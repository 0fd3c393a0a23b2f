"""Benchmark of the GGUF Q4_0 linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: the 26-layer decoder linear stack at batch-1 decode
(hidden 3072, GQA 32Q/8KV, FFN 9216; Q4_0 weights N(0, 0.02^2) quantized on
the device, activation N(0, 1) fp32).  A step is one decode token: 104
dependent fused dequant-GEMV launches (per layer: [wq;wk;wv], wo, [w1;w3], w2)
with programmatic dependent launch, replayed from CUDA graphs.  `value` is
weight GB/s = Q4 bytes streamed per step x steps / device time.  The weights
(1.70 GB) are ~13x the 126 MB L2, so every step reads them from HBM.

The same line carries: the roofline of the GEMV kernel against the measured
HBM copy bandwidth; `e2e` (per step: host->device copy of the token's input
from pinned memory, the step, device->host copy of the layer-stack output);
the prefill/encoder GEMM (32 layers x 4 linears of the 1280-wide encoder at
3000 frames) in TFLOP/s against the measured bf16 peak; the batch-1 output
head and embedding gather; and the CPU oracle timed on a bounded sample.

--impl reference times the CPU oracle (plain C, fp64 sums) on the host cores,
one decoder layer's [wq;wk;wv] product per step, same metric and unit.
Under torchrun each rank runs an independent replica (no collective on the
data path); timing is the max over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_0 decode GEMV weight GB/s (% of HBM peak); prefill GEMM TFLOP/s (% peak)"
WORKLOAD = ("decoder linear stack, 26 layers, batch-1 decode: per layer Q4_0 "
            "wq 3072->4096, wk/wv 3072->1024, wo 4096->3072, w1/w3 3072->9216, w2 9216->3072")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _barrier_max(value: float, world: int, torch):
    """Max of `value` over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _oracle_sample(seconds: float = 12.0, mats=("qkv", "wo", "w13", "w2")):
    """CPU oracle on one decoder layer (bounded): weight GB/s on all host cores."""
    import numpy as np

    import oracle
    import synth
    threads = oracle.cpu_count()
    shapes = {"qkv": [(4096, 3072), (1024, 3072), (1024, 3072)], "wo": [(3072, 4096)],
              "w13": [(9216, 3072), (9216, 3072)], "w2": [(3072, 9216)]}
    packed = []
    for name in mats:
        blocks = [oracle.quantize(synth.np_weights(n, k, seed=synth.seed_for(2, 0, i)))[0]
                  for i, (n, k) in enumerate(shapes[name])]
        W = np.concatenate(blocks, axis=0)
        n = W.shape[0]
        k = shapes[name][0][1]
        packed.append((W, n, k, synth.np_activations(1, k, seed=synth.activation_seed(2000))))
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        for W, n, k, x in packed:
            oracle.matmul(W, n, k, x, nthreads=threads)
            done_bytes += W.nbytes
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 50:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"decoder layer 0 linears ({'+'.join(mats)}), {reps} pass(es), "
                      f"{done_bytes / 1e9:.2f} GB of Q4 weights in {el:.1f} s, fp64 sums, "
                      f"{threads} threads"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import synth
    threads = oracle.cpu_count()
    blocks = [oracle.quantize(synth.np_weights(n, 3072, seed=synth.seed_for(2, 0, i)))[0]
              for i, n in enumerate((4096, 1024, 1024))]
    W = np.concatenate(blocks, axis=0)
    n, k = W.shape[0], 3072
    xs = [synth.np_activations(1, k, seed=synth.activation_seed(2000, s))
          for s in range(min(args.steps + args.warmup, 64))]
    for s in range(args.warmup):
        oracle.matmul(W, n, k, xs[s % len(xs)], nthreads=threads)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.matmul(W, n, k, xs[s % len(xs)], nthreads=threads)
    el = time.perf_counter() - t0
    value = W.nbytes * args.steps / el / 1e9
    sample = (f"one decoder layer's [wq;wk;wv] product (6144x3072 Q4_0, {W.nbytes} B) per "
              f"step, fp64 sums, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "reference_step": sample},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _time_graph_replays(graphs, stream, torch):
    """Replay (graph, count) pairs back to back; return device ms."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for g, cnt in graphs:
            for _ in range(cnt):
                g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def _region_count(est_ms: float, world: int, torch, min_regions: int = 5,
                  min_total_ms: float = 500.0, max_regions: int = 200) -> int:
    """How many timed regions of K steps to run: at least `min_regions` and
    enough to cover `min_total_ms`; the same count on every rank."""
    n = max(min_regions, int(min_total_ms / max(est_ms, 1e-3)) + 1)
    n = min(n, max_regions)
    return int(_barrier_max(float(n), world, torch))


def _timed_regions(fn, regions: int, world: int, dev, torch):
    """Run `fn` (one timed region, returns device ms) `regions` times, each
    bracketed by a barrier and a synchronize, with the clocks sampled across
    all of them; returns ((max over ranks of the median ms, stats), clocks)."""
    times = []
    with ClockSampler(dev.index) as clk:
        for _ in range(regions):
            torch.cuda.synchronize()
            _barrier(world)
            torch.cuda.synchronize()
            times.append(fn())
            torch.cuda.synchronize()
    med = _barrier_max(statistics.median(times), world, torch)
    return (med, {"regions": regions, "min_ms": min(times), "max_ms": max(times)}), clk.summary()


def run_ours(args):
    import torch

    from bit_weight_quantized_03_b300 import lib

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    lib()
    hbm, bf16_burst, bf16_sust, peak_src = _peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream()

    line = {
        "metric": METRIC, "value": None, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded N(0,0.02^2) weights quantized on device, N(0,1) activations)",
    }
    if args.only in ("all", "stack"):
        line.update(_run_stack(args, world, dev, stream, hbm, peak_src, torch))
    extra = {}
    if args.only in ("all", "single"):
        extra["single_gemv"] = _run_single_gemv(args, dev, stream, hbm, torch)
    if args.only in ("all", "head", "gather"):
        extra.update(_run_head_gather(args, dev, stream, hbm, torch))
    gemm = None
    if args.only in ("all", "gemm"):
        gemm = _run_gemm(args, world, dev, stream, bf16_burst, bf16_sust, peak_src, torch)
    if args.only in ("all", "crossover"):
        line["crossover"] = _run_crossover(args, dev, stream, hbm, bf16_burst, torch)
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = _oracle_sample(seconds=args.cpu_seconds)
    line["cpu_baseline"] = cpu
    line["prefill_gemm"] = gemm
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# DRAM bytes (read + write) per decode step from ncu captures of the kernels
# as they stand (profiles/decode_step_dram_traffic.md): a 2-layer step
# captured, scaled to 26 layers (every layer has the same four shapes, so the
# traffic grows with the layer count).  Each entry is used only while the
# kernel sources hash to what they were when captured, else it is null.
STEP_TRAFFIC = {
    "per_launch": {"bytes_per_step": 13 * 133_615_616,
                   "sources": ("q4_gemv_b1.cu", "q4_gemv_tile.cuh"),
                   "sha16": "356d83a8628bbfcf"},
    "fused": {"bytes_per_step": 13 * 135_205_376,
              "sources": ("q4_chain.cu", "q4r_tile.cuh"),
              "sha16": "5e9eade3da070177"},
}


def _sources_sha16(names):
    import hashlib
    h = hashlib.sha256()
    for nm in names:
        with open(os.path.join(ROOT, "bit_weight_quantized_03_b300", "csrc", nm), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _step_traffic(path):
    t = STEP_TRAFFIC.get(path)
    if t is None or _sources_sha16(t["sources"]) != t["sha16"]:
        return None
    return t["bytes_per_step"]


def _run_stack(args, world, dev, stream, hbm, peak_src, torch):
    """Decoder linear stack at batch-1 decode (headline).  The step runs as one
    q4_gemv_chain launch (104 dependent products); the same step as 104 q4_gemv
    launches with programmatic dependent launch is timed beside it."""
    import synth
    from bit_weight_quantized_03_b300.stacks import DecoderStack

    dec = DecoderStack(device=dev, **({} if args.layers is None else {"layers": args.layers}))
    wbytes = dec.weight_bytes()
    abytes = dec.activation_bytes()
    G = 8
    inputs = [synth.torch_activations(1, 3072, seed=synth.activation_seed(2000, s), device=dev)
              for s in range(G)]

    def timed(kind):
        if kind == "fused":
            g_multi = dec.capture_fused(inputs, stream)
            g_one = dec.capture_fused(inputs[:1], stream)
        else:
            g_multi = dec.capture(inputs, stream, chain=kind == "chain")
            g_one = dec.capture(inputs[:1], stream, chain=kind == "chain")

        def plan(steps):
            return [(g_multi, steps // G), (g_one, steps % G)]

        # Warm-up: every graph that the timed region replays is replayed here
        # first (a graph's first replay uploads it), whatever --warmup is.
        _time_graph_replays([(g_multi, max(1, args.warmup // G)),
                             (g_one, max(1, args.warmup % G))], stream, torch)
        torch.cuda.synchronize()
        est = _time_graph_replays(plan(args.steps), stream, torch)
        regions = _region_count(est, world, torch)
        res = _timed_regions(lambda: _time_graph_replays(plan(args.steps), stream, torch),
                             regions, world, dev, torch)
        del g_multi, g_one
        return res

    paths = {}
    for kind in ("fused", "chain", "per_launch"):
        (ms_k, reg_k), clk_k = timed(kind)
        paths[kind] = (ms_k, reg_k, clk_k)
    # headline: the fastest way of running a step
    best = min(paths, key=lambda k: paths[k][0])
    ms, reg, clocks = paths[best]
    ms_step = ms / args.steps
    value = world * wbytes * args.steps / (ms * 1e-3) / 1e9
    achieved = (wbytes + abytes) / (ms_step * 1e-3) / 1e9

    # ---------------- where the per-launch step's time goes: each kind of
    # product (one per layer) timed as its own PDL chain
    breakdown = {}
    for key in ("qkv", "wo", "w13", "w2"):
        gk = dec.capture_only(key, G, stream)
        _time_graph_replays([(gk, 1)], stream, torch)
        kms = statistics.median(_time_graph_replays([(gk, 1)], stream, torch)
                                for _ in range(5)) / G
        n_k, k_k = dec.shapes[key]
        kbytes = dec.layers * (n_k * k_k // 32 * 18)
        breakdown[key] = {"ms_per_step": kms, "launches": dec.layers,
                          "us_per_launch": kms * 1e3 / dec.layers,
                          "weight_gbs": kbytes / (kms * 1e-3) / 1e9}
        del gk
    breakdown["sum_ms"] = sum(v["ms_per_step"] for v in breakdown.values())
    breakdown["note"] = ("each kind's products of a step timed as their own PDL chain of "
                         "q4_gemv launches (CUDA events, graphs of 8 steps); their sum against "
                         "step_paths.per_launch.ms_per_step shows what running the four kinds "
                         "back to back adds or saves")

    # ---------------- e2e: host input -> step -> host output, every step
    rows = max(args.steps, 3)  # the 3 untimed warm-up steps use rows 0..2 too
    x_host = torch.empty((rows, 3072), dtype=torch.float32).pin_memory()
    x_host.copy_(torch.randn((rows, 3072), generator=torch.Generator().manual_seed(7)))
    y_host = torch.empty((rows, 3072), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((1, 3072), dtype=torch.float32, device=dev)
    if best == "fused":
        g_e2e, y_dev = dec.capture_fused([x_dev], stream), dec.x_fused
    else:
        g_e2e, y_dev = dec.capture([x_dev], stream, chain=best == "chain"), dec.x
    with torch.cuda.stream(stream):
        for s in range(3):
            x_dev.copy_(x_host[s:s + 1], non_blocking=True)
            g_e2e.replay()
            y_host[s:s + 1].copy_(y_dev, non_blocking=True)
    stream.synchronize()

    def e2e_region():
        _barrier(world)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for s in range(args.steps):
                x_dev.copy_(x_host[s:s + 1], non_blocking=True)
                g_e2e.replay()
                y_host[s:s + 1].copy_(y_dev, non_blocking=True)
        stream.synchronize()
        return (time.perf_counter() - t0) * 1e3

    e2e_times = [e2e_region() for _ in range(reg["regions"])]
    e2e_s = _barrier_max(statistics.median(e2e_times), world, torch) * 1e-3
    e2e = {"value": world * wbytes * args.steps / e2e_s / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": 3072 * 4, "d2h_bytes_per_step": 3072 * 4,
           "ms_per_step": e2e_s / args.steps * 1e3,
           "timing": f"host clock, median of {reg['regions']} regions of {args.steps} steps"}
    del g_e2e
    return {
        "value": value, "ms_per_step": ms_step,
        "config": {"workload": WORKLOAD, "layers": dec.layers, "hidden": 3072,
                   "gqa": "32Q/8KV", "ffn": 9216, "batch": 1,
                   "weight_bytes_per_step": wbytes, "activation_bytes_per_step": abytes,
                   "l2": "inputs larger than L2: 1.70 GB of weights per step vs 126 MB L2",
                   "timing": (f"CUDA events on the launching stream; median of "
                              f"{reg['regions']} timed regions of exactly {args.steps} steps "
                              f"(min {reg['min_ms'] / args.steps:.4f}, max "
                              f"{reg['max_ms'] / args.steps:.4f} ms/step), each bracketed by a "
                              f"barrier and synchronize; every graph replayed before timing"),
                   "graph": f"CUDA graphs of {G} steps, {PATH_NOTES[best]}",
                   "step_function": STEP_FUNCTION[best],
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": (args.traffic if args.traffic is not None else
                                 (_step_traffic(best) if dec.layers == 26 else None)),
                     "traffic_note": ("DRAM read + write bytes per step (ncu, a 2-layer step "
                                      "scaled to 26 layers); algorithmic bytes per step "
                                      f"{wbytes + abytes}"),
                     "kernel": KERNELS[best],
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "per_launch": ("algorithmic bytes of the 104 launches of a step / step time "
                                    "(every launch of the step is this kernel)"
                                    if best == "per_launch" else
                                    "algorithmic bytes of one step (one launch) / its time")},
        "step_paths": {k: {"ms_per_step": v[0] / args.steps,
                           "gbs": world * wbytes * args.steps / (v[0] * 1e-3) / 1e9,
                           "frac_of_hbm": wbytes * args.steps / (v[0] * 1e-3) / 1e9 / hbm,
                           "regions": v[1]["regions"], "note": PATH_NOTES[k],
                           "step_function": STEP_FUNCTION[k]}
                       for k, v in paths.items()},
        "per_launch_breakdown": breakdown,
        "e2e": e2e,
        "gpu_launches": args.steps * (dec.launches_per_step() if best == "per_launch" else 1),
        "clocks": clocks,
    }


def _run_single_gemv(args, dev, stream, hbm, torch):
    """Single batch-1 GEMV on the 4096 x 3072 decoder shape: Q4_0 weights
    N(0, 0.02^2), x N(0, 1) fp32, y fp32.  L2-cold: 36 distinct weight copies
    (255 MB, twice the L2) are rotated, 72 calls per CUDA graph."""
    import synth
    from bit_weight_quantized_03_b300 import FLAG_PDL, Workspace, q4_gemv, q4_quantize
    n, k, copies, reps = 4096, 3072, 36, 72
    Ws = []
    for c in range(copies):
        w = synth.torch_weights(n, k, seed=synth.seed_for(1, 0, c), device=dev)
        Ws.append(q4_quantize(w))
        del w
    x = synth.torch_activations(1, k, seed=synth.activation_seed(1000), device=dev)
    y = torch.empty((1, n), device=dev)
    ws = Workspace(dev)
    algo = n * k // 32 * 18 + 4 * (k + n)
    out = {"workload": "single Q4_0 GEMV 4096x3072, batch 1, fp32 x and y",
           "algorithmic_bytes_per_call": algo,
           "l2": f"{copies} weight copies rotated ({copies * n * k // 32 * 18 / 1e6:.0f} MB)"}
    from bit_weight_quantized_03_b300 import q4_gemv_q8, q4_gemv_r, q4_repack
    Rs = [q4_repack(W, n, k) for W in Ws]
    wsr = Workspace(dev)
    calls = {
        "q4_gemv_pdl": lambda i: q4_gemv(Ws[i % copies], n, k, x, y=y, workspace=ws,
                                         flags=FLAG_PDL, stream=stream),
        "q4_gemv": lambda i: q4_gemv(Ws[i % copies], n, k, x, y=y, workspace=ws, stream=stream),
        "q4_gemv_r": lambda i: q4_gemv_r(Rs[i % copies], n, k, x, y=y, workspace=wsr,
                                         stream=stream),
        "q4_gemv_r_pdl": lambda i: q4_gemv_r(Rs[i % copies], n, k, x, y=y, workspace=wsr,
                                             flags=FLAG_PDL, stream=stream),
        # the Q4 x Q8 integer path (x quantized per 32 inside the kernel)
        "q4_gemv_q8": lambda i: q4_gemv_q8(Ws[i % copies], n, k, x, y=y[0], stream=stream),
    }
    for name, call in calls.items():
        with torch.cuda.stream(stream):
            call(0)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    call(i)
        _time_graph_replays([(g, 2)], stream, torch)
        us = statistics.median(_time_graph_replays([(g, 1)], stream, torch) for _ in range(7)) \
            / reps * 1e3
        out[name] = {"us_per_call": us, "gbs": algo / (us * 1e-6) / 1e9,
                     "frac_of_hbm": algo / (us * 1e-6) / 1e9 / hbm}
        del g
    # the fastest fp32 path (the integer path computes a different product)
    best = min((v["us_per_call"], key) for key, v in out.items()
               if isinstance(v, dict) and key != "q4_gemv_q8")
    out["best"] = best[1]
    return out


PATH_NOTES = {
    "fused": "one q4_chain launch per step on the repacked weights",
    "chain": "one q4_gemv_chain launch per step on the GGUF weights",
    "per_launch": ("104 q4_gemv_prefetch launches per step with programmatic dependent launch, "
                   "each prefetching the next product's weights into L2"),
}
STEP_FUNCTION = {
    "fused": "per layer: qkv = Wqkv x; h = x + Wo q; g = W1h sigmoid(W1h) W3h; x' = h + W2 g",
    "chain": "per layer: qkv = Wqkv x; o = Wo q; g = W13 o; x' = W2 g1",
    "per_launch": "per layer: qkv = Wqkv x; o = Wo q; g = W13 o; x' = W2 g1",
}
KERNELS = {"fused": "chain_kernel", "chain": "gemv_chain_kernel", "per_launch": "gemv_b1_kernel"}


def _run_head_gather(args, dev, stream, hbm, torch):
    import synth
    from bit_weight_quantized_03_b300 import FLAG_PDL, Workspace, q4_embed_gather, q4_gemv, \
        q4_quantize

    # ---------------- output head GEMV and embedding gather (131072 x 3072 table)
    extra = {}
    if True:
        V, H = synth.VOCAB, 3072
        table = torch.empty((V, H // 32 * 18), dtype=torch.uint8, device=dev)
        for r0 in range(0, V, 16384):
            w = synth.torch_weights(16384, H, seed=synth.seed_for(3, 0, r0 // 16384), device=dev)
            q4_quantize(w, blocks=table[r0:r0 + 16384])
            del w
        xh = synth.torch_activations(1, H, seed=synth.activation_seed(3000), device=dev)
        logits = torch.empty((1, V), device=dev)
        ws = Workspace(dev)
        reps = 20
        gh = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            q4_gemv(table, V, H, xh, y=logits, workspace=ws, stream=stream)
            stream.synchronize()
            with torch.cuda.graph(gh, stream=stream):
                for _ in range(reps):
                    q4_gemv(table, V, H, xh, y=logits, workspace=ws, flags=FLAG_PDL,
                            stream=stream)
        _time_graph_replays([(gh, 2)], stream, torch)
        hms = _time_graph_replays([(gh, 3)], stream, torch) / (3 * reps)
        head_bytes = table.numel()
        extra["head_gemv"] = {"workload": "output head 3072->131072, batch 1",
                              "us_per_call": hms * 1e3,
                              "weight_gbs": head_bytes / (hms * 1e-3) / 1e9,
                              "frac_of_hbm": head_bytes / (hms * 1e-3) / 1e9 / hbm,
                              "note": "226 MB table > L2; consecutive calls re-read it"}
        del gh
        # the same head on the repacked table: the product, and the argmax of
        # the logits without writing them (one q4_chain link)
        from bit_weight_quantized_03_b300 import (OP_ARGMAX, Link, q4_chain, q4_gemv_r,
                                                  q4_repack)
        Rt = q4_repack(table, V, H)
        wsr = Workspace(dev)
        am = torch.zeros(2, dtype=torch.int32, device=dev)
        from bit_weight_quantized_03_b300 import q4_gemv_q8
        variants = {
            "q4_gemv_r": lambda: q4_gemv_r(Rt, V, H, xh, y=logits, workspace=wsr, stream=stream),
            "q4_gemv_q8": lambda: q4_gemv_q8(table, V, H, xh, y=logits[0], stream=stream),
            "argmax_no_logits": lambda: q4_chain([Link(Rt, V, H, xh, argmax=am, ops=OP_ARGMAX)],
                                                 workspace=wsr, stream=stream),
        }
        for name, call in variants.items():
            with torch.cuda.stream(stream):
                call()
                stream.synchronize()
                gv = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gv, stream=stream):
                    for _ in range(reps):
                        call()
            _time_graph_replays([(gv, 2)], stream, torch)
            vms = statistics.median(_time_graph_replays([(gv, 1)], stream, torch)
                                    for _ in range(5)) / reps
            algo = head_bytes + 4 * H + (8 if name == "argmax_no_logits" else 4 * V)
            extra["head_gemv"][name] = {"us_per_call": vms * 1e3,
                                        "weight_gbs": head_bytes / (vms * 1e-3) / 1e9,
                                        "frac_of_hbm": algo / (vms * 1e-3) / 1e9 / hbm}
            del gv
        del Rt
        gather = {}
        for B in (1, 64, 4096):
            ids = synth.torch_token_ids(B, V, seed=B, device=dev)
            out = torch.empty((B, H), device=dev)
            gg = torch.cuda.CUDAGraph()
            r = 50 if B < 4096 else 20
            with torch.cuda.stream(stream):
                q4_embed_gather(table, V, H, ids, out=out, stream=stream)
                stream.synchronize()
                with torch.cuda.graph(gg, stream=stream):
                    for _ in range(r):
                        q4_embed_gather(table, V, H, ids, out=out, stream=stream)
            _time_graph_replays([(gg, 2)], stream, torch)
            gms = _time_graph_replays([(gg, 3)], stream, torch) / (3 * r)
            nbytes = B * (H // 32 * 18 + H * 4 + 4)
            gather[str(B)] = {"us_per_call": gms * 1e3, "gbs": nbytes / (gms * 1e-3) / 1e9}
        extra["embed_gather"] = gather
        del table
    return extra


def _run_gemm(args, world, dev, stream, bf16_burst, bf16_sust, peak_src, torch):
    """Encoder/prefill GEMM stack at M = 375, 1500 and 3000 frames (headline: 3000)."""
    import synth
    from bit_weight_quantized_03_b300.stacks import EncoderStack

    try:
        enc = EncoderStack(frames=3000, device=dev)
        per_m = {}
        for M in (375, 1500, 3000):
            x0 = synth.torch_activations(M, 1280, seed=synth.activation_seed(4000), device=dev,
                                         dtype=torch.bfloat16)
            ge = enc.capture(x0, stream)
            _time_graph_replays([(ge, 2)], stream, torch)
            _barrier(world)
            gms = _barrier_max(_time_graph_replays([(ge, 5)], stream, torch) / 5, world, torch)
            per_m[M] = (gms, enc.flops(M) / (gms * 1e-3) / 1e12)
            del ge
        gms, tflops = per_m[3000]
        gemm = {"workload": "encoder linear stack, 32 layers x (qkv 1280->3840, out "
                            "1280->1280, up 1280->5120, down 5120->1280), M=3000 frames",
                "value": world * tflops, "unit": "TFLOP/s", "ms_per_pass": gms,
                "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_burst,
                             "unit": "TFLOP/s", "frac": tflops / bf16_burst,
                             "kernel": "gemm_tc_kernel",
                             "peak_source": f"{peak_src} bf16 burst (cuBLAS 8192^3)"},
                "frac_of_sustained": tflops / bf16_sust,
                "by_frames": {str(M): {"ms_per_pass": v[0], "tflops": v[1],
                                       "frac_of_peak": v[1] / bf16_burst}
                              for M, v in per_m.items()},
                "gpu_launches_per_pass": enc.launches_per_pass()}
        del enc
    except Exception as e:  # reported, never silently replaced
        gemm = {"error": f"{type(e).__name__}: {e}"}
    return gemm


def _fp32_fma_peak(dev, stream, torch):
    """Measured fp32 FMA ceiling of this GPU: cuBLAS SGEMM 8192^3 with TF32 off
    (a denominator only; nothing on the Q4 path uses it)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        g = torch.Generator(device=dev).manual_seed(11)
        a = torch.randn((8192, 8192), device=dev, generator=g)
        b = torch.randn((8192, 8192), device=dev, generator=g)
        c = torch.empty((8192, 8192), device=dev)
        with torch.cuda.stream(stream):
            for _ in range(2):
                torch.matmul(a, b, out=c)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                torch.matmul(a, b, out=c)
            e1.record(stream)
        stream.synchronize()
        secs = e0.elapsed_time(e1) * 1e-3 / 5
        return 2 * 8192 ** 3 / secs / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


CROSSOVER_SHAPES = [(4096, 3072), (1024, 3072), (3072, 4096), (9216, 3072), (3072, 9216),
                    (3840, 1280), (1280, 1280), (5120, 1280), (1280, 5120)]


def _crossover_by_shape(dev, stream, torch, ms=(1, 2, 3, 4, 5, 6, 8, 12, 16)):
    """Per decoder and encoder shape: fp32 GEMV vs bf16 tensor-core GEMM time at
    each M the GEMV takes, L2-cold (weight copies rotated, >= 256 MB), and the
    largest M at which the GEMV is still faster for every M up to it (the
    value q4_linear_crossover_m returns for that shape)."""
    import synth
    from bit_weight_quantized_03_b300 import FLAG_PDL, Workspace, q4_gemm, q4_gemv, q4_quantize
    out = {}
    for n, k in CROSSOVER_SHAPES:
        wbytes = n * k // 32 * 18
        copies = max(2, -(-(256 << 20) // wbytes))
        Ws = []
        for c in range(copies):
            w = synth.torch_weights(n, k, seed=synth.seed_for(5, 1, c), device=dev)
            Ws.append(q4_quantize(w))
            del w
        reps = max(copies, 24)
        ws = Workspace(dev)
        times = {}
        for M in ms:
            x32 = synth.torch_activations(M, k, seed=synth.activation_seed(5100, M), device=dev)
            xbf = x32.to(torch.bfloat16)
            y = torch.empty((M, n), device=dev)
            t = {}
            for name, fn in (("gemv", lambda W: q4_gemv(W, n, k, x32, y=y, workspace=ws,
                                                        flags=FLAG_PDL, stream=stream)),
                             ("gemm", lambda W: q4_gemm(W, n, k, xbf, Y=y, workspace=ws,
                                                        flags=FLAG_PDL, stream=stream))):
                with torch.cuda.stream(stream):
                    fn(Ws[0])
                    stream.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(reps):
                            fn(Ws[i % copies])
                _time_graph_replays([(g, 1)], stream, torch)
                t[name] = statistics.median(_time_graph_replays([(g, 1)], stream, torch)
                                            for _ in range(3)) / reps * 1e3
                del g
            times[str(M)] = {"gemv_us": t["gemv"], "gemm_us": t["gemm"]}
        last = 0
        for M in ms:
            if times[str(M)]["gemv_us"] <= times[str(M)]["gemm_us"]:
                last = M
            else:
                break
        out[f"{n}x{k}"] = {"by_m": times, "gemv_up_to_m": last, "copies": copies}
        del Ws
    return out


def _run_crossover(args, dev, stream, hbm, bf16_burst, torch):
    """Batched decode on the 4096x3072 decoder shape: fp32 GEMV vs bf16 tensor-core
    GEMM for M in 1..128 concurrent streams, L2-cold (72 weight copies, 510 MB)."""
    import synth
    from bit_weight_quantized_03_b300 import (FLAG_PDL, GEMV_MAX_M, Workspace, q4_gemm, q4_gemv,
                                              q4_quantize)
    n, k, copies, reps = 4096, 3072, 72, 72
    Ws = []
    for c in range(copies):
        w = synth.torch_weights(n, k, seed=synth.seed_for(5, 0, c), device=dev)
        Ws.append(q4_quantize(w))
        del w
    wbytes = n * k // 32 * 18
    ws = Workspace(dev)
    rows = {}
    for M in (1, 2, 4, 8, 16, 32, 64, 128):
        x32 = synth.torch_activations(M, k, seed=synth.activation_seed(5000, M), device=dev)
        xbf = x32.to(torch.bfloat16)
        y = torch.empty((M, n), device=dev)
        res = {}
        paths = [("gemm", lambda W: q4_gemm(W, n, k, xbf, Y=y, workspace=ws, flags=FLAG_PDL,
                                           stream=stream))]
        if M <= GEMV_MAX_M:
            paths.insert(0, ("gemv", lambda W: q4_gemv(W, n, k, x32, y=y, workspace=ws,
                                                       flags=FLAG_PDL, stream=stream)))
        for name, fn in paths:
            with torch.cuda.stream(stream):
                fn(Ws[0])
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(reps):
                        fn(Ws[i % copies])
            _time_graph_replays([(g, 1)], stream, torch)
            us = _time_graph_replays([(g, 3)], stream, torch) / (3 * reps) * 1e3
            byts = wbytes + M * k * (4 if name == "gemv" else 2) + M * n * 4
            res[name] = {"us": us, "gbs": byts / (us * 1e-6) / 1e9,
                         "tflops": 2 * M * n * k / (us * 1e-6) / 1e12}
            del g
        rows[str(M)] = res
    fp32_peak = _fp32_fma_peak(dev, stream, torch)
    for r in rows.values():
        if "gemv" in r:
            r["gemv"]["frac_of_fp32_peak"] = r["gemv"]["tflops"] / fp32_peak
    cross = None
    for M in (1, 2, 4, 8, 16, 32, 64, 128):
        r = rows[str(M)]
        if "gemv" not in r or r["gemm"]["us"] < r["gemv"]["us"]:
            cross = M
            break
    del Ws
    by_shape = _crossover_by_shape(dev, stream, torch)
    return {"workload": "batched decode, 4096x3072 Q4_0, M concurrent streams, fp32 x (GEMV) / "
                        "bf16 x (tensor-core GEMM), fp32 y; 72 weight copies rotated (L2-cold)",
            "by_m": rows, "crossover_m": cross, "by_shape": by_shape,
            "fp32_peak_tflops": {"value": fp32_peak,
                                 "source": "cuBLAS SGEMM 8192^3, TF32 off, measured in this run"},
            "note": "crossover_m = smallest M at which the tensor-core GEMM is faster; "
                    "gemv frac_of_fp32_peak = its 2*M*n*k flop rate over the measured fp32 "
                    "FMA ceiling"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["all", "stack", "single", "head", "gather", "gemm",
                                       "crossover"],
                    default="all",
                    help="run one section (profiling runs); the default runs all of them")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=None,
                    help="decoder layers of the stack (default 26; fewer only for profiling)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="per-launch DRAM bytes of the GEMV kernel from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
