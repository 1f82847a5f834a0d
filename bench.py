#!/usr/bin/env python3
"""Benchmark: nvfp4_gemv us/call and achieved HBM GB/s on the Llama-3-8B-shaped
decode linears (qkv 6144x4096, o_proj 4096x4096, gate_up 28672x4096 with
silu_mul, down 4096x14336) at M = 1, 2, 4, 8, 16, 32 tokens.

One step = one pass of the NVFP4 GEMV over all 4 layers x 6 token counts (24
launches, chained with programmatic dependent launch).  Inputs are synthetic
(seeded) and resident in HBM; the weights are rotated over 5 replicas so a
layer's weights are re-read at a reuse distance of ~490 MB (> 3 x the 129 MB
L2): every call streams its weights from HBM.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the FP64 CPU oracle
on a bounded sample of the same workload instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

import torch  # noqa: E402

from moe_nvfp4_gemv_gb300 import synth  # noqa: E402

METRIC = "nvfp4_gemv µs/call and achieved HBM GB/s (% of GB300 peak) at M=1..32"
LAYERS = synth.LLAMA8B_LAYERS
MS = synth.LLAMA8B_M
GS = 0.01
PHASES = 7  # replica rotation of the step (see run_gpu)
WORKLOAD = "llama3-8b decode linears (qkv, o_proj, gate_up+silu_mul, down), NVFP4, M=1,2,4,8,16,32"


def nvfp4_bytes(M, N, K, silu):
    """Algorithmic bytes of one call: codes + scales + activations + output
    (the output of silu_mul is [M, N/2])."""
    n_out = N // 2 if silu else N
    return N * K // 2 + N * K // 16 + 2 * M * K + 2 * M * n_out


def step_bytes():
    return sum(nvfp4_bytes(M, N, K, s) for M in MS for (N, K, s) in LAYERS.values())


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_nvfp4_gemv_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "nvfp4_gemv_llama8b_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, local, world, dist
    return rank, local, world, None


def max_over_ranks(v, dist, device):
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# --------------------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------------------

def oracle_sample(budget_s=15.0, threads=None):
    """Time the FP64 oracle on a bounded sample of the workload: for each
    (layer, M) a slice of output rows, until ~budget_s of work.  Returns
    (GB/s-equivalent of the sampled algorithmic bytes, threads, description)."""
    import numpy as np
    import oracle
    threads = threads or (os.cpu_count() or 1)
    rows_per_call = 64
    done_bytes, spent = 0.0, 0.0
    calls = 0
    cache = {}
    rounds = 0
    while spent < budget_s and rounds < 50:
        rounds += 1
        for name, (N, K, silu) in LAYERS.items():
            if name not in cache:
                w = synth.fp4_bytes(N, K, seed=1).numpy()
                sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=2).numpy()
                cache[name] = (w, sf)
            w, sf = cache[name]
            n_out = N // 2 if silu else N
            for M in MS:
                x = synth.activations(M, K, seed=3 + M).view(torch.int16).numpy().view(np.uint16)
                rows = np.arange(rows_per_call, dtype=np.int64) + (rounds * rows_per_call) % (n_out - rows_per_call)
                t0 = time.perf_counter()
                oracle.nvfp4_gemv(x, w, sf, GS, silu_mul=silu, rows=rows, threads=threads)
                spent += time.perf_counter() - t0
                frac = rows_per_call / n_out
                done_bytes += nvfp4_bytes(M, N, K, silu) * frac
                calls += 1
            if spent >= budget_s:
                break
    desc = (f"{calls} oracle calls of {rows_per_call} output rows each over the 24 (layer, M) cases, "
            f"{spent:.1f} s; bytes scaled by the sampled fraction of each call")
    return done_bytes / spent / 1e9, threads, desc


def run_reference(args):
    rank, local, world, dist = dist_setup(args.gpus)
    if rank != 0:
        return 0
    value, threads, desc = oracle_sample(budget_s=max(5.0, 20.0 / max(1, args.steps)))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_bytes() / (value * 1e9) * 1e3, 3),
            "ms_per_step_kind": "extrapolated: one step's algorithmic bytes / the sampled oracle throughput",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "device": "host CPU (FP64 oracle)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------------------

def capture_graph(fn, dev):
    """A CUDA graph of the launches `fn` makes (called once eagerly first, so
    every lazily-configured attribute is set before capture)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        fn()
        side.synchronize()
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    return g


def run_gpu(args):
    rank, local, world, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from moe_nvfp4_gemv_gb300 import fp4gemv

    # Weights: every layer has a pool of replicas, at least PHASES and at
    # least 400 MB.  In the step, call c of a layer (c = step * 6 + m_index)
    # reads replica c % PHASES, so a replica comes back only after 6 other
    # calls of each of the 4 layers (~740 MB of other weights, > 5 x L2).
    weights = {}
    for name, (N, K, silu) in LAYERS.items():
        nb = N * K // 2 + fp4gemv.scale_bytes(N, K)
        weights[name] = [(synth.fp4_bytes(N, K, seed=1000 * r + 1, device=dev),
                          synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=1000 * r + 2, device=dev))
                         for r in range(max(PHASES, replicas_for(nb)))]
    gs = torch.tensor([GS], dtype=torch.float32, device=dev)
    # The step's activations and outputs each live in one buffer (16-byte
    # aligned views per call), so end to end a step is one host-to-device
    # copy of its inputs and one device-to-host copy of its results.
    def packed(shapes):
        offs, n = {}, 0
        for k, (r, c) in shapes.items():
            offs[k] = n
            n += (r * c + 7) // 8 * 8
        flat = torch.empty(n, dtype=torch.bfloat16, device=dev)
        return flat, {k: flat[o:o + r * c].view(r, c) for (k, (r, c)), o in zip(shapes.items(), offs.values())}
    x_flat, xs = packed({(name, M): (M, LAYERS[name][1]) for name in LAYERS for M in MS})
    for (name, M), v in xs.items():
        v.copy_(synth.activations(M, LAYERS[name][1], seed=10 * M + 3, device=dev))
    out_flat, outs = packed({(name, M): (M, LAYERS[name][0] // (2 if LAYERS[name][2] else 1))
                             for name in LAYERS for M in MS})
    stream = torch.cuda.current_stream(dev)

    def step_with(phase, xv=None, ov=None, keep=lambda M: True):
        """The step's calls in phase `phase` of the replica rotation (all 24,
        or those whose token count passes `keep`)."""
        xv = xs if xv is None else xv
        ov = outs if ov is None else ov

        def fn():
            for mi, M in enumerate(MS):
                if not keep(M):
                    continue
                for name, (N, K, silu) in LAYERS.items():
                    w, sf = weights[name][(phase * len(MS) + mi) % PHASES]
                    fp4gemv.nvfp4_gemv(xv[(name, M)], w, sf, gs, silu_mul=silu, pdl=True, out=ov[(name, M)])
        return fn

    # A decode server replays its step as a CUDA graph: one graph per phase
    # of the replica rotation, replayed in turn.
    launches0 = fp4gemv.launch_count()
    graphs = [capture_graph(step_with(ph), dev) for ph in range(PHASES)]
    launches_per_step = (fp4gemv.launch_count() - launches0) // (2 * PHASES)
    for i in range(max(args.warmup, PHASES)):
        graphs[i % PHASES].replay()
    torch.cuda.synchronize()
    assert fp4gemv.get_device_error() == 0, "device error during warm-up"

    # ---- timed region (device-resident inputs) ----
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for i in range(args.steps):
            graphs[i % PHASES].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    launches = launches_per_step * args.steps
    ms_total = e0.elapsed_time(e1)
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    total_bytes = step_bytes() * args.steps * world
    value = total_bytes / (ms_total * 1e-3) / 1e9
    del graphs

    # ---- each kernel alone: the step's calls of one kernel, same rotation ----
    # (register-fed kernels: the 20 calls with M <= 16; tcgen05 kernel: M = 32)
    kernels = {}
    for kname, keep in (("gemv_rf_kernel", lambda M: M <= 16), ("gemv_kernel", lambda M: M > 16)):
        gk = [capture_graph(step_with(ph, keep=keep), dev) for ph in range(PHASES)]
        for i in range(PHASES):
            gk[i % PHASES].replay()
        reps = max(args.steps, PHASES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            gk[i % PHASES].replay()
        b.record(stream)
        torch.cuda.synchronize()
        n_calls = sum(1 for M in MS if keep(M)) * len(LAYERS)
        kb = sum(nvfp4_bytes(M, N, K, s) for M in MS if keep(M) for (N, K, s) in LAYERS.values())
        us = a.elapsed_time(b) * 1e3 / (reps * n_calls)
        kernels[kname] = {"launches_per_step": n_calls, "bytes_per_launch": round(kb / n_calls),
                          "us_per_launch": round(us, 3), "GB/s": round(kb / n_calls / (us * 1e-6) / 1e9, 1)}
        del gk

    # ---- per-call us: each (layer, M) alone, every replica of the layer's
    # pool (>= 400 MB) in turn within one graph ----
    per_call = {}
    for name, (N, K, silu) in LAYERS.items():
        per_call[name] = {}
        pool = weights[name]
        calls = max(20, len(pool))
        for M in MS:
            def fn(name=name, M=M, silu=silu, pool=pool, calls=calls):
                for i in range(calls):
                    w, sf = pool[i % len(pool)]
                    fp4gemv.nvfp4_gemv(xs[(name, M)], w, sf, gs, silu_mul=silu, pdl=True, out=outs[(name, M)])
            g = capture_graph(fn, dev)
            g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(3):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (3 * calls)
            per_call[name][str(M)] = {"us": round(us, 2),
                                      "GB/s": round(nvfp4_bytes(M, N, K, silu) / (us * 1e-6) / 1e9, 1)}
            del g

    # ---- end to end through the public API with pinned host buffers ----
    # A serving loop: every step uploads its 24 activation blocks (one copy
    # from pinned host memory), runs the 24 GEMVs and downloads their outputs
    # (one copy).  The copies run on their own stream with double-buffered
    # device blocks, so the upload of step i+1 and the download of step i
    # overlap the GEMVs of step i; every copy of every step is inside the
    # timed region.
    host_x = x_flat.cpu().pin_memory()
    host_out = torch.empty(out_flat.shape, dtype=out_flat.dtype).pin_memory()
    h2d = host_x.numel() * host_x.element_size()
    d2h = host_out.numel() * host_out.element_size()
    x_flat2, xs2 = packed({(name, M): (M, LAYERS[name][1]) for name in LAYERS for M in MS})
    out_flat2, outs2 = packed({(name, M): (M, LAYERS[name][0] // (2 if LAYERS[name][2] else 1))
                               for name in LAYERS for M in MS})
    bufs = [(x_flat, xs, out_flat, outs), (x_flat2, xs2, out_flat2, outs2)]
    copy_stream = torch.cuda.Stream(dev)

    def e2e_pipelined(nsteps):
        graphs_b = [[capture_graph(step_with(ph, bufs[b][1], bufs[b][3]), dev) for b in range(2)]
                    for ph in range(PHASES)]
        h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
        comp_done = [torch.cuda.Event(), torch.cuda.Event()]

        def run(n):
            copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                bufs[0][0].copy_(host_x, non_blocking=True)
                h2d_done[0].record(copy_stream)
            for i in range(n):
                b = i % 2
                stream.wait_event(h2d_done[b])
                graphs_b[i % PHASES][b].replay()
                comp_done[b].record(stream)
                with torch.cuda.stream(copy_stream):
                    if i + 1 < n:  # (buffer 1-b: step i-1 is done with it, in this stream's order)
                        bufs[1 - b][0].copy_(host_x, non_blocking=True)
                        h2d_done[1 - b].record(copy_stream)
                    copy_stream.wait_event(comp_done[b])
                    host_out.copy_(bufs[b][2], non_blocking=True)
            stream.wait_stream(copy_stream)
        run(2 * PHASES)  # warm-up
        torch.cuda.synchronize()
        barrier(dist)
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run(nsteps)
        b2.record(stream)
        torch.cuda.synchronize()
        del graphs_b
        return max_over_ranks(a.elapsed_time(b2), dist, dev)

    def e2e_with(ph):
        def fn():
            x_flat.copy_(host_x, non_blocking=True)  # the step's inputs
            step_with(ph)()
            host_out.copy_(out_flat, non_blocking=True)  # the step's results
        return fn

    def timed(step_fns, nsteps):
        barrier(dist)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(nsteps):
            step_fns[i % len(step_fns)]()
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b), dist, dev)

    # (a) graph-replayed GEMVs with pipelined copies; (b) the same calls and
    # copies issued eagerly, one stream
    e2e_ms = e2e_pipelined(args.steps)
    eager_fns = [e2e_with(ph) for ph in range(PHASES)]
    for f in eager_fns[:2]:
        f()
    eager_ms = timed(eager_fns, args.steps)
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9
    eager_value = total_bytes / (eager_ms * 1e-3) / 1e9
    assert fp4gemv.get_device_error() == 0, "device error during the timed region"
    del weights

    peak, peak_kind = read_peaks()
    dom = kernels["gemv_rf_kernel"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, threads, desc = oracle_sample(budget_s=args.cpu_budget)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc}
    extra = None
    if rank == 0 and not args.no_configs:
        extra = config_results(dev, compact=True)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "launches_per_step": launches_per_step,
                       "us_per_call_avg": round(ms_step * 1e3 / launches_per_step, 3),
                       "l2": (f"inputs larger than L2 instead of a flush: call c of a layer (c = step * 6 + "
                              f"m_index) reads weight replica c % {PHASES}, so each replica comes back after 6 "
                              f"calls of each of the 4 layers (~740 MB > 5 x the 129 MB L2); per-call timing "
                              f"rotates >= 400 MB of replicas of the one layer"),
                       "global_scale": GS, "pdl": True,
                       "launch": f"one CUDA graph per rotation phase ({PHASES}), PDL edges between the launches"},
            "roofline": {"bound": "hbm", "achieved": dom["GB/s"], "peak": peak, "unit": "GB/s",
                         "frac": round(dom["GB/s"] / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                         "traffic": traffic_from_profile(),
                         "kernel": "fp4::gemv_rf_kernel / fp4::gemv_slab_kernel (the register-fed kernels: M <= 16)",
                         "bytes_per_launch": dom["bytes_per_launch"], "us_per_launch": dom["us_per_launch"],
                         "timing": "CUDA events around graph replays of the step's 20 M <= 16 calls, same rotation"},
            "kernels": kernels,
            "step_frac": round(value / world / peak, 4),
            "per_call": per_call,
            "clocks": clk.summary(),
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "launch": "CUDA graph of the step's GEMVs; its input upload and output download on a copy stream, overlapped with the neighbouring steps",
                    "eager_value": round(eager_value, 1)},
            "gpu_launches": launches,
            "cpu_baseline": cpu,
            "configs": extra,
        }
        print(json.dumps(line))
    if rank == 0 and args.extended:
        with open(args.extended, "w") as f:
            json.dump(config_results(dev, compact=False), f, indent=1)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------------------
# Extended suite (--extended PATH): every configuration, L2-cold, one JSON file
# --------------------------------------------------------------------------------------

def time_calls(fn_list, reps, stream):
    """Average device time (us) of one call when the calls in fn_list are
    issued round-robin (each fn uses its own weight replica), replayed from a
    CUDA graph so host launch cost does not leak into the number."""
    dev = stream.device

    def fn():
        for i in range(reps):
            fn_list[i % len(fn_list)]()
    g = capture_graph(fn, dev)
    g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (2 * reps)


def replicas_for(nbytes, min_reps=2, target=400 << 20):
    return max(min_reps, -(-target // max(1, nbytes)))


def read_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def config_results(dev, compact=True):
    """Every configuration besides the default step, L2-cold (weights rotated
    over >= 400 MB of replicas, MoE over 8 routings): the 70B layers and
    their dequantize_rows, the 8B layers with BF16 weights, the MoE block,
    the N = K = 8192 sweep of the GEMV against dequantize + GEMM (with
    `compact`, the sweep at M = 1, 8, 32, 128 only) and the W4A4 path on
    that layer."""
    from moe_nvfp4_gemv_gb300 import fp4gemv
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = read_peaks()
    tpeak, tpeak_kind = read_tflops()
    gs = torch.tensor([GS], dtype=torch.float32, device=dev)
    res = {"peak_hbm_gbs": peak, "peak_kind": peak_kind, "peak_bf16_tflops": tpeak, "tflops_kind": tpeak_kind,
           "l2_policy": "weights rotated over replicas, >= 400 MB"}

    def fp4_layer(N, K, seed):
        nb = N * K // 2 + N * K // 16
        reps = replicas_for(nb)
        return [(synth.fp4_bytes(N, K, seed=seed + 10 * r, device=dev),
                 synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=seed + 10 * r + 1, device=dev))
                for r in range(reps)]

    # 70B layers (nvfp4_gemv) + dequantize_rows
    t70 = {}
    for name, (N, K, silu) in synth.LLAMA70B_LAYERS.items():
        ws = fp4_layer(N, K, 7)
        t70[name] = {}
        for M in synth.LLAMA70B_M:
            x = synth.activations(M, K, seed=M, device=dev)
            out = torch.empty(M, N // 2 if silu else N, dtype=torch.bfloat16, device=dev)
            fns = [lambda w=w, sf=sf: fp4gemv.nvfp4_gemv(x, w, sf, gs, silu_mul=silu, out=out) for w, sf in ws]
            us = time_calls(fns, 20, stream)
            gbs = nvfp4_bytes(M, N, K, silu) / (us * 1e-6) / 1e9
            t70[name][str(M)] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 3)}
        dq = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
        fns = [lambda w=w, sf=sf: fp4gemv.dequantize_rows(w, sf, out=dq) for w, sf in ws[:2]]
        us = time_calls(fns, 10, stream)
        gbs = N * K * (0.5 + 1 / 16 + 2) / (us * 1e-6) / 1e9
        t70[name]["dequantize_rows"] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 3)}
        del ws, dq
    res["llama70b"] = t70

    # BF16 weights on the 8B layers
    tb = {}
    for name, (N, K, silu) in LAYERS.items():
        nb = 2 * N * K
        ws = [synth.bf16_weight(N, K, seed=r, device=dev) for r in range(replicas_for(nb))]
        tb[name] = {}
        for M in MS:
            x = synth.activations(M, K, seed=M, device=dev)
            out = torch.empty(M, N // 2 if silu else N, dtype=torch.bfloat16, device=dev)
            fns = [lambda w=w: fp4gemv.bf16_gemv(x, w, silu_mul=silu, out=out) for w in ws]
            us = time_calls(fns, 20, stream)
            byts = nb + 2 * M * K + 2 * M * (N // 2 if silu else N)
            tb[name][str(M)] = {"us": round(us, 2), "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                                "frac": round(byts / (us * 1e-6) / 1e9 / peak, 3)}
        del ws
    res["llama8b_bf16"] = tb

    res["decode_chain"] = decode_chain(dev, gs, peak, Ms=(1, 4, 8) if compact else (1, 2, 4, 8, 16, 32))

    # BF16 GEMV against cuBLAS (torch.nn.functional.linear) on the 8B layers
    bc = {}
    for name, (N, K, silu) in LAYERS.items():
        ws = [synth.bf16_weight(N, K, seed=r, device=dev) for r in range(replicas_for(2 * N * K))]
        bc[name] = {}
        for M in ((1, 8, 32, 128) if compact else (1, 2, 4, 8, 16, 32, 64, 128)):
            x = synth.activations(M, K, seed=M, device=dev)
            out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            us_g = time_calls([lambda w=w: fp4gemv.bf16_gemv(x, w, out=out) for w in ws], 20, stream)
            us_c = time_calls([lambda w=w: torch.matmul(x, w.t(), out=out) for w in ws], 20, stream)
            bc[name][str(M)] = {"gemv_us": round(us_g, 2), "cublas_us": round(us_c, 2)}
        del ws
    res["bf16_gemv_vs_cublas"] = bc

    # MoE block
    c = synth.MOE
    E, H, I, SI, topk = c["E"], c["H"], c["I"], c["SI"], c["topk"]
    w1 = synth.fp4_bytes(E * 2 * I, H, seed=1, device=dev).view(E, 2 * I, H // 2)
    w1_sf = synth.e4m3_bytes(E * fp4gemv.scale_bytes(2 * I, H), seed=2, device=dev)
    w2 = synth.fp4_bytes(E * H, I, seed=3, device=dev).view(E, H, I // 2)
    w2_sf = synth.e4m3_bytes(E * fp4gemv.scale_bytes(H, I), seed=4, device=dev)
    wsh = synth.fp4_bytes(2 * SI, H, seed=5, device=dev)
    ssh = synth.e4m3_bytes(fp4gemv.scale_bytes(2 * SI, H), seed=6, device=dev)
    wsd = synth.fp4_bytes(H, SI, seed=7, device=dev)
    ssd = synth.e4m3_bytes(fp4gemv.scale_bytes(H, SI), seed=8, device=dev)
    alpha = synth.expert_alphas(E, device=dev)
    gsh = torch.tensor([0.01], device=dev)
    tm = {}
    ex_gu = 2 * I * H // 2 + fp4gemv.scale_bytes(2 * I, H)
    ex_dn = H * I // 2 + fp4gemv.scale_bytes(H, I)
    # Each kernel timed from a CUDA graph (host launch cost excluded, as for
    # the dense layers) over R routings of the same batch size: every call
    # touches other experts, so the ~8 experts of one call are not in L2 from
    # the previous call.
    R = 8
    for M in synth.MOE_M:
        rts = [synth.routing(M, E, topk, seed=M * 1000 + r, device=dev) for r in range(R)]
        x = synth.activations(M, H, seed=M, device=dev)
        act = torch.empty(M * topk, I, dtype=torch.bfloat16, device=dev)
        sact = torch.empty(M, SI, dtype=torch.bfloat16, device=dev)
        out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        distinct = statistics.mean(int(torch.unique(ids).numel()) for ids, _ in rts)
        gu_b = (distinct + 1) * ex_gu + 2 * M * H + 2 * M * topk * I + 2 * M * SI + 4 * M * topk
        dn_b = (distinct + 1) * ex_dn + 2 * M * topk * I + 2 * M * SI + 2 * M * H + 8 * M * topk
        gu_fns = [lambda ids=ids: fp4gemv.moe_gate_up(x, ids, w1, w1_sf, alpha, act, wsh, ssh, gsh, sact)
                  for ids, _ in rts]
        dn_fns = [lambda ids=ids, tw=tw: fp4gemv.moe_down_combine(act, ids, tw, w2, w2_sf, alpha, sact, wsd, ssd,
                                                                  gsh, out)
                  for ids, tw in rts]
        ug = time_calls(gu_fns, 2 * R, stream)
        ud = time_calls(dn_fns, 2 * R, stream)
        tm[str(M)] = {"distinct_experts": round(distinct, 1),
                      "gate_up": {"us": round(ug, 2), "GB/s": round(gu_b / (ug * 1e-6) / 1e9, 1),
                                  "frac": round(gu_b / (ug * 1e-6) / 1e9 / peak, 3)},
                      "down_combine": {"us": round(ud, 2), "GB/s": round(dn_b / (ud * 1e-6) / 1e9, 1),
                                       "frac": round(dn_b / (ud * 1e-6) / 1e9 / peak, 3)}}
    res["moe"] = tm
    del w1, w2, w1_sf, w2_sf

    # M sweep on N = K = 8192: nvfp4_gemv vs dequantize_rows + bf16 GEMM
    N = K = synth.SWEEP_NK
    ws = fp4_layer(N, K, 11)
    wb = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
    wbs = [torch.empty(N, K, dtype=torch.bfloat16, device=dev) for _ in range(replicas_for(2 * N * K))]
    for (w, sf), b in zip(ws * len(wbs), wbs):
        fp4gemv.dequantize_rows(w, sf, out=b)
    sw = {}
    for M in ((1, 8, 32, 128) if compact else synth.SWEEP_M):
        x = synth.activations(M, K, seed=M, device=dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        fns = [lambda w=w, sf=sf: fp4gemv.nvfp4_gemv(x, w, sf, gs, out=out) for w, sf in ws]
        us_g = time_calls(fns, 20, stream)
        fns2 = [lambda w=w, sf=sf: fp4gemv.dequant_gemm(x, w, sf, gs, w_bf16=wb, out=out) for w, sf in ws]
        us_d = time_calls(fns2, 10, stream)
        b_g = nvfp4_bytes(M, N, K, False)
        b_d = N * K * (0.5 + 1 / 16 + 2) + 2 * N * K + 2 * M * K + 2 * M * N
        # the GEMM half alone (bf16 weights already dequantized, rotated)
        fns3 = [lambda b=b: fp4gemv.bf16_gemv(x, b, out=out) for b in wbs]
        us_m = time_calls(fns3, 10, stream)
        tf = 2 * M * N * K / (us_m * 1e-6) / 1e12
        sw[str(M)] = {"gemv_us": round(us_g, 2), "gemv_GB/s": round(b_g / (us_g * 1e-6) / 1e9, 1),
                      "gemv_frac": round(b_g / (us_g * 1e-6) / 1e9 / peak, 3),
                      "gemv_TFLOP/s": round(2 * M * N * K / (us_g * 1e-6) / 1e12, 2),
                      "dequant_gemm_us": round(us_d, 2), "dequant_gemm_GB/s": round(b_d / (us_d * 1e-6) / 1e9, 1),
                      "dequant_gemm_frac": round(b_d / (us_d * 1e-6) / 1e9 / peak, 3),
                      "gemm_us": round(us_m, 2), "gemm_TFLOP/s": round(tf, 1), "gemm_tflops_frac": round(tf / tpeak, 4)}
    rows_m = [int(m) for m in sw]
    cross = next((m for m in rows_m if sw[str(m)]["dequant_gemm_us"] < sw[str(m)]["gemv_us"]), None)
    res["sweep_8192"] = {"rows": sw, "crossover_M": cross}
    del wbs, wb

    # W4A4 on the same layer: quantise the activations, then the NVFP4 x NVFP4
    # GEMM (w4a4_linear: one quantisation launch writing codes, scales and
    # the exact dequantised operand, then the GEMM launches), against the
    # W4A16 GEMV of the sweep; and the quantisation alone on an 8192 x 8192
    # activation block (HBM-bound: larger than L2, so every call is cold)
    gsi_v = 448.0 * 6 / 4.0
    gsi = torch.tensor([gsi_v], dtype=torch.float32, device=dev)
    alpha = torch.tensor([GS / gsi_v], dtype=torch.float32, device=dev)
    w4 = {}
    for M in ((1, 32, 128) if compact else (1, 8, 32, 128, 512)):
        x = synth.activations(M, K, seed=M, device=dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        xq = torch.empty(M, K // 2, dtype=torch.uint8, device=dev)
        xsf = torch.empty(fp4gemv.scale_bytes(M, K), dtype=torch.uint8, device=dev)
        wsp = torch.empty(fp4gemv.w4a4_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
        fns = [lambda w=w, sf=sf: fp4gemv.w4a4_linear(x, gsi, w, sf, alpha, out=out, x_fp4=xq, x_sf=xsf,
                                                      workspace=wsp) for w, sf in ws]
        us_l = time_calls(fns, 20, stream)
        us_q = time_calls([lambda: fp4gemv.quantize_act(x, gsi, x_fp4=xq, x_sf=xsf)], 20, stream)
        w4[str(M)] = {"w4a4_linear_us": round(us_l, 2), "quantize_us": round(us_q, 2),
                      "w4a16_gemv_us": sw[str(M)]["gemv_us"] if str(M) in sw else None}
    Mq = 8192
    xl = synth.activations(Mq, K, seed=3, device=dev)
    ql = torch.empty(Mq, K // 2, dtype=torch.uint8, device=dev)
    sfl = torch.empty(fp4gemv.scale_bytes(Mq, K), dtype=torch.uint8, device=dev)
    us_big = time_calls([lambda: fp4gemv.quantize_act(xl, gsi, x_fp4=ql, x_sf=sfl)], 10, stream)
    bq = Mq * K * 2 + Mq * K // 2 + fp4gemv.scale_bytes(Mq, K)
    res["w4a4_8192"] = {"rows": w4, "quantize_8192x8192": {
        "us": round(us_big, 2), "GB/s": round(bq / (us_big * 1e-6) / 1e9, 1),
        "frac": round(bq / (us_big * 1e-6) / 1e9 / peak, 3), "bytes": bq}}
    del ws, xl, ql, sfl
    assert fp4gemv.get_device_error() == 0
    return res


def decode_chain(dev, gs, peak, Ms=(1, 4, 8)):
    """The four decode linears of a Llama-3-8B layer chained with their real
    data dependencies -- x -> qkv; o_proj on the first 4096 columns of the
    qkv output (a strided view standing in for attention's output);
    gate_up + silu_mul on o_proj's output; down on that; down's output is the
    next layer's x -- over 7 layers of distinct weights (L2-cold), replayed as
    one CUDA graph.  Reported per layer: with PDL on every launch; with PDL
    off on o_proj (the launch after attention, a kernel that needs the whole
    GPU); with PDL off everywhere; and the sum of the four calls timed alone
    (per_call), whose difference to the chain is the overlap PDL buys."""
    from moe_nvfp4_gemv_gb300 import fp4gemv
    stream = torch.cuda.current_stream(dev)
    nl = 7
    ws = {name: [(synth.fp4_bytes(N, K, seed=100 * l + 1, device=dev),
                  synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=100 * l + 2, device=dev)) for l in range(nl)]
          for name, (N, K, silu) in LAYERS.items()}
    layer_bytes = {M: sum(nvfp4_bytes(M, N, K, s) for (N, K, s) in LAYERS.values()) for M in Ms}
    res = {}
    for M in Ms:
        H = LAYERS["o_proj"][1]
        x0 = synth.activations(M, H, seed=M, device=dev)
        bufs = {"x": [x0] + [torch.empty(M, H, dtype=torch.bfloat16, device=dev) for _ in range(nl)],
                "qkv": torch.empty(M, LAYERS["qkv"][0], dtype=torch.bfloat16, device=dev),
                "o": torch.empty(M, H, dtype=torch.bfloat16, device=dev),
                "gu": torch.empty(M, LAYERS["gate_up"][0] // 2, dtype=torch.bfloat16, device=dev)}

        def chain(pdl_o, pdl_rest):
            def fn():
                for l in range(nl):
                    x = bufs["x"][l]
                    fp4gemv.nvfp4_gemv(x, *ws["qkv"][l], gs, pdl=pdl_rest, out=bufs["qkv"])
                    fp4gemv.nvfp4_gemv(bufs["qkv"][:, :H], *ws["o_proj"][l], gs, pdl=pdl_o, out=bufs["o"])
                    fp4gemv.nvfp4_gemv(bufs["o"], *ws["gate_up"][l], gs, silu_mul=True, pdl=pdl_rest, out=bufs["gu"])
                    fp4gemv.nvfp4_gemv(bufs["gu"], *ws["down"][l], gs, pdl=pdl_rest, out=bufs["x"][l + 1])
            return fn

        row = {}
        for key, (po, pr) in (("pdl", (True, True)), ("pdl_off_after_attention", (False, True)),
                              ("no_pdl", (False, False))):
            us = time_calls([chain(po, pr)], 1, stream) / nl
            row[key] = {"us_per_layer": round(us, 2), "GB/s": round(layer_bytes[M] / (us * 1e-6) / 1e9, 1),
                        "frac": round(layer_bytes[M] / (us * 1e-6) / 1e9 / peak, 3)}
        res[str(M)] = row
    del ws
    return res


def run_profile_case(spec):
    """A few launches of one case, for ncu captures: LAYER:M[:bf16] with
    LAYER in qkv, o_proj, gate_up, down; moe:M; dequantize_rows:N (N x N);
    sweep_gemm:M (dequantize + GEMM, N = K = 8192); quantize:M (the W4A4
    activation quantisation of M x 8192); w4a4:M (w4a4_linear, N = K = 8192)."""
    from moe_nvfp4_gemv_gb300 import fp4gemv
    dev = torch.device("cuda", 0)
    parts = spec.split(":")
    M = int(parts[1])
    gs = torch.tensor([GS], dtype=torch.float32, device=dev)
    if parts[0] == "sweep_gemm":
        # the dequantize + GEMM path on N = K = 8192 (dequantize_rows, then the
        # tcgen05 GEMM on the bf16 weight)
        N = K = synth.SWEEP_NK
        w = synth.fp4_bytes(N, K, seed=1, device=dev)
        sf = synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=2, device=dev)
        x = synth.activations(M, K, seed=M, device=dev)
        wb = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
        for _ in range(4):
            fp4gemv.dequant_gemm(x, w, sf, gs, w_bf16=wb)
    elif parts[0] == "dequantize_rows":
        N = M
        w = synth.fp4_bytes(N, N, seed=1, device=dev)
        sf = synth.e4m3_bytes(fp4gemv.scale_bytes(N, N), seed=2, device=dev)
        out = torch.empty(N, N, dtype=torch.bfloat16, device=dev)
        for _ in range(4):
            fp4gemv.dequantize_rows(w, sf, out=out)
    elif parts[0] == "quantize":
        # the W4A4 activation quantisation of M x 8192 bf16 activations
        K = synth.SWEEP_NK
        x = synth.activations(M, K, seed=1, device=dev)
        g = torch.tensor([448.0 * 6 / 4.0], dtype=torch.float32, device=dev)
        for _ in range(4):
            fp4gemv.quantize_act(x, g)
    elif parts[0] == "w4a4":
        # w4a4_linear on the N = K = 8192 layer at M tokens (quantisation, then the GEMM)
        N = K = synth.SWEEP_NK
        x = synth.activations(M, K, seed=1, device=dev)
        w = synth.fp4_bytes(N, K, seed=1, device=dev)
        sf = synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=2, device=dev)
        g = torch.tensor([448.0 * 6 / 4.0], dtype=torch.float32, device=dev)
        a = torch.tensor([GS / (448.0 * 6 / 4.0)], dtype=torch.float32, device=dev)
        for _ in range(4):
            fp4gemv.w4a4_linear(x, g, w, sf, a)
    elif parts[0] == "moe":
        c = synth.MOE
        E, H, I, SI, topk = c["E"], c["H"], c["I"], c["SI"], c["topk"]
        w1 = synth.fp4_bytes(E * 2 * I, H, seed=1, device=dev).view(E, 2 * I, H // 2)
        w1_sf = synth.e4m3_bytes(E * fp4gemv.scale_bytes(2 * I, H), seed=2, device=dev)
        w2 = synth.fp4_bytes(E * H, I, seed=3, device=dev).view(E, H, I // 2)
        w2_sf = synth.e4m3_bytes(E * fp4gemv.scale_bytes(H, I), seed=4, device=dev)
        wsh = synth.fp4_bytes(2 * SI, H, seed=5, device=dev)
        ssh = synth.e4m3_bytes(fp4gemv.scale_bytes(2 * SI, H), seed=6, device=dev)
        wsd = synth.fp4_bytes(H, SI, seed=7, device=dev)
        ssd = synth.e4m3_bytes(fp4gemv.scale_bytes(H, SI), seed=8, device=dev)
        alpha = synth.expert_alphas(E, device=dev)
        ids, tw = synth.routing(M, E, topk, seed=M, device=dev)
        x = synth.activations(M, H, seed=M, device=dev)
        act = torch.empty(M * topk, I, dtype=torch.bfloat16, device=dev)
        sact = torch.empty(M, SI, dtype=torch.bfloat16, device=dev)
        out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        for _ in range(4):
            fp4gemv.moe_gate_up(x, ids, w1, w1_sf, alpha, act, wsh, ssh, gs, sact)
            fp4gemv.moe_down_combine(act, ids, tw, w2, w2_sf, alpha, sact, wsd, ssd, gs, out)
    else:
        N, K, silu = LAYERS[parts[0]]
        x = synth.activations(M, K, seed=M, device=dev)
        if len(parts) > 2 and parts[2] == "bf16":
            w = synth.bf16_weight(N, K, seed=1, device=dev)
            for _ in range(4):
                fp4gemv.bf16_gemv(x, w, silu_mul=silu)
        else:
            w = synth.fp4_bytes(N, K, seed=1, device=dev)
            sf = synth.e4m3_bytes(fp4gemv.scale_bytes(N, K), seed=2, device=dev)
            for _ in range(4):
                fp4gemv.nvfp4_gemv(x, w, sf, gs, silu_mul=silu)
    torch.cuda.synchronize()
    assert fp4gemv.get_device_error() == 0
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extended", metavar="PATH", help="also time every configuration into a JSON file")
    ap.add_argument("--no-configs", action="store_true", help="leave the other configurations out of the line")
    ap.add_argument("--profile", metavar="CASE", help="run a few launches of one case (for ncu) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile:
        return run_profile_case(args.profile)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
