#!/usr/bin/env python3
"""Benchmark of the weightless linear projection path on GB300.

One step = one pass of a Gemma-3-1B-shaped decoder layer stack at decode
(T = 1): per layer fused Q/K/V (1152 -> 1024/256/256), O (1024 -> 1152) and
the fused GeGLU MLP (1152 -> 6912 -> 1152), rank r = 4, bf16, seeded synthetic
weights.  The stack has 26 layers with one W0 per layer (G = 26), so every
step streams 1.4 GB of distinct weights: far larger than L2 (no flush needed;
each layer's weights are cold when read).

value = algorithmic bytes of the step / device time of the step (GB/s).
Also reported: us per token per layer, the roofline of the dominant kernel
(the fused MLP), the end-to-end rate through the public API with host
buffers, and the fp64 CPU oracle on the host cores as a baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl wl|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L_LAYERS = 26
SHAPES = dict(hidden=1152, q=1024, kv=256, inter=6912)
METRIC = "weightless-linear HBM GB/s (T=1) & TFLOP/s (T=2048) vs roofline; µs/token/layer"


def proj_list(shapes):
    h, q, kv, i = shapes["hidden"], shapes["q"], shapes["kv"], shapes["inter"]
    return [(h, q), (h, kv), (h, kv), (q, h), (h, i), (h, i), (i, h)]  # (in, out)


def layer_bytes(shapes, T, r):
    """Algorithmic HBM bytes of one layer: W0 (2 B/elem), s (4 B/row),
    U and V (2 B/elem), every projection's input and output activations."""
    b = 0
    for inp, out in proj_list(shapes):
        b += 2 * out * inp + 4 * out + 2 * r * (inp + out) + 2 * T * (inp + out)
    return b


def mlp_bytes(shapes, T, r):
    h, i = shapes["hidden"], shapes["inter"]
    b = 0
    for inp, out in ((h, i), (h, i), (i, h)):
        b += 2 * out * inp + 4 * out + 2 * r * (inp + out)
    return b + 2 * T * 2 * h


def layer_flops(shapes, T, r):
    return sum(2 * T * (out * inp + r * (inp + out)) for inp, out in proj_list(shapes))


# The nominal HBM rate the decode target is stated against (about 8 TB/s);
# every fraction is also given against the measured copy rate.
NOMINAL_HBM_GBS = 8000.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: wait for its first sample (taken
        # before the timed region, and dropped in stop()) so that the samples
        # kept all fall inside the region
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.split(",") for ln in self.f.read().strip().splitlines() if ln.strip()][1:]
        os.unlink(self.f.name)
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = max(smax, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------- ranks (replicas)
def max_over_ranks(value: float, device=None) -> float:
    """The largest of every rank's value (the slowest replica sets the job's
    time); the value itself without a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units all replicas processed over the
    slowest replica's time (units per second)."""
    return units_per_rank * world / (ms * 1e-3)


# --------------------------------------------------------------- reference
def run_reference(args):
    """The fp64 CPU oracle on the host cores, as it stands, on the same
    workload: each timed step is one whole pass over the 26-layer stack at
    T = 1 (every layer's output feeds the next, as on the GPU)."""
    import oracle
    import torch
    import wl_synth

    oracle.build()
    r = args.rank
    cores = oracle.get_threads()
    dims = proj_list(SHAPES)
    g = wl_synth.make_generator(0)
    x = wl_synth.draw_x(g, 1, SHAPES["hidden"])
    # one layer's theta bundles, reused by every layer of the step: the oracle's
    # time does not depend on the weights' values, and 26 distinct layers would
    # cost 26 draws of 54 MB on the host
    thetas = [wl_synth.draw_theta(g, inp, out, r) for inp, out in dims]

    def one_layer(xin):
        q = oracle.linear(xin, thetas[0])
        oracle.linear(xin, thetas[1])
        oracle.linear(xin, thetas[2])
        o = oracle.linear(torch.from_numpy(q).to(torch.bfloat16), thetas[3])
        y = oracle.mlp_geglu(torch.from_numpy(o).to(torch.bfloat16), thetas[4], thetas[5], thetas[6])
        return torch.from_numpy(y).to(torch.bfloat16)

    def one_step(xin):
        for _ in range(L_LAYERS):
            xin = one_layer(xin)
        return xin

    for _ in range(args.warmup):
        one_step(x)
    t_all = time.perf_counter()
    for _ in range(args.steps):
        one_step(x)
    wall = time.perf_counter() - t_all
    per_step = wall / args.steps
    step_bytes = layer_bytes(SHAPES, 1, r) * L_LAYERS
    value = step_bytes / per_step / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"gemma3-1b decode layer stack: {L_LAYERS} layers x (fused QKV "
                               f"1152->1024/256/256, O 1024->1152, fused GeGLU MLP 1152->6912->1152), "
                               f"T=1, r={r}, bf16 inputs",
                   "T": 1, "r": r, "layers": L_LAYERS, "step_bytes": step_bytes,
                   "us_per_token_per_layer": round(per_step * 1e6 / L_LAYERS, 3),
                   "L2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{args.steps} whole {L_LAYERS}-layer steps at T=1 after {args.warmup} "
                                   f"warm-up steps; wall {wall:.1f}s"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def time_oracle_sample(r, budget_s=12.0):
    """cpu_baseline of the wl arm: oracle on a bounded sample (whole layers)."""
    import oracle
    import torch
    import wl_synth

    oracle.build()
    dims = proj_list(SHAPES)
    g = wl_synth.make_generator(1)
    x = wl_synth.draw_x(g, 1, SHAPES["hidden"])
    thetas = [wl_synth.draw_theta(g, inp, out, r) for inp, out in dims]
    n = 0
    t0 = time.perf_counter()
    while True:
        q = oracle.linear(x, thetas[0])
        oracle.linear(x, thetas[1])
        oracle.linear(x, thetas[2])
        o = oracle.linear(torch.from_numpy(q).to(torch.bfloat16), thetas[3])
        oracle.mlp_geglu(torch.from_numpy(o).to(torch.bfloat16), *thetas[4:])
        n += 1
        el = time.perf_counter() - t0
        if el > budget_s or n >= 5000:
            break
    value = layer_bytes(SHAPES, 1, r) * n / el / 1e9
    cores = oracle.get_threads()
    # the same layer on one host thread (a short sample)
    oracle.set_threads(1)
    try:
        n1 = 0
        t1 = time.perf_counter()
        while True:
            q = oracle.linear(x, thetas[0])
            oracle.linear(x, thetas[1])
            oracle.linear(x, thetas[2])
            o = oracle.linear(torch.from_numpy(q).to(torch.bfloat16), thetas[3])
            oracle.mlp_geglu(torch.from_numpy(o).to(torch.bfloat16), *thetas[4:])
            n1 += 1
            el1 = time.perf_counter() - t1
            if el1 > budget_s / 4 or n1 >= 100:
                break
    finally:
        oracle.set_threads(cores)
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": f"{n} layers of the T=1 stack (of {L_LAYERS}), {el:.1f}s",
            "one_thread": {"value": round(layer_bytes(SHAPES, 1, r) * n1 / el1 / 1e9, 4), "unit": "GB/s",
                           "cores": 1, "sample": f"{n1} layers, {el1:.1f}s"}}


def time_oracle_prefill(r=16, T=2048, rows=64):
    """The oracle on the prefill layer (T tokens, r): QKV, O and the MLP on
    fixed subsets of `rows` and 2*`rows` token rows (rows are independent),
    timed; the whole layer's time is the fixed part (the oracle forms each
    W_eff row once per call) plus the per-row part, extrapolated linearly to
    T rows; TFLOP/s of the layer's algorithmic FLOPs.  A reported CPU
    baseline, not a target."""
    import oracle
    import torch
    import wl_synth

    oracle.build()
    dims = proj_list(SHAPES)
    g = wl_synth.make_generator(2)
    thetas = [wl_synth.draw_theta(g, inp, out, r) for inp, out in dims]
    xs = wl_synth.draw_x(g, 2 * rows, SHAPES["hidden"])

    def layer(x):
        t0 = time.perf_counter()
        q = oracle.linear(x, thetas[0])
        oracle.linear(x, thetas[1])
        oracle.linear(x, thetas[2])
        o = oracle.linear(torch.from_numpy(q).to(torch.bfloat16), thetas[3])
        oracle.mlp_geglu(torch.from_numpy(o).to(torch.bfloat16), *thetas[4:])
        return time.perf_counter() - t0

    t1 = layer(xs[:rows])
    t2 = layer(xs)
    per_row = max(t2 - t1, 1e-9) / rows
    sec_full = max(t1 - per_row * rows, 0.0) + per_row * T
    return {"value": round(layer_flops(SHAPES, T, r) / sec_full / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.get_threads(), "kind": "oracle",
            "sample": f"{rows} and {2 * rows} of {T} token rows of the r={r} layer ({t1:.2f}s, {t2:.2f}s); "
                      f"fixed + per-row time extrapolated to {T} rows ({sec_full:.1f}s)"}


# ---------------------------------------------------------------- wl arm --
def run_wl(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import rank_weight_reconstruction_wl_gb300 as wl
    from rank_weight_reconstruction_wl_gb300.stack import DecoderStack, build_layers

    r = args.rank
    T = 1
    nl = args.layers
    layers = build_layers(nl, nl, T, SHAPES, r, seed=rank, device=dev)
    stack = DecoderStack(layers, T, SHAPES["hidden"], SHAPES["q"], SHAPES["inter"], r, device=dev,
                         engine=args.engine)
    gx = torch.Generator(device=dev)
    gx.manual_seed(100 + rank)
    stack.x.copy_(torch.randn(T, SHAPES["hidden"], generator=gx, device=dev).to(torch.bfloat16))
    stack.capture()

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    # ---- device-timed steps (graph replay) ----
    for _ in range(args.warmup):
        stack.step()
    barrier()
    clocks = Clocks(local)
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stack.stream)
    for _ in range(args.steps):
        stack.step()
    ev1.record(stack.stream)
    barrier()
    ck = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms, dev)
    step_bytes = layer_bytes(SHAPES, T, r) * nl
    value = job_rate(step_bytes, world, ms) / 1e9
    status = wl.wl_device_status(stack.stream)

    # ---- dominant kernel, timed per launch with events on its stream ----
    hbm_peak, _, peak_kind = load_peaks()
    if stack.engine == "stack":
        # the step is the V^T pass (about 7 us) and nchunk back-to-back launches
        # of the stack kernel, each over an equal share of the layers; the
        # per-launch time below includes the V^T pass (it understates the
        # kernel's rate by about 1 %)
        nchunk = stack.kernel_launches_per_step
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(3, min(args.steps, 20)))]
        for a0, a1 in evs:
            a0.record(stack.stream)
            stack.step()
            a1.record(stack.stream)
        stack.stream.synchronize()
        launch_ms = statistics.mean(a.elapsed_time(b) for a, b in evs) / nchunk
        kb = step_bytes / nchunk
        kname = f"stack_kernel ({nl // nchunk} layers per launch, {nchunk} launches per step)"
        traffic = load_traffic("stack_kernel")
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nl)]
        mlp_ms = []
        for _ in range(max(3, min(args.steps, 10))):
            stack.step(mlp_events=evs)
            stack.stream.synchronize()
            mlp_ms.extend(a.elapsed_time(b) for a, b in evs)
        launch_ms = statistics.mean(mlp_ms)
        kb = mlp_bytes(SHAPES, T, r)
        kname = "dec_gateup_kernel + dec_down_kernel (fused GeGLU MLP call, T=1)"
        traffic = load_traffic("dec_mlp")
    achieved = kb / (launch_ms * 1e-3) / 1e9

    # ---- end to end through the public API with pinned host buffers ----
    xh = torch.empty(T, SHAPES["hidden"], dtype=torch.bfloat16).pin_memory()
    yh = torch.empty(T, SHAPES["hidden"], dtype=torch.bfloat16).pin_memory()
    xh.copy_(stack.x.cpu())
    for _ in range(args.warmup):
        stack.forward_host(xh, yh)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stack.stream)
    for _ in range(args.steps):
        stack.forward_host(xh, yh)
    t1.record(stack.stream)
    barrier()
    e2e_ms = t0.elapsed_time(t1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = job_rate(step_bytes, world, e2e_ms) / 1e9

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"gemma3-1b decode layer stack: {nl} layers x (fused QKV "
                                   f"1152->1024/256/256, O 1024->1152, fused GeGLU MLP 1152->6912->1152), "
                                   f"T=1, r={r}, G={nl} (one W0 per layer)",
                       "T": T, "r": r, "layers": nl,
                       "l2": "inputs larger than L2 (1.4 GB of distinct weights per step), no flush",
                       "parallelism": f"replicas x{world}",
                       "step_bytes": step_bytes,
                       "us_per_token_per_layer": round(ms * 1e3 / (T * nl), 3),
                       "us_per_token_per_stack": round(ms * 1e3 / T, 2),
                       "engine": stack.engine,
                       "graph": ("a V^T pass, then one stack-kernel launch per 24 layers" if stack.engine == "stack"
                                 else "CUDA graph replay of the per-projection calls")},
            "roofline": {"bound": "hbm", "kernel": kname,
                         "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                         "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                         "bytes_per_launch": int(kb), "avg_launch_us": round(launch_ms * 1e3, 3),
                         "traffic": traffic},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": T * SHAPES["hidden"] * 2,
                    "d2h_bytes_per_step": T * SHAPES["hidden"] * 2,
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": stack.launches_per_step * args.steps,
            "device_status": wl.STATUS_NAMES.get(status, status),
        }
        if ck is not None:
            line["clocks"] = ck
        if stack.engine == "stack" and not args.no_compare:
            line["per_call_graph"] = measure_graph_engine(layers, T, r, dev)
            line["precompute_path"] = measure_precompute(layers, T, r, dev, ms)
        from rank_weight_reconstruction_wl_gb300.metrics import compression_ratio
        line["compression"] = {"r": r, "layers": nl,
                               f"G={nl}": round(compression_ratio(SHAPES, nl, nl, r), 5),
                               "G=1": round(compression_ratio(SHAPES, nl, 1, r), 5),
                               "definition": "theta bytes (W0 + s + U + V, all layers and families) / bf16 "
                                             "dense projection bytes"}
        if not args.no_grid:
            line["stack_grid"] = measure_stack_grid(dev)
            line["materialize"] = measure_materialize(dev)
            line["f32_encoding"] = measure_f32(dev)
            line["decompose"] = measure_decompose(dev)
        if not args.no_prefill:
            line["prefill_T2048"] = measure_prefill(dev)
            line["prefill_T2048_r32"] = measure_prefill(dev, r=32, reps=2)
            line["matmul_yardstick_T2048"] = measure_matmul_yardstick(dev)
            line["large_set"] = measure_large(dev)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = time_oracle_sample(r)
            if not args.no_prefill:
                line["cpu_baseline_prefill_T2048"] = time_oracle_prefill()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def measure_precompute(layers, T, r, dev, ms_weightless, steps=100):
    """The precompute path ("Serve and generate with weightless", fast path):
    W_eff of every projection formed once by wl_materialize (bf16), then the
    same stack run as dense weights (rank 0) on the stack engine."""
    import torch
    from rank_weight_reconstruction_wl_gb300.stack import DecoderStack, materialize_layers

    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        materialize_layers(layers[:1])  # warm-up
        st.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        dense = materialize_layers(layers)
        e1.record(st)
        st.synchronize()
    mat_ms = e0.elapsed_time(e1)
    stk = DecoderStack(dense, T, SHAPES["hidden"], SHAPES["q"], SHAPES["inter"], 0, device=dev, engine="stack")
    stk.x.normal_()
    stk.capture()
    for _ in range(5):
        stk.step()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stk.stream)
    for _ in range(steps):
        stk.step()
    a1.record(stk.stream)
    stk.stream.synchronize()
    ms = a0.elapsed_time(a1) / steps
    b = layer_bytes(SHAPES, T, 0) * len(layers)
    return {"value": round(b / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "us_per_token_per_layer": round(ms * 1e3 / (T * len(layers)), 3),
            "step_speed_vs_weightless": round(ms_weightless / ms, 3),
            "materialize_ms_all_layers": round(mat_ms, 3),
            "note": "W_eff bf16 of all 182 projections formed once (wl_materialize), then the stack kernel at r=0"}


def measure_graph_engine(layers, T, r, dev, steps=30):
    """The same step through the per-projection calls replayed as a CUDA
    graph (the other engine), for comparison."""
    import torch
    from rank_weight_reconstruction_wl_gb300.stack import DecoderStack

    st = DecoderStack(layers, T, SHAPES["hidden"], SHAPES["q"], SHAPES["inter"], r, device=dev, engine="graph")
    st.x.normal_()
    st.capture()
    for _ in range(3):
        st.step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st.stream)
    for _ in range(steps):
        st.step()
    e1.record(st.stream)
    st.stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    b = layer_bytes(SHAPES, T, r) * len(layers)
    return {"value": round(b / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "us_per_token_per_layer": round(ms * 1e3 / (T * len(layers)), 3)}


def measure_prefill(dev, T=2048, r=16, nlayers=4, reps=5):
    """TFLOP/s of the Gemma-1B layer at prefill (T tokens): fused QKV, O and
    the fused MLP on the tensor-core path, rotating over `nlayers` distinct
    weight sets (216 MB at r=16, larger than L2)."""
    import torch
    import rank_weight_reconstruction_wl_gb300 as wl
    from rank_weight_reconstruction_wl_gb300.stack import build_layers

    layers = build_layers(nlayers, nlayers, T, SHAPES, r, seed=7, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    z = dict(dtype=torch.bfloat16, device=dev)
    x = torch.randn(T, SHAPES["hidden"], generator=g, device=dev).to(torch.bfloat16)
    yq = torch.empty(T, SHAPES["q"], **z)
    yk = torch.empty(T, SHAPES["kv"], **z)
    yv = torch.empty(T, SHAPES["kv"], **z)
    yo = torch.empty(T, SHAPES["hidden"], **z)
    ym = torch.empty(T, SHAPES["hidden"], **z)
    ws = wl.mlp_workspace(T, SHAPES["hidden"], SHAPES["inter"], r, torch.bfloat16, dev)
    st = torch.cuda.Stream(dev)
    # The layer's launches are captured once as CUDA graphs and replayed, so
    # that the timings are device time (no host launch overhead inside).
    parts = {"qkv": lambda th: wl.wl_qkv_fused(x, th.q, th.k, th.v, outs=(yq, yk, yv), stream=st),
             "o": lambda th: wl.wl_linear(yq, th.o.W0, th.o.s, th.o.U, th.o.V, y=yo, stream=st),
             "mlp": lambda th: wl.wl_mlp_geglu_fused(yo, th.gate, th.up, th.down, y=ym, workspace=ws, stream=st)}

    def capture(fns):
        with torch.cuda.stream(st):
            for th in layers:
                for f in fns:
                    f(th)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for _ in range(reps):
                    for th in layers:
                        for f in fns:
                            f(th)
        return g

    def time_graph(g):
        with torch.cuda.stream(st):
            g.replay()
            st.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(st)
            g.replay()
            a1.record(st)
            st.synchronize()
        return a0.elapsed_time(a1) / (reps * nlayers)

    ms = time_graph(capture(list(parts.values())))
    part_ms = {k: time_graph(capture([f])) for k, f in parts.items()}
    flops = layer_flops(SHAPES, T, r)
    h, q, kv, i = SHAPES["hidden"], SHAPES["q"], SHAPES["kv"], SHAPES["inter"]
    part_flops = {"qkv": 2 * T * (h * (q + 2 * kv) + r * 3 * h + r * (q + 2 * kv)),
                  "o": 2 * T * (q * h + r * (q + h)),
                  "mlp": 2 * T * (3 * h * i + r * 3 * (h + i))}
    out_parts = {}
    for k, pms in part_ms.items():
        out_parts[k] = {"us": round(pms * 1e3, 2), "tflops": round(part_flops[k] / (pms * 1e-3) / 1e12, 1)}
    _, bf16_peak, kind = load_peaks()
    tf = flops / (ms * 1e-3) / 1e12
    return {"T": T, "r": r, "ms_per_layer": round(ms, 4), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / bf16_peak, 4), "peak_tflops": bf16_peak, "peak_kind": kind,
            "layer_gflop": round(flops / 1e9, 2), "parts": out_parts,
            "timing": "CUDA graph replay of the layer's launches (device time)",
            "l2": f"{nlayers} weight sets rotated (larger than L2)"}


def measure_matmul_yardstick(dev, T=2048, reps=20):
    """A measurement only, not a hot-path option: torch.matmul (the vendor
    library) in bf16 on the dense products of the prefill MLP at T tokens,
    [T x 1152] x [1152 x 13824] (gate and up) and [T x 6912] x [6912 x 1152]
    (down), over 4 weight sets (larger than L2).  Gives the rate a library GEMM
    attains at these K, against which the weightless prefill kernel is read."""
    import torch

    h, i = SHAPES["hidden"], SHAPES["inter"]
    g = torch.Generator(device=dev)
    g.manual_seed(23)
    bf = dict(dtype=torch.bfloat16, device=dev)
    out = {"timing": f"CUDA events over {reps} passes of 4 weight sets"}
    _, bf16_peak, kind = load_peaks()
    for name, K, N in (("gate_up", h, 2 * i), ("down", i, h)):
        a = torch.randn(T, K, generator=g, device=dev).to(torch.bfloat16)
        bs = [torch.randn(K, N, generator=g, device=dev).to(torch.bfloat16) for _ in range(4)]
        c = torch.empty(T, N, **bf)
        for b in bs:
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for b in bs:
                torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * len(bs))
        tf = 2 * T * K * N / (ms * 1e-3) / 1e12
        out[name] = {"shape": f"[{T} x {K}] x [{K} x {N}]", "us": round(ms * 1e3, 2), "tflops": round(tf, 1),
                     "frac_of_bf16_peak": round(tf / bf16_peak, 4)}
        del a, bs, c
    out["peak_kind"] = kind
    return out


def unique_bytes(shapes, L, G, T, r):
    """Distinct bytes one step touches: G W0 blocks per family, every layer's
    s, U, V and activations (W0 shared by the layers of a band is counted
    once)."""
    b = 0
    for inp, out in proj_list(shapes):
        b += G * 2 * out * inp + L * (4 * out + 2 * r * (inp + out) + 2 * T * (inp + out))
    return b


def measure_stack_grid(dev, steps=20, Ts=(1, 32), Gs=(L_LAYERS, 1), ranks=(4, 16, 32), nlayers=L_LAYERS):
    """The 26-layer stack on the stack engine over T (1: one request; 32: 32
    requests decoded together), G (26: one W0 per layer, every step streams
    1.4 GB of distinct weights; 1: one shared W0 set of 53.7 MB, which may stay
    in L2) and r.  Streamed bytes count every layer's W0 read (the algorithmic
    bytes of the step); unique bytes count a shared W0 once.  nlayers < 26 is
    for profiling only (G = 26 then means one W0 per layer)."""
    import torch
    from rank_weight_reconstruction_wl_gb300.stack import DecoderStack, build_layers

    hbm_peak, _, kind = load_peaks()
    out = {"l2_bytes": torch.cuda.get_device_properties(dev).L2_cache_size, "peak_gbs": hbm_peak,
           "peak_kind": kind, "timing": f"CUDA events over {steps} steps after 3 warm-up steps"}
    for T in Ts:
        for G in Gs:
            for r in ranks:
                G_ = min(G, nlayers)
                layers = build_layers(nlayers, G_, T, SHAPES, r, seed=17 + r, device=dev)
                st = DecoderStack(layers, T, SHAPES["hidden"], SHAPES["q"], SHAPES["inter"], r, device=dev,
                                  engine="stack")
                gx = torch.Generator(device=dev)
                gx.manual_seed(5)
                st.x.copy_(torch.randn(T, SHAPES["hidden"], generator=gx, device=dev).to(torch.bfloat16))
                st.capture()
                for _ in range(3):
                    st.step()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st.stream)
                for _ in range(steps):
                    st.step()
                e1.record(st.stream)
                st.stream.synchronize()
                ms = e0.elapsed_time(e1) / steps
                streamed = layer_bytes(SHAPES, T, r) * nlayers
                uniq = unique_bytes(SHAPES, nlayers, G_, T, r)
                gbs = streamed / (ms * 1e-3) / 1e9
                out[f"T{T}_G{G}_r{r}"] = {
                    "ms_per_step": round(ms, 4),
                    "us_per_token_per_stack": round(ms * 1e3 / T, 3),
                    "us_per_token_per_layer": round(ms * 1e3 / (T * nlayers), 4),
                    "streamed_MB": round(streamed / 1e6, 1), "GBs_streamed": round(gbs, 1),
                    "frac_of_hbm_streamed": round(gbs / hbm_peak, 4),
                    "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                    "unique_MB": round(uniq / 1e6, 1),
                    "GBs_unique": round(uniq / (ms * 1e-3) / 1e9, 1),
                    "tflops": round(layer_flops(SHAPES, T, r) * nlayers / (ms * 1e-3) / 1e12, 2)}
                del st, layers
                torch.cuda.empty_cache()
    return out


def measure_materialize(dev, r=4, nsets=2, reps=10):
    """wl_materialize alone: W_eff of the seven Gemma-3-1B projections (one
    layer) in fp32 and in bf16, output tensors allocated before timing, the
    launches replayed as a CUDA graph over `nsets` weight sets.  Algorithmic
    bytes per layer: W0 (2 B/element), s, U and V read once, W_eff written once
    (4 or 2 B/element)."""
    import torch
    import rank_weight_reconstruction_wl_gb300 as wl
    import wl_synth

    hbm_peak, _, kind = load_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    sets = [[wl_synth.draw_theta(g, inp, o, r) for inp, o in proj_list(SHAPES)] for _ in range(nsets)]
    st = torch.cuda.Stream(dev)
    res = {"r": r, "peak_gbs": hbm_peak, "peak_kind": kind,
           "timing": f"CUDA graph replay, {nsets} weight sets rotated, {reps} passes"}
    for name, dt, esz in (("f32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        outs = [[torch.empty(o, inp, dtype=dt, device=dev) for inp, o in proj_list(SHAPES)] for _ in range(nsets)]

        def issue():
            for w, ob in zip(sets, outs):
                for th, y in zip(w, ob):
                    wl.wl_materialize(th.W0, th.s, th.U, th.V, dt=dt, out=y, stream=st)

        with torch.cuda.stream(st):
            issue()
            st.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=st):
                for _ in range(reps):
                    issue()
            gr.replay()
            st.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(st)
            gr.replay()
            a1.record(st)
            st.synchronize()
        ms = a0.elapsed_time(a1) / (reps * nsets)
        b = sum(2 * o * inp + 4 * o + 2 * r * (inp + o) + esz * o * inp for inp, o in proj_list(SHAPES))
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"us_per_layer": round(ms * 1e3, 2), "MB_per_layer": round(b / 1e6, 1),
                     "GBs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                     "launches_per_layer": 7}
        del outs
    return res


# fp32 arithmetic peak of the CUDA cores (the fp32 encoding runs on them):
# 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (maximum SM clock)
F32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def measure_f32(dev, r=4, reps=10):
    """The fp32 encoding ("Serve and generate with weightless", "Supported
    encodings and devices"): fused Q/K/V of the Gemma-3-1B layer with fp32 x,
    W0, s, U, V.  T = 1: GB/s of algorithmic bytes (4-byte weights) against
    HBM; T = 2048: TFLOP/s against the fp32 CUDA-core peak.  CUDA-graph
    replay rotating weight sets: at T = 1 enough sets (7.1 MB each) to hold
    twice the L2, so that W0 comes from HBM; at T = 2048 two sets."""
    import torch
    import rank_weight_reconstruction_wl_gb300 as wl
    import wl_synth

    hbm_peak, _, kind = load_peaks()
    h, q, kv = SHAPES["hidden"], SHAPES["q"], SHAPES["kv"]
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    set_bytes = sum(4 * o * (h + 1 + 2 * r) for o in (q, kv, kv))
    nsets = max(2, -(-2 * torch.cuda.get_device_properties(dev).L2_cache_size // set_bytes))
    sets = [[wl_synth.draw_theta_f32(g, h, o, r) for o in (q, kv, kv)] for _ in range(nsets)]
    st = torch.cuda.Stream(dev)
    res = {"r": r, "peak_gbs": hbm_peak, "peak_kind": kind, "alu_peak_tflops": round(F32_ALU_PEAK_TFLOPS, 1),
           "alu_peak": "152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (nominal, maximum clock)"}
    for T in (1, 2048):
        x = torch.randn(T, h, generator=g, device=dev)
        outs = [torch.empty(T, o, dtype=torch.float32, device=dev) for o in (q, kv, kv)]
        use = sets if T == 1 else sets[:2]
        with torch.cuda.stream(st):
            for w in use:
                wl.wl_qkv_fused(x, *w, outs=outs, ydt=torch.float32, stream=st)
            st.synchronize()
            gr = torch.cuda.CUDAGraph()
            n = reps if T == 1 else 2
            with torch.cuda.graph(gr, stream=st):
                for _ in range(n):
                    for w in use:
                        wl.wl_qkv_fused(x, *w, outs=outs, ydt=torch.float32, stream=st)
            gr.replay()
            st.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(st)
            gr.replay()
            a1.record(st)
            st.synchronize()
        sec = a0.elapsed_time(a1) * 1e-3 / (n * len(use))
        if T == 1:
            b = sum(4 * o * h + 4 * o + 4 * r * (h + o) for o in (q, kv, kv)) + 4 * T * (h + q + 2 * kv)
            res["T1"] = {"qkv_us": round(sec * 1e6, 2), "GBs": round(b / sec / 1e9, 1),
                         "frac_of_hbm": round(b / sec / 1e9 / hbm_peak, 4), "weight_sets": len(use)}
        else:
            f = 2 * T * (h * (q + 2 * kv) + r * 3 * h + r * (q + 2 * kv))
            res["T2048"] = {"qkv_us": round(sec * 1e6, 1), "TFLOPs": round(f / sec / 1e12, 2),
                            "frac_of_alu_peak": round(f / sec / 1e12 / F32_ALU_PEAK_TFLOPS, 4)}
    return res


def measure_decompose(dev, r=16, p=8, iters=4, n=2):
    """Dense weights -> theta (wl_decompose_band) for one band of n layers of
    each Gemma-3-1B projection shape.  Algorithmic bytes per layer: one pass
    over W and W0 for s and 2 * iters + 2 passes for the subspace iteration
    (R is re-formed from W, W0 and s on every pass), plus the band mean (n
    weights read, W0 written); reported as GB/s against HBM."""
    import torch
    import rank_weight_reconstruction_wl_gb300 as wl
    import wl_synth

    hbm_peak, _, kind = load_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(23)
    res = {"r": r, "p": p, "iters": iters, "layers_per_band": n, "peak_gbs": hbm_peak, "peak_kind": kind}
    tot_ms, tot_b = 0.0, 0
    for name, (inp, out) in (("q", (1152, 1024)), ("o", (1024, 1152)), ("gate", (1152, 6912)),
                             ("down", (6912, 1152))):
        Ws = [wl_synth.draw_theta(g, inp, out, 0).W0 for _ in range(n)]
        wl.wl_decompose_band(Ws, r, p, iters, seed=1)  # warm-up
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        reps = 3
        for _ in range(reps):
            wl.wl_decompose_band(Ws, r, p, iters, seed=1)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        w = 2 * out * inp
        b = (n + 1) * w + n * (2 * iters + 3) * 2 * w
        res[name] = {"ms_per_band": round(ms, 3), "GBs": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)}
        tot_ms += ms
        tot_b += b
    res["all"] = {"ms": round(tot_ms, 3), "GBs": round(tot_b / (tot_ms * 1e-3) / 1e9, 1)}
    return res


LARGE = dict(hidden=5376, q=4096, kv=2048, inter=21504, r=64)


def measure_large(dev, nsets=2, Ts=(1, 64, 4096), reps_small=10):
    """The large projection set (hidden 5376, intermediate 21504, Q/K/V
    5376 -> 4096/2048/2048, r = 64): fused Q/K/V and fused MLP calls at 1, 64
    and 4096 tokens, rotating over `nsets` weight sets (1.56 GB, larger than
    L2), timed by CUDA-graph replay.  GB/s of algorithmic bytes at 1 and 64
    tokens (with the fraction of the measured HBM copy rate), TFLOP/s at 4096
    (with the fraction of the measured bf16 burst rate)."""
    import torch
    import rank_weight_reconstruction_wl_gb300 as wl
    import wl_synth

    H, Q, KV, I, r = LARGE["hidden"], LARGE["q"], LARGE["kv"], LARGE["inter"], LARGE["r"]
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    sets = [dict(q=wl_synth.draw_theta(g, H, Q, r), k=wl_synth.draw_theta(g, H, KV, r),
                 v=wl_synth.draw_theta(g, H, KV, r), gate=wl_synth.draw_theta(g, H, I, r),
                 up=wl_synth.draw_theta(g, H, I, r), down=wl_synth.draw_theta(g, I, H, r))
            for _ in range(nsets)]
    st = torch.cuda.Stream(dev)

    def timeit(fn, reps):
        with torch.cuda.stream(st):
            for w in sets:
                fn(w)
            st.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=st):
                for _ in range(reps):
                    for w in sets:
                        fn(w)
            gr.replay()
            st.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(st)
            gr.replay()
            a1.record(st)
            st.synchronize()
        return a0.elapsed_time(a1) / (reps * nsets) * 1e-3  # s

    hbm_peak, tc_peak, kind = load_peaks()
    out = {"shapes": "hidden 5376, inter 21504, q/k/v 4096/2048/2048, r=64, bf16",
           "l2": f"{nsets} weight sets rotated ({0.78 * nsets:.2f} GB, larger than L2)",
           "peaks": f"{hbm_peak} GB/s, {tc_peak} TFLOP/s bf16 burst ({kind})"}
    bf = dict(dtype=torch.bfloat16, device=dev)
    for T in Ts:
        x = torch.randn(T, H, generator=g, device=dev).to(torch.bfloat16)
        yq, yk, yv = torch.empty(T, Q, **bf), torch.empty(T, KV, **bf), torch.empty(T, KV, **bf)
        ym = torch.empty(T, H, **bf)
        ws = wl.mlp_workspace(T, H, I, r, torch.bfloat16, dev)
        reps = reps_small if T < 4096 else 2
        tq = timeit(lambda w: wl.wl_qkv_fused(x, w["q"], w["k"], w["v"], outs=(yq, yk, yv), stream=st), reps)
        tm = timeit(lambda w: wl.wl_mlp_geglu_fused(x, w["gate"], w["up"], w["down"], y=ym, workspace=ws,
                                                    stream=st), reps)
        if T < 4096:
            bq = sum(2 * o * H + 4 * o + 2 * r * (H + o) for o in (Q, KV, KV)) + 2 * T * (H + Q + 2 * KV)
            bm = (2 * (2 * I * H + 4 * I + 2 * r * (H + I)) + (2 * H * I + 4 * H + 2 * r * (I + H))
                  + 2 * T * 2 * H)
            out[f"T{T}"] = {"qkv_us": round(tq * 1e6, 1), "qkv_GBs": round(bq / tq / 1e9, 1),
                            "qkv_frac": round(bq / tq / 1e9 / hbm_peak, 3),
                            "mlp_us": round(tm * 1e6, 1), "mlp_GBs": round(bm / tm / 1e9, 1),
                            "mlp_frac": round(bm / tm / 1e9 / hbm_peak, 3)}
        else:
            fq = 2 * T * (H * (Q + 2 * KV) + r * 3 * H + r * (Q + 2 * KV))
            fm = 2 * T * (3 * H * I + r * 3 * (H + I))
            out[f"T{T}"] = {"qkv_us": round(tq * 1e6, 1), "qkv_TFLOPs": round(fq / tq / 1e12, 1),
                            "qkv_frac": round(fq / tq / 1e12 / tc_peak, 3),
                            "mlp_us": round(tm * 1e6, 1), "mlp_TFLOPs": round(fm / tm / 1e12, 1),
                            "mlp_frac": round(fm / tm / 1e12 / tc_peak, 3)}
        del ws
    return out


def load_traffic(kernel):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (null if none was taken for the current kernel)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d.get(kernel)
    except Exception:
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="wl", choices=["wl", "reference"])
    ap.add_argument("--rank", type=int, default=4, help="LoRA rank r of the theta bundles")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the T=2048 prefill measurement")
    ap.add_argument("--no-compare", action="store_true", help="skip timing the per-projection graph engine")
    ap.add_argument("--no-grid", action="store_true",
                    help="skip the stack grid (T, G, r) and the wl_materialize measurement")
    ap.add_argument("--engine", default="auto", choices=["auto", "stack", "graph"],
                    help="stack kernel (one launch per 24 layers) or per-projection CUDA graph")
    ap.add_argument("--only-prefill", action="store_true",
                    help="run only the T=2048 prefill layer measurement (for profiling)")
    ap.add_argument("--only", default=None, choices=["large1", "stack32", "materialize", "f32"],
                    help="run one measurement alone, for profiling: the large set at one token "
                         "(one weight set), a 4-layer stack at 32 tokens, wl_materialize, or the fp32 encoding")
    ap.add_argument("--layers", type=int, default=L_LAYERS,
                    help="layers in the stack (smaller values are for profiling only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        if args.steps > 20:
            args.steps = 20
        run_reference(args)
        return
    if args.only_prefill:
        import torch

        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        print(json.dumps({"prefill_T2048": measure_prefill(dev, nlayers=min(args.layers, 4), reps=1)}))
        return
    if args.only:
        import torch

        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        if args.only == "large1":
            res = measure_large(dev, nsets=1, Ts=(1,), reps_small=2)
        elif args.only == "stack32":
            res = measure_stack_grid(dev, steps=3, Ts=(32,), Gs=(L_LAYERS,), ranks=(args.rank,),
                                     nlayers=min(args.layers, 4))
        elif args.only == "f32":
            res = measure_f32(dev, r=args.rank)
        else:
            res = measure_materialize(dev, r=args.rank, nsets=1, reps=2)
        print(json.dumps({args.only: res}))
        return
    run_wl(args)


if __name__ == "__main__":
    main()
