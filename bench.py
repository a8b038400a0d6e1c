"""Benchmark: routed MoE expert-MLP layer, forward + backward, on GB300.

One step = the whole hot path on one batch of synthetic input already resident in
HBM: moe_route_permute -> moe_expert_mlp_fwd -> moe_combine (Y) ->
moe_expert_mlp_bwd -> moe_combine (dX).  FLOPs are counted algorithmically:
forward 6*R*D*I, backward 12*R*D*I (R = T*K routed rows; the backward's
activation recompute is not counted as work).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica of the layer on its own GPU (weak scaling, no collective).
``--impl reference`` times the CPU oracle on a bounded sample instead.
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
sys.path.insert(0, ROOT)

METRIC = "MoE expert-MLP TFLOP/s fwd & bwd on 1 GB300 (% of BF16 dense peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Algorithmic FLOPs of each tensor-core kernel per launch, in units of R*D*I (R = T*K
# routed rows; padding rows excluded).
GEMM_FLOPS_RDI = {"gemm_gateup_swiglu": 4, "gemm_down": 2, "gemm_dA": 2, "gemm_bwd_gateup": 4,
                  "gemm_dx": 4, "gemm_dw_gateup": 4, "gemm_dw_down": 2}


def gemm_bytes(s):
    """Algorithmic bytes per launch of each grouped GEMM: the expert weights it reads once,
    the routed rows it reads and writes once (padding excluded), and its fp32 weight
    gradients.  Rows: x and dY bf16 / fp16 (2 B), intermediates 2 B, dA fp16."""
    R, D, I, E = s.R, s.D, s.I, s.E
    w1 = E * D * I * 2          # one weight matrix, bf16
    return {"gemm_gateup_swiglu": 2 * w1 + R * D * 2 + R * I * 2,
            "gemm_down": w1 + R * I * 2 + R * D * 2,
            "gemm_dA": w1 + R * D * 2 + R * I * 2,
            "gemm_bwd_gateup": 2 * w1 + R * D * 2 + R * I * 2 + R * I * 2 + 2 * (R * 2 * I * 2),
            "gemm_dx": 2 * w1 + R * 2 * I * 2 + R * D * 2,
            "gemm_dw_gateup": R * D * 2 + R * 2 * I * 2 + 2 * E * D * I * 4,
            "gemm_dw_down": R * I * 2 + R * D * 2 + E * I * D * 4}


def movement_bytes(s):
    """Algorithmic bytes per launch of the HBM-bound kernels (what each must read and
    write at the minimum): permute (x rows in, sorted rows out, slot ids and weights),
    combine (sorted rows in, token rows out, inverse permutation and weights), the
    backward's dX reduction (the same without weights; it runs beside the dW_down GEMM,
    so its time there is shared time) and the
    backward's row preparation (dY and x rows in; dY_perm, its fp16 copy and the fp16
    copy of x_perm out)."""
    T, R, D = s.T, s.R, s.D
    return {"gather_x": T * D * 2 + R * D * 2 + 8 * R,
            "combine": R * D * 2 + 8 * R + T * D * 2,
            "combine_dx": R * D * 2 + 4 * R + T * D * 2,
            "bwd_prep_rows": 2 * T * D * 2 + 3 * R * D * 2 + 4 * R}


def direction_bytes(s):
    """Minimum bytes each direction must move: forward X, all expert weights, Y;
    backward X, dY, the weights, dX and the fp32 weight gradients."""
    w = 3 * s.E * s.D * s.I
    return {"fwd": 2 * s.T * s.D * 2 + w * 2, "bwd": 3 * s.T * s.D * 2 + w * 2 + w * 4}


def pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="qwen3_30b_a3b")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def get_shape(name):
    from mixture_experts_expert_gb300 import synth
    try:
        return synth.shape_by_name(name)
    except ValueError as e:
        raise SystemExit(str(e))


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every 20 ms while running;
    only the samples taken inside the marked window count."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []     # (host time the line arrived, line)
        self.thread = None
        self.window = (0.0, float("inf"))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if not (self.window[0] <= t <= self.window[1]):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the architecture)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def workload_config(s, world=1):
    """The `config` object of every line this script prints for workload `s`."""
    return {"workload": s.name, "T": s.T, "D": s.D, "I": s.I, "E": s.E, "K": s.K,
            "align": 128, "router": s.router,
            "l2": "working set larger than L2 (expert weights alone 3*E*D*I*2 bytes)",
            "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"}


class OracleSample:
    """The oracle as it stands, on this host's cores, expert by expert: the workload's
    inputs and sorted rows are prepared once; run(e) times the forward and the backward of
    expert e, each on its own."""

    def __init__(self, shape):
        import numpy as np

        import oracle
        from mixture_experts_expert_gb300 import synth
        self.s = s = shape
        self.oracle = oracle
        inp = synth.make_inputs(s)
        x = inp["x"].double().numpy()
        self.dy = inp["dy"].double().numpy()
        ids = inp["topk_ids"].numpy().astype(np.int64)
        w = inp["topk_w"].double().numpy()
        self.r = oracle.route_permute(ids, w, x, s.E, 128)
        self.wg, self.wu, self.wd = ([t[e].double().numpy() for e in range(s.E)]
                                     for t in (inp["w_gate"], inp["w_up"], inp["w_down"]))

    def run(self, e):
        """(routed rows of expert e, forward seconds, backward seconds)."""
        o, r = self.oracle, self.r
        t0 = time.perf_counter()
        o.expert_mlp_fwd(r["x_perm"], self.wg, self.wu, self.wd, r["offsets"], experts=[e])
        t1 = time.perf_counter()
        o.expert_mlp_bwd(self.dy, r["x_perm"], r["perm_src"], r["w_perm"], r["offsets"],
                         self.wg, self.wu, self.wd, self.s.K, experts=[e])
        t2 = time.perf_counter()
        return int(r["counts"][e]), t1 - t0, t2 - t1


def cpu_baseline(shape, budget_s=12.0, router=None):
    """The oracle timed on this host's cores over a bounded sample of the workload, forward
    and backward separately (FLOPs counted as for the GPU: 6 and 12 R*D*I).  With
    `router` = (logits, ids) (host arrays: the logits the router kernel was given and the
    ids it chose) the leg also checks that choice against the oracle's router."""
    smp = OracleSample(shape)
    rows, t_f, t_b, done = 0, 0.0, 0.0, []
    for e in range(shape.E):
        r_e, f_e, b_e = smp.run(e)
        rows, t_f, t_b = rows + r_e, t_f + f_e, t_b + b_e
        done.append(e)
        if t_f + t_b > budget_s:
            break
    s = shape
    rdi = rows * s.D * s.I
    out = {"value": 18.0 * rdi / (t_f + t_b) / 1e12, "unit": "TFLOP/s",
           "fwd": 6.0 * rdi / t_f / 1e12, "bwd": 12.0 * rdi / t_b / 1e12,
           "cores": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
           "sample": f"fp64 forward and backward of experts {done[0]}..{done[-1]} ({rows} "
                     f"routed rows of {s.R}) of the {s.name} layer, {t_f:.1f} s forward + "
                     f"{t_b:.1f} s backward"}
    if router is not None:
        import numpy as np
        logits, ids = router
        ids_ref, _ = smp.oracle.router_topk(logits, s.K, s.router)
        out["router_choice_matches_oracle"] = bool(np.array_equal(ids, ids_ref))
    return out


def run_reference(args, shape):
    """The CPU oracle as the reference arm: each step is a bounded sample (one expert's
    forward and backward), timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = shape
    smp = OracleSample(s)
    for i in range(args.warmup):
        smp.run(i % s.E)
    rows, t_f, t_b = 0, 0.0, 0.0
    for i in range(args.steps):
        r_i, f_i, b_i = smp.run((args.warmup + i) % s.E)
        rows, t_f, t_b = rows + r_i, t_f + f_i, t_b + b_i
    dt = t_f + t_b
    rdi = rows * s.D * s.I
    value = 18.0 * rdi / dt / 1e12
    sample = (f"fp64 forward and backward of one expert per step ({rows} routed rows in "
              f"{args.steps} steps) of the {s.name} layer")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(s, args.gpus),
            "fwd_tflops": 6.0 * rdi / t_f / 1e12, "bwd_tflops": 12.0 * rdi / t_b / 1e12,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    shape = get_shape(args.workload)
    if args.impl == "reference":
        run_reference(args, shape)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist

    from mixture_experts_expert_gb300 import binding as B
    from mixture_experts_expert_gb300 import build as Bld
    from mixture_experts_expert_gb300 import synth
    from mixture_experts_expert_gb300.layer import MoEExpertMLP
    from mixture_experts_expert_gb300.replicas import job_throughput, max_over_ranks

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_status = None
    if rank == 0 or world == 1:
        Bld.build()
        build_status = Bld.last_status
        print(f"libmoe_gb300: {build_status} {Bld.LIB_PATH}", file=sys.stderr, flush=True)
    if world > 1:
        dist.barrier()
    B.lib()

    s = shape
    inp = synth.make_inputs(s, device=dev)
    layer = MoEExpertMLP(s.T, s.K, s.E, s.D, s.I, align=128, device=dev)
    wg, wu, wd = inp["w_gate"], inp["w_up"], inp["w_down"]
    stream = torch.cuda.current_stream(dev)

    def step():
        layer.forward(inp["x"], inp["topk_ids"], inp["topk_w"], wg, wu, wd)
        ev_mid.record(stream)
        layer.backward(inp["dy"], wg, wu, wd)

    ev_mid = torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK

    sampler = ClockSampler(local)   # nvidia-smi needs a moment to start
    sampler.start()
    time.sleep(0.3)

    # ---------------- per-kernel table: a separate pass with every launch bracketed by
    # CUDA events (the events cost ~2% of a step, so the timed region below brackets only
    # the dominant GEMM)
    kpass = min(args.steps, 10)
    B.moe_timing_collect()   # drop anything recorded before
    B.moe_timing_enable(True)
    for _ in range(kpass):
        step()
    torch.cuda.synchronize()
    B.moe_timing_enable(False)
    per_kernel = B.moe_timing_collect()
    gemm_times = {k: v[0] for k, v in per_kernel.items() if k in GEMM_FLOPS_RDI}
    dom = max(gemm_times, key=gemm_times.get) if gemm_times else None

    # ---------------- timed region (device-resident inputs)
    launches0, _ = B.moe_launch_count()
    B.moe_timing_enable_only([dom] if dom else [])
    t_load0 = time.perf_counter()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        starts[i].record(stream)
        ev_mid = mids[i]
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    B.moe_timing_enable(False)
    launches1, _ = B.moe_launch_count()
    dom_timed = B.moe_timing_collect()   # the dominant GEMM's launches inside the timed region
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    fwd_ms = [a.elapsed_time(b) for a, b in zip(starts, mids)]
    bwd_ms = [a.elapsed_time(b) for a, b in zip(mids, ends)]
    total_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), dev)
    ms_per_step = total_ms / args.steps
    step_flops = s.fwd_flops() + s.bwd_flops()
    value = job_throughput(step_flops, world, ms_per_step * 1e-3) / 1e12
    fwd_tflops = s.fwd_flops() / (statistics.median(fwd_ms) * 1e-3) / 1e12
    bwd_tflops = s.bwd_flops() / (statistics.median(bwd_ms) * 1e-3) / 1e12

    # ---------------- end to end through host buffers (pinned), same step
    # Every step copies its inputs (x, ids, w, dY) in from pinned host memory and its
    # results (Y, dX) out.  The copies run on a second stream and are double-buffered:
    # step i+2's inputs are copied in and step i's results copied out while step i+1
    # computes (the layer writes Y and dX into one of two device output sets).
    keys = ("x", "topk_ids", "topk_w", "dy")
    host = {k: inp[k].cpu().pin_memory() for k in keys}
    out_y = [torch.empty(s.T, s.D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    out_dx = [torch.empty(s.T, s.D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    stage_y = [torch.empty(s.T, s.D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    stage_dx = [torch.empty(s.T, s.D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_y[0].numel() * out_y[0].element_size() + out_dx[0].numel() * out_dx[0].element_size()
    copy = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, staged, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def prefetch(b):
        with torch.cuda.stream(copy):
            for k in keys:
                dev_in[b][k].copy_(host[k], non_blocking=True)
            h2d_done[b].record(copy)

    def e2e_step(i, n):
        b = i % 2
        stream.wait_event(h2d_done[b])
        d = dev_in[b]
        stream.wait_event(d2h_done[b])          # output set b has been copied out
        layer.forward(d["x"], d["topk_ids"], d["topk_w"], wg, wu, wd, out=stage_y[b])
        layer.backward(d["dy"], wg, wu, wd, dx_out=stage_dx[b])
        staged[b].record(stream)
        with torch.cuda.stream(copy):
            copy.wait_event(staged[b])
            out_y[b].copy_(stage_y[b], non_blocking=True)
            out_dx[b].copy_(stage_dx[b], non_blocking=True)
            d2h_done[b].record(copy)
        if i + 2 < n:
            prefetch(b)                          # inputs of step i + 2 (slot b is free)

    def e2e_run(n):
        copy.wait_stream(stream)
        prefetch(0)
        if n > 1:
            prefetch(1)
        for i in range(n):
            e2e_step(i, n)
        stream.wait_stream(copy)                 # the last results have reached the host

    e2e_run(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    t_load1 = time.perf_counter()
    sampler.mark(t_load0, t_load1)   # clocks under load: the timed region and the e2e run
    clocks = sampler.stop()
    clocks["window"] = "timed region and end-to-end run"
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = job_throughput(step_flops, world, e2e_ms / args.steps * 1e-3) / 1e12
    assert layer.device_error()[0] == B.MOE_OK
    # the host copy of the last step's Y equals the device-resident result of the same inputs
    assert torch.equal(out_y[(args.steps - 1) % 2].to(dev), layer.y)

    # ---------------- the same step captured once as a CUDA graph and replayed
    def graph_step():
        layer.forward(inp["x"], inp["topk_ids"], inp["topk_w"], wg, wu, wd)
        layer.backward(inp["dy"], wg, wu, wd)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graph_step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), dev) / args.steps
    assert layer.device_error()[0] == B.MOE_OK

    # ---------------- the router step (not part of the expert-MLP metric): routing from
    # the workload's logits, and the logit gradient after the backward
    logits = inp["logits"].to(dev)

    def router_step():
        layer.route(logits, s.router)
        layer.router_backward(inp["dy"])

    router_step()
    torch.cuda.synchronize()
    B.moe_timing_collect()
    B.moe_timing_enable_only(["router_topk", "router_weight_grad", "router_backward"])
    for _ in range(args.steps):
        router_step()
    torch.cuda.synchronize()
    B.moe_timing_enable(False)
    router_ms = {k: v[0] / v[1] for k, v in B.moe_timing_collect().items()}
    router_choice = (logits.cpu().numpy(), layer.topk_ids.cpu().numpy())

    # ---------------- roofline of the dominant kernel (largest share of the step)
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    rdi = s.R * s.D * s.I
    kernels = {}
    hbm_gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gb = gemm_bytes(s)
    ridge = peak * 1e12 / (hbm_gbs * 1e9)   # FLOP per byte where the two roofs meet
    for k, (ms_k, n_k) in sorted(per_kernel.items()):
        ent = {"ms_per_launch": ms_k / n_k, "launches_per_step": n_k / kpass}
        if k in GEMM_FLOPS_RDI:
            sec = ms_k / n_k * 1e-3
            tf = GEMM_FLOPS_RDI[k] * rdi / sec / 1e12
            ai = GEMM_FLOPS_RDI[k] * rdi / gb[k]
            ent["tflops"] = tf
            ent["frac_of_sustained_peak"] = tf / peak
            ent["gbs"] = gb[k] / sec / 1e9
            ent["flop_per_byte"] = ai
            ent["bound"] = "tensor" if ai >= ridge else "hbm"
            ent["frac_of_roof"] = (tf / peak) if ai >= ridge else ent["gbs"] / hbm_gbs
        kernels[k] = ent
    for k, nbytes in movement_bytes(s).items():
        if k in kernels:
            gbs = nbytes / (kernels[k]["ms_per_launch"] * 1e-3) / 1e9
            kernels[k]["gbs"] = gbs
            kernels[k]["frac_of_hbm"] = gbs / hbm_gbs
    db = direction_bytes(s)
    roof_fwd = min(peak_tf, s.fwd_flops() / db["fwd"] * hbm_gbs * 1e9 / 1e12)
    roof_bwd = min(peak_tf, s.bwd_flops() / db["bwd"] * hbm_gbs * 1e9 / 1e12)
    achieved = dom_ms = None
    dom_bound = kernels[dom]["bound"] if dom else "tensor"
    if dom and dom in dom_timed:
        ms_d, n_d = dom_timed[dom]
        dom_ms = ms_d / n_d
        if dom_bound == "tensor":
            achieved = GEMM_FLOPS_RDI[dom] * rdi / (dom_ms * 1e-3) / 1e12
        else:
            achieved = gb[dom] / (dom_ms * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if dom and os.path.exists(prof):
        try:
            with open(prof) as fh:
                traffic = json.load(fh).get(f"{s.name}:{dom}")
        except Exception:
            traffic = None

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(s, world),
        "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "fwd_frac_of_peak": fwd_tflops / peak_tf, "bwd_frac_of_peak": bwd_tflops / peak_tf,
        "peak_bf16_tflops": peak_tf, "peak_source": peak_src,
        "fwd_frac_of_roof": fwd_tflops / roof_fwd, "bwd_frac_of_roof": bwd_tflops / roof_bwd,
        "roof_tflops": {"fwd": roof_fwd, "bwd": roof_bwd,
                        "note": "min(dense bf16 peak, algorithmic FLOP/byte x measured HBM GB/s)"},
        "fwd_ms_median": statistics.median(fwd_ms), "bwd_ms_median": statistics.median(bwd_ms),
        "fwd_ms_p10_p90": [pct(fwd_ms, 0.1), pct(fwd_ms, 0.9)],
        "bwd_ms_p10_p90": [pct(bwd_ms, 0.1), pct(bwd_ms, 0.9)],
        "graph": {"ms_per_step": graph_ms,
                  "value": job_throughput(step_flops, world, graph_ms * 1e-3) / 1e12,
                  "note": "the same step captured once as a CUDA graph and replayed"},
        "step_ms_median": statistics.median(step_ms),
        "roofline": ({"kernel": dom, "bound": "tensor", "achieved": achieved,
                      "ms_per_launch": dom_ms, "peak": peak, "unit": "TFLOP/s",
                      "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                      "peak_source": f"bf16_tflops_sustained ({peak_src})"}
                     if dom_bound == "tensor" else
                     {"kernel": dom, "bound": "hbm", "achieved": achieved,
                      "ms_per_launch": dom_ms, "peak": hbm_gbs, "unit": "GB/s",
                      "frac": (achieved / hbm_gbs) if achieved else None, "traffic": traffic,
                      "algorithmic_bytes": gb[dom],
                      "flop_per_byte": kernels[dom]["flop_per_byte"],
                      "tflops": GEMM_FLOPS_RDI[dom] * rdi / (dom_ms * 1e-3) / 1e12 if dom_ms else None,
                      "peak_source": f"hbm_gbs ({peak_src})"}),
        "kernels": kernels,
        "kernels_pass": f"separate pass of {kpass} steps before the timed region, every "
                        "launch bracketed by CUDA events",
        "gpu_launches": int(launches1 - launches0),
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        "router": {"ms_per_launch": router_ms,
                   "weight_grad_gbs": (s.R * s.D * 2 + s.T * s.D * 2) /
                                      (router_ms.get("router_weight_grad", float("nan")) * 1e-3) / 1e9,
                   "note": "router step, outside the expert-MLP metric"},
    }
    tun, tun_src = B.moe_tuning_get(s.T, s.K, s.E, s.D, s.I)
    line["tuning"] = {"source": tun_src, **tun}
    line["build"] = build_status   # "compiled" on this host, or "reused" (source hash matched)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s, router=router_choice)
        line["router"]["choice_matches_oracle"] = line["cpu_baseline"].pop(
            "router_choice_matches_oracle")
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
