"""Offline tuner of the grouped GEMMs' per-shape launch choices (``moe_tuning_t``).

Runs on one GB300.  For each layer shape it is given it times the layer's kernels (the
library's own per-launch CUDA events, inputs resident in HBM) under candidate choices,
keeps a candidate only when its median time over alternating repetitions beats the
current choice's by more than ``--margin``, and
prints the resulting table; ``--write`` stores it as ``csrc/tuning_table.inc``, which
the library compiles in (rebuild afterwards).  Choices are tuned one at a time, starting
from the defaults:

1. the tile order of each token-row GEMM (row pair by row pair, or N tile by N tile):
   each GEMM's own time decides;
2. transposed odd tail tiles on or off: the token-row GEMMs' summed time;
3. the dA GEMM's tile width (256 or 128 columns): its own time;
4. the dW chunk rows: dW preparation + dA + backward gate/up + both dW GEMMs.

Workloads with the same (T, K, E, D, I) share one table entry; their times are summed,
so an entry serves a uniform and a skewed routing of that size alike.  The choices
change speed only: every choice is covered by the GPU parity tests.

    python -m mixture_experts_expert_gb300.tune [--workloads a,b,...] [--write]
"""
from __future__ import annotations

import argparse
import copy
import json
import os
import sys

KIND_OF_GEMM = {"gate_up": "gemm_gateup_swiglu", "down": "gemm_down", "dA": "gemm_dA",
                "bwd_gate_up": "gemm_bwd_gateup", "dx": "gemm_dx"}
DW_KERNELS = ("dw_prep", "gemm_dA", "gemm_bwd_gateup", "gemm_dw_gateup", "gemm_dw_down")
# The chunk only spreads an expert's rows over tiles (whether its operands are
# compensated depends on its row count alone), so every candidate is equally accurate.
CHUNK_CANDIDATES = (1024, 2048, 4096, 8192, 16384)
DEFAULT_WORKLOADS = ("tiny", "qwen3_30b_a3b_T1024", "qwen3_30b_a3b_T2048",
                     "qwen3_30b_a3b_T4096", "qwen3_30b_a3b", "qwen3_30b_a3b_T16384",
                     "skewed_zipf1.2", "skewed_zipf1.4", "qwen3_30b_a3b_T32768",
                     "qwen3_30b_a3b_T65536", "llama4_scout", "llama4_scout_zipf1.2")
TABLE_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc",
                          "tuning_table.inc")


def default_choices() -> dict:
    return {"order": {g: 0 for g in KIND_OF_GEMM}, "swap_tails": 1, "da_tile_n": 256,
            "dw_chunk_rows": 4096}


class Bench:
    """One workload's inputs and layer; ``times(choices)`` -> mean ms per launch of
    every kernel of a forward + backward step under those choices."""

    def __init__(self, shape, steps: int, warmup: int):
        import torch

        from . import synth
        from .layer import MoEExpertMLP
        self.torch = torch
        self.shape = shape
        self.steps, self.warmup = steps, warmup
        self.inp = synth.make_inputs(shape, device="cuda")
        s = shape
        self.layer = MoEExpertMLP(s.T, s.K, s.E, s.D, s.I, align=128, device="cuda")

    def _step(self):
        i = self.inp
        self.layer.forward(i["x"], i["topk_ids"], i["topk_w"], i["w_gate"], i["w_up"],
                           i["w_down"])
        self.layer.backward(i["dy"], i["w_gate"], i["w_up"], i["w_down"])

    def times(self, choices: dict) -> dict:
        from . import binding as B
        B.moe_tuning_override(choices)
        try:
            for _ in range(self.warmup):
                self._step()
            self.torch.cuda.synchronize()
            B.moe_timing_collect()
            B.moe_timing_enable(True)
            for _ in range(self.steps):
                self._step()
            self.torch.cuda.synchronize()
            B.moe_timing_enable(False)
            per = B.moe_timing_collect()
            code, _ = self.layer.device_error()
            if code != B.MOE_OK:
                raise RuntimeError(f"{self.shape.name}: device error {code} under {choices}")
        finally:
            B.moe_tuning_override(None)
        return {k: ms / n for k, (ms, n) in per.items()}


def tune_key(benches, margin: float, reps: int, log) -> tuple[dict, dict]:
    """Coordinate search over the choices for the workloads of one shape key.  Each
    comparison times the two candidates alternately ``reps`` times and compares medians,
    so that a slow drift of the clocks does not favour either."""
    import statistics

    def timed(ch):
        tot = {}
        for b in benches:
            for k, v in b.times(ch).items():
                tot[k] = tot.get(k, 0.0) + v
        return tot

    def compare(a, b):
        runs_a, runs_b = [], []
        for _ in range(reps):
            runs_a.append(timed(a))
            runs_b.append(timed(b))
        med = lambda runs: {k: statistics.median(r.get(k, 0.0) for r in runs) for k in runs[0]}
        return med(runs_a), med(runs_b)

    def cost(t, kernels):
        return sum(t.get(k, 0.0) for k in kernels)

    def better(t_alt, t_cur, kernels):
        return cost(t_alt, kernels) < (1.0 - margin) * cost(t_cur, kernels)

    best = default_choices()
    # 1. tile order, per GEMM
    flipped = copy.deepcopy(best)
    for g in KIND_OF_GEMM:
        flipped["order"][g] = 1
    t0, t1 = compare(best, flipped)
    base = t0
    for g, kern in KIND_OF_GEMM.items():
        if better(t1, t0, [kern]):
            best["order"][g] = 1
    log(f"  order {best['order']}")
    # 2. transposed tails
    alt = copy.deepcopy(best)
    alt["swap_tails"] = 0
    tc, ta = compare(best, alt)
    if better(ta, tc, list(KIND_OF_GEMM.values())):
        best = alt
    log(f"  swap_tails {best['swap_tails']}")
    # 3. dA tile width (only shapes with I % 256 == 0 have a choice)
    if benches[0].shape.I % 256 == 0:
        alt = copy.deepcopy(best)
        alt["da_tile_n"] = 128
        tc, ta = compare(best, alt)
        if better(ta, tc, ["gemm_dA"]):
            best = alt
    log(f"  da_tile_n {best['da_tile_n']}")
    # 4. dW chunk rows
    for c in CHUNK_CANDIDATES:
        if c == best["dw_chunk_rows"]:
            continue
        alt = copy.deepcopy(best)
        alt["dw_chunk_rows"] = c
        tc, ta = compare(best, alt)
        if better(ta, tc, DW_KERNELS):
            best = alt
    log(f"  dw_chunk_rows {best['dw_chunk_rows']}")
    t_def, t_best = compare(default_choices(), best)
    return best, {"default_ms": sum(t_def.values()), "tuned_ms": sum(t_best.values()),
                  "default": t_def, "tuned": t_best}


def table_text(entries) -> str:
    lines = ["// Per-shape launch choices of the grouped GEMMs, measured on a GB300.",
             "// Written by `python -m mixture_experts_expert_gb300.tune --write`; "
             "do not edit by hand.",
             "// Fields: T, K, E, D, I, order[gate_up, down, dA, bwd_gate_up, dX], "
             "swap_tails, da_tile_n,",
             "// dw_chunk_rows.  The last row (T = 0) ends the table."]
    for (T, K, E, D, I), ch in sorted(entries.items()):
        o = ", ".join(str(ch["order"][g]) for g in KIND_OF_GEMM)
        lines.append(f"{{{T}, {K}, {E}, {D}, {I}, {{{o}}}, {ch['swap_tails']}, "
                     f"{ch['da_tile_n']}, {ch['dw_chunk_rows']}}},")
    lines.append("{0, 0, 0, 0, 0, {0, 0, 0, 0, 0}, 1, 256, 4096},")
    return "\n".join(lines) + "\n"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workloads", default=",".join(DEFAULT_WORKLOADS))
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--margin", type=float, default=0.015,
                    help="a candidate must be this fraction faster to replace the current")
    ap.add_argument("--reps", type=int, default=3,
                    help="alternating repetitions per comparison (medians compared)")
    ap.add_argument("--write", action="store_true", help=f"write {TABLE_PATH}")
    ap.add_argument("--json", default=None, help="also write the measurements here")
    args = ap.parse_args(argv)

    import torch

    from . import binding as B
    from . import synth
    if not torch.cuda.is_available():
        raise SystemExit("the tuner measures kernels: it needs a GPU")
    B.lib()

    def log(msg):
        print(msg, file=sys.stderr, flush=True)

    groups = {}
    for name in args.workloads.split(","):
        s = synth.shape_by_name(name.strip())
        groups.setdefault((s.T, s.K, s.E, s.D, s.I), []).append(s)
    entries, report = {}, {}
    for key, shapes in groups.items():
        log(f"{key}: {[s.name for s in shapes]}")
        benches = [Bench(s, args.steps, args.warmup) for s in shapes]
        ch, rep = tune_key(benches, args.margin, args.reps, log)
        entries[key] = ch
        report[",".join(s.name for s in shapes)] = {"key": key, "choices": ch, **rep}
        log(f"  step {rep['default_ms']:.3f} -> {rep['tuned_ms']:.3f} ms (sum of kernels)")
        del benches
        torch.cuda.empty_cache()
    text = table_text(entries)
    print(text, end="")
    if args.json:
        with open(args.json, "w") as fh:
            json.dump(report, fh, indent=1)
    if args.write:
        with open(TABLE_PATH, "w") as fh:
            fh.write(text)


if __name__ == "__main__":
    main()
