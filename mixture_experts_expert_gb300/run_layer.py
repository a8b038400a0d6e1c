"""Runs the layer's forward + backward on synthetic inputs of a chosen shape.

  python -m mixture_experts_expert_gb300.run_layer --T 2048 --D 2048 --I 768 --E 32 --K 8 --steps 3

A minimal example of driving the library, and the fixed command that kernel
profiles are taken with (a reduced expert count keeps the device footprint small
while each expert sees the same rows per expert as the full layer).
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import binding as B
from . import build as Bld
from . import synth
from .layer import MoEExpertMLP


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--D", type=int, default=2048)
    ap.add_argument("--I", type=int, default=768)
    ap.add_argument("--E", type=int, default=32)
    ap.add_argument("--K", type=int, default=8)
    ap.add_argument("--zipf", type=float, default=None)
    ap.add_argument("--steps", type=int, default=3)
    a = ap.parse_args()
    Bld.build()
    shape = dataclasses.replace(synth.QWEN3_30B_A3B, name="custom", T=a.T, D=a.D, I=a.I, E=a.E,
                                K=a.K, zipf_s=a.zipf)
    inp = synth.make_inputs(shape, device="cuda")
    layer = MoEExpertMLP(a.T, a.K, a.E, a.D, a.I, align=128, device="cuda")
    for _ in range(a.steps):
        layer.forward(inp["x"], inp["topk_ids"], inp["topk_w"], inp["w_gate"], inp["w_up"],
                      inp["w_down"])
        layer.backward(inp["dy"], inp["w_gate"], inp["w_up"], inp["w_down"])
    torch.cuda.synchronize()
    code, raw = layer.device_error()
    if code != B.MOE_OK:
        raise SystemExit(f"device error {raw}")
    print("ok", a)


if __name__ == "__main__":
    main()
