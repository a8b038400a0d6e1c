"""Writes tiny_oracle_fingerprint.json: a regression lock on the oracle.

Calls only the oracle (and the seeded input generator) on the tiny layer
(T=256, D=256, I=128, E=8, K=2, seed 0) and stores the expert counts and
offsets plus the sum and Frobenius norm of every output.  The stored values
are the oracle's own, so they pin the oracle against unintended changes of its
arithmetic, not against the pages (which print no worked example).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mixture_experts_expert_gb300 import synth  # noqa: E402


def fingerprint():
    s = synth.TINY
    inp = synth.make_inputs(s)
    f = {k: inp[k].double().numpy() for k in ("x", "w_gate", "w_up", "w_down", "dy", "topk_w")}
    ids = inp["topk_ids"].numpy().astype(np.int64)
    r = oracle.route_permute(ids, f["topk_w"], f["x"], s.E, 128)
    y = oracle.moe_forward(f["x"], ids, f["topk_w"], f["w_gate"], f["w_up"], f["w_down"])
    dx, dwg, dwu, dwd = oracle.moe_backward(f["x"], ids, f["topk_w"], f["w_gate"], f["w_up"],
                                            f["w_down"], f["dy"])
    out = {"config": "tiny T=256 D=256 I=128 E=8 K=2 seed=0 align=128",
           "counts": r["counts"].tolist(), "offsets": r["offsets"].tolist()}
    for name, a in (("y", y), ("dx", dx), ("dw_gate", dwg), ("dw_up", dwu), ("dw_down", dwd)):
        out[name] = {"sum": float(a.sum()), "fro": float(np.sqrt((a * a).sum()))}
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_fingerprint.json")
    with open(path, "w") as fh:
        json.dump(fingerprint(), fh, indent=1)
    print("wrote", path)
