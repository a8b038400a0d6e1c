"""Seeded synthetic inputs for the routed MoE expert-MLP layer.

This module draws inputs.  It holds none of the expert-MLP layer's arithmetic (no
permutation, no expert MLP, no combine, no gradient).  It does derive the layer's
routing input from the drawn logits (``route_from_logits``, plain torch ops): that
is the input recipe the workloads state, not a reference for the library's own
router kernel, which the tests check against the oracle's router instead.  Both the
CUDA path and the CPU oracle consume the arrays it returns, bit for bit.

Recipe (one generator, fixed draw order):

* ``x``      [T, D]    ~ N(0, 1)
* ``w_gate`` [E, D, I] ~ N(0, w_std)
* ``w_up``   [E, D, I] ~ N(0, w_std)
* ``w_down`` [E, I, D] ~ N(0, w_std)
* ``logits`` [T, E]    ~ N(0, 1), plus ``-zipf_s * ln(e + 1)`` when a Zipf
  popularity bias is requested
* ``dy``     [T, D]    ~ N(0, 1)

Values are drawn in fp32 and rounded to bf16 (round to nearest even) for x,
the weights and dy. Routing is an input of the layer, derived from the logits:

* ``router="softmax"``: softmax over all E logits, the K largest
  probabilities (ties go to the lower expert index, k = 0 is the largest),
  renormalised to sum to one.  Shapes like Qwen3-30B-A3B use this.
* ``router="sigmoid_top1"``: the largest logit's expert, weight
  ``sigmoid(logit)`` with no renormalisation (K must be 1).  Shapes like
  Llama-4-Scout use this.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """One layer configuration: tokens, hidden, intermediate, experts, top-K."""

    name: str
    T: int
    D: int
    I: int
    E: int
    K: int
    w_std: float = 0.02
    router: str = "softmax"
    zipf_s: float | None = None
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.K

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: 2*R*D*I for each of gate, up and down."""
        return 6.0 * self.R * self.D * self.I

    def bwd_flops(self) -> float:
        """Algorithmic backward FLOPs (twice the forward; recompute is overhead)."""
        return 12.0 * self.R * self.D * self.I

    def bwd_flops_executed(self) -> float:
        """Backward FLOPs as executed, counting the gate/up recompute."""
        return 16.0 * self.R * self.D * self.I


# The workloads: a tiny layer, Qwen3-30B-A3B and Llama-4-Scout expert shapes,
# a token sweep at the Qwen shape and a Zipf-skewed routing stress.
TINY = MoEShape("tiny", T=256, D=256, I=128, E=8, K=2, w_std=0.02)
QWEN3_30B_A3B = MoEShape("qwen3_30b_a3b", T=8192, D=2048, I=768, E=128, K=8, w_std=0.02)
LLAMA4_SCOUT = MoEShape("llama4_scout", T=8192, D=5120, I=8192, E=16, K=1, w_std=0.01,
                        router="sigmoid_top1")
SKEWED = MoEShape("skewed_zipf1.2", T=16384, D=2048, I=768, E=128, K=8, w_std=0.02,
                  zipf_s=1.2)
# A steeper profile of the same family (s = 1.4) that leaves 15 experts without a token.
SKEWED_STEEP = MoEShape("skewed_zipf1.4", T=16384, D=2048, I=768, E=128, K=8, w_std=0.02,
                        zipf_s=1.4)
# The Zipf stress at the Llama-4-Scout shape (few, large experts; top-1 sigmoid router).
SCOUT_SKEWED = MoEShape("llama4_scout_zipf1.2", T=8192, D=5120, I=8192, E=16, K=1,
                        w_std=0.01, router="sigmoid_top1", zipf_s=1.2)


def sweep_shape(T: int) -> MoEShape:
    """Token-count sweep point at the Qwen3-30B-A3B expert shape."""
    return dataclasses.replace(QWEN3_30B_A3B, name=f"qwen3_30b_a3b_T{T}", T=T)


SHAPES = {s.name: s for s in (TINY, QWEN3_30B_A3B, LLAMA4_SCOUT, SKEWED, SKEWED_STEEP,
                               SCOUT_SKEWED)}


def shape_by_name(name: str) -> MoEShape:
    """A workload of SHAPES, or a sweep point ``qwen3_30b_a3b_T<T>``."""
    if name in SHAPES:
        return SHAPES[name]
    if name.startswith("qwen3_30b_a3b_T"):
        return sweep_shape(int(name.split("_T")[-1]))
    raise ValueError(f"unknown workload {name!r}")


def route_from_logits(logits: torch.Tensor, K: int, router: str):
    """Top-K expert ids (int32) and fp32 router weights from fp32 logits: the routing
    input of the synthetic workloads (the router step itself is the library's
    moe_router_topk, checked against the oracle, not against this function)."""
    if router == "softmax":
        probs = torch.softmax(logits.float(), dim=-1)
        # stable descending sort: among equal probabilities the lower index wins
        p_sorted, idx = torch.sort(probs, dim=-1, descending=True, stable=True)
        top_p = p_sorted[:, :K]
        ids = idx[:, :K]
        w = top_p / top_p.sum(dim=-1, keepdim=True)
    elif router == "sigmoid_top1":
        if K != 1:
            raise ValueError("sigmoid_top1 routing needs K == 1")
        l_sorted, idx = torch.sort(logits.float(), dim=-1, descending=True, stable=True)
        ids = idx[:, :1]
        w = torch.sigmoid(l_sorted[:, :1])
    else:
        raise ValueError(f"unknown router {router!r}")
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def make_inputs(shape: MoEShape, device: str | torch.device = "cpu", seed: int | None = None):
    """Draw one layer's inputs.  Returns a dict of tensors on ``device``.

    Keys: x, w_gate, w_up, w_down (bf16), logits (fp32), dy (bf16),
    topk_ids (int32 [T, K]), topk_w (fp32 [T, K]).
    """
    s = shape
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(s.seed if seed is None else seed)
    kw = dict(generator=g, device=dev, dtype=torch.float32)
    x = torch.randn(s.T, s.D, **kw).to(torch.bfloat16)
    w_gate = (torch.randn(s.E, s.D, s.I, **kw) * s.w_std).to(torch.bfloat16)
    w_up = (torch.randn(s.E, s.D, s.I, **kw) * s.w_std).to(torch.bfloat16)
    w_down = (torch.randn(s.E, s.I, s.D, **kw) * s.w_std).to(torch.bfloat16)
    logits = torch.randn(s.T, s.E, **kw)
    if s.zipf_s is not None:
        bias = torch.tensor([-s.zipf_s * math.log(e + 1.0) for e in range(s.E)],
                            dtype=torch.float32, device=dev)
        logits = logits + bias
    dy = torch.randn(s.T, s.D, **kw).to(torch.bfloat16)
    ids, w = route_from_logits(logits, s.K, s.router)
    return dict(x=x, w_gate=w_gate, w_up=w_up, w_down=w_down, logits=logits, dy=dy,
                topk_ids=ids, topk_w=w)


def random_routing(T: int, K: int, E: int, seed: int = 0, allow_repeats: bool = False,
                   device="cpu"):
    """Uniform random routing for edge-case tests (ids int32 [T,K], weights fp32 [T,K]).

    With ``allow_repeats`` a token may name the same expert twice, which the
    layer must accept.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    if allow_repeats or K > E:
        ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int64)
    else:
        ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]) if T else \
            torch.zeros(0, K, dtype=torch.int64)
    w = torch.rand(T, K, generator=g) + 0.05
    w = w / w.sum(dim=-1, keepdim=True)
    return ids.to(torch.int32).to(device), w.to(torch.float32).to(device)
