"""CPU oracle for the router step on both sides of the expert-MLP layer.

TEST INFRASTRUCTURE ONLY (same status as moe_oracle): the plain fp64 statement that
the CUDA router kernels are checked against; nothing in the library imports it.

The pages ("LigerCute -- native CUTLASS + NVSHMEM kernels", LigerMoE design, Forward
pass) say only that the final local combine applies the router weights; how the
weights arise is fixed by the workloads the layer is measured on:

* softmax router: p = softmax(z) over all E logits of a token; the K experts of
  largest p (equal p: the lower expert index first; slot k = 0 holds the largest);
  w_k = p_{i_k} / sum_j p_{i_j} (renormalised over the K chosen experts).
* sigmoid top-1 router (the Llama-4-Scout shape): the expert of largest logit (equal
  logits: the lower index), w = sigmoid(z_i), not renormalised.

The router-weight gradient of L = sum(Y * dY), Y[t] = sum_k w[t,k] f_{i_k}(x[t]), is
dL/dw[t,k] = <dY[t], f_{i_k}(x[t])>; the logit gradient follows by the chain rule
through the weights (the choice of experts is piecewise constant in z, so it adds
nothing).

Pins (tests/test_oracle_router.py): the choice against a brute-force scan over all
ordered K-subsets' keys; the weights' sum and order; the gradients against fp64 central
finite differences of the forward; the logit gradient against the equivalent
softmax-over-the-chosen-logits form (an identity that the definition implies).
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import sigmoid

__all__ = ["router_topk", "router_backward", "router_weight_grad", "ROUTERS"]

ROUTERS = ("softmax", "sigmoid_top1")


def _softmax(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def router_topk(logits, K: int, router: str = "softmax"):
    """(topk_ids [T,K] int64, topk_w [T,K] fp64) from logits [T,E]."""
    z = np.asarray(logits, dtype=np.float64)
    T, E = z.shape
    if router == "softmax":
        p = _softmax(z)
        ids = np.zeros((T, K), dtype=np.int64)
        w = np.zeros((T, K))
        for t in range(T):
            # descending p, ties by ascending index: sort on the key (-p, index)
            order = sorted(range(E), key=lambda e: (-p[t, e], e))[:K]
            ids[t] = order
            sel = p[t, order]
            w[t] = sel / sel.sum()
        return ids, w
    if router == "sigmoid_top1":
        if K != 1:
            raise ValueError("the sigmoid top-1 router takes K == 1")
        ids = np.zeros((T, 1), dtype=np.int64)
        for t in range(T):
            ids[t, 0] = min(range(E), key=lambda e: (-z[t, e], e))
        return ids, sigmoid(np.take_along_axis(z, ids, axis=1))
    raise ValueError(f"unknown router {router!r}")


def router_backward(logits, topk_ids, d_topk_w, router: str = "softmax"):
    """dL/dlogits [T,E] given dL/dw [T,K], for the experts chosen in topk_ids."""
    z = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    dw = np.asarray(d_topk_w, dtype=np.float64)
    T, E = z.shape
    dz = np.zeros((T, E))
    if router == "softmax":
        p = _softmax(z)
        for t in range(T):
            sel = ids[t]
            S = p[t, sel].sum()
            # w_k = p_{i_k} / S  =>  dL/dp_{i_k} = dw_k / S - sum_j dw_j p_{i_j} / S^2
            dp = np.zeros(E)
            dp[sel] = dw[t] / S - np.dot(dw[t], p[t, sel]) / S ** 2
            # softmax: dL/dz = p * (dL/dp - <p, dL/dp>)
            dz[t] = p[t] * (dp - np.dot(p[t], dp))
        return dz
    if router == "sigmoid_top1":
        s = sigmoid(np.take_along_axis(z, ids, axis=1))
        np.put_along_axis(dz, ids, dw * s * (1.0 - s), axis=1)
        return dz
    raise ValueError(f"unknown router {router!r}")


def router_weight_grad(x, topk_ids, w_gate, w_up, w_down, dy):
    """dL/dw [T,K] = <dY[t], f_{ids[t,k]}(x[t])> with the SwiGLU expert MLP f_e."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    dy = np.asarray(dy, dtype=np.float64)
    T, K = ids.shape
    dw = np.zeros((T, K))
    for t in range(T):
        for k in range(K):
            e = ids[t, k]
            g = x[t] @ np.asarray(w_gate[e], np.float64)
            u = x[t] @ np.asarray(w_up[e], np.float64)
            a = g * sigmoid(g) * u
            dw[t, k] = np.dot(dy[t], a @ np.asarray(w_down[e], np.float64))
    return dw
