"""Pins for the oracle's forward (expert MLP and combine), independent of the oracle.

* a dense, masked per-token loop over *all* experts, with SiLU written in its
  tanh form, so a slip in the oracle's sparse path or its SiLU shows up;
* K = 1 with weight 1 reduces to a plain SwiGLU MLP computed with torch's own
  fp64 ``silu`` and matmul;
* linearity in the router weights and a hand-derived scalar case;
* a planted mistake in the oracle is caught.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.moe_oracle as om
from mixture_experts_expert_gb300 import synth


def to64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def dense_masked_forward(x, ids, w, wg, wu, wd):
    """y[t] = sum over ALL experts e of m[t,e] * f_e(x[t]), m[t,e] = sum_k w[t,k][ids[t,k]==e]."""
    T = x.shape[0]
    E = wg.shape[0]
    y = np.zeros((T, wd.shape[2]))
    for t in range(T):
        for e in range(E):
            m = sum(float(w[t, k]) for k in range(ids.shape[1]) if ids[t, k] == e)
            if m == 0.0:
                continue
            g = x[t] @ wg[e]
            u = x[t] @ wu[e]
            a = 0.5 * g * (1.0 + np.tanh(0.5 * g)) * u   # silu(g) = g/2 * (1 + tanh(g/2))
            y[t] += m * (a @ wd[e])
    return y


def small_case(T, D, I, E, K, seed, w_std=0.3, repeats=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, D, I, generator=g) * w_std).to(torch.bfloat16)
    wu = (torch.randn(E, D, I, generator=g) * w_std).to(torch.bfloat16)
    wd = (torch.randn(E, I, D, generator=g) * w_std).to(torch.bfloat16)
    ids, w = synth.random_routing(T, K, E, seed=seed + 100, allow_repeats=repeats)
    return to64(x), ids.numpy().astype(np.int64), to64(w), to64(wg), to64(wu), to64(wd)


@pytest.mark.parametrize("T,D,I,E,K,seed,repeats", [
    (8, 16, 8, 4, 2, 0, False),
    (33, 24, 16, 6, 3, 1, True),
    (12, 8, 8, 16, 2, 2, False),   # more experts than tokens
])
def test_forward_matches_dense_masked_loop(T, D, I, E, K, seed, repeats):
    x, ids, w, wg, wu, wd = small_case(T, D, I, E, K, seed, repeats=repeats)
    ref = dense_masked_forward(x, ids, w, wg, wu, wd)
    y = oracle.moe_forward(x, ids, w, wg, wu, wd)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # the permuted path (sort, expert MLP, combine) gives the same result
    for align in (1, 8, 128):
        r = oracle.route_permute(ids, w, x, E, align)
        y_perm = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
        y2 = oracle.combine(y_perm, r["inv_perm"], w, T, K)
        np.testing.assert_allclose(y2, ref, rtol=1e-12, atol=1e-12)
        # padding rows stay exactly zero through the expert MLP
        assert np.all(y_perm[r["perm_src"] < 0] == 0.0)


def test_tiny_config_matches_dense_masked_loop():
    s = synth.TINY
    inp = synth.make_inputs(s)
    x, wg, wu, wd = (to64(inp[k]) for k in ("x", "w_gate", "w_up", "w_down"))
    ids, w = inp["topk_ids"].numpy().astype(np.int64), to64(inp["topk_w"])
    ref = dense_masked_forward(x, ids, w, wg, wu, wd)
    r = oracle.route_permute(ids, w, x, s.E, 128)
    y_perm = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
    y = oracle.combine(y_perm, r["inv_perm"], w, s.T, s.K)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-13)


def test_k1_unit_weight_is_plain_swiglu_mlp():
    """K = 1, w = 1: each token goes through exactly one expert's SwiGLU MLP."""
    T, D, I, E = 20, 16, 12, 3
    x, _, _, wg, wu, wd = small_case(T, D, I, E, 1, seed=7)
    ids = (np.arange(T) % E).reshape(T, 1)
    w = np.ones((T, 1))
    y = oracle.moe_forward(x, ids, w, wg, wu, wd)
    F = torch.nn.functional
    for t in range(T):
        e = int(ids[t, 0])
        xt = torch.from_numpy(x[t:t + 1])
        ref = (F.silu(xt @ torch.from_numpy(wg[e])) * (xt @ torch.from_numpy(wu[e]))) \
            @ torch.from_numpy(wd[e])
        np.testing.assert_allclose(y[t], ref.numpy()[0], rtol=1e-12, atol=1e-14)


def test_linear_in_router_weights():
    x, ids, w, wg, wu, wd = small_case(10, 8, 8, 4, 2, seed=3)
    y1 = oracle.moe_forward(x, ids, w, wg, wu, wd)
    y2 = oracle.moe_forward(x, ids, 2.5 * w, wg, wu, wd)
    np.testing.assert_allclose(y2, 2.5 * y1, rtol=1e-13, atol=1e-15)
    # and additive over the K slots
    ya = oracle.moe_forward(x, ids[:, :1], w[:, :1], wg, wu, wd)
    yb = oracle.moe_forward(x, ids[:, 1:], w[:, 1:], wg, wu, wd)
    np.testing.assert_allclose(ya + yb, y1, rtol=1e-13, atol=1e-15)


def test_scalar_closed_form():
    """D = I = 1, one token, two experts, worked by hand.

    expert 0: g = 1.5*2 = 3, u = 1.5*(-1) = -1.5, a = silu(3)*(-1.5), y0 = a*0.5
    expert 1: g = 1.5*(-0.5) = -0.75, u = 1.5*4 = 6, a = silu(-0.75)*6, y1 = a*(-2)
    Y = 0.75*y0 + 0.25*y1
    """
    def silu_hand(z):
        return z / (1.0 + math.exp(-z))
    x = np.array([[1.5]])
    wg = np.array([[[2.0]], [[-0.5]]])
    wu = np.array([[[-1.0]], [[4.0]]])
    wd = np.array([[[0.5]], [[-2.0]]])
    ids = np.array([[0, 1]])
    w = np.array([[0.75, 0.25]])
    expect = 0.75 * (silu_hand(3.0) * -1.5 * 0.5) + 0.25 * (silu_hand(-0.75) * 6.0 * -2.0)
    y = oracle.moe_forward(x, ids, w, wg, wu, wd)
    assert abs(y[0, 0] - expect) < 1e-15
    r = oracle.route_permute(ids, w, x, 2, 1)
    yp = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
    assert abs(oracle.combine(yp, r["inv_perm"], w, 1, 2)[0, 0] - expect) < 1e-15


def test_combine_unit_weights_sums_rows():
    src = np.arange(12, dtype=np.float64).reshape(6, 2)
    inv = np.array([5, 0, 2, 3])     # T=2, K=2
    out = oracle.combine(src, inv, None, 2, 2)
    assert out.tolist() == [[10 + 0, 11 + 1], [4 + 6, 5 + 7]]


def test_planted_silu_mistake_is_caught(monkeypatch):
    """Plant a wrong activation in the oracle: the dense-loop pin must fail."""
    x, ids, w, wg, wu, wd = small_case(8, 16, 8, 4, 2, seed=0)
    ref = dense_masked_forward(x, ids, w, wg, wu, wd)
    monkeypatch.setattr(om, "silu", lambda z: np.asarray(z) * 0.5)
    y = oracle.moe_forward(x, ids, w, wg, wu, wd)
    assert not np.allclose(y, ref, rtol=1e-6, atol=1e-9)


def test_planted_weight_placement_mistake_is_caught():
    """Router weights scale expert outputs, not inputs: weighting the input instead differs."""
    x, ids, w, wg, wu, wd = small_case(8, 16, 8, 4, 2, seed=0)
    ref = dense_masked_forward(x, ids, w, wg, wu, wd)
    wrong = np.zeros_like(ref)
    for t in range(8):
        for k in range(2):
            e = ids[t, k]
            xs = w[t, k] * x[t]
            wrong[t] += (om.silu(xs @ wg[e]) * (xs @ wu[e])) @ wd[e]
    assert not np.allclose(wrong, ref, rtol=1e-6, atol=1e-9)
