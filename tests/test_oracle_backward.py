"""Pins for the oracle's backward, independent of the oracle's own formulas.

* fp64 central finite differences of L = sum(Y * dY) through the oracle's
  forward (itself pinned by the dense masked loop) for every element of dX and
  dW on a micro layer, and for sampled elements on the tiny layer;
* Y is linear in W_down[e] and in W_up[e], so
  <dW_down[e], W_down[e]> = <dW_up[e], W_up[e]> = sum over e's slots of
  w * <dY[t], f_e(x[t])>, with f_e evaluated here by a separate dense loop;
* experts that receive no token get exactly zero weight gradient;
* the permuted path (expert_mlp_bwd + unit-weight combine) equals the
  per-token definition;
* planted mistakes in the oracle are caught.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.moe_oracle as om
from mixture_experts_expert_gb300 import synth

from test_oracle_forward import small_case, to64


def loss(x, ids, w, wg, wu, wd, dy):
    return float(np.sum(oracle.moe_forward(x, ids, w, wg, wu, wd) * dy))


def fd_grad(arr, idx, f, h=1e-6):
    old = arr[idx]
    arr[idx] = old + h
    lp = f()
    arr[idx] = old - h
    lm = f()
    arr[idx] = old
    return (lp - lm) / (2 * h)


def assert_fd_close(an, fd, what):
    scale = max(1.0, float(np.max(np.abs(an))))
    err = np.max(np.abs(an - fd)) / scale
    assert err <= 1e-6, f"{what}: finite-difference mismatch {err:.3e}"


def micro():
    T, D, I, E, K = 8, 16, 8, 4, 2
    x, ids, w, wg, wu, wd = small_case(T, D, I, E, K, seed=11, w_std=0.5)
    dy = np.random.default_rng(12).standard_normal((T, D))
    return x, ids, w, wg, wu, wd, dy


def test_backward_all_elements_finite_difference_micro():
    x, ids, w, wg, wu, wd, dy = micro()
    dx, dwg, dwu, dwd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    f = lambda: loss(x, ids, w, wg, wu, wd, dy)  # noqa: E731
    for name, arr, an in (("dX", x, dx), ("dW_gate", wg, dwg), ("dW_up", wu, dwu),
                          ("dW_down", wd, dwd)):
        fd = np.zeros_like(an)
        for idx in np.ndindex(arr.shape):
            fd[idx] = fd_grad(arr, idx, f)
        assert_fd_close(an, fd, name)


def test_backward_sampled_finite_difference_tiny():
    s = synth.TINY
    inp = synth.make_inputs(s)
    x, wg, wu, wd, dy = (to64(inp[k]) for k in ("x", "w_gate", "w_up", "w_down", "dy"))
    ids, w = inp["topk_ids"].numpy().astype(np.int64), to64(inp["topk_w"])
    dx, dwg, dwu, dwd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    f = lambda: loss(x, ids, w, wg, wu, wd, dy)  # noqa: E731
    rng = np.random.default_rng(5)
    for name, arr, an in (("dX", x, dx), ("dW_gate", wg, dwg), ("dW_up", wu, dwu),
                          ("dW_down", wd, dwd)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            fd = fd_grad(arr, idx, f, h=1e-5)
            scale = max(1e-3, float(np.max(np.abs(an))))
            assert abs(fd - an[idx]) / scale <= 1e-6, (name, idx, fd, an[idx])


def test_linear_weight_identity():
    x, ids, w, wg, wu, wd, dy = micro()
    _, _, dwu, dwd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    E = wg.shape[0]
    for e in range(E):
        rhs = 0.0
        for t in range(x.shape[0]):
            for k in range(ids.shape[1]):
                if ids[t, k] != e:
                    continue
                g = x[t] @ wg[e]
                a = g / (1.0 + np.exp(-g)) * (x[t] @ wu[e])
                rhs += w[t, k] * float(dy[t] @ (a @ wd[e]))
        assert abs(np.sum(dwd[e] * wd[e]) - rhs) <= 1e-12 * max(1.0, abs(rhs))
        assert abs(np.sum(dwu[e] * wu[e]) - rhs) <= 1e-12 * max(1.0, abs(rhs))


def test_empty_experts_get_zero_weight_gradient():
    T, D, I, E, K = 6, 8, 8, 10, 2
    x, _, w, wg, wu, wd = small_case(T, D, I, E, K, seed=3)
    ids = np.array([[0, 1], [1, 2], [0, 2], [2, 1], [0, 1], [1, 0]])
    dy = np.random.default_rng(1).standard_normal((T, D))
    _, dwg, dwu, dwd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    for e in range(3, E):
        assert np.all(dwg[e] == 0) and np.all(dwu[e] == 0) and np.all(dwd[e] == 0)
    r = oracle.route_permute(ids, w, x, E, 16)
    _, pg, pu, pd = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"],
                                           r["offsets"], wg, wu, wd, K)
    for e in range(3, E):
        assert np.all(pg[e] == 0) and np.all(pu[e] == 0) and np.all(pd[e] == 0)


@pytest.mark.parametrize("align", [1, 16, 128])
def test_permuted_backward_matches_definition(align):
    x, ids, w, wg, wu, wd, dy = micro()
    T, K = ids.shape
    E = wg.shape[0]
    dx, dwg, dwu, dwd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    r = oracle.route_permute(ids, w, x, E, align)
    dxp, pg, pu, pd = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"],
                                             r["offsets"], wg, wu, wd, K)
    assert np.all(dxp[r["perm_src"] < 0] == 0)
    np.testing.assert_allclose(oracle.combine(dxp, r["inv_perm"], None, T, K), dx,
                               rtol=1e-12, atol=1e-14)
    for a, b in ((pg, dwg), (pu, dwu), (pd, dwd)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_expert_subset_matches_full():
    x, ids, w, wg, wu, wd, dy = micro()
    T, K = ids.shape
    r = oracle.route_permute(ids, w, x, wg.shape[0], 16)
    full = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"], r["offsets"],
                                 wg, wu, wd, K)
    sub = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"], r["offsets"],
                                wg, wu, wd, K, experts=[1, 3])
    for e in (1, 3):
        rows = slice(int(r["offsets"][e]), int(r["offsets"][e + 1]))
        assert np.array_equal(sub[0][rows], full[0][rows])
        for a, b in zip(sub[1:], full[1:]):
            assert np.array_equal(a[e], b[e])
    assert sorted(sub[1]) == [1, 3]
    yf = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
    ys = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"], experts=[2])
    rows = slice(int(r["offsets"][2]), int(r["offsets"][3]))
    assert np.array_equal(ys[rows], yf[rows])


def _fd_mismatch(x, ids, w, wg, wu, wd, dy):
    """Largest scaled finite-difference error over all of dW_gate (micro layer)."""
    _, dwg, _, _ = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    f = lambda: loss(x, ids, w, wg, wu, wd, dy)  # noqa: E731
    fd = np.zeros_like(dwg)
    for idx in np.ndindex(wg.shape):
        fd[idx] = fd_grad(wg, idx, f)
    return np.max(np.abs(dwg - fd)) / max(1.0, float(np.max(np.abs(dwg))))


def test_planted_silu_derivative_mistake_is_caught(monkeypatch):
    """Drop the (1 + g(1 - sigmoid g)) factor of SiLU' in the oracle: FD must object."""
    x, ids, w, wg, wu, wd, dy = micro()
    assert _fd_mismatch(x, ids, w, wg, wu, wd, dy) <= 1e-6
    monkeypatch.setattr(om, "silu_grad", lambda z: om.sigmoid(z))
    assert _fd_mismatch(x, ids, w, wg, wu, wd, dy) > 1e-3


def test_planted_missing_router_weight_in_backward_is_caught(monkeypatch):
    """Backward that forgets the router weight on dY: the identity pin must object."""
    x, ids, w, wg, wu, wd, dy = micro()
    _, _, _, dwd_good = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    _, _, _, dwd_bad = oracle.moe_backward(x, ids, np.ones_like(w), wg, wu, wd, dy)
    e = int(ids[0, 0])
    rhs = 0.0
    for t in range(x.shape[0]):
        for k in range(ids.shape[1]):
            if ids[t, k] == e:
                g = x[t] @ wg[e]
                a = g / (1.0 + np.exp(-g)) * (x[t] @ wu[e])
                rhs += w[t, k] * float(dy[t] @ (a @ wd[e]))
    assert abs(np.sum(dwd_good[e] * wd[e]) - rhs) <= 1e-12 * max(1, abs(rhs))
    assert abs(np.sum(dwd_bad[e] * wd[e]) - rhs) > 1e-6 * max(1, abs(rhs))
