"""Pins of the router oracle against what the definition and the mathematics fix
(CPU).  Each check is independent of the oracle's own code path: a selection by
repeated argmax instead of a sort, the library softmax / logistic functions, finite
differences of the forward, the layer's linearity in the router weights."""
import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle


def rng_logits(T, E, seed):
    return np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)


def select_by_repeated_argmax(p, K):
    """K rounds of: the remaining expert of largest p, the lower index on ties."""
    left = list(range(len(p)))
    out = []
    for _ in range(K):
        best = left[0]
        for e in left[1:]:
            if p[e] > p[best]:
                best = e
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("T,E,K,seed", [(50, 8, 2, 0), (40, 16, 5, 1), (20, 128, 8, 2)])
def test_softmax_choice_matches_repeated_argmax(T, E, K, seed):
    z = rng_logits(T, E, seed)
    ids, w = oracle.router_topk(z, K, "softmax")
    p = softmax(z.astype(np.float64), axis=-1)
    for t in range(T):
        assert list(ids[t]) == select_by_repeated_argmax(p[t], K)
    assert np.allclose(w.sum(-1), 1.0, atol=1e-15)
    assert np.all(np.diff(w, axis=-1) <= 0)


def test_ties_take_the_lower_index():
    z = np.zeros((3, 6), np.float32)
    z[1, [1, 4]] = 2.0           # two equal maxima
    z[2] = [1, 3, 3, 3, 0, 3]
    ids, w = oracle.router_topk(z, 3, "softmax")
    assert list(ids[0]) == [0, 1, 2]
    assert list(ids[1]) == [1, 4, 0]
    assert list(ids[2]) == [1, 2, 3]
    assert np.allclose(w[0], 1 / 3) and np.allclose(w[2], 1 / 3)
    i1, _ = oracle.router_topk(z, 1, "sigmoid_top1")
    assert list(i1[:, 0]) == [0, 1, 1]


def test_all_experts_chosen_is_the_plain_softmax():
    z = rng_logits(30, 7, 3)
    ids, w = oracle.router_topk(z, 7, "softmax")
    p = softmax(z.astype(np.float64), axis=-1)
    assert np.allclose(w, np.take_along_axis(p, ids, axis=1), rtol=1e-13, atol=0)


def test_renormalised_top_k_is_softmax_of_the_chosen_logits():
    z = rng_logits(30, 32, 4)
    ids, w = oracle.router_topk(z, 4, "softmax")
    ref = softmax(np.take_along_axis(z.astype(np.float64), ids, axis=1), axis=-1)
    assert np.allclose(w, ref, rtol=1e-13, atol=0)


def test_sigmoid_top1_is_the_logistic_of_the_largest_logit():
    z = rng_logits(40, 16, 5)
    ids, w = oracle.router_topk(z, 1, "sigmoid_top1")
    assert np.array_equal(ids[:, 0], np.argmax(z, axis=1))
    assert np.allclose(w[:, 0], expit(z.max(axis=1).astype(np.float64)), rtol=1e-15)


@pytest.mark.parametrize("router,K", [("softmax", 3), ("sigmoid_top1", 1)])
def test_logit_gradient_matches_finite_differences(router, K):
    T, E = 6, 9
    z = rng_logits(T, E, 6).astype(np.float64)
    ids, _ = oracle.router_topk(z, K, router)
    dw = np.random.default_rng(7).standard_normal((T, K))
    dz = oracle.router_backward(z, ids, dw, router)
    h = 1e-6
    num = np.zeros_like(z)
    for t in range(T):
        for e in range(E):
            zp, zm = z.copy(), z.copy()
            zp[t, e] += h
            zm[t, e] -= h
            ip, wp = oracle.router_topk(zp, K, router)
            im, wm = oracle.router_topk(zm, K, router)
            assert np.array_equal(ip, ids) and np.array_equal(im, ids)   # choice unchanged
            num[t, e] = np.sum(dw * (wp - wm)) / (2 * h)
    assert np.allclose(dz, num, rtol=1e-6, atol=1e-9)


def test_logit_gradient_closed_form():
    """Renormalised top-K = softmax over the chosen logits, so dz_i = w_k (dw_k - <w, dw>)
    on the chosen experts and 0 elsewhere."""
    z = rng_logits(20, 16, 8)
    ids, w = oracle.router_topk(z, 4, "softmax")
    dw = np.random.default_rng(9).standard_normal(w.shape)
    dz = oracle.router_backward(z, ids, dw, "softmax")
    ref = np.zeros_like(dz)
    np.put_along_axis(ref, ids, w * (dw - (w * dw).sum(-1, keepdims=True)), axis=1)
    assert np.allclose(dz, ref, rtol=1e-12, atol=1e-15)


def test_router_weight_gradient_from_the_layer():
    """L = sum(Y * dY) is linear in the router weights: its derivative in w[t,k] is the
    difference quotient of the layer forward (exact up to rounding), and
    sum w * dL/dw = L."""
    rng = np.random.default_rng(10)
    T, D, I, E, K = 5, 8, 6, 4, 2
    x = rng.standard_normal((T, D))
    wg, wu, wd = (rng.standard_normal(s) * 0.3 for s in ((E, D, I), (E, D, I), (E, I, D)))
    dy = rng.standard_normal((T, D))
    ids, w = oracle.router_topk(rng.standard_normal((T, E)), K, "softmax")
    dw = oracle.router_weight_grad(x, ids, wg, wu, wd, dy)
    L = lambda ww: float(np.sum(oracle.moe_forward(x, ids, ww, wg, wu, wd) * dy))  # noqa: E731
    for t in range(T):
        for k in range(K):
            wp, wm = w.copy(), w.copy()
            wp[t, k] += 0.5
            wm[t, k] -= 0.5
            assert abs((L(wp) - L(wm)) - dw[t, k]) < 1e-10
    assert abs(np.sum(w * dw) - L(w)) < 1e-10
