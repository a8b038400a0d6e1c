"""Pins for the oracle's expert sort (route_permute), independent of the oracle.

The reference point is a brute-force scan written here from the definition
("sort routed tokens by expert", stable inside an expert, each expert's segment
padded to ``align`` rows), plus the invariants every correct sort satisfies.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_expert_gb300 import synth


def brute_force_sort(ids, E, align):
    """O(R*E) scan: for each expert in order, list its flat slots ascending."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    R = len(flat)
    counts = [sum(1 for v in flat if v == e) for e in range(E)]
    offsets = [0]
    for e in range(E):
        padded = -(-counts[e] // align) * align
        offsets.append(offsets[-1] + padded)
    T, K = np.asarray(ids).shape
    cap = oracle.capacity(T, K, E, align)
    perm = [-1] * cap
    inv = [None] * R
    for e in range(E):
        row = offsets[e]
        for j in range(R):
            if flat[j] == e:
                perm[row] = j
                inv[j] = row
                row += 1
    return counts, offsets, perm, inv


def check_invariants(out, ids, w, x, E, align):
    ids = np.asarray(ids)
    T, K = ids.shape
    R = T * K
    counts, offsets, perm, inv = out["counts"], out["offsets"], out["perm_src"], out["inv_perm"]
    assert counts.sum() == R
    assert offsets[0] == 0 and np.all(np.diff(offsets) >= 0)
    assert np.all(offsets % align == 0)
    assert np.all(np.diff(offsets) - counts < align) and np.all(np.diff(offsets) >= counts)
    cap = oracle.capacity(T, K, E, align)
    assert offsets[-1] <= cap and perm.shape == (cap,)
    real = perm >= 0
    # bijection between non-padding rows and [0, R)
    assert real.sum() == R
    assert np.array_equal(np.sort(perm[real]), np.arange(R))
    assert np.array_equal(inv[perm[real]], np.nonzero(real)[0])
    for j in range(R):
        assert perm[inv[j]] == j
    # each row belongs to the segment of its expert, in ascending slot order
    flat = ids.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        got = seg[seg >= 0]
        assert np.all(flat[got] == e)
        assert np.all(np.diff(got) > 0)
        assert np.all(seg[:len(got)] >= 0)  # padding only at the end of the segment
    assert np.all(out["w_perm"][real] == np.asarray(w, np.float64).reshape(-1)[perm[real]])
    assert np.all(out["w_perm"][~real] == 0)
    if x is not None:
        xp = out["x_perm"]
        assert np.array_equal(xp[real], np.asarray(x, np.float64)[perm[real] // K])
        assert np.all(xp[~real] == 0)


@pytest.mark.parametrize("T,K,E,align,seed,repeats", [
    (16, 2, 4, 1, 0, False),
    (37, 3, 5, 4, 1, False),
    (64, 8, 16, 16, 2, False),
    (50, 4, 3, 8, 3, True),      # a token may pick the same expert twice
    (5, 2, 12, 16, 4, False),    # more experts than tokens: empty experts
    (1, 1, 1, 128, 5, False),    # a single slot
    (0, 2, 4, 16, 6, False),     # no tokens at all
])
def test_route_matches_brute_force(T, K, E, align, seed, repeats):
    ids, w = synth.random_routing(T, K, E, seed=seed, allow_repeats=repeats)
    x = torch.randn(T, 8, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    out = oracle.route_permute(ids.numpy(), w.numpy(), x.double().numpy(), E, align)
    counts, offsets, perm, inv = brute_force_sort(ids.numpy(), E, align)
    assert out["counts"].tolist() == counts
    assert out["offsets"].tolist() == offsets
    assert out["perm_src"].tolist() == perm
    assert out["inv_perm"].tolist() == inv
    check_invariants(out, ids.numpy(), w.numpy(), x.double().numpy(), E, align)


def test_route_all_tokens_one_expert():
    T, K, E, align = 40, 1, 6, 16
    ids = np.full((T, K), 3, dtype=np.int32)
    w = np.ones((T, K), np.float32)
    out = oracle.route_permute(ids, w, None, E, align)
    assert out["counts"].tolist() == [0, 0, 0, 40, 0, 0]
    assert out["offsets"].tolist() == [0, 0, 0, 0, 48, 48, 48]
    assert out["perm_src"][:40].tolist() == list(range(40))
    assert np.all(out["perm_src"][40:] == -1)


def test_route_tiny_config_invariants():
    inp = synth.make_inputs(synth.TINY)
    s = synth.TINY
    out = oracle.route_permute(inp["topk_ids"].numpy(), inp["topk_w"].numpy(),
                               inp["x"].double().numpy(), s.E, 128)
    check_invariants(out, inp["topk_ids"].numpy(), inp["topk_w"].numpy(),
                     inp["x"].double().numpy(), s.E, 128)


def test_capacity_bounds_every_routing():
    # the padded total never exceeds the capacity, for the worst-case spread too
    for T, K, E, align in [(7, 3, 5, 4), (256, 2, 8, 128), (3, 2, 64, 16)]:
        cap = oracle.capacity(T, K, E, align)
        assert cap % align == 0
        worst = T * K + min(E, T * K) * (align - 1)
        assert cap >= worst


def test_route_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.route_permute(np.array([[0, 9]]), np.ones((1, 2)), None, 4, 16)


def test_planted_unstable_sort_is_caught(monkeypatch):
    """A sort that is not stable inside an expert must fail the brute-force pin."""
    ids, w = synth.random_routing(24, 2, 3, seed=9)
    ref = brute_force_sort(ids.numpy(), 3, 4)
    good = oracle.route_permute(ids.numpy(), w.numpy(), None, 3, 4)
    bad_perm = good["perm_src"].copy()
    seg = slice(int(good["offsets"][0]), int(good["offsets"][0] + good["counts"][0]))
    bad_perm[seg] = bad_perm[seg][::-1]
    assert bad_perm.tolist() != ref[2]
    assert good["perm_src"].tolist() == ref[2]
