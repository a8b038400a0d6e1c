"""GPU parity of the expert-MLP forward and backward (through the C ABI) against
the fp64 oracle on the same bf16 inputs.

Small layers are compared element by element in full: they span several 128-row
tiles per expert with ragged expert tails (padding rows), several N tiles, empty
experts, and an expert large enough to be split for the weight gradient.  The
full-size workloads (Qwen3-30B-A3B, Llama-4-Scout and the Zipf-skewed layer) are
run in the launch configuration the benchmark uses and compared on sampled
tokens (Y, dX) and sampled experts (y_perm, dx_perm, dW: the hottest, the
coldest, an empty one when there is one, and a random one).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import MAX_ABS_TOL, REL_FRO_TOL, PerExpert, assert_close, f64, i64
from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import synth
from mixture_experts_expert_gb300.layer import MoEExpertMLP

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()


def random_layer(T, D, I, E, K, seed, ids=None, w_std=0.02):
    """Inputs drawn like the workloads: x, dY ~ N(0,1), weights ~ N(0, 0.02)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, D, I, generator=g) * w_std).to(torch.bfloat16)
    wu = (torch.randn(E, D, I, generator=g) * w_std).to(torch.bfloat16)
    wd = (torch.randn(E, I, D, generator=g) * w_std).to(torch.bfloat16)
    dy = torch.randn(T, D, generator=g).to(torch.bfloat16)
    if ids is None:
        ids, w = synth.random_routing(T, K, E, seed=seed + 1)
    else:
        w = torch.rand(T, K, generator=g) + 0.1
        w = w / w.sum(-1, keepdim=True)
    return dict(x=x, w_gate=wg, w_up=wu, w_down=wd, dy=dy, topk_ids=ids, topk_w=w.float())


def run_gpu(inp, T, D, I, E, K, align=128):
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoEExpertMLP(T, K, E, D, I, align=align, device=DEV)
    y = layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
    dx, dwg, dwu, dwd = layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])
    torch.cuda.synchronize()
    code, raw = layer.device_error()
    assert code == B.MOE_OK, f"device error word {raw}"
    return layer


def check_full(inp, T, D, I, E, K, align=128, grad_unit=1.0):
    """Every output against the oracle.  `grad_unit` (a power of two): the scale dY was
    drawn at; gradients are compared in that unit (both sides divided by it, exactly), so
    the absolute bar means the same at every scale of dY."""
    layer = run_gpu(inp, T, D, I, E, K, align)
    gu = float(grad_unit)
    x, wg, wu, wd, dy, w = (f64(inp[k]) for k in ("x", "w_gate", "w_up", "w_down", "dy", "topk_w"))
    ids = i64(inp["topk_ids"])
    r = oracle.route_permute(ids, w, x, E, align)
    used = int(r["offsets"][-1])
    assert np.array_equal(i64(layer.offsets), r["offsets"])
    # per-call parity: expert MLP forward on the oracle's own sorted rows
    y_perm = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
    assert_close(layer.y_perm[:used], y_perm[:used], "y_perm")
    # padding rows come out exactly zero
    pad = r["perm_src"][:used] < 0
    if pad.any():
        assert np.all(f64(layer.y_perm[:used])[pad] == 0)
    assert_close(layer.y, oracle.moe_forward(x, ids, w, wg, wu, wd), "Y")
    dxp, pg, pu, pd = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"],
                                            r["offsets"], wg, wu, wd, K)
    assert_close(f64(layer.dx_perm[:used]) / gu, dxp[:used] / gu, "dx_perm")
    dX, dWg, dWu, dWd = oracle.moe_backward(x, ids, w, wg, wu, wd, dy)
    assert_close(f64(layer.dx) / gu, dX / gu, "dX")
    assert_close(f64(layer.dw_gate) / gu, dWg / gu, "dW_gate")
    assert_close(f64(layer.dw_up) / gu, dWu / gu, "dW_up")
    assert_close(f64(layer.dw_down) / gu, dWd / gu, "dW_down")
    counts = r["counts"]
    for e in np.nonzero(counts == 0)[0]:
        assert bool((layer.dw_gate[e] == 0).all() and (layer.dw_up[e] == 0).all()
                    and (layer.dw_down[e] == 0).all())
    return layer


def test_tiny_layer():
    s = synth.TINY
    check_full(synth.make_inputs(s), s.T, s.D, s.I, s.E, s.K)


@pytest.mark.parametrize("T,D,I,E,K,seed", [
    (600, 512, 384, 6, 2, 0),     # several M tiles per expert with ragged tails, 3x2 N tiles
    (40, 256, 128, 16, 2, 1),     # most experts empty
    (1, 256, 128, 4, 1, 2),       # a single token
    (300, 768, 256, 3, 3, 3),     # D = 3 x 256, I = 2 x 128
    (200, 256, 128, 1, 1, 4),     # a single expert
    (512, 256, 128, 256, 8, 5),   # many experts with a handful of rows each (mostly padding)
    (64, 256, 128, 1024, 32, 6),  # the largest expert count and top-K
])
def test_small_layers(T, D, I, E, K, seed):
    check_full(random_layer(T, D, I, E, K, seed), T, D, I, E, K)


@pytest.mark.parametrize("align", [256, 384])
def test_coarser_padding(align):
    """Experts padded to 256 or 384 rows: every expert then spans whole row pairs (256)
    or one and a half (384: an odd tile count whose last tile is padding)."""
    T, D, I, E, K = 500, 256, 256, 6, 2
    check_full(random_layer(T, D, I, E, K, seed=14), T, D, I, E, K, align=align)


@pytest.mark.parametrize("I", [256, 384])
def test_tail_tile_sizes(I):
    """Experts whose last row tile has 1, 31, 32, 33, 127, 128 real rows (one tile), 129
    (two tiles), 300, 352, 353 (three) and 513, 640 (five): every odd last tile is computed
    transposed over its real rows rounded up to 32, the rest of it written as zeros.  With
    I = 384 the dA GEMM has 128-column tiles and runs those tiles with an idle CTA half
    instead."""
    counts = [1, 31, 32, 33, 127, 128, 129, 300, 0, 352, 353, 513, 640]
    E, K, D = len(counts), 1, 256
    T = sum(counts)
    ids = torch.cat([torch.full((c, 1), e, dtype=torch.int32) for e, c in enumerate(counts)])
    ids = ids[torch.randperm(T, generator=torch.Generator().manual_seed(3))]
    check_full(random_layer(T, D, I, E, K, seed=12, ids=ids), T, D, I, E, K)


def test_padding_skip_changes_nothing():
    """The GEMMs given the real row counts produce exactly what they produce computing
    every padded row (padding rows of the inputs are zero)."""
    T, D, I, E, K = 700, 512, 256, 6, 2
    g = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=11).items()}
    outs = []
    for skip in (True, False):
        layer = MoEExpertMLP(T, K, E, D, I, align=128, device=DEV, skip_padding=skip)
        layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
        layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])
        torch.cuda.synchronize()
        assert layer.device_error()[0] == B.MOE_OK
        outs.append([t.clone() for t in (layer.y_perm, layer.y, layer.dx_perm, layer.dx,
                                          layer.dw_gate, layer.dw_up, layer.dw_down)])
    used = int(layer.offsets[-1])
    for name, a, b in zip(("y_perm", "y", "dx_perm", "dx", "dW_gate", "dW_up", "dW_down"), *outs):
        if name.endswith("_perm"):
            a, b = a[:used], b[:used]
        assert torch.equal(a, b), name


def test_backward_without_unsorted_x():
    """Without the unsorted x the backward reads its fp16 copy of the sorted rows from
    x_perm: the same values, so the same results bit for bit."""
    T, D, I, E, K = 300, 256, 256, 4, 2
    g = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=13).items()}
    layer = MoEExpertMLP(T, K, E, D, I, align=128, device=DEV)
    layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
    ref = [t.clone() for t in layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])]
    layer._x = None
    out = layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    for a, b in zip(ref, out):
        assert torch.equal(a, b)


def test_layer_without_tokens():
    """T = 0: nothing is routed; Y and dX are empty and every weight gradient is exactly
    zero (every expert is empty)."""
    T, D, I, E, K = 0, 256, 128, 4, 2
    g = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=30).items()}
    layer = MoEExpertMLP(T, K, E, D, I, align=128, device=DEV)
    layer.dw_gate.fill_(1.0)
    layer.dw_up.fill_(1.0)
    layer.dw_down.fill_(1.0)
    y = layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
    dx, dwg, dwu, dwd = layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    assert y.shape == (0, D) and dx.shape == (0, D)
    assert int(layer.offsets[-1]) == 0
    for t in (dwg, dwu, dwd):
        assert bool((t == 0).all())


def test_compensated_expert():
    """One expert holds 7000 rows (more than 4096): its weight gradients take the
    compensated operands (a value pass and a residual pass) and are split into two
    4096-row chunks that are TMA reduce-added."""
    T, D, I, E, K = 7300, 256, 128, 4, 1
    ids = torch.full((T, K), 1, dtype=torch.int32)
    ids[:200, 0] = 0
    ids[200:300, 0] = 3
    check_full(random_layer(T, D, I, E, K, seed=31, ids=ids), T, D, I, E, K)


def test_split_expert_reduce_add():
    """One expert holds 5000 rows (> 4096): its weight gradient is split into two
    token chunks that are TMA reduce-added, with compensation (5000 > 4096); the
    other experts are empty or small."""
    T, D, I, E, K = 5200, 256, 128, 4, 1
    ids = torch.full((T, K), 2, dtype=torch.int32)
    ids[:150, 0] = 0
    ids[150:200, 0] = 3
    check_full(random_layer(T, D, I, E, K, seed=9, ids=ids), T, D, I, E, K)


def _sample_experts(counts, rng):
    nz = np.nonzero(counts)[0]
    picks = {int(np.argmax(counts)), int(nz[np.argmin(counts[nz])]), int(rng.choice(nz))}
    empty = np.nonzero(counts == 0)[0]
    if empty.size:
        picks.add(int(empty[0]))
    return sorted(picks)


def check_sampled(s, dy_scale=1.0):
    """A full-size workload in the benchmark's launch configuration, compared with the
    oracle on sampled tokens (Y, dX) and sampled experts (y_perm, dx_perm, dW).  dY is
    multiplied by `dy_scale` (a power of two, exact in bf16); gradients are compared in
    that unit."""
    inp_dev = synth.make_inputs(s, device=DEV)
    if dy_scale != 1.0:
        inp_dev["dy"] = inp_dev["dy"] * dy_scale
    layer = MoEExpertMLP(s.T, s.K, s.E, s.D, s.I, align=128, device=DEV)
    y = layer.forward(inp_dev["x"], inp_dev["topk_ids"], inp_dev["topk_w"], inp_dev["w_gate"],
                      inp_dev["w_up"], inp_dev["w_down"])
    layer.backward(inp_dev["dy"], inp_dev["w_gate"], inp_dev["w_up"], inp_dev["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK

    x, dy, w = f64(inp_dev["x"]), f64(inp_dev["dy"]), f64(inp_dev["topk_w"])
    ids = i64(inp_dev["topk_ids"])
    wg, wu, wd = (PerExpert(inp_dev[k]) for k in ("w_gate", "w_up", "w_down"))
    rng = np.random.default_rng(0)

    # sampled tokens: Y and dX depend only on their own token
    tok = np.sort(rng.choice(s.T, size=96, replace=False))
    y_ref = oracle.moe_forward(x[tok], ids[tok], w[tok], wg, wu, wd)
    assert_close(f64(y)[tok], y_ref, "Y (sampled tokens)")
    dx_ref = oracle.moe_backward(x[tok], ids[tok], w[tok], wg, wu, wd, dy[tok],
                                 weight_grads=False)[0]
    gu = float(dy_scale)
    assert_close(f64(layer.dx)[tok] / gu, dx_ref / gu, "dX (sampled tokens)")

    # sampled experts: sorted-row outputs and weight gradients
    r = oracle.route_permute(ids, w, x, s.E, 128)
    assert np.array_equal(i64(layer.offsets), r["offsets"])
    experts = _sample_experts(r["counts"], rng)
    yp = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"], experts=experts)
    dxp, dwg, dwu, dwd = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"],
                                               r["offsets"], wg, wu, wd, s.K, experts=experts)
    for e in experts:
        rows = slice(int(r["offsets"][e]), int(r["offsets"][e + 1]))
        if rows.stop > rows.start:
            assert_close(layer.y_perm[rows], yp[rows], f"y_perm[e={e}]")
            assert_close(f64(layer.dx_perm[rows]) / gu, dxp[rows] / gu, f"dx_perm[e={e}]")
        assert_close(f64(layer.dw_gate[e]) / gu, dwg[e] / gu, f"dW_gate[e={e}]")
        assert_close(f64(layer.dw_up[e]) / gu, dwu[e] / gu, f"dW_up[e={e}]")
        assert_close(f64(layer.dw_down[e]) / gu, dwd[e] / gu, f"dW_down[e={e}]")
        if r["counts"][e] == 0:
            assert bool((layer.dw_gate[e] == 0).all() and (layer.dw_down[e] == 0).all())
    return layer


@pytest.mark.parametrize("shape", [synth.QWEN3_30B_A3B, synth.sweep_shape(1024),
                                   synth.sweep_shape(2048), synth.sweep_shape(4096),
                                   synth.sweep_shape(16384), synth.sweep_shape(32768),
                                   synth.sweep_shape(65536), synth.SKEWED, synth.SKEWED_STEEP,
                                   synth.LLAMA4_SCOUT, synth.SCOUT_SKEWED], ids=lambda s: s.name)
def test_full_size_workloads_sampled(shape):
    check_sampled(shape)


def test_qwen3_30b_a3b_full_tensors():
    """The headline workload (Qwen3-30B-A3B shape, T = 8192) in the benchmark's launch
    configuration, compared with the oracle on every element: Y, y_perm, dx_perm, dX and all
    3 x 128 weight-gradient matrices, each as one tensor (relative Frobenius error over the
    whole tensor, max-abs over all its elements).  The oracle runs expert by expert, 16
    experts at a time, to bound host memory."""
    s = synth.QWEN3_30B_A3B
    inp_dev = synth.make_inputs(s, device=DEV)
    layer = MoEExpertMLP(s.T, s.K, s.E, s.D, s.I, align=128, device=DEV)
    y = layer.forward(inp_dev["x"], inp_dev["topk_ids"], inp_dev["topk_w"], inp_dev["w_gate"],
                      inp_dev["w_up"], inp_dev["w_down"])
    layer.backward(inp_dev["dy"], inp_dev["w_gate"], inp_dev["w_up"], inp_dev["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK

    x, dy, w = f64(inp_dev["x"]), f64(inp_dev["dy"]), f64(inp_dev["topk_w"])
    ids = i64(inp_dev["topk_ids"])
    wg, wu, wd = (PerExpert(inp_dev[k]) for k in ("w_gate", "w_up", "w_down"))
    r = oracle.route_permute(ids, w, x, s.E, 128)
    assert np.array_equal(i64(layer.offsets), r["offsets"])
    used = int(r["offsets"][-1])
    y_perm = oracle.expert_mlp_fwd(r["x_perm"], wg, wu, wd, r["offsets"])
    assert_close(layer.y_perm[:used], y_perm[:used], "y_perm")
    assert_close(y, oracle.combine(y_perm, r["inv_perm"], w, s.T, s.K), "Y")
    del y_perm

    dx_perm = np.zeros(r["x_perm"].shape)
    stats = {n: [0.0, 0.0, 0.0] for n in ("dW_gate", "dW_up", "dW_down")}   # err^2, ref^2, max
    for e0 in range(0, s.E, 16):
        batch = list(range(e0, min(s.E, e0 + 16)))
        dxp, dwg, dwu, dwd = oracle.expert_mlp_bwd(dy, r["x_perm"], r["perm_src"], r["w_perm"],
                                                   r["offsets"], wg, wu, wd, s.K, experts=batch)
        for e in batch:
            rows = slice(int(r["offsets"][e]), int(r["offsets"][e + 1]))
            dx_perm[rows] = dxp[rows]
            for name, got, ref in (("dW_gate", layer.dw_gate[e], dwg[e]),
                                   ("dW_up", layer.dw_up[e], dwu[e]),
                                   ("dW_down", layer.dw_down[e], dwd[e])):
                diff = f64(got) - ref
                st = stats[name]
                st[0] += float(np.sum(diff * diff))
                st[1] += float(np.sum(ref * ref))
                st[2] = max(st[2], float(np.max(np.abs(diff))))
    for name, (e2, r2, mx) in stats.items():
        rel = (e2 ** 0.5) / (r2 ** 0.5)
        assert mx <= MAX_ABS_TOL and rel <= REL_FRO_TOL, \
            f"{name}: max abs {mx:.3e}, rel fro {rel:.3e}"
    assert_close(layer.dx_perm[:used], dx_perm[:used], "dx_perm")
    assert_close(layer.dx, oracle.combine(dx_perm, r["inv_perm"], None, s.T, s.K), "dX")


def test_repeated_calls_are_bitwise_stable():
    """Without split experts every output is written by exactly one tile, so two runs
    agree bit for bit."""
    T, D, I, E, K = 600, 512, 384, 6, 2
    inp = random_layer(T, D, I, E, K, seed=4)
    a = run_gpu(inp, T, D, I, E, K)
    outs_a = [t.clone() for t in (a.y, a.dx, a.dw_gate, a.dw_up, a.dw_down)]
    b = run_gpu(inp, T, D, I, E, K)
    for ta, tb in zip(outs_a, (b.y, b.dx, b.dw_gate, b.dw_up, b.dw_down)):
        assert torch.equal(ta, tb)
