"""Scales of x and dY in the backward (through the C ABI).

The weight-gradient GEMMs read fp16 operands (x, dY and the intermediates w*act, dG, dU,
dA), whose exponent range is far narrower than bf16's: a loss averaged over many tokens
gives gradients near 1e-6, where unscaled fp16 keeps only a few significant bits.  The
backward therefore scales every fp16 operand by a power of two chosen on the GPU from
max|x| and max|dY| and undoes it in fp32 (multiplying by 2^k is exact).  Checks:

* dY scaled by 2^-20, 2^-10 and 2^8 on the tiny layer, on a layer with a compensated
  expert (7000 rows) and on the full Qwen3-30B-A3B workload (sampled): the oracle bar
  holds with the gradients measured in units of 2^k (both sides divided by 2^k, exactly;
  the absolute 3e-2 bar is stated for dY of unit scale), and the gradients are exactly
  2^k times the unscaled ones, bit for bit (the scaling makes the backward equivariant
  under power-of-two scales of dY);
* x scaled down by 2^-12 / 2^-6, and x with a large outlier: the oracle bar holds
  (for the outlier, with errors measured relative to each output's largest magnitude);
* inf in dY, and weights so large that a scaled intermediate overflows fp16, are
  reported as MOE_ERR_FP16_RANGE instead of passing silently.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f64, i64
from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import synth
from mixture_experts_expert_gb300.layer import MoEExpertMLP

from test_gpu_mlp import check_full, check_sampled, random_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALES = [-20, -10, 8]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()


def scaled(inp, key, k):
    out = dict(inp)
    out[key] = (inp[key].float() * 2.0 ** k).to(torch.bfloat16)
    assert torch.equal(out[key].float(), inp[key].float() * 2.0 ** k)   # exact in bf16
    return out


def grads(layer, g, dy):
    layer.backward(dy, g["w_gate"], g["w_up"], g["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    return [t.clone() for t in (layer.dx_perm, layer.dx, layer.dw_gate, layer.dw_up,
                                layer.dw_down)]


def check_equivariant(inp, T, D, I, E, K, ks):
    """One forward, then the backward with dY and with 2^k dY: every gradient of the
    second is 2^k times the first's, bit for bit."""
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoEExpertMLP(T, K, E, D, I, align=128, device=DEV)
    layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
    base = grads(layer, g, g["dy"])
    used = int(layer.offsets[-1])
    for k in ks:
        out = grads(layer, g, (g["dy"].float() * 2.0 ** k).to(torch.bfloat16))
        for name, a, b in zip(("dx_perm", "dx", "dW_gate", "dW_up", "dW_down"), base, out):
            if name == "dx_perm":
                a, b = a[:used], b[:used]
            want = (a.float() * 2.0 ** k).to(a.dtype)
            assert torch.equal(b, want), f"{name} at dY * 2^{k}"


@pytest.mark.parametrize("k", SCALES)
def test_tiny_layer_gradient_scale(k):
    s = synth.TINY
    check_full(scaled(synth.make_inputs(s), "dy", k), s.T, s.D, s.I, s.E, s.K,
               grad_unit=2.0 ** k)


@pytest.mark.parametrize("k", [-20, 8])
def test_compensated_expert_gradient_scale(k):
    T, D, I, E, K = 7300, 256, 128, 4, 1
    ids = torch.full((T, K), 1, dtype=torch.int32)
    ids[:200, 0] = 0
    ids[200:300, 0] = 3
    inp = random_layer(T, D, I, E, K, seed=31, ids=ids)
    check_full(scaled(inp, "dy", k), T, D, I, E, K, grad_unit=2.0 ** k)


def test_qwen3_30b_a3b_gradient_scale_sampled():
    check_sampled(synth.QWEN3_30B_A3B, dy_scale=2.0 ** -20)


def test_backward_is_equivariant_in_dy_scale():
    s = synth.TINY
    check_equivariant(synth.make_inputs(s), s.T, s.D, s.I, s.E, s.K, SCALES)
    # a compensated expert (fp16 residuals) and split dW chunks
    T, D, I, E, K = 7300, 256, 128, 4, 1
    ids = torch.full((T, K), 1, dtype=torch.int32)
    ids[:200, 0] = 0
    check_equivariant(random_layer(T, D, I, E, K, seed=32, ids=ids), T, D, I, E, K, [-20, 8])


@pytest.mark.parametrize("k", [-12, -6])
def test_small_x(k):
    s = synth.TINY
    check_full(scaled(synth.make_inputs(s), "x", k), s.T, s.D, s.I, s.E, s.K)


def test_x_outlier():
    """One x value of 70000 (beyond fp16's 65504: unscaled, the fp16 copy of x could not
    hold it).  Outputs that grow with it are compared relative to their own magnitude."""
    T, D, I, E, K = 600, 512, 384, 6, 2
    inp = random_layer(T, D, I, E, K, seed=24)
    inp["x"][T // 2, 7] = 70000.0
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoEExpertMLP(T, K, E, D, I, align=128, device=DEV)
    layer.forward(g["x"], g["topk_ids"], g["topk_w"], g["w_gate"], g["w_up"], g["w_down"])
    layer.backward(g["dy"], g["w_gate"], g["w_up"], g["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    x, wg, wu, wd, dy, w = (f64(inp[k]) for k in ("x", "w_gate", "w_up", "w_down", "dy", "topk_w"))
    ids = i64(inp["topk_ids"])
    refs = (oracle.moe_forward(x, ids, w, wg, wu, wd),) + tuple(
        oracle.moe_backward(x, ids, w, wg, wu, wd, dy))
    for name, got, ref in zip(("Y", "dX", "dW_gate", "dW_up", "dW_down"),
                              (layer.y, layer.dx, layer.dw_gate, layer.dw_up, layer.dw_down), refs):
        m = max(float(np.abs(ref).max()), 1.0)   # errors relative to the largest magnitude
        assert_close(f64(got) / m, ref / m, f"{name} (relative to {m:.3g})")


def test_nonfinite_dy_is_reported():
    T, D, I, E, K = 600, 512, 384, 6, 2
    t = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=25).items()}
    layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
    layer.forward(t["x"], t["topk_ids"], t["topk_w"], t["w_gate"], t["w_up"], t["w_down"])
    t["dy"][T // 3, 5] = float("inf")
    layer.backward(t["dy"], t["w_gate"], t["w_up"], t["w_down"])
    code, raw = layer.device_error()
    assert code == B.MOE_ERR_FP16_RANGE and raw == 7, raw
    assert layer.device_error()[0] == B.MOE_OK   # reading cleared the word


def test_intermediate_overflow_is_reported():
    """W_down 4096 times larger: dA = w dY W_down^T outgrows the headroom its scale leaves
    (about 2^6 over max|dY|) and overflows fp16; reported, not passed on silently."""
    T, D, I, E, K = 600, 512, 384, 6, 2
    inp = random_layer(T, D, I, E, K, seed=26)
    t = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
    layer.forward(t["x"], t["topk_ids"], t["topk_w"], t["w_gate"], t["w_up"], t["w_down"])
    layer.backward(t["dy"], t["w_gate"], t["w_up"], t["w_down"])
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    big = (t["w_down"].float() * 4096.0).to(torch.bfloat16)
    layer.backward(t["dy"], t["w_gate"], t["w_up"], big)
    code, raw = layer.device_error()
    assert code == B.MOE_ERR_FP16_RANGE and raw == 7, raw
