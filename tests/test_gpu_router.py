"""GPU parity of the router step (through the C ABI) against the fp64 router oracle:
expert ids bit for bit (the choice is made on the fp32 logits, equal logits -> lower
index), weights and gradients within the floating-point bar."""
import numpy as np
import pytest
import torch

import oracle
from helpers import PerExpert, assert_close, f64, i64
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


def run_topk(z, K, router):
    T, E = z.shape
    zd = torch.as_tensor(z, dtype=torch.float32, device=DEV)
    ids = torch.empty(T, K, dtype=torch.int32, device=DEV)
    w = torch.empty(T, K, dtype=torch.float32, device=DEV)
    B.moe_router_topk(zd, T, E, K, router, ids, w)
    return zd, ids, w


def check_topk_and_backward(z, K, router, seed=0):
    T, E = z.shape
    zd, ids, w = run_topk(z, K, router)
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.router_topk(z, K, router)
    assert np.array_equal(i64(ids), ids_ref)
    assert_close(w, w_ref, "topk_w")
    assert np.max(np.abs(f64(w) - w_ref)) < 1e-5          # fp32 arithmetic, far inside the bar
    dw = torch.randn(T, K, generator=torch.Generator().manual_seed(seed)).to(DEV)
    dz = torch.empty(T, E, dtype=torch.float32, device=DEV)
    B.moe_router_backward(ids, w, dw, T, E, K, router, dz)
    torch.cuda.synchronize()
    dz_ref = oracle.router_backward(z, ids_ref, f64(dw), router)
    assert_close(dz, dz_ref, "d_logits")
    assert np.max(np.abs(f64(dz) - dz_ref)) < 1e-5


@pytest.mark.parametrize("T,E,K,router", [
    (300, 128, 8, "softmax"),     # the Qwen3-30B-A3B router shape
    (77, 40, 5, "softmax"),       # E not a multiple of 32
    (64, 1024, 32, "softmax"),    # the largest E and K
    (50, 6, 6, "softmax"),        # every expert chosen: the plain softmax
    (200, 16, 1, "sigmoid_top1"), # the Llama-4-Scout router
])
def test_router_random_logits(T, E, K, router):
    z = np.random.default_rng(T + E + K).standard_normal((T, E)).astype(np.float32)
    check_topk_and_backward(z, K, router)


def test_router_ties_and_extremes():
    z = np.zeros((6, 40), np.float32)
    z[1, [3, 35]] = 1.5                        # equal maxima in different lanes
    z[2, ::3] = 2.0                            # many equal values
    z[3] = -np.inf
    z[3, [7, 9]] = 0.0                         # -inf logits are never chosen ahead of finite ones
    z[4] = np.linspace(-60.0, 60.0, 40)        # exp range edges
    z[5, 39] = 80.0
    check_topk_and_backward(z, 4, "softmax")
    check_topk_and_backward(z[:, :16].copy(), 1, "sigmoid_top1")


def test_router_empty_batch():
    zd, ids, w = run_topk(np.zeros((0, 8), np.float32), 2, "softmax")
    torch.cuda.synchronize()
    assert ids.numel() == 0 and w.numel() == 0


def test_router_on_the_qwen_workload_logits():
    s = synth.QWEN3_30B_A3B
    z = synth.make_inputs(s)["logits"].numpy()
    zd, ids, w = run_topk(z, s.K, "softmax")
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.router_topk(z, s.K, "softmax")
    assert np.array_equal(i64(ids), ids_ref)
    assert_close(w, w_ref, "topk_w (Qwen logits)")


@pytest.mark.parametrize("T,D,I,E,K", [(300, 256, 128, 6, 2), (64, 512, 256, 16, 8)])
def test_router_weight_gradient(T, D, I, E, K):
    g = torch.Generator().manual_seed(T + K)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    wg, wu, wd = ((torch.randn(*sh, generator=g) * 0.02).to(torch.bfloat16)
                  for sh in ((E, D, I), (E, D, I), (E, I, D)))
    dy = torch.randn(T, D, generator=g).to(torch.bfloat16)
    z = torch.randn(T, E, generator=g)
    ids_ref, w_ref = oracle.router_topk(z.numpy(), K, "softmax")
    ids = torch.as_tensor(ids_ref, dtype=torch.int32)
    w = torch.as_tensor(w_ref, dtype=torch.float32)
    layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
    dev = {k: v.to(DEV) for k, v in dict(x=x, wg=wg, wu=wu, wd=wd, dy=dy, ids=ids, w=w).items()}
    layer.forward(dev["x"], dev["ids"], dev["w"], dev["wg"], dev["wu"], dev["wd"])
    dw = torch.empty(T, K, dtype=torch.float32, device=DEV)
    B.moe_router_weight_grad(dev["dy"], layer.y_perm, layer.inv_perm, T, K, D, dw)
    torch.cuda.synchronize()
    ref = oracle.router_weight_grad(f64(x), ids_ref, PerExpert(wg), PerExpert(wu), PerExpert(wd),
                                    f64(dy))
    assert_close(dw, ref, "d_topk_w")
