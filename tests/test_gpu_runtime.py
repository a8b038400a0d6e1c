"""Runtime properties of the CUDA path (through the C ABI):

* a forward + backward captured once in a CUDA graph and replayed with new inputs and a
  new routing reproduces eager execution bit for bit (launch shapes depend only on the
  sizes, never on the routing);
* a grouped GEMM whose waits run out reports MOE_ERR_DEVICE_TIMEOUT through the device
  error word instead of hanging, and the context stays usable afterwards;
* the backward's in-call dX reduction equals a separate moe_combine, and two layers
  driven from two host threads on two streams at once give what each gives alone.
(Values outside the range of the backward's scaled fp16 operands: test_gpu_scales.py.)
"""
import pytest
import torch

from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300.layer import MoEExpertMLP

from test_gpu_mlp import random_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHAPE = dict(T=600, D=512, I=384, E=6, K=2)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()


def step(layer, t):
    layer.forward(t["x"], t["topk_ids"], t["topk_w"], t["w_gate"], t["w_up"], t["w_down"])
    layer.backward(t["dy"], t["w_gate"], t["w_up"], t["w_down"])


def outputs(layer):
    return [o.clone() for o in (layer.y, layer.dx, layer.dw_gate, layer.dw_up, layer.dw_down)]


def test_cuda_graph_replay_matches_eager():
    T, D, I, E, K = (SHAPE[k] for k in ("T", "D", "I", "E", "K"))
    first = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=21).items()}
    second = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=22).items()}
    assert not torch.equal(first["topk_ids"], second["topk_ids"])

    eager = MoEExpertMLP(T, K, E, D, I, device=DEV)
    step(eager, second)
    torch.cuda.synchronize()
    want = outputs(eager)

    layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
    static = {k: v.clone() for k, v in first.items()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(layer, static)          # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(layer, static)
    for k in static:
        static[k].copy_(second[k])
    graph.replay()
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    for got, ref in zip(outputs(layer), want):
        assert torch.equal(got, ref)


def test_expired_wait_reports_timeout_and_context_survives():
    T, D, I, E, K = (SHAPE[k] for k in ("T", "D", "I", "E", "K"))
    t = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=23).items()}
    layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
    B.moe_debug_drop_next_loads()
    layer.forward(t["x"], t["topk_ids"], t["topk_w"], t["w_gate"], t["w_up"], t["w_down"])
    code, raw = layer.device_error()          # waits for the kernel (about one second)
    assert code == B.MOE_ERR_DEVICE_TIMEOUT and raw in (3, 4), raw
    assert layer.device_error()[0] == B.MOE_OK  # reading cleared the word
    # the same context still runs the layer correctly
    step(layer, t)
    torch.cuda.synchronize()
    assert layer.device_error()[0] == B.MOE_OK
    ref = MoEExpertMLP(T, K, E, D, I, device=DEV)
    step(ref, t)
    torch.cuda.synchronize()
    for got, want in zip(outputs(layer), outputs(ref)):
        assert torch.equal(got, want)


def test_reduction_inside_backward_matches_separate_combine():
    """moe_expert_mlp_bwd reducing dx_perm to tokens itself (on its side stream, beside the
    weight-gradient GEMMs) gives exactly what a separate moe_combine call gives."""
    T, D, I, E, K = (SHAPE[k] for k in ("T", "D", "I", "E", "K"))
    t = {k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=27).items()}
    runs = []
    for fused in (True, False):
        layer = MoEExpertMLP(T, K, E, D, I, device=DEV, reduce_in_backward=fused)
        step(layer, t)
        torch.cuda.synchronize()
        assert layer.device_error()[0] == B.MOE_OK
        runs.append(outputs(layer))
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_concurrent_layers_on_two_streams_and_threads():
    """Two host threads drive two layers on two CUDA streams at once, each backward
    forking the library's side stream for its dX reduction: every result equals the same
    layer run alone, bit for bit (the side stream is shared, its use serialised per call,
    and each call joins it back into its own stream)."""
    import threading

    T, D, I, E, K = (SHAPE[k] for k in ("T", "D", "I", "E", "K"))
    inputs = [{k: v.to(DEV) for k, v in random_layer(T, D, I, E, K, seed=s).items()}
              for s in (28, 29)]
    want = []
    for t in inputs:
        layer = MoEExpertMLP(T, K, E, D, I, device=DEV)
        step(layer, t)
        torch.cuda.synchronize()
        want.append(outputs(layer))

    layers = [MoEExpertMLP(T, K, E, D, I, device=DEV) for _ in inputs]
    streams = [torch.cuda.Stream() for _ in inputs]
    errors = []

    def run(i):
        try:
            with torch.cuda.stream(streams[i]):
                for _ in range(5):
                    step(layers[i], inputs[i])
            streams[i].synchronize()
        except Exception as e:   # reported below, on the main thread
            errors.append(e)

    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(inputs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for layer, ref in zip(layers, want):
        assert layer.device_error()[0] == B.MOE_OK
        for got, exp in zip(outputs(layer), ref):
            assert torch.equal(got, exp)
