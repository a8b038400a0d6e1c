"""moe_route_permute_noalloc: routing for callers that cannot allocate device memory
(a framework plugin handed only tensor pointers, or an engine whose device memory is
fixed up front).  Its counters live in an array compiled into the library instead of
a caller workspace; its results must equal moe_route_permute's, call after call, since
the array keeps whatever the previous call left in it.

This file is named to be collected last."""
import pytest
import torch

from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()


def outputs(T, K, E, D, align, with_x):
    cap = B.moe_capacity(T, K, E, align)
    i32 = dict(dtype=torch.int32, device=DEV)
    return dict(counts=torch.full((E,), -9, **i32), offsets=torch.full((E + 1,), -9, **i32),
                perm_src=torch.full((cap,), -9, **i32),
                inv_perm=torch.full((max(T * K, 1),), -9, **i32),
                w_perm=torch.full((cap,), -9.0, dtype=torch.float32, device=DEV),
                x_perm=torch.full((cap, D), 9.0, dtype=torch.bfloat16, device=DEV)
                if with_x else None)


def route_both(ids, w, x, E, align, want_ws_error=B.MOE_OK):
    T, K = ids.shape
    D = x.shape[1]
    ref = outputs(T, K, E, D, align, True)
    ws = torch.empty(B.moe_workspace_bytes(T, K, E, D, 128, align), dtype=torch.uint8,
                     device=DEV)
    B.moe_workspace_init(ws)
    B.moe_route_permute(ids, w, x, T, K, E, D, align, ref["counts"], ref["offsets"],
                        ref["perm_src"], ref["inv_perm"], ref["w_perm"], ref["x_perm"], ws)
    assert B.moe_get_device_error(ws)[0] == want_ws_error
    got = outputs(T, K, E, D, align, True)
    B.moe_route_permute_noalloc(ids, w, x, T, K, E, D, align, got["counts"], got["offsets"],
                                got["perm_src"], got["inv_perm"], got["w_perm"], got["x_perm"])
    torch.cuda.synchronize()
    used = int(ref["offsets"][-1])
    for k in ("counts", "offsets", "perm_src", "w_perm"):
        assert torch.equal(got[k], ref[k]), k
    assert torch.equal(got["inv_perm"][:T * K], ref["inv_perm"][:T * K])
    assert torch.equal(got["x_perm"][:used].view(torch.int16),
                       ref["x_perm"][:used].view(torch.int16))


def test_matches_workspace_routing_on_consecutive_calls():
    # two different layers back to back: the second call must not see the first's counters
    s = synth.QWEN3_30B_A3B
    inp = synth.make_inputs(s, device=DEV)
    route_both(inp["topk_ids"], inp["topk_w"], inp["x"], s.E, 128)
    ids, w = synth.random_routing(3000, 4, 37, seed=5, device=DEV)
    x = torch.randn(3000, 256, device=DEV).to(torch.bfloat16)
    route_both(ids, w, x, 37, 16)
    # and the first layer again, after the second one rewrote the array
    route_both(inp["topk_ids"], inp["topk_w"], inp["x"], s.E, 128)


def test_rejects_sizes_beyond_the_fixed_array():
    T, K, E = 9600, 8, 1024          # E * ceil(T*K/256) = 1024 * 300 > 262080
    with pytest.raises(B.MoEError) as ei:
        B.moe_route_permute_noalloc(torch.zeros(T, K, dtype=torch.int32, device=DEV),
                                    torch.zeros(T, K, device=DEV), None, T, K, E, 8, 128,
                                    *[torch.zeros(n, dtype=torch.int32, device=DEV)
                                      for n in (E, E + 1, B.moe_capacity(T, K, E, 128), T * K)],
                                    torch.zeros(B.moe_capacity(T, K, E, 128), device=DEV), None)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED


def test_no_tokens_with_x_given():
    """T = 0 with x given: nothing is routed or gathered; counts and offsets are zero and
    every row is padding, exactly as moe_route_permute leaves them."""
    E, K, D = 6, 2, 256
    x = torch.randn(1, D, device=DEV).to(torch.bfloat16)   # non-NULL, never read
    ids = torch.zeros(0, K, dtype=torch.int32, device=DEV)
    w = torch.zeros(0, K, dtype=torch.float32, device=DEV)
    route_both(ids, w, x, E, 128)


def test_expert_ids_outside_the_range_are_skipped():
    """Slots whose expert id lies outside [0, E) reach no row in either entry point (the
    workspace version also reports them); every other output agrees bit for bit."""
    T, K, E, D = 500, 3, 9, 256
    ids, w = synth.random_routing(T, K, E, seed=11, device=DEV)
    ids[7, 1] = E
    ids[100, 0] = -1
    ids[333, 2] = 1 << 20
    x = torch.randn(T, D, device=DEV).to(torch.bfloat16)
    route_both(ids, w, x, E, 128, want_ws_error=B.MOE_ERR_BAD_INDEX)
