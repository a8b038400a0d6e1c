"""GPU parity of the routing and data-movement kernels (through the C ABI).

Integer and byte outputs are compared bit for bit with the oracle: counts,
offsets, perm_src, inv_perm, w_perm and x_perm.  The combine is compared with the
oracle's fp64 sum under the floating-point bar.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f64, i64
from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()


def run_route(ids, w, x, T, K, E, D, align):
    cap = B.moe_capacity(T, K, E, align)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts = torch.full((E,), -7, **i32)
    offsets = torch.full((E + 1,), -7, **i32)
    perm_src = torch.full((cap,), -7, **i32)
    inv = torch.full((max(T * K, 1),), -7, **i32)
    w_perm = torch.full((cap,), -7.0, dtype=torch.float32, device=DEV)
    x_perm = torch.full((cap, D), 7.0, dtype=torch.bfloat16, device=DEV) if x is not None else None
    ws = torch.empty(B.moe_workspace_bytes(T, K, E, D, 128, align), dtype=torch.uint8, device=DEV)
    B.moe_workspace_init(ws)
    B.moe_route_permute(ids, w, x, T, K, E, D, align, counts, offsets, perm_src, inv, w_perm,
                        x_perm, ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ws)[0] == B.MOE_OK
    return dict(counts=counts, offsets=offsets, perm_src=perm_src, inv_perm=inv, w_perm=w_perm,
                x_perm=x_perm)


def check_route_exact(ids, w, x, E, align):
    T, K = ids.shape
    D = x.shape[1] if x is not None else 8
    got = run_route(ids.to(DEV), w.to(DEV), x.to(DEV) if x is not None else None, T, K, E, D,
                    align)
    ref = oracle.route_permute(ids.numpy(), w.numpy(), f64(x) if x is not None else None, E,
                               align)
    assert np.array_equal(i64(got["counts"]), ref["counts"])
    assert np.array_equal(i64(got["offsets"]), ref["offsets"])
    assert np.array_equal(i64(got["perm_src"]), ref["perm_src"])
    if T * K:
        assert np.array_equal(i64(got["inv_perm"])[:T * K], ref["inv_perm"])
    # router weights are copied, so they match the fp32 input bit for bit
    assert np.array_equal(got["w_perm"].cpu().numpy(), ref["w_perm"].astype(np.float32))
    if x is not None:
        used = int(ref["offsets"][-1])
        gx = got["x_perm"][:used].cpu()
        rx = torch.from_numpy(ref["x_perm"][:used]).to(torch.bfloat16)
        assert torch.equal(gx.view(torch.int16), rx.view(torch.int16))
    return got, ref


@pytest.mark.parametrize("T,K,E,align,seed,repeats", [
    (16, 2, 4, 1, 0, False),
    (37, 3, 5, 16, 1, False),
    (300, 8, 16, 128, 2, False),
    (50, 4, 3, 8, 3, True),
    (5, 2, 12, 128, 4, False),
    (1, 1, 1, 128, 5, False),
    (1000, 8, 1024, 16, 6, False),   # the largest expert count the kernels accept
    (777, 32, 64, 128, 7, True),     # the largest K
])
def test_route_bit_exact_small(T, K, E, align, seed, repeats):
    ids, w = synth.random_routing(T, K, E, seed=seed, allow_repeats=repeats)
    x = torch.randn(T, 64, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    check_route_exact(ids, w, x, E, align)


def test_route_no_tokens():
    ids = torch.zeros(0, 2, dtype=torch.int32)
    w = torch.zeros(0, 2, dtype=torch.float32)
    got = run_route(None, None, None, 0, 2, 4, 8, 128)
    assert got["counts"].tolist() == [0, 0, 0, 0]
    assert got["offsets"].tolist() == [0] * 5
    assert bool((got["perm_src"] == -1).all())
    del ids, w


def test_route_all_tokens_one_expert():
    T, K, E = 1000, 1, 6
    ids = torch.full((T, K), 5, dtype=torch.int32)
    w = torch.rand(T, K)
    x = torch.randn(T, 32).to(torch.bfloat16)
    check_route_exact(ids, w, x, E, 128)


@pytest.mark.parametrize("shape", [synth.TINY, synth.QWEN3_30B_A3B, synth.SKEWED,
                                   synth.SKEWED_STEEP, synth.LLAMA4_SCOUT],
                         ids=lambda s: s.name)
def test_route_bit_exact_workloads(shape):
    g = torch.Generator().manual_seed(0)
    logits = torch.randn(shape.T, shape.E, generator=g)
    if shape.zipf_s is not None:
        logits += torch.tensor([-shape.zipf_s * np.log(e + 1.0) for e in range(shape.E)])
    ids, w = synth.route_from_logits(logits, shape.K, shape.router)
    x = torch.randn(shape.T, shape.D, generator=g).to(torch.bfloat16)
    got, ref = check_route_exact(ids, w, x, shape.E, 128)
    if shape.zipf_s is not None:
        # the Zipf popularity profile puts more than 10% of all routed slots on one expert
        # and leaves at least one expert without tokens
        counts = ref["counts"]
        assert counts.max() > 0.10 * shape.R and (counts == 0).sum() >= 1


def test_bad_expert_id_is_reported_not_faulted():
    T, K, E = 64, 2, 4
    ids = torch.randint(0, E, (T, K), dtype=torch.int32)
    ids[3, 1] = 9
    ids[10, 0] = -1
    w = torch.rand(T, K)
    cap = B.moe_capacity(T, K, E, 128)
    i32 = dict(dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_workspace_bytes(T, K, E, 64, 128, 128), dtype=torch.uint8, device=DEV)
    B.moe_workspace_init(ws)
    B.moe_route_permute(ids.to(DEV), w.to(DEV), None, T, K, E, 64, 128,
                        torch.empty(E, **i32), torch.empty(E + 1, **i32),
                        torch.empty(cap, **i32), torch.empty(T * K, **i32),
                        torch.empty(cap, dtype=torch.float32, device=DEV), None, ws)
    code, raw = B.moe_get_device_error(ws)
    assert code == B.MOE_ERR_BAD_INDEX
    assert B.moe_get_device_error(ws)[0] == B.MOE_OK   # reading clears the word


@pytest.mark.parametrize("T,K,D,weighted", [(1, 1, 8, True), (257, 8, 2048, True),
                                            (100, 3, 520, False), (64, 32, 256, True),
                                            (8192, 8, 2048, True)])
def test_combine_matches_oracle(T, K, D, weighted):
    g = torch.Generator().manual_seed(T + K)
    rows = T * K + 17
    # expert outputs of the workloads' magnitude (a few tenths)
    src = (0.3 * torch.randn(rows, D, generator=g)).to(torch.bfloat16)
    inv = torch.randperm(rows, generator=g)[:T * K].to(torch.int32)
    w = torch.rand(T, K, generator=g) if weighted else None
    if w is not None:
        w = w / w.sum(-1, keepdim=True)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=DEV)
    B.moe_combine(src.to(DEV), inv.to(DEV), w.to(DEV) if w is not None else None, T, K, D, out)
    ref = oracle.combine(f64(src), i64(inv), None if w is None else w.double().numpy(), T, K)
    assert_close(out, ref, "combine")
    # the only rounding is the final bf16 store: within half an ulp of the fp32 sum
    assert np.all(np.abs(f64(out) - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)


def test_combine_no_tokens():
    B.moe_combine(None, None, None, 0, 2, 64, None)
    torch.cuda.synchronize()
