"""GPU parity of the layer under every per-shape launch choice (moe_tuning_override),
against the fp64 oracle, element by element.  The tile order changes no arithmetic, so
its outputs must also equal the default order's bit for bit."""
import pytest
import torch

from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import tune
from test_gpu_mlp import check_full, random_layer, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()
    yield
    B.moe_tuning_override(None)

# Experts of 1-5 row pairs with ragged (odd) last tiles, one expert large enough to be
# split for dW at a 512-row chunk, and an empty expert.
COUNTS = [700, 130, 1100, 257, 0, 520, 383]
D, I, K = 512, 256, 1


def skewed_ids(seed=5):
    E = len(COUNTS)
    T = sum(COUNTS)
    ids = torch.cat([torch.full((c, 1), e, dtype=torch.int32) for e, c in enumerate(COUNTS)])
    return ids[torch.randperm(T, generator=torch.Generator().manual_seed(seed))], T, E


def with_choices(ch, fn):
    B.moe_tuning_override(ch)
    try:
        return fn()
    finally:
        B.moe_tuning_override(None)


def choices(**kw):
    ch = tune.default_choices()
    for k, v in kw.items():
        if k == "order":
            ch["order"] = {g: v for g in tune.KIND_OF_GEMM}
        else:
            ch[k] = v
    return ch


@pytest.mark.parametrize("ch", [
    choices(order=1),
    choices(swap_tails=0),
    choices(da_tile_n=128),
    choices(dw_chunk_rows=512),                 # three experts split, compensated operands
    choices(order=1, swap_tails=0, da_tile_n=128, dw_chunk_rows=256),
], ids=["order1", "noswap", "da128", "chunk512", "all"])
def test_choices_match_oracle(ch):
    ids, T, E = skewed_ids()
    inp = random_layer(T, D, I, E, K, seed=21, ids=ids)
    with_choices(ch, lambda: check_full(inp, T, D, I, E, K))


def test_compensated_expert_unsplit():
    """A 7000-row expert with 16384-row chunks: compensated operands in one chunk (no
    reduce-add)."""
    T, D, I, E, K = 7300, 256, 128, 3, 1
    ids = torch.full((T, K), 2, dtype=torch.int32)
    ids[:300, 0] = 0
    inp = random_layer(T, D, I, E, K, seed=23, ids=ids)
    with_choices(choices(dw_chunk_rows=16384), lambda: check_full(inp, T, D, I, E, K))


def test_tile_order_changes_no_bit():
    ids, T, E = skewed_ids(seed=6)
    inp = random_layer(T, D, I, E, K, seed=22, ids=ids)
    outs = []
    for order in (0, 1):
        layer = with_choices(choices(order=order), lambda: run_gpu(inp, T, D, I, E, K))
        used = int(layer.offsets[-1])   # rows past the last expert are never written
        outs.append([t.clone() for t in (layer.y_perm[:used], layer.y, layer.dx_perm[:used],
                                         layer.dx, layer.dw_gate, layer.dw_up,
                                         layer.dw_down)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_tuner_runs_on_the_tiny_layer(capsys, tmp_path):
    """The tuner measures every choice on a workload and prints a table the library can
    compile (it leaves no override behind)."""
    out = tmp_path / "t.json"
    tune.main(["--workloads", "tiny", "--steps", "2", "--warmup", "1", "--reps", "1",
               "--json", str(out)])
    text = capsys.readouterr().out
    assert "{256, 2, 8, 256, 128, {" in text and text.rstrip().endswith("1, 256, 4096},")
    assert B.moe_tuning_get(256, 2, 8, 256, 128)[1] != "override"
    assert out.exists()
