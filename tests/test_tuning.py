"""Per-shape tuning table and override (host logic only: no GPU needed).

The library picks the grouped GEMMs' launch choices per shape from a table compiled in
from ``csrc/tuning_table.inc``: the entry with the same K, E, D, I and the nearest T.
These tests read that file independently and check the library's lookup against it, the
override's validation, and that the tuner's table writer round-trips."""
import os
import re

import pytest

from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld
from mixture_experts_expert_gb300 import tune

TABLE = os.path.join(os.path.dirname(B.PKG_DIR), "mixture_experts_expert_gb300", "csrc",
                     "tuning_table.inc")
ROW = re.compile(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), \{(\d), (\d), (\d), (\d), (\d)\}, "
                 r"(\d), (\d+), (\d+)\},")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Bld.build()
    B.lib()
    yield
    B.moe_tuning_override(None)


def table_rows(text):
    rows = []
    for m in ROW.finditer(text):
        v = [int(g) for g in m.groups()]
        if v[0] == 0:
            continue
        rows.append(((v[0], v[1], v[2], v[3], v[4]),
                     {"order": dict(zip(tune.KIND_OF_GEMM, v[5:10])), "swap_tails": v[10],
                      "da_tile_n": v[11], "dw_chunk_rows": v[12]}))
    return rows


def test_table_file_ends_with_sentinel():
    text = open(TABLE).read()
    last = [l for l in text.splitlines() if l.startswith("{")][-1]
    assert last.startswith("{0, 0, 0, 0, 0,")


def test_unlisted_shape_gets_defaults():
    ch, src = B.moe_tuning_get(4096, 3, 7, 512, 384)
    assert src == "default"
    assert ch == tune.default_choices()


def test_lookup_matches_table_entries():
    rows = table_rows(open(TABLE).read())
    for (T, K, E, D, I), ch in rows:
        got, src = B.moe_tuning_get(T, K, E, D, I)
        assert src == "table" and got == ch, (T, K, E, D, I)


def test_lookup_takes_nearest_token_count():
    rows = table_rows(open(TABLE).read())
    by_shape = {}
    for (T, K, E, D, I), ch in rows:
        by_shape.setdefault((K, E, D, I), []).append((T, ch))
    for (K, E, D, I), entries in by_shape.items():
        for Tq in (1, 3000, 5000, 12000, 100000):
            # nearest by ratio; on a tie the smaller T
            best = min(entries, key=lambda e: (max(Tq / e[0], e[0] / Tq), e[0]))
            got, src = B.moe_tuning_get(Tq, K, E, D, I)
            assert src == "table" and got == best[1], (Tq, K, E, D, I)


def test_override_round_trip_and_clear():
    ch = tune.default_choices()
    ch["order"]["down"] = 1
    ch["order"]["dx"] = 1
    ch["swap_tails"] = 0
    ch["da_tile_n"] = 128
    ch["dw_chunk_rows"] = 512
    B.moe_tuning_override(ch)
    try:
        got, src = B.moe_tuning_get(8192, 8, 128, 2048, 768)
        assert src == "override" and got == ch
        got, src = B.moe_tuning_get(100, 1, 3, 256, 128)   # any shape
        assert src == "override" and got == ch
    finally:
        B.moe_tuning_override(None)
    assert B.moe_tuning_get(100, 1, 3, 256, 128)[1] == "default"


@pytest.mark.parametrize("bad", [
    {"order": {"gate_up": 2}},
    {"swap_tails": 3},
    {"da_tile_n": 192},
    {"dw_chunk_rows": 100},      # not a multiple of 64
    {"dw_chunk_rows": 128},      # below 256
    {"dw_chunk_rows": 131072},   # above 65536
])
def test_override_rejects_out_of_range(bad):
    good = tune.default_choices()
    good["dw_chunk_rows"] = 1024
    B.moe_tuning_override(good)
    try:
        with pytest.raises(B.MoEError):
            B.moe_tuning_override(bad)
        assert B.moe_tuning_get(64, 2, 4, 256, 128) == (good, "override")   # unchanged
    finally:
        B.moe_tuning_override(None)


def test_get_rejects_bad_sizes():
    with pytest.raises(B.MoEError):
        B.moe_tuning_get(-1, 8, 128, 2048, 768)
    with pytest.raises(B.MoEError):
        B.moe_tuning_get(10, 0, 128, 2048, 768)


def test_table_writer_round_trips():
    entries = {(8192, 8, 128, 2048, 768): tune.default_choices(),
               (16384, 1, 16, 5120, 8192): {"order": dict(zip(tune.KIND_OF_GEMM, [1, 0, 1, 1, 0])),
                                            "swap_tails": 0, "da_tile_n": 128,
                                            "dw_chunk_rows": 2048}}
    rows = dict(table_rows(tune.table_text(entries)))
    assert rows == entries
