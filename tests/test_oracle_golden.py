"""The oracle still reproduces its stored tiny-layer fingerprint (regression lock)."""
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fingerprint_unchanged():
    import sys
    sys.path.insert(0, os.path.join(HERE, "golden"))
    from make_golden import fingerprint
    with open(os.path.join(HERE, "golden", "tiny_oracle_fingerprint.json")) as fh:
        ref = json.load(fh)
    got = fingerprint()
    assert got["counts"] == ref["counts"] and got["offsets"] == ref["offsets"]
    for k in ("y", "dx", "dw_gate", "dw_up", "dw_down"):
        assert got[k]["sum"] == pytest.approx(ref[k]["sum"], rel=1e-9, abs=1e-12)
        assert got[k]["fro"] == pytest.approx(ref[k]["fro"], rel=1e-12)
