"""The oracle still reproduces its committed regression snapshot."""
import importlib.util
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_snapshot_unchanged():
    spec = importlib.util.spec_from_file_location(
        "make_oracle_snapshot", os.path.join(HERE, "golden", "make_oracle_snapshot.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(HERE, "golden", "tiny_oracle_snapshot.json")) as f:
        ref = json.load(f)
    now = mod.snapshot()
    np.testing.assert_allclose(now["q"], ref["q"], rtol=1e-14, atol=0)
    assert now["codes"] == ref["codes"] and now["scales"] == ref["scales"]
