"""The seeded input generators: deterministic, right shapes, right spreads."""
import numpy as np
import torch

import synth


def test_inputs_deterministic_and_shaped():
    w = synth.workload("tiny")
    a = synth.make_inputs(w, seed=0)
    b = synth.make_inputs(w, seed=0)
    for k in ("x", "W", "b", "dq", "cos", "sin", "pos"):
        assert torch.equal(a[k], b[k]), k
    assert a["x"].shape == (w.T, w.K) and a["x"].dtype == torch.bfloat16
    assert a["W"].shape == (w.N, w.K) and a["dq"].shape == (w.T, w.H, w.D)
    assert a["cos"].shape == (w.cs_rows, w.Dr) and a["cos"].dtype == torch.float32
    assert torch.equal(a["pos"], torch.arange(w.T, dtype=torch.int32))
    c = synth.make_inputs(w, seed=1)
    assert not torch.equal(a["x"], c["x"])


def test_spreads_and_outliers():
    x = synth.normal_bf16((512, 1536), 1.0, 5, outlier_frac=0.01, outlier_mult=50.0).float()
    big = (x.abs() > 8).float().mean().item()
    assert 0.005 < big < 0.015
    W = synth.normal_bf16((1024, 256), 0.02, 6).float()
    assert abs(W.std().item() - 0.02) < 0.001


def test_positions_restart_per_sequence():
    p = synth.positions(8192, 4096)
    assert p[4095] == 4095 and p[4096] == 0 and p.dtype == torch.int32


def test_yarn_ramp_bounds():
    cos, sin = synth.rope_table_yarn(4096, 64)
    ang = np.arctan2(sin[1].double().numpy(), cos[1].double().numpy())  # angle at pos 1 = freq
    inv = 10000.0 ** (-2.0 * np.arange(32) / 64)
    np.testing.assert_allclose(ang[:10], inv[:10], rtol=1e-6)        # below low: unchanged
    np.testing.assert_allclose(ang[24:32], inv[24:32] / 40.0, rtol=1e-5)  # above high: / factor
