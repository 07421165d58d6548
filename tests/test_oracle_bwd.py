"""Pins of the oracle's backward: RoPE backward, then dgrad / wgrad / bgrad.

TransformerEngine PR "Add a backwards linear function to be used with the
fused mla q up-proj": sequence diagram (query gradient -> RoPE backward ->
pre-RoPE gradient -> linear backward with the saved input and the weight ->
input and weight gradients) and the review comment "BF16 bias gradient
remains missing" (the bias gradient is part of that backward). Megatron-LM PR
"Fix fused MLA YaRN RoPE query kernel corrupting upstream tensor in-place",
discussion: the weight gradient is dy^T x with the linear's saved input.

Pins: the adjoint identity of the RoPE pair (any table), inverse of the
rotation for unit tables, library matmuls for dgrad/wgrad, a numpy sum for
bgrad, and central finite differences of L = sum(q * G) for every gradient.
"""
import numpy as np
import torch

import oracle
import synth


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_rope_adjoint_identity_any_table():
    """<RoPE(u), v> == <u, RoPE_bwd(v)> for arbitrary (non-unit, unequal-column) tables."""
    T, H, Dn, Dr = 9, 3, 4, 6
    rng = np.random.default_rng(0)
    cos = rng.standard_normal((12, 8)).astype(np.float32)
    sin = rng.standard_normal((12, 8)).astype(np.float32)
    pos = rng.integers(0, 12, T).astype(np.int32)
    u = _rand((T, H * (Dn + Dr)), 1)
    v = _rand((T, H, Dn + Dr), 2)
    lhs = np.sum(oracle.rope_fwd(u, H, Dn, Dr, cos, sin, pos) * v)
    rhs = np.sum(u.reshape(T, H, -1) * oracle.rope_bwd(v, H, Dn, Dr, cos, sin, pos))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0)


def test_rope_bwd_hand_example():
    """g' = J^T g with a = channel i, c = channel i+1 (Dr = 2, distinct columns)."""
    g = np.array([[[3.0, -2.0]]])
    cos = np.array([[0.5, 0.25]], np.float32)
    sin = np.array([[0.75, 0.125]], np.float32)
    gp = oracle.rope_bwd(g, 1, 0, 2, cos, sin, None)
    # d/da = g0*cos0 + g1*sin1 = 1.5 - 0.25 ; d/dc = -g0*sin0 + g1*cos1 = -2.25 - 0.5
    np.testing.assert_array_equal(gp[0, 0], [1.25, -2.75])


def test_rope_bwd_inverts_forward_for_unit_tables():
    w = synth.workload("tiny")
    for tabs in (synth.rope_table_standard(w.T, w.Dr),
                 synth.rope_table_yarn(w.T, w.Dr, 10000.0, 40.0, 64, 32.0, 1.0, 1.0)):
        cos, sin = (t.numpy() for t in tabs)
        u = _rand((w.T, w.N), 3)
        back = oracle.rope_bwd(oracle.rope_fwd(u, w.H, w.Dn, w.Dr, cos, sin), w.H, w.Dn, w.Dr,
                               cos, sin)
        np.testing.assert_allclose(back.reshape(w.T, -1), u, rtol=0, atol=1e-6)
        assert np.array_equal(back[..., :w.Dn], u.reshape(w.T, w.H, -1)[..., :w.Dn])


def test_dgrad_wgrad_bgrad_match_library():
    T, N, K = 37, 24, 11
    g = _rand((T, N), 4)
    W = _rand((N, K), 5)
    x = _rand((T, K), 6)
    tg, tW, tx = (torch.from_numpy(a) for a in (g, W, x))
    np.testing.assert_allclose(oracle.dgrad(g, W), (tg @ tW).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.wgrad(g, x), (tg.T @ tx).numpy(), rtol=1e-12, atol=1e-12)
    rows = np.array([5, 0, 23])
    np.testing.assert_allclose(oracle.wgrad(g, x, rows), (tg.T @ tx).numpy()[rows], rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(oracle.bgrad(g), g.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_finite_difference_gradients():
    """L(x, W, b) = sum(q * G) is linear in each argument, so central differences are
    exact up to fp64 rounding; the oracle's dx, dW, db must match them."""
    T, K, H, Dn, Dr = 5, 7, 2, 2, 4
    N = H * (Dn + Dr)
    rng = np.random.default_rng(8)
    cos = rng.standard_normal((6, Dr)).astype(np.float32)  # any table: gradient is J^T
    sin = rng.standard_normal((6, Dr)).astype(np.float32)
    pos = np.array([3, 0, 5, 5, 1], np.int32)
    x, W, b = _rand((T, K), 9), _rand((N, K), 10), _rand((N,), 11)
    G = _rand((T, H, Dn + Dr), 12)

    def loss(x_, W_, b_):
        return float(np.sum(oracle.forward(x_, W_, H, Dn, Dr, cos, sin, pos, b_) * G))

    g = oracle.backward(G, x, W, H, Dn, Dr, cos, sin, pos)
    h = 0.5
    for (arr, grad) in ((x, g["dx"]), (W, g["dW"]), (b, g["db"])):
        flat = arr.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(x, W, b)
            flat[i] = old - h
            lm = loss(x, W, b)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad.reshape(-1)[i]) <= 1e-8 * (abs(fd) + 1.0), (arr.shape, i)


def test_backward_uses_saved_input_not_output():
    """wgrad takes the forward's input x (what the linear saves), not q."""
    T, K, H, Dn, Dr = 4, 3, 1, 2, 2
    x, W = _rand((T, K), 13), _rand((H * (Dn + Dr), K), 14)
    cos, sin = (t.numpy() for t in synth.rope_table_standard(T, Dr))
    dq = _rand((T, H, Dn + Dr), 15)
    g = oracle.backward(dq, x, W, H, Dn, Dr, cos, sin)
    np.testing.assert_allclose(g["dW"], g["dq_pre"].T @ x, rtol=1e-12, atol=1e-12)
