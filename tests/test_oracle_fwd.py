"""Pins of the oracle's forward: linear (+bias) then rotate-half RoPE.

Forward of the fused MLA query up-projection (TransformerEngine PR "Add
support for fused Q Up-Proj GEMM/RoPE/Quant", description paragraph: the Q
up-proj GEMM followed by RoPE; Megatron-LM PR "Fix fused MLA YaRN RoPE query
kernel corrupting upstream tensor in-place", Problem section: RoPE applied to
the up-projection's output q, which must not be overwritten).

Pins: a library matmul at the position where RoPE is the identity, hand
expansions on tiny shapes, a hand-computed rotation with distinct table
columns (fixes which column each output reads), norm preservation, untouched
pass-through channels and the rejection of a too-narrow table.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_linear_matches_library_matmul_at_identity_rotation():
    """pos = 0 has cos = 1, sin = 0: q reduces to x W^T + b (torch fp64 matmul)."""
    w = synth.workload("tiny")
    inp = synth.make_inputs(w, seed=0)
    x = oracle.decode_bf16(synth.bf16_bits(inp["x"]))
    W = oracle.decode_bf16(synth.bf16_bits(inp["W"]))
    b = oracle.decode_bf16(synth.bf16_bits(inp["b"]))
    cos, sin = inp["cos"].numpy(), inp["sin"].numpy()
    assert (cos[0] == 1).all() and (sin[0] == 0).all()
    pos = np.zeros(w.T, np.int32)
    q = oracle.forward(x, W, w.H, w.Dn, w.Dr, cos, sin, pos, b)
    ref = (torch.from_numpy(x) @ torch.from_numpy(W).T + torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(q.reshape(w.T, -1), ref, rtol=1e-12, atol=1e-12)


def test_linear_hand_expansion_tiny():
    x = np.array([[1.0, 2.0, -1.0, 0.5, 3.0], [0.0, -2.0, 4.0, 1.0, -1.0], [2.0, 2.0, 2.0, 2.0, 2.0]])
    W = np.array([[1.0, 0.0, 0.0, 0.0, 0.0], [0.5, 0.5, 0.5, 0.5, 0.5], [-1.0, 1.0, -1.0, 1.0, -1.0],
                  [0.0, 0.0, 2.0, 0.0, 0.0]])
    b = np.array([10.0, 0.0, -1.0, 0.25])
    y = oracle.linear(x, W, b)
    # row 0: [1, 0.5*(1+2-1+0.5+3)=2.75, -1+2+1+0.5-3=-0.5, 2*-1=-2] + b
    np.testing.assert_array_equal(y[0], [11.0, 2.75, -1.5, -1.75])
    np.testing.assert_array_equal(y[1], [10.0, 1.0, -5.0, 8.25])  # 0-2-4+1+1-1
    np.testing.assert_array_equal(y[2], [12.0, 5.0, -3.0, 4.25])


def test_rope_quarter_turn_hand_example():
    """Dr = 2 with cos = 0, sin = 1 maps (a, c) to (-c, a)."""
    y = np.array([[7.0, 3.0, -5.0]])  # H = 1, Dn = 1, Dr = 2
    cos = np.zeros((1, 2), np.float32)
    sin = np.ones((1, 2), np.float32)
    q = oracle.rope_fwd(y, 1, 1, 2, cos, sin, np.zeros(1, np.int32))
    np.testing.assert_array_equal(q[0, 0], [7.0, 5.0, 3.0])


def test_rope_distinct_columns_hand_example():
    """Columns i and i+Dr/2 distinct: out[i] = a cos[i] - c sin[i]; out[i+h] = c cos[i+h] + a sin[i+h]."""
    y = np.array([[2.0, -4.0]])  # H = 1, Dn = 0, Dr = 2: a = 2, c = -4
    cos = np.array([[0.5, 0.25]], np.float32)
    sin = np.array([[0.75, 0.125]], np.float32)
    q = oracle.rope_fwd(y, 1, 0, 2, cos, sin, None)
    # a*cos0 - c*sin0 = 1 + 3 = 4 ; c*cos1 + a*sin1 = -1 + 0.25 = -0.75
    np.testing.assert_array_equal(q[0, 0], [4.0, -0.75])


def test_rope_positions_select_rows():
    """Token t reads table row pos[t] (rows differ only in the chosen row)."""
    H, Dn, Dr = 2, 2, 4
    y = _rand((3, H * (Dn + Dr)), 0)
    cos = np.array([[1, 1, 1, 1], [0, 0, 0, 0], [0.5, 0.5, 0.5, 0.5]], np.float32)
    sin = np.array([[0, 0, 0, 0], [1, 1, 1, 1], [0.5, 0.5, 0.5, 0.5]], np.float32)
    q = oracle.rope_fwd(y, H, Dn, Dr, cos, sin, np.array([0, 1, 2], np.int32))
    yr = y.reshape(3, H, Dn + Dr)
    np.testing.assert_array_equal(q[0], yr[0])  # identity row
    a, c = yr[1, :, Dn:Dn + 2], yr[1, :, Dn + 2:]
    np.testing.assert_array_equal(q[1, :, Dn:Dn + 2], -c)
    np.testing.assert_array_equal(q[1, :, Dn + 2:], a)


def test_rope_preserves_pair_norm_and_passthrough():
    w = synth.workload("tiny")
    cos, sin = synth.rope_table_standard(w.T, w.Dr)
    y = _rand((w.T, w.N), 1)
    q = oracle.rope_fwd(y, w.H, w.Dn, w.Dr, cos.numpy(), sin.numpy(), None)
    yr = y.reshape(w.T, w.H, w.D)
    assert np.array_equal(q[..., :w.Dn], yr[..., :w.Dn])  # bit-identical pass-through
    h = w.Dr // 2
    n_in = np.hypot(yr[..., w.Dn:w.Dn + h], yr[..., w.Dn + h:])
    n_out = np.hypot(q[..., w.Dn:w.Dn + h], q[..., w.Dn + h:])
    np.testing.assert_allclose(n_out, n_in, rtol=2e-7)


def test_rope_yarn_table_unit_amplitude():
    cos, sin = synth.rope_table_yarn(4096, 64, 10000.0, 40.0, 4096, 32.0, 1.0, 1.0)
    c, s = cos.double().numpy(), sin.double().numpy()
    np.testing.assert_allclose(c * c + s * s, 1.0, atol=2e-7)
    assert np.array_equal(c[:, :32], c[:, 32:])


def test_rope_rejects_narrow_table():
    """A table narrower than Dr is an error, never an out-of-bounds read."""
    y = _rand((4, 8), 2)
    cos = np.ones((4, 3), np.float32)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.rope_fwd(y, 1, 4, 4, cos, cos, None)
    assert ei.value.status == oracle.ERR_ROPE_WIDTH


def test_rope_rejects_position_out_of_range():
    y = _rand((2, 8), 3)
    cos = np.ones((4, 4), np.float32)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.rope_fwd(y, 1, 4, 4, cos, cos, np.array([0, 4], np.int32))
    assert ei.value.status == oracle.ERR_POS_RANGE


def test_wider_table_uses_leading_columns():
    """cs_width > Dr: row stride is cs_width, channel j reads column j."""
    y = _rand((3, 6), 4)
    rng = np.random.default_rng(5)
    cos = rng.standard_normal((3, 7)).astype(np.float32)
    sin = rng.standard_normal((3, 7)).astype(np.float32)
    q_wide = oracle.rope_fwd(y, 1, 2, 4, cos, sin, None)
    q_narrow = oracle.rope_fwd(y, 1, 2, 4, cos[:, :4].copy(), sin[:, :4].copy(), None)
    np.testing.assert_array_equal(q_wide, q_narrow)


def test_forward_input_not_modified():
    w = synth.workload("tiny", T=16)
    inp = synth.make_inputs(w, seed=1)
    x = oracle.decode_bf16(synth.bf16_bits(inp["x"]))
    W = oracle.decode_bf16(synth.bf16_bits(inp["W"]))
    x0, W0 = x.copy(), W.copy()
    oracle.forward(x, W, w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), None, None,
                   quantize=True)
    assert np.array_equal(x, x0) and np.array_equal(W, W0)


def test_forward_quantized_blocks_per_head():
    """MXFP8 blocks run along each head's channels: ceil(D/32) scales per (t, h)."""
    w = synth.workload("tiny", T=8)
    inp = synth.make_inputs(w, seed=2)
    x = oracle.decode_bf16(synth.bf16_bits(inp["x"]))
    W = oracle.decode_bf16(synth.bf16_bits(inp["W"]))
    q, codes, scales = oracle.forward(x, W, w.H, w.Dn, w.Dr, inp["cos"].numpy(),
                                      inp["sin"].numpy(), None, None, quantize=True)
    assert codes.shape == (8, w.H, w.D) and scales.shape == (8, w.H, math.ceil(w.D / 32))
    # the second block of each head holds only its 16 rope channels
    for t in range(8):
        for h in range(w.H):
            amax = np.abs(q[t, h, 32:]).max()
            assert scales[t, h, 1] == oracle.e8m0_exponent(amax) + 127
