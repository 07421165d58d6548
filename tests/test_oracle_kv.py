"""Pins of the oracle's KV side (kv = c_kv W^T split per head; o_key = k_nope
followed by the shared k_pe under rotate-half RoPE, broadcast to every head;
o_value = v). The pages only say the KV path writes fresh o_key and o_value
buffers (Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting
upstream tensor in-place", Solution section); the split and broadcast
follow the MLA attention block.

Pins independent of the oracle's own code: a hand expansion of every output
on a tiny case (quarter-turn table), the identity rotation at position 0,
and the inputs left unchanged.
"""
import math

import numpy as np

import oracle


def test_kv_hand_expansion_quarter_turn():
    # T=2 tokens, K=3, H=2 heads, Dn=1, Dv=1, Dr=2; positions: token 0 -> row 0
    # (angle 0), token 1 -> row 1 (angle pi/2: (a, c) -> (-c, a))
    c_kv = np.array([[1.0, 2.0, 3.0], [-1.0, 0.5, 2.0]])
    W = np.array([[1.0, 0.0, 0.0],    # head 0: nope
                  [0.0, 1.0, 0.0],    # head 0: v
                  [0.0, 0.0, 1.0],    # head 1: nope
                  [1.0, 1.0, 1.0]])   # head 1: v
    k_pe = np.array([[3.0, 4.0], [5.0, 7.0]])
    cos = np.array([[1.0, 1.0], [0.0, 0.0]], np.float32)
    sin = np.array([[0.0, 0.0], [1.0, 1.0]], np.float32)
    o_key, o_value = oracle.kv_forward(c_kv, W, k_pe, 2, 1, 1, 2, cos, sin, np.array([0, 1], np.int32))
    # token 0: nope_h0 = 1, v_h0 = 2, nope_h1 = 3, v_h1 = 6; rope part = (3, 4) unrotated
    assert o_key[0].tolist() == [[1.0, 3.0, 4.0], [3.0, 3.0, 4.0]]
    assert o_value[0].tolist() == [[2.0], [6.0]]
    # token 1: nope_h0 = -1, v_h0 = 0.5, nope_h1 = 2, v_h1 = 1.5; rope part (5, 7) -> (-7, 5)
    assert o_key[1].tolist() == [[-1.0, -7.0, 5.0], [2.0, -7.0, 5.0]]
    assert o_value[1].tolist() == [[0.5], [1.5]]


def test_kv_identity_rotation_and_unchanged_inputs():
    rng = np.random.default_rng(3)
    T, K, H, Dn, Dv, Dr = 5, 16, 3, 8, 4, 8
    c_kv = rng.standard_normal((T, K))
    W = rng.standard_normal((H * (Dn + Dv), K))
    k_pe = rng.standard_normal((T, Dr))
    ang = np.zeros((1, Dr))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    before = (c_kv.copy(), W.copy(), k_pe.copy())
    o_key, o_value = oracle.kv_forward(c_kv, W, k_pe, H, Dn, Dv, Dr, cos, sin, np.zeros(T, np.int32))
    for h in range(H):
        assert np.array_equal(o_key[:, h, Dn:], k_pe)
        rows = W[h * (Dn + Dv):(h + 1) * (Dn + Dv)]
        for t in range(T):
            for c in range(Dn):
                assert math.isclose(o_key[t, h, c], sum(c_kv[t, k] * rows[c, k] for k in range(K)), rel_tol=1e-12,
                                    abs_tol=1e-12)
            for c in range(Dv):
                assert math.isclose(o_value[t, h, c], sum(c_kv[t, k] * rows[Dn + c, k] for k in range(K)),
                                    rel_tol=1e-12, abs_tol=1e-12)
    assert all(np.array_equal(a, b) for a, b in zip(before, (c_kv, W, k_pe)))


def test_kv_rope_pairs_turn_by_their_table_angle():
    """Geometry of rotate-half RoPE on the shared k_pe, with a distinct angle
    per channel pair: each pair (j, j + Dr/2) keeps its length and turns by
    exactly the angle its table row gives, at every position, for every head.
    A wrong pairing (adjacent channels) or a wrong direction fails this."""
    rng = np.random.default_rng(11)
    T, K, H, Dn, Dv, Dr = 6, 8, 3, 4, 4, 8
    half = Dr // 2
    rows = 9
    theta = rng.uniform(-math.pi, math.pi, size=(rows, half))
    cos = np.cos(np.concatenate([theta, theta], axis=1)).astype(np.float32)
    sin = np.sin(np.concatenate([theta, theta], axis=1)).astype(np.float32)
    pos = rng.integers(0, rows, size=T).astype(np.int32)
    k_pe = rng.standard_normal((T, Dr))
    o_key, _ = oracle.kv_forward(rng.standard_normal((T, K)), rng.standard_normal((H * (Dn + Dv), K)), k_pe,
                                 H, Dn, Dv, Dr, cos, sin, pos)
    for t in range(T):
        for h in range(H):
            assert np.array_equal(o_key[t, h, Dn:], o_key[t, 0, Dn:])  # one rope part for all heads
        out = o_key[t, 0, Dn:]
        for j in range(half):
            a_in, b_in = k_pe[t, j], k_pe[t, j + half]
            a_out, b_out = out[j], out[j + half]
            assert math.isclose(math.hypot(a_out, b_out), math.hypot(a_in, b_in), rel_tol=1e-6)
            # the table holds the angle in float32: compare with the angle it encodes
            want = math.atan2(float(sin[pos[t], j]), float(cos[pos[t], j]))
            turn = math.atan2(b_out, a_out) - math.atan2(b_in, a_in)
            d = (turn - want + math.pi) % (2 * math.pi) - math.pi
            assert abs(d) < 1e-6, (t, j, turn, want)
