"""Pins of the oracle's MXFP8 backward and of its float32 inverse rotation.

The pages name the MXFP8 quantization helpers (TransformerEngine PR "Add
support for fused Q Up-Proj GEMM/RoPE/Quant") but give no formula for a
low-precision backward; the oracle takes the plain reading (operands
quantized along their reduction dimension, exact products). Pins: a hand
example of the float32 rotation, its single-rounding order computed through
float64, the fp64 rotation within float32 rounding, lossless quantization on
E4M3-exact inputs, and the whole chain rebuilt from the brute-force block
quantizer of test_oracle_quant and a float64 matmul.
"""
import numpy as np

import oracle
from test_oracle_quant import _all_code_values_torch, _expected_block


def test_rope_bwd_f32_hand_example():
    dq = np.array([[[7.0, 1.0, 2.0]]])                  # T=1, H=1, Dn=1, Dr=2
    cos = np.array([[0.5, 0.5]], np.float32)
    sin = np.array([[0.25, 0.25]], np.float32)
    out = oracle.rope_bwd_f32(dq, 1, 1, 2, cos, sin)
    assert out.dtype == np.float32
    assert out.tolist() == [[[7.0, 1.0 * 0.5 + 2.0 * 0.25, 2.0 * 0.5 - 1.0 * 0.25]]]


def test_rope_bwd_f32_rounding_order():
    rng = np.random.default_rng(0)
    T, H, Dn, Dr = 64, 2, 4, 8
    dq = rng.standard_normal((T, H, Dn + Dr)).astype(np.float32).astype(np.float64)
    ang = rng.uniform(0, 6.3, (T, Dr))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    out = oracle.rope_bwd_f32(dq, H, Dn, Dr, cos, sin)
    h = Dr // 2
    f32 = lambda v: np.float32(v)  # from float64: products of two float32 are exact there
    for t in range(T):
        for hd in range(H):
            for i in range(h):
                a, c = dq[t, hd, Dn + i], dq[t, hd, Dn + h + i]
                p1, p2 = f32(a * float(cos[t, i])), f32(c * float(sin[t, h + i]))
                q1, q2 = f32(c * float(cos[t, h + i])), f32(a * float(sin[t, i]))
                assert out[t, hd, Dn + i] == f32(float(p1) + float(p2))
                assert out[t, hd, Dn + h + i] == f32(float(q1) - float(q2))
    ref = oracle.rope_bwd(dq, H, Dn, Dr, cos, sin)
    assert np.max(np.abs(out - ref)) <= 4 * 2.0 ** -24 * np.max(np.abs(ref)) * 2


def test_backward_mxfp8_lossless_on_e4m3_values():
    """Powers of two up to 2^8 quantize exactly (scale 1 or larger), so the
    MXFP8 products equal the exact float64 products."""
    rng = np.random.default_rng(1)
    T, H, Dn, Dr, K = 64, 1, 32, 32, 64
    pick = lambda shape: rng.choice([-4.0, -1.0, -0.5, 0.0, 0.25, 1.0, 2.0, 8.0], size=shape)
    dq = pick((T, H, Dn + Dr))
    x, W = pick((T, K)), pick((H * (Dn + Dr), K))
    cos = np.ones((T, Dr), np.float32)
    sin = np.zeros((T, Dr), np.float32)
    g = oracle.backward_mxfp8(dq, x, W, H, Dn, Dr, cos, sin)
    dqp = dq.reshape(T, -1)
    assert np.array_equal(g["dx"], dqp @ W)
    assert np.array_equal(g["dW"], dqp.T @ x)
    assert np.array_equal(g["db"], dqp.sum(0))


def test_backward_mxfp8_rebuilt_from_brute_force_blocks():
    rng = np.random.default_rng(2)
    T, H, Dn, Dr, K = 40, 1, 32, 16, 36
    dq = rng.standard_normal((T, H, Dn + Dr)).astype(np.float32).astype(np.float64)
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((H * (Dn + Dr), K)) * 0.02
    ang = rng.uniform(0, 6.3, (T, Dr))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    g = oracle.backward_mxfp8(dq, x, W, H, Dn, Dr, cos, sin)
    table = _all_code_values_torch()

    def deq_blocks(v):  # rows quantized in blocks of 32, dequantized by the brute-force reference
        out = np.zeros_like(v)
        for r in range(v.shape[0]):
            for b0 in range(0, v.shape[1], 32):
                sb, codes = _expected_block(v[r, b0:b0 + 32], table)
                out[r, b0:b0 + len(codes)] = table[np.array(codes)] * 2.0 ** (sb - 127)
        return out

    dqp = oracle.rope_bwd_f32(dq, H, Dn, Dr, cos, sin).reshape(T, -1).astype(np.float64)
    A = deq_blocks(dqp)            # blocks along the channels
    B = deq_blocks(W.T)            # W^T rows = columns of W, blocks along the channels
    assert np.allclose(g["dx"], A @ B.T, rtol=0, atol=1e-12)
    Ac = deq_blocks(dqp.T)         # blocks along the tokens
    Xc = deq_blocks(x.T)
    assert np.allclose(g["dW"], Ac @ Xc.T, rtol=0, atol=1e-12)
