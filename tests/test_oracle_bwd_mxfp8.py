"""Pins of the oracle's MXFP8 backward.

The pages name the MXFP8 quantization helpers (TransformerEngine PR "Add
support for fused Q Up-Proj GEMM/RoPE/Quant") but give no formula for a
low-precision backward; the oracle takes the plain reading: the exact RoPE
backward, operands quantized along their reduction dimension, exact
products. Pins: lossless quantization on E4M3-exact inputs, the whole chain
rebuilt from the brute-force block quantizer of test_oracle_quant and a
float64 matmul (which catches a block along the wrong axis or a transposed
operand), and the quantization error bound against the unquantized
gradients.
"""
import numpy as np

import oracle
from test_oracle_quant import _all_code_values_torch, _expected_block


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

    # the rotation: the pinned fp64 RoPE backward (test_oracle_bwd), not this chain's own
    dqp = oracle.rope_bwd(dq, H, Dn, Dr, cos, sin).reshape(T, -1)
    assert np.array_equal(g["dq_pre"], dqp)
    A = deq_blocks(dqp)            # blocks along the channels
    B = deq_blocks(W.T)            # W^T rows = columns of W, blocks along the channels
    assert np.allclose(g["dx"], A @ B.T, rtol=0, atol=1e-12)
    Ac = deq_blocks(dqp.T)         # blocks along the tokens
    Xc = deq_blocks(x.T)
    assert np.allclose(g["dW"], Ac @ Xc.T, rtol=0, atol=1e-12)


def test_backward_mxfp8_within_the_quantization_bound():
    """Against the unquantized fp64 gradients: each operand element moves by
    at most half an E4M3 step, |q - v| <= 2^-4 |v| + 2^-10 2^e (normal
    relative half-step, plus the subnormal step of the block), so each
    product term by at most ((1 + 2^-4)^2 - 1) |a b| plus the subnormal
    terms; summed, that bounds |dx_mx - dx| and |dW_mx - dW|."""
    rng = np.random.default_rng(3)
    T, H, Dn, Dr, K = 96, 2, 32, 32, 64
    dq = rng.standard_normal((T, H, Dn + Dr))
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((H * (Dn + Dr), K)) * 0.02
    ang = rng.uniform(0, 6.3, (T, Dr))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    g = oracle.backward_mxfp8(dq, x, W, H, Dn, Dr, cos, sin)
    ex = oracle.backward(dq, x, W, H, Dn, Dr, cos, sin)

    def half_step(v, axis):  # bound on |quantized - v| with blocks of 32 along `axis`
        a = np.moveaxis(np.abs(v), axis, -1)
        n = a.shape[-1]
        pad = (-n) % 32
        blk = np.pad(a, [(0, 0)] * (a.ndim - 1) + [(0, pad)]).reshape(a.shape[:-1] + (-1, 32))
        e = np.ceil(np.log2(np.maximum(blk.max(-1), 1e-300) / 448.0))
        sub = np.repeat(2.0 ** (e - 10), 32, axis=-1)[..., :n]
        return np.moveaxis(2.0 ** -4 * a + sub, -1, axis)

    A, B = ex["dq_pre"], W
    dA, dB = half_step(A, 1), half_step(B, 0)
    bound_dx = np.abs(A) @ dB + dA @ np.abs(B) + dA @ dB
    assert (np.abs(g["dx"] - ex["dx"]) <= bound_dx * (1 + 1e-9)).all()
    dAt, dX = half_step(A, 0), half_step(x, 0)
    bound_dw = np.abs(A).T @ dX + dAt.T @ np.abs(x) + dAt.T @ dX
    assert (np.abs(g["dW"] - ex["dW"]) <= bound_dw * (1 + 1e-9)).all()
    assert np.allclose(g["db"], ex["db"], rtol=0, atol=0)
