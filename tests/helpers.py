"""Shared helpers of the GPU parity tests: oracle calls on seeded inputs and
the tolerance checks (all written out here, in the tests, not in the library).

Tolerances (fixed by the problem statement of the fused up-projection):
  bf16 q:    |gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref), per element
  MXFP8 q:   >= 99.9% of E8M0 scale bytes identical; every element within one
             E4M3 step of the GPU's own grid: |deq_gpu - q_ref| <=
             ulp_e4m3(|q_ref| 2^-e_gpu) 2^e_gpu; where the scales agree the
             code ordinals differ by at most one
  dx, dW, db: ||gpu - ref||_F / ||ref||_F <= 5e-3
  quantizer: bit-exact
"""
import numpy as np
import torch

import oracle
import synth

_E4M3_LUT = None


def e4m3_lut():
    global _E4M3_LUT
    if _E4M3_LUT is None:
        _E4M3_LUT = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3_LUT


def f64(t_bf16):
    return oracle.decode_bf16(synth.bf16_bits(t_bf16.cpu()))


def bf16_to_f64(t):
    """bf16 CUDA/CPU tensor -> float64 numpy (exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_bf16_close(gpu, ref, what="q"):
    g = bf16_to_f64(gpu).reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol = 8e-3 * np.abs(ref) + 2e-3 * rms
    err = np.abs(g - ref)
    bad = err > tol
    assert not np.isnan(g).any(), f"{what}: NaN in GPU output"
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; "
                           f"worst at {np.unravel_index(np.argmax(err - tol), err.shape)}: "
                           f"gpu {g.reshape(-1)[np.argmax(err - tol)]} ref "
                           f"{ref.reshape(-1)[np.argmax(err - tol)]}")


def ulp_e4m3(u):
    u = np.abs(u)
    return np.where(u < 2.0 ** -6, 2.0 ** -9,
                    np.exp2(np.minimum(np.floor(np.log2(np.maximum(u, 1e-300))), 8.0) - 3))


def check_mxfp8_close(codes, scales, q_ref, ref_codes, ref_scales, what="q"):
    """codes [T, H, D] uint8, scales [T, H, NB] uint8 (numpy, from the GPU)."""
    codes = np.asarray(codes)
    scales = np.asarray(scales)
    T, H, D = q_ref.shape
    same = scales == ref_scales
    frac = same.mean()
    assert frac >= 0.999, f"{what}: only {frac:.5f} of scale bytes identical"
    assert (scales != 0xFF).all(), f"{what}: NaN scale on finite input"
    e = scales.astype(np.int64) - 127
    e_el = np.repeat(e, 32, axis=2)[:, :, :D].astype(np.float64)
    deq = e4m3_lut()[codes] * np.exp2(e_el)
    u = np.abs(q_ref) * np.exp2(-e_el)
    tol = ulp_e4m3(u) * np.exp2(e_el)
    err = np.abs(deq - q_ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond one E4M3 step; first "
                           f"{np.argwhere(bad)[:5].tolist()}")
    same_el = np.repeat(same, 32, axis=2)[:, :, :D]
    ordv = lambda c: np.where(c & 0x80, -(c & 0x7F).astype(np.int64), (c & 0x7F).astype(np.int64))
    d_ord = np.abs(ordv(codes) - ordv(ref_codes))
    assert (d_ord[same_el] <= 1).all(), f"{what}: code ordinals differ by more than one"
    return frac


def frob_rel(gpu, ref):
    g = bf16_to_f64(gpu).reshape(ref.shape)
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))


def oracle_forward(inp, w, tokens=None, quantize=False):
    """Oracle forward on the workload's seeded inputs (optionally a token subset)."""
    x = f64(inp["x"])
    W = f64(inp["W"])
    b = f64(inp["b"]) if inp.get("b") is not None else None
    pos = inp["pos"].numpy()
    if tokens is not None:
        x = x[tokens]
        pos = pos[tokens]
    return oracle.forward(x, W, w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), pos, b,
                          quantize=quantize)


def to_dev(inp, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def sf_tiled_offsets(rows, cols, G):
    """Byte offsets of scale (r, c), r < rows, c < cols, in the block-scaled
    GEMMs' tiled scale order with row groups of G (mla_mxfp8_bwd_layout):
    groups padded to whole 128-row chunks, chunk i of group g and K step kt
    at tile (g * ceil(G/128) + i) * ceil(cols/4) + kt of 512 bytes, inside it
    (rr % 32) * 16 + (rr // 32) * 4 + c % 4."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    c = np.arange(cols, dtype=np.int64)[None, :]
    nsub, nkt = -(-G // 128), -(-cols // 4)
    g, rg = r // G, r % G
    i, rr = rg // 128, rg % 128
    return ((g * nsub + i) * nkt + c // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + c % 4


def sf_untile(buf, rows, cols, G):
    """Row-major [rows, cols] scales read back from the tiled order."""
    buf = np.asarray(buf)
    return buf[sf_tiled_offsets(rows, cols, G)]
