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


def e8m0_exponent_vec(amax):
    """The MXFP8 scale exponent of each block amax (float64 array, >= 0): the
    smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127]. With
    amax = m * 2^k (m in [0.5, 1), numpy.frexp) and 448 = 0.875 * 2^9 this is
    k - 9, or k - 8 when m > 0.875; exact, no logarithm."""
    m, k = np.frexp(np.asarray(amax, np.float64))
    e = k.astype(np.int64) - 9 + (m > 0.875)
    e = np.where(m == 0, -127, e)
    return np.clip(e, -127, 127)


def mxfp8_decided(v, eb):
    """Which rowwise MXFP8 scales and codes of float64 values v [R, C] (blocks
    of 32 along C) are fixed by the quantization rule for every value within
    +-eb [R, C] of v, i.e. whatever rounding a float32 evaluation of v made:
    a block's scale is fixed when the exponents of its smallest and largest
    possible amax agree; an element's code when, on that scale, no rounding
    midpoint of the E4M3 grid lies in its interval and its sign is fixed (an
    exact value, eb = 0, is always decided: ties round to even).
    Returns (scale_fixed [R, nb], code_fixed [R, C], e_lo [R, nb], e_hi [R, nb])."""
    v = np.asarray(v, np.float64)
    eb = np.asarray(eb, np.float64)
    R, C = v.shape
    nb = (C + 31) // 32
    pad = nb * 32 - C
    a = np.pad(np.abs(v), ((0, 0), (0, pad))).reshape(R, nb, 32)
    b = np.pad(eb, ((0, 0), (0, pad))).reshape(R, nb, 32)
    e_lo = e8m0_exponent_vec(np.maximum(a - b, 0.0).max(-1))
    e_hi = e8m0_exponent_vec((a + b).max(-1))
    scale_fixed = e_lo == e_hi
    s = np.repeat(np.exp2(-e_lo.astype(np.float64)), 32, axis=1)[:, :C]
    lut = e4m3_lut()[:127]                     # codes 0x00..0x7E: 0 .. 448, increasing
    mids = (lut[:-1] + lut[1:]) / 2
    lo = (np.abs(v) - eb) * s
    hi = (np.abs(v) + eb) * s
    # an exact value (eb = 0) is decided even on a rounding tie (ties go to even)
    no_mid = (eb == 0) | (np.searchsorted(mids, lo, side="left") == np.searchsorted(mids, hi, side="right"))
    sign_fixed = (np.abs(v) > eb) | (eb == 0)
    code_fixed = no_mid & sign_fixed & np.repeat(scale_fixed, 32, axis=1)[:, :C]
    return scale_fixed, code_fixed, e_lo, e_hi


def check_mxfp8_decided(codes, scales, v, eb, ref_codes, ref_scales, what, min_fixed=0.9):
    """GPU MXFP8 rows (codes [R, C], scales [R, nb], numpy) of values the GPU
    evaluated within +-eb of the float64 v: bit-exact against the oracle's
    quantization of v (ref_codes, ref_scales) wherever the rule fixes the
    result (mxfp8_decided); elsewhere every element within one E4M3 step of
    v on the GPU's own grid. At least `min_fixed` of the elements must be
    fixed (so the bound is not vacuous). Returns the undecided mask."""
    codes, scales = np.asarray(codes), np.asarray(scales)
    R, C = v.shape
    sf, cf, _, _ = mxfp8_decided(v, eb)
    assert cf.mean() >= min_fixed, f"{what}: only {cf.mean():.5f} of the codes are decided"
    assert np.array_equal(scales[sf], ref_scales[sf]), f"{what}: decided scales differ"
    assert np.array_equal(codes[cf], ref_codes[cf]), (
        f"{what}: {(codes[cf] != ref_codes[cf]).sum()} decided codes differ")
    und = ~cf
    if und.any():
        e = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)[:, :C].astype(np.float64)[und]
        deq = e4m3_lut()[codes[und]] * np.exp2(e)
        tol = ulp_e4m3(np.abs(v[und]) * np.exp2(-e)) * np.exp2(e)
        assert (np.abs(deq - v[und]) <= tol).all(), f"{what}: an undecided element is beyond one E4M3 step"
    return und


# ------------------------------------------------------- full-tensor checks
class FrobAcc:
    """The relative Frobenius error of a tensor compared chunk by chunk."""

    def __init__(self):
        self.num = 0.0
        self.den = 0.0

    def add(self, gpu, ref):
        g = bf16_to_f64(gpu).reshape(ref.shape)
        assert not np.isnan(g).any(), "NaN in GPU output"
        self.num += float(np.sum((g - ref) ** 2))
        self.den += float(np.sum(ref * ref))

    def rel(self):
        return float(np.sqrt(self.num) / max(np.sqrt(self.den), 1e-300))


def check_fwd_all_tokens(inp, w, q=None, codes=None, scales=None, x64=None, W64=None, chunk=2048):
    """Every element of a forward output against the oracle, in token chunks
    (tokens are independent in the forward): bf16 q (``q``) with the bf16 bar
    (the rms of the bar taken over each chunk of ``chunk`` tokens, which on
    these homogeneous synthetic inputs equals the whole tensor's to well
    under 1%), and/or MXFP8 q (``codes``, ``scales``: [T, H, D] and
    [T, H, ceil(D/32)]) with the MXFP8 bar. ``x64``, ``W64``: the float64
    operands (default: the decoded bf16 inputs; the MXFP8-weight path passes
    its dequantized operands)."""
    x = f64(inp["x"]) if x64 is None else x64
    W = f64(inp["W"]) if W64 is None else W64
    b = f64(inp["b"]) if inp.get("b") is not None else None
    pos, cos, sin = inp["pos"].numpy(), inp["cos"].numpy(), inp["sin"].numpy()
    q_h = None if q is None else q.cpu()
    c_h = None if codes is None else codes.cpu().numpy()
    s_h = None if scales is None else scales.cpu().numpy()
    for t0 in range(0, w.T, chunk):
        t1 = min(w.T, t0 + chunk)
        if c_h is not None:
            q_ref, rc, rs = oracle.forward(x[t0:t1], W, w.H, w.Dn, w.Dr, cos, sin, pos[t0:t1], b, quantize=True)
            check_mxfp8_close(c_h[t0:t1], s_h[t0:t1], q_ref, rc, rs, what=f"q tokens {t0}:{t1}")
        else:
            q_ref = oracle.forward(x[t0:t1], W, w.H, w.Dn, w.Dr, cos, sin, pos[t0:t1], b)
        if q_h is not None:
            check_bf16_close(q_h[t0:t1], q_ref, what=f"q tokens {t0}:{t1}")


def check_bwd_all(inp, w, dx=None, dW=None, db=None, rope=None, tol=5e-3, tok_chunk=2048, head_chunk=16):
    """Every element of the backward's outputs against the oracle: dx
    (relative Frobenius error over the whole tensor <= tol) and the stored
    rope channels dq_pre_rope [T, H, Dr] (bf16 bar) token chunk by token
    chunk; dW and db (relative Frobenius <= tol) head group by head group
    (a head's rows need only that head's dq, over every token)."""
    pos, cos, sin = inp["pos"].numpy(), inp["cos"].numpy(), inp["sin"].numpy()
    T, H, D, Dn, Dr = w.T, w.H, w.D, w.Dn, w.Dr
    if dx is not None or rope is not None:
        W64 = f64(inp["W"])
        dx_h = None if dx is None else dx.cpu()
        rope_h = None if rope is None else rope.cpu()
        acc = FrobAcc()
        for t0 in range(0, T, tok_chunk):
            t1 = min(T, t0 + tok_chunk)
            dqp = oracle.rope_bwd(f64(inp["dq"][t0:t1]), H, Dn, Dr, cos, sin, pos[t0:t1])
            if rope_h is not None:
                check_bf16_close(rope_h[t0:t1], dqp[:, :, Dn:], what=f"dq_pre_rope tokens {t0}:{t1}")
            if dx_h is not None:
                acc.add(dx_h[t0:t1], oracle.dgrad(dqp.reshape(t1 - t0, -1), W64))
        if dx_h is not None:
            assert acc.rel() <= tol, f"dx: relative Frobenius error {acc.rel():.3e}"
    if dW is not None or db is not None:
        x64 = f64(inp["x"])
        dW_h = None if dW is None else dW.cpu()
        db_h = None if db is None else db.cpu()
        accw, accb = FrobAcc(), FrobAcc()
        for h0 in range(0, H, head_chunk):
            h1 = min(H, h0 + head_chunk)
            dqp = oracle.rope_bwd(f64(inp["dq"][:, h0:h1].contiguous()), h1 - h0, Dn, Dr, cos, sin,
                                  pos).reshape(T, -1)
            rows = slice(h0 * D, h1 * D)
            if dW_h is not None:
                accw.add(dW_h[rows], oracle.wgrad(dqp, x64))
            if db_h is not None:
                accb.add(db_h[rows], oracle.bgrad(dqp))
        if dW_h is not None:
            assert accw.rel() <= tol, f"dW: relative Frobenius error {accw.rel():.3e}"
        if db_h is not None:
            assert accb.rel() <= tol, f"db: relative Frobenius error {accb.rel():.3e}"
