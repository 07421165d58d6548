"""Pins of the oracle's MXFP8 quantizer (E4M3 elements, E8M0 block scales).

The rule pinned here: scale exponent e = the smallest integer with
amax <= 448 * 2^e (= ceil(log2(amax/448))), clamped to [-127, 127], stored as
the byte e + 127; elements encoded as round-to-nearest-even E4M3 (OCP "FN":
max 448, no infinity) of v * 2^-e with saturation. It is the MXFP8 output of
the fused up-projection (TransformerEngine PR "Add support for fused Q
Up-Proj GEMM/RoPE/Quant", description paragraph) and the standalone
quantization helper of the same PR (Greptile summary: "two-phase MXFP8
quantization" helpers).

Pins are independent of the oracle's own code: torch's float8_e4m3fn
conversion (a library routine), an exhaustive nearest-value search over the
256 codes, hand-derived closed forms and the rounding error bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _all_code_values_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_all_codes_match_torch():
    ref = _all_code_values_torch()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert (nan_ref == nan_got).all()
    assert nan_got.sum() == 2  # 0x7F and 0xFF only (no infinity in E4M3 "FN")
    assert np.array_equal(ref[~nan_ref], got[~nan_got])
    # sign of zero
    assert math.copysign(1.0, got[0x80]) == -1.0


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x3C, 1.5), (0x70, 2.0 ** 7), (0x78, 2.0 ** 8), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_decode_closed_form(code, value):
    # sign bit, exponent field (bias 7), 3 mantissa bits; field 0 = subnormal m * 2^-9
    assert oracle.e4m3_decode(code) == value


def test_decode_bf16_every_pattern_matches_torch():
    """All 65 536 bf16 bit patterns decode to torch's own bf16 -> float64
    conversion (a library routine): same value, same sign of zero, NaN
    exactly where torch gives NaN. Every oracle test feeds its inputs through
    this decode, so it is pinned on its own."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert np.array_equal(nan_ref, nan_got)
    assert nan_got.sum() == 2 * 127  # exponent field 255, mantissa != 0, both signs
    assert np.array_equal(got[~nan_got], ref[~nan_ref])
    assert np.array_equal(np.signbit(got[~nan_got]), np.signbit(ref[~nan_ref]))
    # closed forms: 1.0, -2.0, the smallest subnormal, the largest finite, infinity
    for b, v in ((0x3F80, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -133),
                 (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127), (0x7F80, np.inf), (0x8000, -0.0)):
        assert oracle.decode_bf16(np.array([b], np.uint16))[0] == v
        assert math.copysign(1.0, oracle.decode_bf16(np.array([b], np.uint16))[0]) == math.copysign(1.0, v)


def test_encode_every_bf16_matches_torch_rne():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode_bf16(bits)
    finite = np.isfinite(vals) & (np.abs(vals) < 464.0)  # torch maps >= 464 to NaN
    v = vals[finite]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_encode_bruteforce_nearest_ties_even():
    """Nearest of the finite codes by exhaustive search, ties to the even code."""
    rng = np.random.default_rng(1234)
    table = _all_code_values_torch()
    pos_codes = np.array([c for c in range(0x7F)])  # 0x00..0x7E: non-negative finite
    pos_vals = table[pos_codes]
    # random magnitudes over the whole range, plus every exact midpoint between codes
    mids = (pos_vals[:-1] + pos_vals[1:]) / 2.0
    rnd = np.concatenate([rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-12, 8.8, 20000)), mids])
    rnd = rnd[rnd <= 448.0]
    for a in rnd:
        d = np.abs(pos_vals - a)
        best = np.flatnonzero(d == d.min())
        if best.size == 2:  # a tie: pick the even code
            best = best[(pos_codes[best] & 1) == 0]
        exp_code = int(pos_codes[best[0]])
        assert oracle.e4m3_encode(a) == exp_code, a
        assert oracle.e4m3_encode(-a) == (exp_code | 0x80), -a


def test_encode_saturates_and_nan():
    for v in [448.0, 449.0, 463.9, 464.0, 500.0, 1e30, float("inf")]:
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00  # below half the smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # exact tie with 0 -> even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie 1.5 steps -> 2 (even)


@pytest.mark.parametrize("e", [-127, -126, -20, -8, -1, 0, 1, 7, 60, 119])
def test_scale_exponent_edges(e):
    edge = math.ldexp(448.0, e)
    assert oracle.e8m0_exponent(edge) == e  # exactly 448*2^e -> e, not e+1
    if e < 127:
        assert oracle.e8m0_exponent(np.nextafter(edge, np.inf)) == e + 1
    if e > -127:
        assert oracle.e8m0_exponent(np.nextafter(edge, 0.0)) == e
        assert oracle.e8m0_exponent(math.ldexp(448.0, e - 1)) == e - 1


def test_scale_exponent_matches_ceil_log2():
    rng = np.random.default_rng(7)
    for a in np.exp2(rng.uniform(-100, 100, 5000)):
        # away from exact powers of two the float log is safe to compare against
        e_ref = math.ceil(math.log2(a / 448.0))
        if abs(math.log2(a / 448.0) - round(math.log2(a / 448.0))) > 1e-9:
            assert oracle.e8m0_exponent(a) == max(-127, min(127, e_ref))


def test_scale_exponent_zero_and_tiny():
    assert oracle.e8m0_exponent(0.0) == -127
    assert oracle.e8m0_exponent(1e-45) == -127
    assert oracle.e8m0_exponent(math.ldexp(448.0, -130)) == -127


def test_block_hand_example():
    # amax 2 -> e = -7 (448/128 = 3.5 >= 2 > 448/256); byte 120
    # 1.0 * 2^7 = 128 = 2^7 -> 0x70; -2 * 2^7 = -256 -> 0xF8; 0.5 * 2^7 = 64 -> 0x68;
    # 0.1 * 128 = 12.8 -> step 1 in [8,16) -> 13 = 1.625 * 8 -> exp field 10, m 5 -> 0x55
    blk = np.zeros((1, 32))
    blk[0, :4] = [1.0, -2.0, 0.5, 0.1]
    codes, scales = oracle.mxfp8_quantize(blk)
    assert scales[0, 0] == 120
    assert list(codes[0, :4]) == [0x70, 0xF8, 0x68, 0x55]
    assert (codes[0, 4:] == 0).all()


def test_block_rules_partial_zero_nonfinite_signed_zero():
    v = np.zeros((3, 48))
    v[0, :] = np.linspace(-3, 3, 48)           # two blocks: 32 + partial 16
    v[1, :] = -0.0                             # all-zero block, signed zeros kept
    v[2, :] = 1.0
    v[2, 5] = np.nan
    v[2, 40] = -np.inf
    codes, scales = oracle.mxfp8_quantize(v)
    assert scales.shape == (3, 2)
    # partial block: amax over its 16 valid values only
    assert scales[0, 1] == oracle.e8m0_exponent(np.abs(v[0, 32:]).max()) + 127
    assert (scales[1] == 0).all() and (codes[1] == 0x80).all()
    assert scales[2, 0] == 0xFF and scales[2, 1] == 0xFF
    assert (codes[2, :32] == 0x7F).all()
    assert codes[2, 40] == 0xFF and (np.delete(codes[2, 32:], 8) == 0x7F).all()


def test_roundtrip_error_bound_and_saturation_free():
    """|deq - v| <= half an E4M3 step at v * 2^-e on that grid; never saturates."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-30, 30, (64, 1)))
    codes, scales = oracle.mxfp8_quantize(v)
    deq = oracle.mxfp8_dequantize(codes, scales)
    e = scales.astype(np.int64).repeat(32, axis=1)[:, :96] - 127
    u = np.abs(v) * np.exp2(-e.astype(np.float64))
    assert (u <= 448.0).all()
    step = np.where(u < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(u, 1e-300))) - 3))
    err = np.abs(deq - v) * np.exp2(-e.astype(np.float64))
    assert (err <= step / 2 + 1e-300).all()
    # each block's largest magnitude rounds into [224, 448]
    amax_codes = (codes & 0x7F).reshape(64, 3, 32).max(axis=2)
    assert (amax_codes >= 0x76).all()  # amax * 2^-e lies in (224, 448]


def _expected_block(vals, table):
    """Independent reference for one block: scale byte and codes, from the
    definition (smallest e with amax <= 448 * 2^e, clamped; nearest E4M3 of
    v * 2^-e by exhaustive search, ties to the even code; NaN/Inf blocks ->
    scale 0xFF and 0x7F codes with the element's sign)."""
    pos_codes = np.arange(0x7F)
    pos_vals = table[pos_codes]
    if not np.all(np.isfinite(vals)):
        return 0xFF, [0x7F | (0x80 if math.copysign(1.0, v) < 0 else 0) for v in vals]
    amax = float(np.max(np.abs(vals))) if len(vals) else 0.0
    if amax == 0.0:
        e = -127
    else:
        e = math.ceil(math.log2(amax / 448.0))
        while amax <= 448.0 * 2.0 ** (e - 1):
            e -= 1
        while amax > 448.0 * 2.0 ** e:
            e += 1
        e = max(-127, min(127, e))
    codes = []
    for v in vals:
        a = abs(v) * 2.0 ** (-e)
        d = np.abs(pos_vals - min(a, 448.0))
        best = np.flatnonzero(d == d.min())
        if best.size == 2:
            best = best[(pos_codes[best] & 1) == 0]
        c = int(pos_codes[best[0]])
        codes.append(c | (0x80 if math.copysign(1.0, v) < 0 else 0))
    return e + 127, codes


def test_columnwise_blocks_run_down_columns():
    """Columnwise quantization = blocks of 32 consecutive rows of a column,
    written transposed: every code and scale of a 70 x 5 matrix (partial last
    block, a zero block, a NaN block, signed zeros, wide magnitudes) against
    the brute-force reference."""
    rng = np.random.default_rng(77)
    R, C = 70, 5
    v = rng.standard_normal((R, C)) * np.exp2(rng.integers(-20, 20, (R, C)))
    v[0:32, 1] = 0.0
    v[5, 1] = -0.0
    v[40, 2] = np.nan
    v[64:70, 3] *= 1e-3
    table = _all_code_values_torch()
    codes_t, scales_t = oracle.mxfp8_quantize_columns(v)
    assert codes_t.shape == (C, R) and scales_t.shape == (C, 3)
    for c in range(C):
        for blk in range(3):
            rows = v[32 * blk:min(R, 32 * blk + 32), c]
            sb, codes = _expected_block(rows, table)
            assert scales_t[c, blk] == sb, (c, blk)
            assert list(codes_t[c, 32 * blk:32 * blk + len(rows)]) == codes, (c, blk)


def test_swizzle_hand_positions():
    """Byte positions of the GEMM scale order, derived by hand from its
    definition (tiles of 128 rows x 4 columns, 512 bytes; inside a tile row
    r, column c at (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4) for a
    130 x 5 scale matrix: 2 x 2 tiles, 2048 bytes."""
    s = np.zeros((130, 5), np.uint8)
    marks = {(0, 0): 1, (1, 0): 2, (32, 0): 3, (0, 1): 4, (127, 3): 5, (129, 4): 6, (2, 4): 7}
    for (r, c), v in marks.items():
        s[r, c] = v
    out = oracle.mxfp8_swizzle_scales(s)
    assert out.shape == (2048,)
    expect = {0: 1, 16: 2, 4: 3, 1: 4, 31 * 16 + 3 * 4 + 3: 5,
              3 * 512 + 1 * 16: 6,          # tile (1, 1): row 129 -> r % 32 = 1, block 0; column 4 -> 0
              1 * 512 + 2 * 16: 7}          # tile (0, 1): row 2, column 4 -> 0
    for pos, v in expect.items():
        assert out[pos] == v, (pos, out[pos], v)
    assert int(np.count_nonzero(out)) == len(marks)


def test_swizzle_is_a_permutation_with_zero_padding():
    rng = np.random.default_rng(5)
    for rows, cols in ((1, 1), (37, 3), (128, 4), (300, 9)):
        s = rng.integers(1, 256, (rows, cols)).astype(np.uint8)
        out = oracle.mxfp8_swizzle_scales(s)
        assert out.size == ((rows + 127) // 128) * 128 * ((cols + 3) // 4) * 4
        assert np.array_equal(np.sort(out[out != 0]), np.sort(s.reshape(-1)))
        assert int(np.count_nonzero(out)) == rows * cols


def test_tiled_scale_order_is_the_swizzle_for_128_row_groups():
    """The tests' reader of the GEMM tiled scale order agrees with the
    oracle's swizzle (written from the definition) when groups are 128 rows,
    and with the swizzle of each padded group otherwise."""
    import helpers
    rng = np.random.default_rng(3)
    for rows, cols in ((130, 7), (256, 24), (1, 1), (300, 9)):
        s = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
        sw = oracle.mxfp8_swizzle_scales(s)
        assert np.array_equal(helpers.sf_untile(sw, rows, cols, 128), s)
    for G in (192, 96, 32):
        rows, cols = 2 * G, 10
        s = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
        buf = np.concatenate([oracle.mxfp8_swizzle_scales(s[g * G:(g + 1) * G]) for g in range(2)])
        assert np.array_equal(helpers.sf_untile(buf, rows, cols, G), s)
