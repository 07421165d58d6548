"""GPU parity of the fused forward (bf16 weights): GEMM + bias + RoPE, bf16 or
MXFP8 output, against the fp64 oracle.

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
description paragraph and flowchart; Megatron-LM PR "Fix fused MLA YaRN RoPE
query kernel corrupting upstream tensor in-place", Problem section (the
input must be unchanged afterwards).
"""
import numpy as np
import pytest
import torch

import helpers
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu

# (name, overrides): several tiles, ragged token / K tails, both rope widths
SHAPES = [
    ("tiny", {}),
    ("tiny", dict(T=300, K=200, H=6)),                    # 3 token tiles (44 ragged), K tail 8
    ("tiny", dict(T=1, K=8, H=1)),                        # single token, single partial k tile
    ("tiny", dict(T=129, K=64, H=16, Dn=64, Dr=32, w_std=0.1)),
    ("dsv3_fwd_bf16w", dict(T=300, H=8)),                 # 256-wide tiles cut heads at 64/128
    ("dsv3_fwd_bf16w", dict(T=260, K=1000, H=3, bias=True)),
    ("dsv3_fwd_bf16w", dict(T=513, H=2, K=256, bias=True)),   # ragged last token tile, bias
    ("dsv3_fwd_bf16w", dict(T=100, H=6, Dn=64, K=128)),       # D = 128: rope regions at channel 64 mod 128
    ("tiny", dict(T=1, K=64, H=4, Dn=64, Dr=32)),             # single token, Dr = 32
    # 128-channel tiles (N = 128): MXFP8 scales written byte by byte
    ("dsv3_fwd_bf16w", dict(T=100, H=2, Dn=0, K=128)),        # Dn = 0: heads are all rope
    ("tiny", dict(T=200, K=64, H=2, Dn=32, Dr=32)),
]


def _run(w, inp, dev, out_mode, status=None):
    d = helpers.to_dev(inp, dev)
    return mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=d.get("b"),
                    pos=d["pos"], out_mode=out_mode, status=status)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_fwd_bf16_out(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=0)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    q = _run(w, inp, cuda_device, "bf16", st)
    mlaq.check_status(st)
    ref = helpers.oracle_forward(inp, w)
    helpers.check_bf16_close(q, ref)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_fwd_mxfp8_out(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=1)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    codes, scales = _run(w, inp, cuda_device, "mxfp8", st)
    mlaq.check_status(st)
    q_ref, rc, rs = helpers.oracle_forward(inp, w, quantize=True)
    helpers.check_mxfp8_close(codes.cpu().numpy(), scales.cpu().numpy(), q_ref, rc, rs)


def test_fwd_passthrough_equals_plain_gemm(cuda_device):
    """The first Dn channels of each head are the GEMM (+bias) itself: run once
    at position 0 (cos = 1, sin = 0, so RoPE is the identity) and once at real
    positions; the pass-through channels must agree bit for bit."""
    w = synth.workload("tiny", T=200)
    inp = synth.make_inputs(w, seed=2)
    q1 = _run(w, inp, cuda_device, "bf16")
    inp0 = dict(inp, pos=torch.zeros(w.T, dtype=torch.int32))
    q0 = _run(w, inp0, cuda_device, "bf16")
    assert torch.equal(q1[..., :w.Dn], q0[..., :w.Dn])
    ref = helpers.oracle_forward(inp0, w)  # = x W^T + b
    helpers.check_bf16_close(q0, ref)


def test_fwd_inputs_unchanged(cuda_device):
    w = synth.workload("tiny", T=333, H=8)
    inp = helpers.to_dev(synth.make_inputs(w, seed=3), cuda_device)
    before = {k: v.clone() for k, v in inp.items() if isinstance(v, torch.Tensor)}
    mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"],
             pos=inp["pos"], out_mode="mxfp8")
    mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"],
             pos=inp["pos"], out_mode="bf16")
    torch.cuda.synchronize()
    for k, v in before.items():
        assert torch.equal(inp[k], v), k


# a Dr = 16 shape and a DeepSeek-V3 head shape (Dr = 64)
KERNELS = [("tiny", {}), ("dsv3_fwd_bf16w", dict(K=128, H=2, bias=True))]


@pytest.mark.parametrize("name,ov", KERNELS)
def test_fwd_writes_nothing_outside_outputs(cuda_device, name, ov):
    """Canary bytes around q and its scales stay untouched."""
    w = synth.workload(name, **dict(ov, T=130))
    inp = helpers.to_dev(synth.make_inputs(w, seed=4), cuda_device)
    pad = 4096
    nb = (w.D + 31) // 32
    nq, ns = w.T * w.H * w.D, w.T * w.H * nb
    qbuf = torch.full((nq + 2 * pad,), 0xA5, dtype=torch.uint8, device=cuda_device)
    sbuf = torch.full((ns + 2 * pad,), 0x5A, dtype=torch.uint8, device=cuda_device)
    q = qbuf[pad:pad + nq].view(w.T, w.H, w.D)
    s = sbuf[pad:pad + ns].view(w.T, w.H, nb)
    mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"],
             pos=inp["pos"], out_mode="mxfp8", q_out=q, q_scales=s)
    torch.cuda.synchronize()
    assert (qbuf[:pad] == 0xA5).all() and (qbuf[pad + nq:] == 0xA5).all()
    assert (sbuf[:pad] == 0x5A).all() and (sbuf[pad + ns:] == 0x5A).all()


@pytest.mark.parametrize("name,ov", KERNELS)
def test_fwd_position_out_of_range_reports_status(cuda_device, name, ov):
    w = synth.workload(name, **dict(ov, T=64))
    inp = synth.make_inputs(w, seed=5)
    inp["pos"] = inp["pos"].clone()
    inp["pos"][7] = w.cs_rows + 3  # outside the table: reported, never read
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    _run(w, inp, cuda_device, "bf16", st)
    assert int(st.item()) == mlaq.STATUS["MLA_ERR_POS_RANGE"]


@pytest.mark.parametrize("name,ov", KERNELS)
def test_fwd_wide_table_and_packed_positions(cuda_device, name, ov):
    """cs_width > Dr (row pitch = cs_width) and positions restarting per sequence."""
    w = synth.workload(name, **dict(ov, T=256, seq_len=100))
    inp = synth.make_inputs(w, seed=6)
    cos, sin = synth.rope_table_standard(100, w.Dr + 8)  # the kernel reads the first Dr columns
    inp["cos"], inp["sin"] = cos, sin
    q = _run(w, inp, cuda_device, "bf16")
    ref = helpers.oracle_forward(inp, w)
    helpers.check_bf16_close(q, ref)


def test_fwd_full_size(cuda_device):
    """DeepSeek-V3 shape (T=4096, K=1536, H=128, Dn=128, Dr=64) in the launch
    configuration the benchmark times: every element of the bf16 q and of
    the MXFP8 q (codes and scales) against one oracle pass."""
    w = synth.workload("dsv3_fwd_bf16w")
    inp = synth.make_inputs(w, seed=0)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    codes, scales = mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                             out_mode="mxfp8", status=st)
    q = mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], out_mode="bf16", status=st)
    mlaq.check_status(st)
    helpers.check_fwd_all_tokens(inp, w, q=q, codes=codes, scales=scales)


@pytest.mark.parametrize("name,ov", KERNELS)
def test_fwd_nonfinite_blocks(cuda_device, name, ov):
    """An Inf weight element makes its channel non-finite for every token (and,
    through the rotation, its rope partner). Every MXFP8 block holding a
    non-finite value gets scale 0xFF and NaN codes (0x7F with the element's
    sign); the other blocks are unaffected. The oracle decides which blocks."""
    w = synth.workload(name, **dict(ov, T=150))
    inp = synth.make_inputs(w, seed=9)
    W = inp["W"].clone()
    W[w.Dn + 3, 5] = float("inf")            # a rope channel of head 0
    W[w.D + min(w.Dn - 1, 40), 2] = float("-inf")  # a pass-through channel of head 1
    inp["W"] = W
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    codes, scales = _run(w, inp, cuda_device, "mxfp8", st)
    mlaq.check_status(st)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    q_ref, rc, rs = helpers.oracle_forward(inp, w, quantize=True)
    bad = rs == 0xFF
    assert bad.any() and (~bad).any()
    assert np.array_equal(scales == 0xFF, bad)
    nb = rs.shape[2]
    bad_el = np.repeat(bad, 32, axis=2)[:, :, :w.D]
    assert ((codes[bad_el] & 0x7F) == 0x7F).all()
    # finite elements of those blocks keep their sign
    fin = bad_el & np.isfinite(q_ref) & (np.abs(q_ref) > 1e-6)
    assert np.array_equal(codes[fin] >> 7, (q_ref[fin] < 0).astype(np.uint8))
    # every other block as usual: scales as the oracle's (>= 99.9%), elements
    # within one E4M3 step of the reference
    ok_blk = ~bad
    assert (scales[ok_blk] == rs[ok_blk]).mean() >= 0.999
    e_el = np.repeat(scales.astype(np.int64) - 127, 32, axis=2)[:, :, :w.D].astype(np.float64)
    ok_el = ~bad_el
    deq = helpers.e4m3_lut()[codes[ok_el]] * np.exp2(e_el[ok_el])
    tol = helpers.ulp_e4m3(np.abs(q_ref[ok_el]) * np.exp2(-e_el[ok_el])) * np.exp2(e_el[ok_el])
    assert (np.abs(deq - q_ref[ok_el]) <= tol).all()
    assert nb == (w.D + 31) // 32
