"""GPU parity of the forward with MXFP8 weights (block-scaled tcgen05 MMA).

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
description paragraph ("supports both 16-bit projection and mxfp8
projection") and flowchart ("BF16 or MXFP8 weight"). x and W are quantized
rowwise (1 x 32 blocks along K) by the library's quantizer; the oracle
quantizes the same bf16 values itself and the two must agree byte for byte
before the products are compared, so the oracle's operands never come from
the CUDA path.
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu

SHAPES = [
    ("tiny", dict(T=300, K=512, H=8)),                        # BN 192 = 4 heads of 48
    ("tiny", dict(T=77, K=256, H=6)),                         # BN 96 (2 heads), ragged tokens
    ("dsv3_fwd_mxfp8w", dict(T=260, H=4)),                    # one head per 192-wide tile
    ("dsv3_fwd_mxfp8w", dict(T=140, H=2, K=1024, bias=True)),
    ("dsv3_fwd_mxfp8w", dict(T=200, H=3, K=256)),
    ("tiny", dict(T=450, K=256, H=4, Dn=64, Dr=32)),          # Dr = 32, 4 token tiles (ragged)
]


def _quantized_operands(inp, dev):
    xs = inp["x"].to(dev)
    Ws = inp["W"].to(dev)
    xq, xsc = mlaq.mxfp8_quantize_rows(xs)
    Wq, Wsc = mlaq.mxfp8_quantize_rows(Ws)
    torch.cuda.synchronize()
    # the oracle's own quantization of the same values
    oxq, oxs = oracle.mxfp8_quantize(helpers.f64(inp["x"]))
    oWq, oWs = oracle.mxfp8_quantize(helpers.f64(inp["W"]))
    assert np.array_equal(xq.cpu().numpy(), oxq) and np.array_equal(xsc.cpu().numpy(), oxs)
    assert np.array_equal(Wq.cpu().numpy(), oWq) and np.array_equal(Wsc.cpu().numpy(), oWs)
    x_deq = oracle.mxfp8_dequantize(oxq, oxs)
    W_deq = oracle.mxfp8_dequantize(oWq, oWs)
    return (xq, xsc, Wq, Wsc), (x_deq, W_deq)


def _oracle(inp, w, x_deq, W_deq, tokens=None, quantize=False):
    b = helpers.f64(inp["b"]) if inp.get("b") is not None else None
    pos = inp["pos"].numpy()
    if tokens is not None:
        x_deq, pos = x_deq[tokens], pos[tokens]
    return oracle.forward(x_deq, W_deq, w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), pos, b,
                          quantize=quantize)


@pytest.mark.parametrize("out_mode", ["bf16", "mxfp8"])
@pytest.mark.parametrize("name,ov", SHAPES)
def test_fwd_mxfp8_weights(cuda_device, name, ov, out_mode):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=2)
    (xq, xsc, Wq, Wsc), (x_deq, W_deq) = _quantized_operands(inp, cuda_device)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = mlaq.fwd(xq, Wq, d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=d.get("b"), pos=d["pos"],
                   weight_mode="mxfp8", out_mode=out_mode, x_scales=xsc, w_scales=Wsc, status=st)
    mlaq.check_status(st)
    if out_mode == "bf16":
        helpers.check_bf16_close(out, _oracle(inp, w, x_deq, W_deq))
    else:
        q_ref, rc, rs = _oracle(inp, w, x_deq, W_deq, quantize=True)
        helpers.check_mxfp8_close(out[0].cpu().numpy(), out[1].cpu().numpy(), q_ref, rc, rs)


def test_fwd_mxfp8_weights_full_size(cuda_device):
    """DeepSeek-V3 shape with 1% x50 activation outliers, MXFP8 x and W, MXFP8
    out, in the benchmark's launch configuration (scales in the GEMM's tiled
    order): every code and scale against the oracle on the dequantized
    operands; the row-major-scale call gives the same bytes."""
    w = synth.workload("dsv3_fwd_mxfp8w")
    inp = synth.make_inputs(w, seed=0)
    (xq, xsc, Wq, Wsc), (x_deq, W_deq) = _quantized_operands(inp, cuda_device)
    xst, Wst = _tiled_scales(xsc, Wsc, w)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (xq, Wq, d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    c1, s1 = mlaq.fwd(*args, pos=d["pos"], weight_mode="mxfp8_tiled", out_mode="mxfp8", x_scales=xst,
                      w_scales=Wst, status=st)
    c2, s2 = mlaq.fwd(*args, pos=d["pos"], weight_mode="mxfp8", out_mode="mxfp8", x_scales=xsc, w_scales=Wsc,
                      status=st)
    mlaq.check_status(st)
    assert torch.equal(c1, c2) and torch.equal(s1, s2)
    helpers.check_fwd_all_tokens(inp, w, codes=c1, scales=s1, x64=x_deq, W64=W_deq)
    # context only: error of the quantized path against the unquantized bf16 operands
    toks = np.arange(0, w.T, 97)
    q_ref = _oracle(inp, w, x_deq, W_deq, tokens=toks)
    q_bf = helpers.oracle_forward(inp, w, tokens=toks)
    rel = np.linalg.norm(q_ref - q_bf) / np.linalg.norm(q_bf)
    assert rel < 0.1


def _tiled_scales(xsc, Wsc, w):
    """The two scale tensors in the GEMM's tiled order (x: 128-row groups;
    W: groups of the kernel's channel tile, from the library's query)."""
    G = mlaq.w_scale_group(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr)
    assert G > 0
    return mlaq.mxfp8_swizzle_scales(xsc), mlaq.mxfp8_swizzle_scales(Wsc, group=G)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_fwd_tiled_scales_bit_identical(cuda_device, name, ov):
    """weight_mode mxfp8_tiled (scales pre-tiled, fetched by bulk copies) gives
    exactly the outputs of weight_mode mxfp8 (per-row scale gather), which
    test_fwd_mxfp8_weights checks against the oracle."""
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=4)
    d = helpers.to_dev(inp, cuda_device)
    xq, xsc = mlaq.mxfp8_quantize_rows(d["x"])
    Wq, Wsc = mlaq.mxfp8_quantize_rows(d["W"])
    xst, Wst = _tiled_scales(xsc, Wsc, w)
    args = (xq, Wq, d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw = dict(bias=d.get("b"), pos=d["pos"], out_mode="mxfp8")
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    c1, s1 = mlaq.fwd(*args, weight_mode="mxfp8", x_scales=xsc, w_scales=Wsc, status=st, **kw)
    c2, s2 = mlaq.fwd(*args, weight_mode="mxfp8_tiled", x_scales=xst, w_scales=Wst, status=st, **kw)
    mlaq.check_status(st)
    assert torch.equal(c1, c2) and torch.equal(s1, s2)


TILED_CASES = [
    # (workload, overrides, out_mode, packed table)
    ("dsv3_fwd_mxfp8w", dict(T=300, H=4), "mxfp8", True),                 # ragged last token tile
    ("dsv3_fwd_mxfp8w", dict(T=129, H=2, bias=True), "mxfp8_bhsd", False),  # one token in the last tile
    ("dsv3_fwd_mxfp8w", dict(T=64, H=3), "mxfp8_bhsd_swizzled", True),      # one partial tile
    ("dsv3_fwd_mxfp8w", dict(T=520, H=5, K=512), "bf16", True),
    ("tiny", dict(T=390, K=256, H=8, Dn=64, Dr=32), "mxfp8", False),        # Dr = 32
    ("tiny", dict(T=1, K=128, H=4), "mxfp8", True),                         # one token, Dr = 16
    # weight scales resident in TMEM per channel tile, CTAs on contiguous tile ranges:
    ("dsv3_fwd_mxfp8w", dict(T=2000, H=24), "mxfp8", True),      # 384 tiles: ranges cross channel tiles
    ("dsv3_fwd_mxfp8w", dict(T=130, H=200, K=512), "mxfp8", True),  # K steps = stages, 2 token tiles
    ("dsv3_fwd_mxfp8w", dict(T=700, H=40, K=1792), "mxfp8_bhsd", False),  # 14 K steps: the most held
    ("dsv3_fwd_mxfp8w", dict(T=300, H=40, K=1920), "bf16", True),   # 15 K steps: scales per stage again
    ("dsv3_fwd_mxfp8w", dict(T=900, H=30, K=1408), "mxfp8", True),  # 11 K steps, 8 token tiles (ragged)
    ("dsv3_fwd_mxfp8w", dict(T=640, H=34, K=1664), "mxfp8_bhsd_swizzled", True),  # 13 K steps
]


@pytest.mark.parametrize("name,ov,out_mode,packed", TILED_CASES)
def test_fwd_tiled_scales_every_mode(cuda_device, name, ov, out_mode, packed):
    """The tiled-scale forward (bulk copies of scale tiles; when they fit, the
    weight scales kept in TMEM across a CTA's tiles of one channel tile and
    each tile's x scales fetched in one copy) equals the per-row-gather
    forward, which test_fwd_mxfp8_weights checks
    against the oracle, for every output mode, both table layouts and
    ragged token counts."""
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=23)
    d = helpers.to_dev(inp, cuda_device)
    xq, xsc = mlaq.mxfp8_quantize_rows(d["x"])
    Wq, Wsc = mlaq.mxfp8_quantize_rows(d["W"])
    xst, Wst = _tiled_scales(xsc, Wsc, w)
    args = (xq, Wq, d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw = dict(bias=d.get("b"), pos=d["pos"], out_mode=out_mode)
    if packed:
        kw["rope_packed"] = mlaq.rope_table_pack(d["cos"], d["sin"], w.Dr)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    a = mlaq.fwd(*args, weight_mode="mxfp8", x_scales=xsc, w_scales=Wsc, status=st, **kw)
    b = mlaq.fwd(*args, weight_mode="mxfp8_tiled", x_scales=xst, w_scales=Wst, status=st, **kw)
    mlaq.check_status(st)
    a = a if isinstance(a, tuple) else (a,)
    b = b if isinstance(b, tuple) else (b,)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
