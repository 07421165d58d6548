"""GPU parity of the MXFP8 backward (mla_q_uproj_bwd_mxfp8).

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
Greptile summary: the MXFP8 helpers (rowwise, the transpose copy) that feed
block-scaled GEMMs. The pages give no backward formula; the oracle's reading
(oracle.backward_mxfp8): dq_pre is the float32 inverse rotation with single
roundings, each GEMM operand is quantized along its reduction dimension, and
dx, dW are exact products of the decoded operands.

Bars:
  * the four quantized operands (codes and scales) are bit-exact, including
    the zero padding of the token axis to a multiple of 128;
  * dx, dW: |gpu - ref| <= 2^-8 |ref| + 2^-14 S elementwise, S = the sum of
    |products| (bf16 output rounding plus fp32 accumulation of exact
    products), and the relative Frobenius error <= 2^-8;
  * db: |gpu - ref| <= 2^-8 |ref| + T 2^-23 sum|dq_pre| (bf16 rounding plus
    fp32 sequential sums).
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
    ("tiny", dict(T=200, K=96, H=2, Dn=64, Dr=64)),        # ragged T (neither 32- nor 128-aligned)
    ("tiny", dict(T=256, K=64, H=4, Dn=32, Dr=32)),
    ("tiny", dict(T=1, K=32, H=2, Dn=32, Dr=32)),          # one token, smallest N
    ("tiny", dict(T=416, K=224, H=3, Dn=64, Dr=64, seq_len=128)),  # 3 heads (N = 384), positions restart
    ("dsv3_bwd", dict(T=300, H=4, seq_len=None)),           # DeepSeek-V3 heads, K = 1536 (256-channel path)
    ("dsv3_long_yarn", dict(T=160, H=2, seq_len=None)),     # YaRN table; N = 384: per-head path
]


def _inputs(w, seed, dev):
    inp = synth.make_inputs(w, seed=seed)
    return inp, helpers.to_dev(inp, dev)


def _np(t):
    return t.cpu().numpy()


def _check_gemm(got, ref, S, what):
    got = helpers.bf16_to_f64(got)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * S
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bound"
    assert np.linalg.norm(got - ref) <= 2.0 ** -8 * np.linalg.norm(ref), what


def _check_db(got, dqp, what="db"):
    ref = dqp.sum(0)
    got = helpers.bf16_to_f64(got)
    bound = 2.0 ** -8 * np.abs(ref) + dqp.shape[0] * 2.0 ** -23 * np.abs(dqp).sum(0)
    assert np.all(np.abs(got - ref) <= bound), what


def _run(w, d, st, ws=None, **kw):
    return mlaq.bwd_mxfp8(d["dq"], d["W"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                          status=st, workspace=ws, **kw)


def _workspace(w, d, dev):
    n = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, d["cos"].shape[0], d["cos"].shape[1], 3)
    return torch.empty((n,), dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_bwd_mxfp8_matches_oracle(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp, d = _inputs(w, 0, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = _workspace(w, d, cuda_device)
    dx, dW, db = _run(w, d, st, ws)
    mlaq.check_status(st)
    g = oracle.backward_mxfp8(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H,
                              w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy())
    ops = mlaq.bwd_mxfp8_operands(ws, w.T, w.K, w.H, w.Dn, w.Dr, d["cos"].shape[0], d["cos"].shape[1])
    T, N, K, nbt, Tp, G = w.T, w.N, w.K, (w.T + 31) // 32, ops["t_pad"], ops["b_group"]
    assert Tp % 128 == 0 and Tp - 128 < T <= Tp
    for key in ("qa", "wt"):
        assert np.array_equal(_np(ops[key]), g[key]), key
    for key in ("qb", "xt"):
        assert np.array_equal(_np(ops[key])[:, :T], g[key]), key
    assert not _np(ops["qb"])[:, T:].any(), "qb: padding tokens must be 0"
    # A operands: the whole tiled array is the oracle's swizzle of the zero-padded scales
    qa_s = np.zeros((Tp, N // 32), np.uint8)
    qa_s[:T] = g["qa_s"]
    assert np.array_equal(_np(ops["qa_s"]), oracle.mxfp8_swizzle_scales(qa_s)), "qa_s"
    qb_s = np.zeros((N, Tp // 32), np.uint8)
    qb_s[:, :nbt] = g["qb_s"]
    assert np.array_equal(_np(ops["qb_s"]), oracle.mxfp8_swizzle_scales(qb_s)), "qb_s"
    # B operands: groups of G rows
    assert np.array_equal(helpers.sf_untile(_np(ops["wt_s"]), K, N // 32, G), g["wt_s"]), "wt_s"
    xt_s = helpers.sf_untile(_np(ops["xt_s"]), K, Tp // 32, G)
    assert np.array_equal(xt_s[:, :nbt], g["xt_s"]), "xt_s"
    assert not xt_s[:, nbt:].any(), "xt_s: padding token blocks must be 0"
    A = np.abs(oracle.mxfp8_dequantize(g["qa"], g["qa_s"]))
    B = np.abs(oracle.mxfp8_dequantize(g["wt"], g["wt_s"]))
    _check_gemm(dx, g["dx"], A @ B.T, "dx")
    A = np.abs(oracle.mxfp8_dequantize(g["qb"], g["qb_s"]))
    B = np.abs(oracle.mxfp8_dequantize(g["xt"], g["xt_s"]))
    _check_gemm(dW, g["dW"], A @ B.T, "dW")
    dqp = oracle.rope_bwd_f32(helpers.f64(inp["dq"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(),
                              inp["sin"].numpy(), inp["pos"].numpy()).reshape(T, -1).astype(np.float64)
    _check_db(db, dqp)


def test_bwd_mxfp8_subsets_are_the_same_bits(cuda_device):
    """Each gradient alone (the other operand absent) equals the same gradient
    of the full call, written over every element of a prefilled output."""
    w = synth.workload("tiny", T=200, K=96, H=2, Dn=64, Dr=64)
    _, d = _inputs(w, 3, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dx, dW, db = _run(w, d, st)
    canary = lambda shape: torch.full(shape, 5.0, dtype=torch.bfloat16, device=cuda_device)
    only_dx = _run(w, dict(d, x=None), st, dx=canary(dx.shape), dW=None, db=None)
    only_dw = _run(w, dict(d, W=None), st, dx=None, dW=canary(dW.shape), db=None)
    only_db = _run(w, dict(d, W=None), st, dx=None, dW=None, db=canary(db.shape))  # x only gives K
    mlaq.check_status(st)
    assert torch.equal(only_dx[0], dx) and only_dx[1] is None and only_dx[2] is None
    assert torch.equal(only_dw[1], dW) and only_dw[0] is None and only_dw[2] is None
    assert torch.equal(only_db[2], db) and only_db[0] is None and only_db[1] is None


def test_bwd_mxfp8_inputs_unchanged_and_deterministic(cuda_device):
    w = synth.workload("tiny", T=256, K=64, H=4, Dn=32, Dr=32)
    _, d = _inputs(w, 4, cuda_device)
    before = {k: v.clone() for k, v in d.items() if isinstance(v, torch.Tensor)}
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    a = _run(w, d, st)
    b = _run(w, d, st)
    mlaq.check_status(st)
    for k, v in before.items():
        assert torch.equal(d[k], v), k
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_mxfp8_zero_tokens(cuda_device):
    w = synth.workload("tiny", T=0, K=64, H=4, Dn=32, Dr=32)
    _, d = _inputs(w, 5, cuda_device)
    dW = torch.full((w.N, w.K), 3.0, dtype=torch.bfloat16, device=cuda_device)
    db = torch.full((w.N,), 3.0, dtype=torch.bfloat16, device=cuda_device)
    dx, dW2, db2 = _run(w, d, None, dx=True, dW=dW, db=db)
    torch.cuda.synchronize()
    assert dx.shape == (0, w.K)
    assert not dW2.any() and not db2.any()


def test_bwd_mxfp8_position_out_of_range_reports_status(cuda_device):
    w = synth.workload("tiny", T=64, K=64, H=4, Dn=32, Dr=32)
    _, d = _inputs(w, 6, cuda_device)
    pos = d["pos"].clone()
    pos[17] = d["cos"].shape[0]  # one past the table
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    _run(w, dict(d, pos=pos), st)
    torch.cuda.synchronize()
    assert int(st.item()) == mlaq.STATUS["MLA_ERR_POS_RANGE"]


def test_bwd_mxfp8_full_size_sampled(cuda_device):
    """DeepSeek-V3 backward shape (T = 2 x 4096, pos = t mod 4096, K = 1536,
    H = 128), as the benchmark runs it: the quantized operands on sampled
    tokens / channels bit-exact, dx on sampled tokens, dW on sampled
    channels, db on every channel."""
    w = synth.workload("dsv3_bwd")
    inp, d = _inputs(w, 0, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = _workspace(w, d, cuda_device)
    dx, dW, db = _run(w, d, st, ws)
    mlaq.check_status(st)
    cs, sn, pos = inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()
    ops = mlaq.bwd_mxfp8_operands(ws, w.T, w.K, w.H, w.Dn, w.Dr, cs.shape[0], cs.shape[1])
    Tp, G = ops["t_pad"], ops["b_group"]
    rng = np.random.default_rng(7)
    W, x = helpers.f64(inp["W"]), helpers.f64(inp["x"])
    wt, wt_s = oracle.mxfp8_quantize_columns(W)
    xt, xt_s = oracle.mxfp8_quantize_columns(x)
    assert np.array_equal(_np(ops["wt"]), wt)
    assert np.array_equal(helpers.sf_untile(_np(ops["wt_s"]), w.K, w.N // 32, G), wt_s)
    assert np.array_equal(_np(ops["xt"]), xt)
    assert np.array_equal(helpers.sf_untile(_np(ops["xt_s"]), w.K, Tp // 32, G), xt_s)
    qa_s_rows = helpers.sf_untile(_np(ops["qa_s"]), Tp, w.N // 32, 128)
    qb_s_rows = helpers.sf_untile(_np(ops["qb_s"]), w.N, Tp // 32, 128)
    Bw, Bx = oracle.mxfp8_dequantize(wt, wt_s), oracle.mxfp8_dequantize(xt, xt_s)
    # dx and the rowwise operand on sampled tokens (rows are independent)
    toks = np.sort(rng.choice(w.T, 24, replace=False))
    dqp = oracle.rope_bwd_f32(helpers.f64(inp["dq"][torch.from_numpy(toks)]), w.H, w.Dn, w.Dr, cs, sn,
                              pos[toks]).reshape(len(toks), -1).astype(np.float64)
    qa, qa_s = oracle.mxfp8_quantize(dqp)
    assert np.array_equal(_np(ops["qa"])[toks], qa) and np.array_equal(qa_s_rows[toks], qa_s)
    A = oracle.mxfp8_dequantize(qa, qa_s)
    _check_gemm(dx[torch.from_numpy(toks).to(cuda_device)], A @ Bw.T, np.abs(A) @ np.abs(Bw).T, "dx")
    # dW and the columnwise operand on sampled heads (a head's channels need only that head's dq)
    heads = np.array([0, 45, 127])
    dqp_h = oracle.rope_bwd_f32(helpers.f64(inp["dq"][:, torch.from_numpy(heads)].contiguous()), len(heads),
                                w.Dn, w.Dr, cs, sn, pos).reshape(w.T, -1).astype(np.float64)
    qb, qb_s = oracle.mxfp8_quantize_columns(dqp_h)
    ch = (heads[:, None] * w.D + np.arange(w.D)[None, :]).reshape(-1)
    assert np.array_equal(_np(ops["qb"])[ch], qb) and np.array_equal(qb_s_rows[ch], qb_s)
    A = oracle.mxfp8_dequantize(qb, qb_s)
    _check_gemm(dW[torch.from_numpy(ch).to(cuda_device)], A @ Bx.T, np.abs(A) @ np.abs(Bx).T, "dW")
    # db on every channel, 16 heads at a time
    for h0 in range(0, w.H, 16):
        dqp_c = oracle.rope_bwd_f32(helpers.f64(inp["dq"][:, h0:h0 + 16].contiguous()), 16, w.Dn, w.Dr,
                                    cs, sn, pos).reshape(w.T, -1).astype(np.float64)
        _check_db(db[h0 * w.D:(h0 + 16) * w.D], dqp_c, f"db heads {h0}+")


@pytest.mark.parametrize("name,ov", [SHAPES[0], SHAPES[3], SHAPES[4]])
def test_prepared_weight_bit_identical(cuda_device, name, ov):
    """mla_q_uproj_bwd_mxfp8_prepared with W's columnwise copy made once
    (mxfp8_quantize_cols_tiled, the layout's b_group) gives the bytes of the
    call that quantizes W itself; the prepared copy equals the one that call
    leaves in its workspace."""
    w = synth.workload(name, **ov)
    inp, d = _inputs(w, 31, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = _workspace(w, d, cuda_device)
    dx1, dW1, db1 = _run(w, d, st, ws)
    ops = mlaq.bwd_mxfp8_operands(ws, w.T, w.K, w.H, w.Dn, w.Dr, d["cos"].shape[0], d["cos"].shape[1])
    wt, wts = mlaq.bwd_mxfp8_prepare_weight(d["W"], w.T, w.H, w.Dn, w.Dr, d["cos"])
    torch.cuda.synchronize()
    assert torch.equal(wt, ops["wt"])
    lay = mlaq.bwd_mxfp8_layout(w.T, w.K, w.H, w.Dn, w.Dr, d["cos"].shape[0], d["cos"].shape[1])
    # the real scale entries agree (the workspace's padding bytes are unspecified)
    G = lay["b_group"]
    ws_s = ws[lay["wt_scales"]:lay["wt_scales"] + wts.numel()].cpu().numpy()
    assert np.array_equal(helpers.sf_untile(wts.cpu().numpy(), w.K, w.N // 32, G),
                          helpers.sf_untile(ws_s, w.K, w.N // 32, G))
    dx2, dW2, db2 = mlaq.bwd_mxfp8(d["dq"], None, d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                                   status=st, prepared=(wt, wts))
    mlaq.check_status(st)
    assert torch.equal(dx1, dx2) and torch.equal(dW1, dW2) and torch.equal(db1, db2)
