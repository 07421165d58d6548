"""GPU parity of the MXFP8 backward (mla_q_uproj_bwd_mxfp8).

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
Greptile summary: the MXFP8 helpers (rowwise, the transpose copy) that feed
block-scaled GEMMs. The pages give no backward formula; the oracle's reading
(oracle.backward_mxfp8): dq_pre is the exact (fp64) RoPE backward, each GEMM
operand is quantized along its reduction dimension, and dx, dW are exact
products of the decoded operands.

The GPU evaluates dq_pre in float32, so its value of each rope channel lies
within eb = 2^-22 (|g_i| + |g_{i+h}|) max|table| of the exact one (at most
three float32 roundings of a two-term sum of products); pass-through
channels are exact. Bars:
  * W's and x's columnwise copies (quantized straight from bf16): bit-exact;
  * dq_pre's two copies: bit-exact wherever the MXFP8 rule decides the scale
    and code for every value within +-eb (helpers.mxfp8_decided: at least
    90% of the elements; a single token at position 0 has rotation ties),
    elsewhere within one E4M3 step on the GPU's grid;
    the token padding to a multiple of 128 is zero;
  * dx, dW: |gpu - ref| <= 2^-8 |ref| + 2^-14 S + F elementwise, S = the sum
    of |products| (bf16 output rounding plus fp32 accumulation of exact
    products), F = the products of two E4M3 steps of the undecided operand
    elements with the other operand (0 when every code is decided), and the
    relative Frobenius error <= 2^-8;
  * db: |gpu - ref| <= 2^-8 |ref| + T 2^-23 sum|dq_pre| + sum eb (bf16
    rounding, float32 sums of float32 values).
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


def rot_error_bound(dq, H, Dn, Dr, cos):
    """eb [T, N]: how far a float32 evaluation of the inverse rotation may be
    from the exact one (see the module docstring); 0 on pass-through channels."""
    T = dq.shape[0]
    g = np.abs(np.asarray(dq, np.float64).reshape(T, H, Dn + Dr))
    h = Dr // 2
    amp = float(np.max(np.abs(cos))) if Dr else 0.0
    eb = np.zeros_like(g)
    pair = g[:, :, Dn:Dn + h] + g[:, :, Dn + h:]
    eb[:, :, Dn:Dn + h] = pair
    eb[:, :, Dn + h:] = pair
    return (eb * 2.0 ** -22 * max(amp, 1.0)).reshape(T, -1)


def _step_max(v, e_hi):
    """One E4M3 step of |v| at the larger of a block's possible exponents."""
    a = np.abs(v)
    normal = np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 3)
    return np.maximum(normal, np.exp2(-9.0 + e_hi))


def _flip_terms(v, eb, other_abs):
    """F: two E4M3 steps of every undecided element of v [R, C] (blocks along
    C) times |other| [C, M], summed: [R, M] (0 when all codes are decided)."""
    _, cf, _, e_hi = helpers.mxfp8_decided(v, eb)
    und = np.argwhere(~cf)
    F = np.zeros((v.shape[0], other_abs.shape[1]))
    for r, c in und:
        F[r] += 2 * _step_max(v[r, c], float(e_hi[r, c // 32])) * other_abs[c]
    return F


def _check_gemm(got, ref, S, what, F=0.0):
    got = helpers.bf16_to_f64(got)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * S + F
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bound"
    assert np.linalg.norm(got - ref) <= 2.0 ** -8 * np.linalg.norm(ref), what


def _check_db(got, dqp, eb, what="db"):
    ref = dqp.sum(0)
    got = helpers.bf16_to_f64(got)
    bound = 2.0 ** -8 * np.abs(ref) + dqp.shape[0] * 2.0 ** -23 * np.abs(dqp).sum(0) + eb.sum(0)
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
    dq64 = helpers.f64(inp["dq"])
    g = oracle.backward_mxfp8(dq64, helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H,
                              w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy())
    ops = mlaq.bwd_mxfp8_operands(ws, w.T, w.K, w.H, w.Dn, w.Dr, d["cos"].shape[0], d["cos"].shape[1])
    T, N, K, nbt, Tp, G = w.T, w.N, w.K, (w.T + 31) // 32, ops["t_pad"], ops["b_group"]
    assert Tp % 128 == 0 and Tp - 128 < T <= Tp
    # W's and x's columnwise copies come straight from bf16: bit-exact
    assert np.array_equal(_np(ops["wt"]), g["wt"]), "wt"
    assert np.array_equal(_np(ops["xt"])[:, :T], g["xt"]), "xt"
    assert np.array_equal(helpers.sf_untile(_np(ops["wt_s"]), K, N // 32, G), g["wt_s"]), "wt_s"
    xt_s = helpers.sf_untile(_np(ops["xt_s"]), K, Tp // 32, G)
    assert np.array_equal(xt_s[:, :nbt], g["xt_s"]), "xt_s"
    assert not xt_s[:, nbt:].any(), "xt_s: padding token blocks must be 0"
    # dq_pre's copies: decided codes bit-exact, the rest within one step
    dqp, eb = g["dq_pre"], rot_error_bound(dq64, w.H, w.Dn, w.Dr, inp["cos"].numpy())
    qa_s = helpers.sf_untile(_np(ops["qa_s"]), Tp, N // 32, 128)
    assert not qa_s[T:].any(), "qa_s: padding rows must be 0"
    helpers.check_mxfp8_decided(_np(ops["qa"]), qa_s[:T], dqp, eb, g["qa"], g["qa_s"], "qa")
    qb = _np(ops["qb"])
    assert not qb[:, T:].any(), "qb: padding tokens must be 0"
    qb_s = helpers.sf_untile(_np(ops["qb_s"]), N, Tp // 32, 128)
    assert not qb_s[:, nbt:].any(), "qb_s: padding token blocks must be 0"
    helpers.check_mxfp8_decided(qb[:, :T], qb_s[:, :nbt], dqp.T.copy(), eb.T.copy(), g["qb"], g["qb_s"], "qb")
    # products against the oracle's operands
    A = np.abs(oracle.mxfp8_dequantize(g["qa"], g["qa_s"]))
    B = np.abs(oracle.mxfp8_dequantize(g["wt"], g["wt_s"]))
    _check_gemm(dx, g["dx"], A @ B.T, "dx", _flip_terms(dqp, eb, B.T))
    A = np.abs(oracle.mxfp8_dequantize(g["qb"], g["qb_s"]))
    B = np.abs(oracle.mxfp8_dequantize(g["xt"], g["xt_s"]))
    _check_gemm(dW, g["dW"], A @ B.T, "dW", _flip_terms(dqp.T.copy(), eb.T.copy(), B.T))
    _check_db(db, dqp, eb)


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
    H = 128), as the benchmark runs it: W's and x's copies bit-exact in
    full; dq_pre's copies and dx on 64 sampled tokens, dq_pre's columnwise
    copy and dW on 8 sampled heads over all tokens; db on every channel."""
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
    toks = np.unique(np.concatenate([[0, 4095, 4096, w.T - 1], rng.choice(w.T, 60, replace=False)]))
    dq_t = helpers.f64(inp["dq"][torch.from_numpy(toks)])
    dqp = oracle.rope_bwd(dq_t, w.H, w.Dn, w.Dr, cs, sn, pos[toks]).reshape(len(toks), -1)
    eb = rot_error_bound(dq_t, w.H, w.Dn, w.Dr, cs)
    qa, qa_s = oracle.mxfp8_quantize(dqp)
    helpers.check_mxfp8_decided(_np(ops["qa"])[toks], qa_s_rows[toks], dqp, eb, qa, qa_s, "qa")
    A = oracle.mxfp8_dequantize(qa, qa_s)
    _check_gemm(dx[torch.from_numpy(toks).to(cuda_device)], A @ Bw.T, np.abs(A) @ np.abs(Bw).T, "dx",
                _flip_terms(dqp, eb, np.abs(Bw).T))
    # dW and the columnwise operand on sampled heads (a head's channels need only that head's dq)
    heads = np.array([0, 17, 45, 64, 90, 101, 126, 127])
    dq_h = helpers.f64(inp["dq"][:, torch.from_numpy(heads)].contiguous())
    dqp_h = oracle.rope_bwd(dq_h, len(heads), w.Dn, w.Dr, cs, sn, pos).reshape(w.T, -1)
    eb_h = rot_error_bound(dq_h, len(heads), w.Dn, w.Dr, cs)
    qb, qb_s = oracle.mxfp8_quantize_columns(dqp_h)
    ch = (heads[:, None] * w.D + np.arange(w.D)[None, :]).reshape(-1)
    helpers.check_mxfp8_decided(_np(ops["qb"])[ch][:, :w.T], qb_s_rows[ch], dqp_h.T.copy(), eb_h.T.copy(),
                                qb, qb_s, "qb")
    A = oracle.mxfp8_dequantize(qb, qb_s)
    _check_gemm(dW[torch.from_numpy(ch).to(cuda_device)], A @ Bx.T, np.abs(A) @ np.abs(Bx).T, "dW",
                _flip_terms(dqp_h.T.copy(), eb_h.T.copy(), np.abs(Bx).T))
    # db on every channel, 16 heads at a time
    for h0 in range(0, w.H, 16):
        dq_c = helpers.f64(inp["dq"][:, h0:h0 + 16].contiguous())
        dqp_c = oracle.rope_bwd(dq_c, 16, w.Dn, w.Dr, cs, sn, pos).reshape(w.T, -1)
        _check_db(db[h0 * w.D:(h0 + 16) * w.D], dqp_c, rot_error_bound(dq_c, 16, w.Dn, w.Dr, cs), f"db heads {h0}+")


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
