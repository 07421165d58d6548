"""GPU parity of the backward: inverse RoPE fused into dgrad and wgrad, plus db.

TransformerEngine PR "Add a backwards linear function to be used with the
fused mla q up-proj": sequence diagram (RoPE backward, then the linear
backward with the saved input and the weight) and the review comment "BF16
bias gradient remains missing" (db must be produced). Megatron-LM PR "Fix
fused MLA YaRN RoPE query kernel corrupting upstream tensor in-place",
discussion: the wgrad must use the linear's saved input and may be delayed
(a separate call). Tolerance: ||gpu - ref||_F / ||ref||_F <= 5e-3.
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu
TOL = 5e-3

SHAPES = [
    ("tiny", {}),
    ("tiny", dict(T=300, K=200, H=6)),                        # ragged tokens, K, channels
    ("tiny", dict(T=1, K=8, H=1)),
    ("tiny", dict(T=130, K=64, H=16, Dn=64, Dr=32)),
    ("dsv3_bwd", dict(T=300, H=8, seq_len=None)),
    ("dsv3_bwd", dict(T=260, K=1000, H=3, seq_len=128)),      # positions restart every 128
    ("dsv3_long_yarn", dict(T=200, H=4, seq_len=None)),       # YaRN table
]


def _dev_inputs(w, seed, dev):
    inp = synth.make_inputs(w, seed=seed)
    return inp, helpers.to_dev(inp, dev)


def _oracle_bwd(inp, w, **kw):
    return oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H,
                           w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy(), **kw)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_bwd_matches_oracle(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp, d = _dev_inputs(w, 0, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
    dW, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                            status=st)
    mlaq.check_status(st)
    g = _oracle_bwd(inp, w)
    for name_, got in (("dx", dx), ("dW", dW), ("db", db)):
        err = helpers.frob_rel(got, g[name_])
        assert err <= TOL, f"{name_}: relative Frobenius error {err:.3e}"


def test_bwd_at_identity_rotation_is_plain_gemm(cuda_device):
    """pos = 0 (cos = 1, sin = 0): dq_pre = dq, so dx = dq W, dW = dq^T x, db = sum dq."""
    w = synth.workload("tiny", T=200, H=8)
    inp = synth.make_inputs(w, seed=3)
    inp["pos"] = torch.zeros(w.T, dtype=torch.int32)
    d = helpers.to_dev(inp, cuda_device)
    dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"])
    dW, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"])
    dq = helpers.f64(inp["dq"]).reshape(w.T, -1)
    x, W = helpers.f64(inp["x"]), helpers.f64(inp["W"])
    assert helpers.frob_rel(dx, dq @ W) <= TOL
    assert helpers.frob_rel(dW, dq.T @ x) <= TOL
    assert helpers.frob_rel(db, dq.sum(0)) <= TOL


def test_wgrad_without_bias_and_inputs_unchanged(cuda_device):
    w = synth.workload("tiny", T=190, H=5)
    inp, d = _dev_inputs(w, 4, cuda_device)
    before = {k: v.clone() for k, v in d.items() if isinstance(v, torch.Tensor)}
    db_canary = torch.full((w.N,), 7.0, dtype=torch.bfloat16, device=cuda_device)
    dW, none = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                              db=None)
    mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"])
    torch.cuda.synchronize()
    assert none is None and (db_canary == 7.0).all()
    for k, v in before.items():
        assert torch.equal(d[k], v), k
    g = _oracle_bwd(inp, w, want=("dW",))
    assert helpers.frob_rel(dW, g["dW"]) <= TOL


def test_wgrad_zero_tokens_gives_zero(cuda_device):
    w = synth.workload("tiny", T=0)
    d = helpers.to_dev(synth.make_inputs(synth.workload("tiny"), seed=5), cuda_device)
    dq = torch.empty((0, w.H, w.D), dtype=torch.bfloat16, device=cuda_device)
    x = torch.empty((0, w.K), dtype=torch.bfloat16, device=cuda_device)
    dW = torch.full((w.N, w.K), 3.0, dtype=torch.bfloat16, device=cuda_device)
    db = torch.full((w.N,), 3.0, dtype=torch.bfloat16, device=cuda_device)
    mlaq.bwd_wgrad(dq, x, d["cos"], d["sin"], w.H, w.Dn, w.Dr, dW=dW, db=db)
    torch.cuda.synchronize()
    assert (dW == 0).all() and (db == 0).all()


def test_bwd_canaries_untouched(cuda_device):
    w = synth.workload("tiny", T=150, H=6)
    inp, d = _dev_inputs(w, 6, cuda_device)
    pad = 2048
    dxb = torch.full((w.T * w.K + 2 * pad,), 9.0, dtype=torch.bfloat16, device=cuda_device)
    dWb = torch.full((w.N * w.K + 2 * pad,), 9.0, dtype=torch.bfloat16, device=cuda_device)
    dbb = torch.full((w.N + 2 * pad,), 9.0, dtype=torch.bfloat16, device=cuda_device)
    mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                   dx=dxb[pad:pad + w.T * w.K].view(w.T, w.K))
    mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                   dW=dWb[pad:pad + w.N * w.K].view(w.N, w.K), db=dbb[pad:pad + w.N])
    torch.cuda.synchronize()
    for buf, n in ((dxb, w.T * w.K), (dWb, w.N * w.K), (dbb, w.N)):
        assert (buf[:pad] == 9.0).all() and (buf[pad + n:] == 9.0).all()


@pytest.mark.parametrize("name,ov", [("tiny", dict(T=64)),                          # fused paths
                                     ("dsv3_bwd", dict(T=300, H=4, seq_len=None))])  # pre-rotated dgrad, hand-off wgrad
def test_bwd_position_out_of_range_reports_status(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=7)
    inp["pos"] = inp["pos"].clone()
    inp["pos"][5] = -1
    d = helpers.to_dev(inp, cuda_device)
    rope = torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=cuda_device)
    for which in ("dgrad", "wgrad"):
        st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        if which == "dgrad":
            mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                           dq_pre_rope=rope)
        else:
            mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
        assert int(st.item()) == mlaq.STATUS["MLA_ERR_POS_RANGE"], which


def test_bwd_full_size(cuda_device):
    """DeepSeek-V3 backward shape (T = 2 x 4096, pos = t mod 4096, K=1536,
    H=128, bias on) in the benchmark's calls (dgrad storing the rotated rope
    channels, wgrad reading them): every element of dx, dW, db and of the
    stored rope channels against the oracle."""
    w = synth.workload("dsv3_bwd")
    inp, d = _dev_inputs(w, 0, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    rope = torch.full((w.T, w.H, w.Dr), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                        dq_pre_rope=rope)
    dW, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                            status=st, dq_pre_rope=rope)
    mlaq.check_status(st)
    helpers.check_bwd_all(inp, w, dx=dx, dW=dW, db=db, rope=rope, tol=TOL)


def test_dgrad_split_reduction(cuda_device):
    """Few tiles for many SMs: dgrad splits each tile's channel reduction,
    writes fp32 partials to the workspace and adds them in a fixed order.
    Sampled tokens against the oracle; two runs are bit-identical; a
    workspace smaller than the least the query reports (which = 4) is
    rejected."""
    import ctypes
    w = synth.workload("dsv3_bwd", T=1024, seq_len=None)
    inp, d = _dev_inputs(w, 9, cuda_device)
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 1)
    assert need > 0  # this shape splits
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dx1 = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
    ws = torch.empty((need,), dtype=torch.uint8, device=cuda_device)
    dx2 = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                         workspace=ws)
    mlaq.check_status(st)
    assert torch.equal(dx1, dx2)
    toks = np.sort(np.random.default_rng(2).choice(w.T, 16, replace=False))
    dqp = oracle.rope_bwd(helpers.f64(inp["dq"][torch.from_numpy(toks)]), w.H, w.Dn, w.Dr,
                          inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()[toks])
    ref = oracle.dgrad(dqp.reshape(len(toks), -1), helpers.f64(inp["W"]))
    assert helpers.frob_rel(dx1[torch.from_numpy(toks).to(cuda_device)], ref) <= TOL
    least = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 4)
    assert 0 < least <= need
    small = torch.empty((least - 16,), dtype=torch.uint8, device=cuda_device)
    with pytest.raises(mlaq.MlaError) as ei:
        mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], workspace=small)
    assert ei.value.status == mlaq.STATUS["MLA_ERR_WORKSPACE"]


@pytest.mark.parametrize("ov", [
    dict(T=3000, seq_len=None),                 # ragged last token tile, split tiles with one later part
    dict(T=300, seq_len=None),                  # 24 groups of 32 K steps: an owner adds 11 partial tiles
    dict(T=2048, K=256, H=16, seq_len=512),     # one column tile: 12 groups, positions restart
])
def test_dgrad_stream_k_schedules(cuda_device, ov):
    """dgrad's stream-K schedule on shapes whose tiles split between groups in
    different ways: every dx element against the oracle, two runs
    bit-identical (the owner adds the parts in a fixed order), and the same
    bits with the rotated rope channels kept in the workspace or handed out
    through dq_pre_rope."""
    w = synth.workload("dsv3_bwd", **ov)
    inp, d = _dev_inputs(w, 17, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 1)
    ws = torch.empty((need,), dtype=torch.uint8, device=cuda_device)
    args = (d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    dx1 = mlaq.bwd_dgrad(*args, pos=d["pos"], status=st, workspace=ws)
    dx2 = mlaq.bwd_dgrad(*args, pos=d["pos"], status=st, workspace=ws)
    rope = torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=cuda_device)
    dx3 = mlaq.bwd_dgrad(*args, pos=d["pos"], status=st, dq_pre_rope=rope)
    mlaq.check_status(st)
    assert torch.equal(dx1, dx2) and torch.equal(dx1, dx3)
    helpers.check_bwd_all(inp, w, dx=dx1, rope=rope, tol=TOL)
