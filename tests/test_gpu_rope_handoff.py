"""GPU parity of the rotated-rope hand-off from dgrad to wgrad.

TransformerEngine PR "Add a backwards linear function to be used with the
fused mla q up-proj", sequence diagram: one RoPE backward (dq -> dq_pre)
feeds both linear-backward products. dgrad rotates dq's rope channels in its
operand path anyway; it can store them (dq_pre_rope [T, H, Dr], bf16, the
values its tensor cores consume) and wgrad then reads them instead of
rotating dq again.

Checks: the stored channels equal the oracle's inverse rotation within the
bf16 tolerance (|err| <= 8e-3 |ref| + 2e-3 rms(ref)); dx is unchanged by
storing them; dW from the hand-off is bit-identical to dW from wgrad's own
rotation (same operand bits, same accumulation order); db stays within the
backward tolerance (its fp32 partial sums are grouped by stage, and the
stages differ in size).
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
    ("tiny", {}),                                             # Dr = 16: wgrad rotates itself
    ("tiny", dict(T=130, K=64, H=16, Dn=64, Dr=32)),          # Dr = 32: likewise
    ("dsv3_bwd", dict(T=300, H=8, seq_len=None)),             # head pairs, ragged tokens
    ("dsv3_bwd", dict(T=260, K=1000, H=6, seq_len=128)),      # ragged K, positions restart
    ("dsv3_bwd", dict(T=1024, seq_len=None)),                 # dgrad splits its reduction
    ("dsv3_long_yarn", dict(T=200, H=4, seq_len=None)),       # YaRN table
    ("dsv3_bwd", dict(T=64, H=2, seq_len=None)),              # one head pair, one stage
]


def _run(w, seed, dev):
    inp = synth.make_inputs(w, seed=seed)
    d = helpers.to_dev(inp, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rope = torch.full((w.T, w.H, w.Dr), float("nan"), dtype=torch.bfloat16, device=dev)
    dx_h = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                          dq_pre_rope=rope)
    dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
    dW_h, db_h = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                                status=st, dq_pre_rope=rope)
    dW, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
    torch.cuda.synchronize()
    mlaq.check_status(st)
    return inp, dict(rope=rope, dx_h=dx_h, dx=dx, dW_h=dW_h, db_h=db_h, dW=dW, db=db)


@pytest.mark.parametrize("name,ov", SHAPES)
def test_rope_handoff(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp, r = _run(w, 5, cuda_device)
    dqp = oracle.rope_bwd(helpers.f64(inp["dq"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                          inp["pos"].numpy())
    helpers.check_bf16_close(r["rope"], dqp[:, :, w.Dn:], what="dq_pre_rope")
    assert torch.equal(r["dx_h"], r["dx"]), "storing the rope channels changed dx"
    assert torch.equal(r["dW_h"], r["dW"]), "dW differs between the hand-off and wgrad's own rotation"
    ref_db = oracle.bgrad(dqp.reshape(w.T, -1))
    for got in (r["db_h"], r["db"]):
        assert helpers.frob_rel(got, ref_db) <= TOL


def test_rope_handoff_full_size(cuda_device):
    """DeepSeek-V3 backward shape at T = 4096 (the training step's size):
    dW bit-identical both ways (compared whole, on the device), the stored
    rope channels against the oracle on 16 sampled tokens, db on all channels
    within tolerance of wgrad's own rotation."""
    w = synth.workload("dsv3_bwd", T=4096, seq_len=None)
    inp, r = _run(w, 6, cuda_device)
    assert torch.equal(r["dW_h"], r["dW"])
    assert torch.equal(r["dx_h"], r["dx"])
    toks = np.sort(np.random.default_rng(3).choice(w.T, 16, replace=False))
    dqp = oracle.rope_bwd(helpers.f64(inp["dq"][torch.from_numpy(toks)]), w.H, w.Dn, w.Dr,
                          inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()[toks])
    helpers.check_bf16_close(r["rope"][torch.from_numpy(toks).to(cuda_device)], dqp[:, :, w.Dn:],
                             what="dq_pre_rope")
    assert not torch.isnan(r["rope"].float()).any()
    assert helpers.frob_rel(r["db_h"], helpers.bf16_to_f64(r["db"])) <= 1e-3


def test_dgrad_paths_agree(cuda_device):
    """The two dgrad paths: with the least workspace (mla_q_uproj_workspace_size
    which = 4) dgrad rotates inside its GEMM (fused transform); with the full
    one (which = 1) it rotates the rope channels in a pass of their own and
    runs a plain GEMM over them. Both store the same rotated bits and both
    dx agree with the oracle (their fp32 accumulation orders differ)."""
    w = synth.workload("dsv3_bwd", T=1024, seq_len=None)
    inp = synth.make_inputs(w, seed=8)
    d = helpers.to_dev(inp, cuda_device)
    cs = d["cos"].shape
    least = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, cs[0], cs[1], 4)
    full = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, cs[0], cs[1], 1)
    assert 0 < least < full
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    outs = {}
    for name, n in (("fused", least), ("pre", full)):
        rope = torch.full((w.T, w.H, w.Dr), float("nan"), dtype=torch.bfloat16, device=cuda_device)
        ws = torch.empty((n,), dtype=torch.uint8, device=cuda_device)
        dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                            workspace=ws, dq_pre_rope=rope)
        outs[name] = (dx, rope)
    torch.cuda.synchronize()
    mlaq.check_status(st)
    assert torch.equal(outs["fused"][1], outs["pre"][1]), "the two paths rotated differently"
    dqp = oracle.rope_bwd(helpers.f64(inp["dq"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                          inp["pos"].numpy()).reshape(w.T, -1)
    ref = oracle.dgrad(dqp, helpers.f64(inp["W"]))
    for name, (dx, _) in outs.items():
        assert helpers.frob_rel(dx, ref) <= TOL, name
    assert helpers.frob_rel(outs["pre"][0], helpers.bf16_to_f64(outs["fused"][0])) <= 2e-3


def test_handoff_wgrad_without_bias(cuda_device):
    """The hand-off wgrad's bias warps share each stage's release with the
    MMA: asking for no db gives the same dW bits and leaves db's buffer
    alone."""
    w = synth.workload("dsv3_bwd", T=300, H=4, seq_len=None)
    inp = synth.make_inputs(w, seed=9)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    rope = torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=cuda_device)
    mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st, dq_pre_rope=rope)
    dW_b, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                              dq_pre_rope=rope)
    dW_n, none = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                                dq_pre_rope=rope, db=None)
    torch.cuda.synchronize()
    mlaq.check_status(st)
    assert none is None
    assert torch.equal(dW_b, dW_n)
    dqp = oracle.rope_bwd(helpers.f64(inp["dq"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                          inp["pos"].numpy())
    assert helpers.frob_rel(db, oracle.bgrad(dqp.reshape(w.T, -1))) <= TOL
