"""The head-sharded path's local calls on the GPU: two shards of the heads
run one after the other on one device (their kernels never wait on each
other; the dx all-reduce is a host-ordered sum, done here by adding the two
partials), against the unsharded GPU calls and the fp64 oracle.

Head sharding follows from the method (TransformerEngine PR "Add a
backwards linear function to be used with the fused mla q up-proj",
sequence diagram): the forward and dW, db are per head; dx sums over heads.
"""
import pytest
import torch

import helpers
import oracle
import synth
import up_proj_gemm_gb300 as mlaq
from up_proj_gemm_gb300 import sharded

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.mark.parametrize("name,ov", [("dsv3_bwd", dict(T=520, H=6, seq_len=256)), ("tiny", dict(T=200, H=5))])
def test_two_head_shards_on_one_gpu(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=13)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    q_full = mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=d.get("b"), pos=d["pos"],
                      out_mode="bf16", status=st)
    partials, dWs, dbs = [], [], []
    for rank in range(2):
        sh = sharded.head_shard(w.H, rank, 2)
        W_l, b_l = sharded.shard_weight(d["W"], d.get("b"), sh, w.D)
        q_l = sharded.sharded_fwd(d["x"], W_l.contiguous(), d["cos"], d["sin"], sh, w.Dn, w.Dr,
                                  bias_local=None if b_l is None else b_l.contiguous(), pos=d["pos"],
                                  out_mode="bf16", status=st)
        # the forward of a head slice is the same bytes as that slice of the full forward
        assert torch.equal(q_l, q_full[:, sh.h0:sh.h1])
        dx_r, dW_l, db_l = sharded.sharded_bwd(d["dq"][:, sh.h0:sh.h1].contiguous(), d["x"], W_l.contiguous(),
                                               d["cos"], d["sin"], sh, w.Dn, w.Dr, pos=d["pos"],
                                               want_db=w.bias, all_reduce=lambda t, g: partials.append(t))
        dWs.append(dW_l)
        dbs.append(db_l)
    mlaq.check_status(st)
    dx = (partials[0].float() + partials[1].float()).to(torch.bfloat16)
    dW = torch.cat(dWs)
    g = oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn, w.Dr,
                        inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy())
    assert helpers.frob_rel(dx, g["dx"]) <= TOL
    assert helpers.frob_rel(dW, g["dW"]) <= TOL
    if w.bias:
        assert helpers.frob_rel(torch.cat(dbs), g["db"]) <= TOL
    # the shards' dW rows agree with the unsharded wgrad's (the kernels may tile the
    # two head counts differently, so compare values, not bytes)
    dW_full, _ = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], db=None)
    assert helpers.frob_rel(dW, helpers.bf16_to_f64(dW_full)) <= 1e-3
