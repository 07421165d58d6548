"""The autograd face (TransformerEngine PR "Add a backwards linear function to
be used with the fused mla q up-proj": an autograd function whose backward
is the RoPE backward then the linear backward with the saved input).

q and the gradients of L = sum(q * G) against the oracle (q within the bf16
tolerance, gradients within relative Frobenius 5e-3), including the cases
where only some inputs need a gradient.
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
import synth
from up_proj_gemm_gb300.autograd import q_up_proj

pytestmark = pytest.mark.gpu
TOL = 5e-3


def _case(name, ov, dev, seed):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=seed)
    d = helpers.to_dev(inp, dev)
    return w, inp, d


@pytest.mark.parametrize("name,ov", [
    ("tiny", {}),
    ("dsv3_bwd", dict(T=300, H=4, seq_len=None)),
])
def test_autograd_matches_oracle(cuda_device, name, ov):
    w, inp, d = _case(name, ov, cuda_device, 21)
    x = d["x"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    b = d["b"].clone().requires_grad_(True) if d.get("b") is not None else None
    q = q_up_proj(x, W, d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=b, pos=d["pos"])
    G = d["dq"]  # the upstream gradient
    (q.float() * G.float()).sum().backward()
    cos, sin, pos = inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()
    bias = helpers.f64(inp["b"]) if inp.get("b") is not None else None
    q_ref = oracle.forward(helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn, w.Dr, cos, sin, pos, bias)
    helpers.check_bf16_close(q.detach(), q_ref, what="q")
    g = oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn, w.Dr,
                        cos, sin, pos)
    assert helpers.frob_rel(x.grad, g["dx"]) <= TOL
    assert helpers.frob_rel(W.grad, g["dW"]) <= TOL
    if b is not None:
        assert helpers.frob_rel(b.grad, g["db"]) <= TOL


def test_autograd_partial_gradients(cuda_device):
    w, inp, d = _case("dsv3_bwd", dict(T=200, H=2, seq_len=None), cuda_device, 22)
    cos, sin, pos = inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()
    g = oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn, w.Dr,
                        cos, sin, pos)
    # frozen weight: only dx
    x = d["x"].clone().requires_grad_(True)
    q = q_up_proj(x, d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"])
    q.backward(d["dq"])
    assert helpers.frob_rel(x.grad, g["dx"]) <= TOL
    # frozen input: only dW (wgrad rotates dq itself)
    W = d["W"].clone().requires_grad_(True)
    q = q_up_proj(d["x"], W, d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"])
    q.backward(d["dq"])
    assert helpers.frob_rel(W.grad, g["dW"]) <= TOL


@pytest.mark.parametrize("out_mode", ["mxfp8", "mxfp8_bhsd", "mxfp8_bhsd_swizzled"])
def test_mxfp8_query_face(cuda_device, out_mode):
    """q_up_proj_mxfp8: the MXFP8 query is the forward's own output for that
    mode (bytes equal to the plain call), and query.backward(dq) with a bf16
    dq gives the gradients of the bf16 face (which the test above checks
    against the oracle), bit for bit."""
    from up_proj_gemm_gb300 import fwd
    from up_proj_gemm_gb300.autograd import q_up_proj_mxfp8
    w, inp, d = _case("dsv3_bwd", dict(T=260, H=4, seq_len=None), cuda_device, 23)
    xa = d["x"].clone().requires_grad_(True)
    Wa = d["W"].clone().requires_grad_(True)
    ba = d["b"].clone().requires_grad_(True)
    qm = q_up_proj_mxfp8(xa, Wa, d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=ba, pos=d["pos"], out_mode=out_mode)
    codes, scales = fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=d["b"], pos=d["pos"],
                        out_mode=out_mode)
    assert torch.equal(qm.codes, codes) and torch.equal(qm.scales, scales)
    assert not qm.codes.requires_grad and qm.anchor.requires_grad
    qm.backward(d["dq"])
    xb = d["x"].clone().requires_grad_(True)
    Wb = d["W"].clone().requires_grad_(True)
    bb = d["b"].clone().requires_grad_(True)
    q = q_up_proj(xb, Wb, d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=bb, pos=d["pos"])
    q.backward(d["dq"])
    torch.cuda.synchronize()
    assert torch.equal(xa.grad, xb.grad) and torch.equal(Wa.grad, Wb.grad) and torch.equal(ba.grad, bb.grad)
    with pytest.raises(ValueError):
        qm.backward(d["dq"].float())
