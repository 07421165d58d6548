"""The failure-detection contract on the device: a pipeline wait that can
never complete gives up after its time limit, the CTA's other role leaves
through the abort flag, MLA_ERR_TIMEOUT reaches the host in the status word,
and the context stays usable.

mla_wait_selftest runs the kernels' own bounded-wait routine on an mbarrier
that nothing arrives at (no copy or MMA is in flight), so the wait runs out
without any fault.
"""
import pytest
import torch

import helpers
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu
S = mlaq.STATUS


def _timed(fn):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def test_wait_completes_when_filled(cuda_device):
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ms = _timed(lambda: mlaq.wait_selftest(True, 50.0, st))
    assert int(st.item()) == S["MLA_OK"]
    assert ms < 25.0, f"a filled barrier still waited {ms:.1f} ms"


def test_wait_gives_up_and_reports(cuda_device):
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ms = _timed(lambda: mlaq.wait_selftest(False, 50.0, st))
    assert int(st.item()) == S["MLA_ERR_TIMEOUT"]
    # role 0 gives up at 50 ms; role 1 leaves through the abort flag, well
    # before its own 100 ms limit
    assert 50.0 <= ms < 90.0, f"{ms:.1f} ms"
    with pytest.raises(mlaq.MlaError):
        mlaq.check_status(st)
    # the status word keeps the first error: a later success leaves it set
    mlaq.wait_selftest(True, 50.0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == S["MLA_ERR_TIMEOUT"]


def test_context_usable_after_timeout(cuda_device):
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mlaq.wait_selftest(False, 10.0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == S["MLA_ERR_TIMEOUT"]
    w = synth.workload("tiny")
    inp = synth.make_inputs(w, seed=3)
    d = helpers.to_dev(inp, cuda_device)
    st2 = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    q = mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], bias=d["b"],
                 out_mode="bf16", status=st2)
    mlaq.check_status(st2)
    helpers.check_bf16_close(q, helpers.oracle_forward(inp, w))


def test_flag_wait_completes_when_raised(cuda_device):
    """The cross-CTA flag wait of dgrad's stream-K owners: a raised flag ends
    the wait at once, nothing is reported."""
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ms = _timed(lambda: mlaq.wait_selftest_flag(True, 50.0, st))
    assert int(st.item()) == S["MLA_OK"]
    assert ms < 25.0, f"a raised flag still waited {ms:.1f} ms"


def test_flag_wait_gives_up_and_reports(cuda_device):
    """A flag nothing raises: the wait gives up at its limit, the other role
    leaves through the abort flag, MLA_ERR_TIMEOUT reaches the host, and the
    context stays usable (a dgrad afterwards matches the oracle)."""
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ms = _timed(lambda: mlaq.wait_selftest_flag(False, 50.0, st))
    assert int(st.item()) == S["MLA_ERR_TIMEOUT"]
    assert 50.0 <= ms < 90.0, f"{ms:.1f} ms"
    w = synth.workload("dsv3_bwd", T=300, H=8, seq_len=None)
    inp = synth.make_inputs(w, seed=19)
    d = helpers.to_dev(inp, cuda_device)
    st2 = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st2)
    mlaq.check_status(st2)
    import oracle
    g = oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn, w.Dr,
                        inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy())
    assert helpers.frob_rel(dx, g["dx"]) <= 5e-3
