"""mla_q_uproj_bwd_dgrad_noalloc: the dgrad entry point for callers that
cannot allocate device memory (a framework that lends a plugin only the
tensors of a call, or a path that cannot afford cudaMalloc's implicit
synchronization). It takes no workspace: its split-reduction partials live
in a fixed scratch array inside the library.

Checked through the C ABI against mla_q_uproj_bwd_dgrad (the entry point
that takes a caller-allocated workspace) on two calls in a row: within the
backward tolerance the other tests use (relative Frobenius error <= 5e-3),
and bit for bit when the allocating call's fastest workspace also fits in
the scratch (then both take the same path with the same schedule). This
file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import helpers
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu
TOL = 5e-3
SCRATCH_BYTES = 64 * 1024 * 1024  # MLA_NOALLOC_SCRATCH_BYTES in include/mlaq.h


def _noalloc_fn():
    f = mlaq.lib().mla_q_uproj_bwd_dgrad_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(mlaq.Shape)] + [ctypes.c_void_p] * 9
    return f


def _call_noalloc(w, d, dx, st):
    s = mlaq.Shape(T=w.T, K=w.K, H=w.H, Dn=w.Dn, Dr=w.Dr, reserved=0, cs_rows=d["cos"].shape[0],
                   cs_width=d["cos"].shape[1])
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    return _noalloc_fn()(ctypes.byref(s), p(d["dq"]), p(d["W"]), p(d["cos"]), p(d["sin"]), p(d["pos"]),
                         p(dx), None, p(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_dgrad_matches_workspace_dgrad(cuda_device):
    # 1024 tokens at the DeepSeek-V3 shape: dgrad splits its reduction here,
    # so the scratch array is really used (partials of about 19 MB)
    w = synth.workload("dsv3_bwd", T=1024, seq_len=None)
    inp = synth.make_inputs(w, seed=11)
    d = helpers.to_dev(inp, cuda_device)
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 4)  # the least dgrad takes
    assert 0 < need <= SCRATCH_BYTES
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ref = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
    # the allocating call takes its fastest path; when that workspace fits in
    # the scratch, the allocation-free call takes the same one
    same_path = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 1) <= SCRATCH_BYTES
    ref64 = helpers.bf16_to_f64(ref)
    for call in range(2):  # the scratch keeps the previous call's contents
        dx = torch.full((w.T, w.K), float("nan"), dtype=torch.bfloat16, device=cuda_device)
        rc = _call_noalloc(w, d, dx, st)
        assert rc == 0, mlaq.status_string(rc)
        torch.cuda.synchronize()
        mlaq.check_status(st)
        err = helpers.frob_rel(dx, ref64)
        assert err <= TOL, f"call {call}: relative Frobenius error {err:.3e}"
        assert not torch.isnan(dx.float()).any()
        if same_path:
            assert torch.equal(dx, ref), f"call {call}: not bit-identical on the same path"


def test_noalloc_dgrad_rejects_shapes_beyond_scratch(cuda_device):
    w = synth.workload("dsv3_bwd", T=4096, seq_len=None)
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr, 4)
    if need <= SCRATCH_BYTES:
        pytest.skip("this device splits the shape into partials that fit the scratch")
    d = helpers.to_dev(synth.make_inputs(synth.workload("dsv3_bwd", T=4096, seq_len=None, H=128),
                                         seed=12, want=("dq", "W", "tables", "pos")), cuda_device)
    dx = torch.empty((w.T, w.K), dtype=torch.bfloat16, device=cuda_device)
    rc = _call_noalloc(w, d, dx, None)
    assert rc == mlaq.STATUS["MLA_ERR_WORKSPACE"]
