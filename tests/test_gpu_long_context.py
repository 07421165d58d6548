"""GPU parity of the long-context step at its full size.

Four packed 4096-token sequences (T = 16384, positions restart at every
4096), the DeepSeek-V3 query up-projection shape (K = 1536, H = 128,
Dn = 128, Dr = 64) and a YaRN context-extension table (factor 40, original
length 4096, beta_fast 32, beta_slow 1, amplitude 1.0). The step runs in the
same calls and the same launch configuration that the benchmark times:
- the forward with MXFP8 output into caller buffers;
- dgrad storing the rotated rope channels;
- wgrad reading them, with no bias gradient.

Every element is checked against the fp64 oracle:
- the forward's codes and scales, with the MXFP8 bar (>= 99.9% of the
  scale bytes identical, every element within one E4M3 step);
- the stored rope channels, within the bf16 bound;
- dx and dW, within the backward's relative Frobenius bound (5e-3).
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


def test_long_context_step_full_size(cuda_device):
    w = synth.workload("dsv3_long_yarn")
    assert (w.T, w.seq_len, w.table) == (16384, 4096, "yarn")
    inp = synth.make_inputs(w, seed=21)
    d = helpers.to_dev(inp, cuda_device)
    dev = cuda_device
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    qc = torch.empty((w.T, w.H, w.D), dtype=torch.uint8, device=dev)
    qs = torch.empty((w.T, w.H, (w.D + 31) // 32), dtype=torch.uint8, device=dev)
    dx = torch.empty((w.T, w.K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
    rope = torch.full((w.T, w.H, w.Dr), float("nan"), dtype=torch.bfloat16, device=dev)

    mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
             out_mode="mxfp8", q_out=qc, q_scales=qs, status=st)
    mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                   dx=dx, status=st, dq_pre_rope=rope)
    _, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                           dW=dW, db=None, status=st, dq_pre_rope=rope)
    torch.cuda.synchronize()
    mlaq.check_status(st)
    assert db is None
    assert not torch.isnan(rope.float()).any(), "rope channels left unwritten"

    cos, sin, pos = inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy()
    assert cos.shape == (4096, w.Dr) and pos.max() == 4095

    helpers.check_fwd_all_tokens(inp, w, codes=qc, scales=qs)
    helpers.check_bwd_all(inp, w, dx=dx, dW=dW, rope=rope, tol=TOL)
