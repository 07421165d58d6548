"""GPU parity of the long-context step at its full size.

Four packed 4096-token sequences (T = 16384, positions restart at every
4096), the DeepSeek-V3 query up-projection shape (K = 1536, H = 128,
Dn = 128, Dr = 64) and a YaRN context-extension table (factor 40, original
length 4096, beta_fast 32, beta_slow 1, amplitude 1.0). The step runs in the
same calls and the same launch configuration that the benchmark times:
- the forward with MXFP8 output into caller buffers;
- dgrad storing the rotated rope channels;
- wgrad reading them, with no bias gradient.

Outputs are checked against the fp64 oracle on samples it can compute one
at a time:
- the forward's codes and scales on sampled tokens, within one E4M3 step;
- the stored rope channels on sampled tokens, within the bf16 bound;
- dx on sampled tokens;
- dW on sampled heads over all 16384 tokens, within the backward's
  relative Frobenius bound (5e-3).
The samples always include the first and last token and both sides of every
sequence restart.
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


def _sample_tokens(T, seq, n, seed):
    """n random tokens plus the edges: 0, T-1 and seq-1, seq at each restart."""
    edges = [0, T - 1] + [t for s in range(seq, T, seq) for t in (s - 1, s)]
    rng = np.random.default_rng(seed)
    rest = rng.choice(T, n, replace=False)
    return np.unique(np.concatenate([np.array(edges), rest]))


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

    # forward: every channel of the sampled tokens
    toks = _sample_tokens(w.T, w.seq_len, 40, seed=2)
    idx = torch.from_numpy(toks).to(dev)
    q_ref, rc, rs = helpers.oracle_forward(inp, w, tokens=toks, quantize=True)
    helpers.check_mxfp8_close(qc[idx].cpu().numpy(), qs[idx].cpu().numpy(), q_ref, rc, rs)

    # dgrad: the stored rope channels and dx on the sampled tokens
    dqp_t = oracle.rope_bwd(helpers.f64(inp["dq"][torch.from_numpy(toks)]), w.H, w.Dn, w.Dr,
                            cos, sin, pos[toks])
    helpers.check_bf16_close(rope[idx], dqp_t[:, :, w.Dn:], what="dq_pre_rope")
    ref_dx = oracle.dgrad(dqp_t.reshape(len(toks), -1), helpers.f64(inp["W"]))
    assert helpers.frob_rel(dx[idx], ref_dx) <= TOL

    # wgrad: sampled heads over every token (a head's rows need only its own dq)
    heads = np.array([0, 45, 90, 127])
    dq_h = helpers.f64(inp["dq"][:, torch.from_numpy(heads)].contiguous())
    dqp_h = oracle.rope_bwd(dq_h, len(heads), w.Dn, w.Dr, cos, sin, pos).reshape(w.T, -1)
    ref_dW = oracle.wgrad(dqp_h, helpers.f64(inp["x"]))
    ch = (heads[:, None] * w.D + np.arange(w.D)[None, :]).reshape(-1)
    assert helpers.frob_rel(dW[torch.from_numpy(ch).to(dev)], ref_dW) <= TOL
