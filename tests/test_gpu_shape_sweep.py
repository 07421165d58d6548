"""GPU parity over a seeded sweep of shapes (beyond the hand-picked cases of
the other files): random T, K, H, Dn, Dr, positions restarting or not, bias
on or off. Each shape runs the forward (bf16 and MXFP8 out; MXFP8 weights,
row-major and pre-tiled scales, where K allows), the backward (dgrad and
wgrad, with and without the rotated-rope hand-off) and, where its limits
allow, the MXFP8 backward, all against the fp64 oracle with the tolerances
the other files use. A shape the kernels do not tile must be rejected with
MLA_ERR_UNSUPPORTED (the documented limits), never computed wrongly.
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


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        Dr = int(rng.choice([16, 32, 64]))
        step = 64 if Dr == 64 else 32
        Dn = int(rng.integers(0, 4)) * step
        H = int(rng.integers(1, 10))
        K = int(rng.integers(1, 140)) * 8
        T = int(rng.integers(1, 600))
        seq = None if rng.random() < 0.5 else int(rng.integers(16, 300))
        bias = bool(rng.random() < 0.5)
        out.append(dict(T=T, K=K, H=H, Dn=Dn, Dr=Dr, seq_len=seq, bias=bias))
    return out


def _shapes_mx(n, seed):
    """Shapes inside the MXFP8 paths' limits more often: Dr 32 or 64, K a
    multiple of 128, an even number of heads."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        Dr = int(rng.choice([32, 64]))
        Dn = int(rng.integers(0, 4)) * 64
        H = 2 * int(rng.integers(1, 5))
        K = 128 * int(rng.integers(1, 10))
        T = int(rng.integers(1, 700))
        seq = None if rng.random() < 0.5 else int(rng.integers(16, 300))
        out.append(dict(T=T, K=K, H=H, Dn=Dn, Dr=Dr, seq_len=seq, bias=bool(rng.random() < 0.5)))
    return out


SHAPES = _shapes(16, 2024) + _shapes_mx(12, 7)


def _unsupported(e):
    return isinstance(e, mlaq.MlaError) and e.status == mlaq.STATUS["MLA_ERR_UNSUPPORTED"]


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_sweep(cuda_device, i):
    ov = SHAPES[i]
    w = synth.workload("tiny", x_std=1.0, w_std=0.05, dq_std=1.0, **ov)
    inp = synth.make_inputs(w, seed=100 + i)
    d = helpers.to_dev(inp, cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw = dict(bias=d.get("b"), pos=d["pos"], status=st)

    # forward, bf16 weights
    q = mlaq.fwd(*args, out_mode="bf16", **kw)
    codes, scales = mlaq.fwd(*args, out_mode="mxfp8", **kw)
    mlaq.check_status(st)
    q_ref, rc, rs = helpers.oracle_forward(inp, w, quantize=True)
    helpers.check_bf16_close(q, q_ref)
    helpers.check_mxfp8_close(codes.cpu().numpy(), scales.cpu().numpy(), q_ref, rc, rs)

    # forward, MXFP8 weights (K % 128 == 0): row-major and pre-tiled scales agree bit for bit
    if w.K % 128 == 0:
        xq, xs = mlaq.mxfp8_quantize_rows(d["x"])
        Wq, Ws = mlaq.mxfp8_quantize_rows(d["W"])
        fa = (xq, Wq, d["cos"], d["sin"], w.H, w.Dn, w.Dr)
        try:
            c1, s1 = mlaq.fwd(*fa, weight_mode="mxfp8", x_scales=xs, w_scales=Ws, **kw)
        except mlaq.MlaError as e:
            assert _unsupported(e) and mlaq.w_scale_group(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr) == 0
        else:
            G = mlaq.w_scale_group(w.T, w.K, w.H, w.Dn, w.Dr, w.cs_rows, w.Dr)
            _, xst = mlaq.mxfp8_quantize_rows(d["x"], group=128)
            _, Wst = mlaq.mxfp8_quantize_rows(d["W"], group=G)
            c2, s2 = mlaq.fwd(*fa, weight_mode="mxfp8_tiled", x_scales=xst, w_scales=Wst, **kw)
            mlaq.check_status(st)
            assert torch.equal(c1, c2) and torch.equal(s1, s2)
            x_deq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(helpers.f64(inp["x"])))
            W_deq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(helpers.f64(inp["W"])))
            b = helpers.f64(inp["b"]) if inp.get("b") is not None else None
            qm, rcm, rsm = oracle.forward(x_deq, W_deq, w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                                          inp["pos"].numpy(), b, quantize=True)
            helpers.check_mxfp8_close(c1.cpu().numpy(), s1.cpu().numpy(), qm, rcm, rsm)

    # backward (Dn % Dr == 0), with and without the hand-off
    if w.Dn % w.Dr == 0:
        g = oracle.backward(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]), w.H, w.Dn,
                            w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy())
        rope = torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=cuda_device)
        dx = mlaq.bwd_dgrad(d["dq"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st,
                            dq_pre_rope=rope)
        dW_h, db_h = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"],
                                    status=st, dq_pre_rope=rope)
        dW, db = mlaq.bwd_wgrad(d["dq"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, pos=d["pos"], status=st)
        mlaq.check_status(st)
        assert torch.equal(dW_h, dW)
        for name, got in (("dx", dx), ("dW", dW), ("db", db), ("db_h", db_h)):
            err = helpers.frob_rel(got, g[name[:2]])
            assert err <= TOL, f"{name}: {err}"

    # MXFP8 backward where its limits allow
    if w.Dr in (32, 64) and w.D % 32 == 0 and w.N % 128 == 0 and w.K % 32 == 0 and w.Dn % w.Dr == 0:
        cs = d["cos"].shape
        try:
            need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, cs[0], cs[1], 3)
            ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=cuda_device)
            mdx, mdW, mdb = mlaq.bwd_mxfp8(d["dq"], d["W"], d["x"], d["cos"], d["sin"], w.H, w.Dn, w.Dr,
                                           pos=d["pos"], status=st, workspace=ws)
        except mlaq.MlaError as e:
            assert _unsupported(e)
        else:
            mlaq.check_status(st)
            gm = oracle.backward_mxfp8(helpers.f64(inp["dq"]), helpers.f64(inp["x"]), helpers.f64(inp["W"]),
                                       w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                                       inp["pos"].numpy())
            for name, got in (("dx", mdx), ("dW", mdW), ("db", mdb)):
                err = helpers.frob_rel(got, gm[name])
                assert err <= 2.0 ** -8, f"MXFP8 {name}: {err}"
