"""The head-sharded query up-projection on two CPU ranks (gloo).

Head sharding (column-parallel W) follows from the method: heads are
independent in the forward (a rope pair and an MXFP8 block never leave a
head), and in the backward (TransformerEngine PR "Add a backwards linear
function to be used with the fused mla q up-proj", sequence diagram) dW and
db of a head need only that head's dq, while dx sums over all heads: one
all-reduce. The host-side logic of up_proj_gemm_gb300.sharded (the head
split, the slices each rank hands to its local calls, the dx all-reduce) is
run here by two gloo ranks whose local calls are the fp64 oracle; the
assembled results must equal the oracle's unsharded ones.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from up_proj_gemm_gb300 import sharded


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_ops():
    """The three local calls, computed by the oracle on CPU tensors (float64 out)."""
    import oracle
    import synth

    def f64(t):
        return oracle.decode_bf16(synth.bf16_bits(t)) if t.dtype == torch.bfloat16 else t.double().numpy()

    def fwd(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None, **kw):
        q = oracle.forward(f64(x), f64(W), H, Dn, Dr, cos.numpy(), sin.numpy(),
                           None if pos is None else pos.numpy(), None if bias is None else f64(bias))
        return torch.from_numpy(q)

    def bwd_dgrad(dq, W, cos, sin, H, Dn, Dr, pos=None, dq_pre_rope=None):
        g = oracle.backward(f64(dq), np.zeros((dq.shape[0], W.shape[1])), f64(W), H, Dn, Dr, cos.numpy(),
                            sin.numpy(), None if pos is None else pos.numpy(), want=("dx",))
        return torch.from_numpy(g["dx"])

    def bwd_wgrad(dq, x, cos, sin, H, Dn, Dr, pos=None, db=False, dq_pre_rope=None):
        g = oracle.backward(f64(dq), f64(x), np.zeros((H * (Dn + Dr), x.shape[1])), H, Dn, Dr, cos.numpy(),
                            sin.numpy(), None if pos is None else pos.numpy(), want=("dW", "db"))
        return torch.from_numpy(g["dW"]), (torch.from_numpy(g["db"]) if db else None)

    return {"fwd": fwd, "bwd_dgrad": bwd_dgrad, "bwd_wgrad": bwd_wgrad}


def _case():
    import synth
    w = synth.workload("tiny", T=96, K=40, H=5, bias=True)  # 5 heads over 2 ranks: 3 + 2
    return w, synth.make_inputs(w, seed=8)


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo")
    w, inp = _case()
    sh = sharded.head_shard(w.H, rank, world)
    W_l, b_l = sharded.shard_weight(inp["W"], inp["b"], sh, w.D)
    ops = _oracle_ops()
    q_l = sharded.sharded_fwd(inp["x"], W_l, inp["cos"], inp["sin"], sh, w.Dn, w.Dr, bias_local=b_l,
                              pos=inp["pos"], ops=ops)
    dq_l = inp["dq"][:, sh.h0:sh.h1].contiguous()
    dx, dW_l, db_l = sharded.sharded_bwd(dq_l, inp["x"], W_l, inp["cos"], inp["sin"], sh, w.Dn, w.Dr,
                                         pos=inp["pos"], want_db=True, ops=ops)
    out.put((rank, sh.h0, sh.h1, q_l.numpy(), dx.numpy(), dW_l.numpy(), db_l.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_head_split_is_contiguous_and_balanced():
    for H in (1, 2, 5, 128):
        for world in range(1, min(H, 8) + 1):
            parts = [sharded.head_shard(H, r, world) for r in range(world)]
            assert parts[0].h0 == 0 and parts[-1].h1 == H
            assert all(a.h1 == b.h0 for a, b in zip(parts, parts[1:]))
            assert max(p.heads for p in parts) - min(p.heads for p in parts) <= 1
    with pytest.raises(ValueError):
        sharded.head_shard(2, 0, 3)


def test_two_rank_head_sharded_step_matches_unsharded_oracle():
    import oracle
    import synth
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=180) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w, inp = _case()
    f64 = lambda t: oracle.decode_bf16(synth.bf16_bits(t))
    q = oracle.forward(f64(inp["x"]), f64(inp["W"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(), inp["sin"].numpy(),
                       inp["pos"].numpy(), f64(inp["b"]))
    g = oracle.backward(f64(inp["dq"]), f64(inp["x"]), f64(inp["W"]), w.H, w.Dn, w.Dr, inp["cos"].numpy(),
                        inp["sin"].numpy(), inp["pos"].numpy())
    assert [r[1:3] for r in res] == [(0, 3), (3, 5)]
    for rank, h0, h1, q_l, dx, dW_l, db_l in res:
        rows = slice(h0 * w.D, h1 * w.D)
        assert np.allclose(q_l, q[:, h0:h1], rtol=1e-12, atol=1e-12)
        # dx: the partial sums of both ranks, all-reduced (the same on every rank)
        assert np.allclose(dx, g["dx"], rtol=1e-12, atol=1e-12)
        assert np.allclose(dW_l, g["dW"][rows], rtol=1e-12, atol=1e-12)
        assert np.allclose(db_l, g["db"][rows], rtol=1e-12, atol=1e-12)
    # one rank's heads alone do not give dx: the all-reduce is what completes it
    part0 = oracle.backward(f64(inp["dq"][:, :3].contiguous()), f64(inp["x"]), f64(inp["W"][:3 * w.D]), 3, w.Dn,
                            w.Dr, inp["cos"].numpy(), inp["sin"].numpy(), inp["pos"].numpy(), want=("dx",))["dx"]
    assert not np.allclose(part0, g["dx"], rtol=1e-3, atol=1e-3)
