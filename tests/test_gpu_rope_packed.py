"""The packed rotary table (mla_rope_table_pack) and the forward that reads
it (mla_q_uproj_fwd_packed).

The table is the per-position cos/sin cache of Megatron-LM PR "Fix fused
MLA YaRN RoPE query kernel corrupting upstream tensor in-place" (Problem
section: a table at least as wide as the rotary dim), re-laid out so the
forward's epilogue reads it fast. Packing is a copy: every entry is
compared with the input tables bit for bit. The forward on the packed table
must give the same bytes as the forward on the plain one (checked against
the fp64 oracle by test_gpu_fwd and test_gpu_fwd_mxfp8w), in every weight
and output mode, and report out-of-range positions the same way.
"""
import numpy as np
import pytest
import torch

import helpers
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,width,Dr", [(256, 16, 16), (100, 72, 64), (4096, 64, 64), (7, 40, 32)])
def test_pack_is_a_bitwise_relayout(cuda_device, rows, width, Dr):
    g = torch.Generator().manual_seed(rows + width)
    cos = torch.randn((rows, width), generator=g)
    sin = torch.randn((rows, width), generator=g)
    packed = mlaq.rope_table_pack(cos.to(cuda_device), sin.to(cuda_device), Dr).cpu().numpy()
    h = Dr // 2
    c, s = cos.numpy(), sin.numpy()
    ref = np.stack([c[:, :h].T, s[:, :h].T, c[:, h:Dr].T, s[:, h:Dr].T], axis=2)  # [h, rows, 4]
    assert packed.shape == (h, rows, 4)
    assert np.array_equal(packed.view(np.uint32), ref.astype(np.float32).view(np.uint32))


MODES = [
    ("tiny", dict(), "bf16", "mxfp8"),
    ("tiny", dict(T=300, K=200, H=6), "bf16", "bf16"),
    ("dsv3_fwd_bf16w", dict(T=300, H=8), "bf16", "mxfp8"),
    ("dsv3_fwd_bf16w", dict(T=260, H=4, bias=True), "bf16", "mxfp8_bhsd"),
    ("dsv3_fwd_bf16w", dict(T=200, H=4), "bf16", "mxfp8_bhsd_swizzled"),
    ("dsv3_long_yarn", dict(T=520, H=4), "bf16", "mxfp8"),            # YaRN table, positions t mod 4096
    ("tiny", dict(T=130, K=64, H=16, Dn=64, Dr=32), "bf16", "bf16"),  # Dr = 32
    ("dsv3_fwd_mxfp8w", dict(T=260, H=4), "mxfp8", "mxfp8"),
    ("dsv3_fwd_mxfp8w", dict(T=140, H=2, K=1024, bias=True), "mxfp8", "bf16"),
]


@pytest.mark.parametrize("name,ov,wmode,omode", MODES)
def test_packed_forward_same_bytes(cuda_device, name, ov, wmode, omode):
    w = synth.workload(name, **ov)
    inp = synth.make_inputs(w, seed=17)
    d = helpers.to_dev(inp, cuda_device)
    x, W, kw = d["x"], d["W"], {}
    if wmode == "mxfp8":
        x, kw["x_scales"] = mlaq.mxfp8_quantize_rows(d["x"])
        W, kw["w_scales"] = mlaq.mxfp8_quantize_rows(d["W"])
    packed = mlaq.rope_table_pack(d["cos"], d["sin"], w.Dr)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (x, W, d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw.update(bias=d.get("b"), pos=d["pos"], weight_mode=wmode, out_mode=omode, status=st)
    a = mlaq.fwd(*args, **kw)
    b = mlaq.fwd(*args, rope_packed=packed, **kw)
    mlaq.check_status(st)
    a = a if isinstance(a, tuple) else (a,)
    b = b if isinstance(b, tuple) else (b,)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_packed_forward_full_size_same_bytes(cuda_device):
    """The long-context step's forward (T = 16384, YaRN, MXFP8 q) as the
    benchmark runs it, plain and packed tables: the same bytes."""
    w = synth.workload("dsv3_long_yarn")
    inp = synth.make_inputs(w, seed=3, want=("x", "W", "tables", "pos"))
    d = helpers.to_dev(inp, cuda_device)
    packed = mlaq.rope_table_pack(d["cos"], d["sin"], w.Dr)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    c1, s1 = mlaq.fwd(*args, pos=d["pos"], status=st)
    c2, s2 = mlaq.fwd(*args, pos=d["pos"], status=st, rope_packed=packed)
    mlaq.check_status(st)
    assert torch.equal(c1, c2) and torch.equal(s1, s2)


def test_packed_forward_position_out_of_range(cuda_device):
    w = synth.workload("tiny", T=64)
    inp = synth.make_inputs(w, seed=5)
    d = helpers.to_dev(inp, cuda_device)
    pos = d["pos"].clone()
    pos[9] = d["cos"].shape[0]  # one past the table
    packed = mlaq.rope_table_pack(d["cos"], d["sin"], w.Dr)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mlaq.fwd(d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr, bias=d["b"], pos=pos, status=st,
             rope_packed=packed)
    torch.cuda.synchronize()
    assert int(st.item()) == mlaq.STATUS["MLA_ERR_POS_RANGE"]
