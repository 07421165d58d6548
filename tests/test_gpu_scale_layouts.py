"""GPU parity of the attention-ready scale layouts and of K/V quantization.

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant":
the query's MXFP8 scales in BHSD order (review thread), the GEMM scale
swizzle among the MXFP8 helpers, and K and V quantized separately with the
same helper. All bit-exact: they are byte permutations of, or the same rule
as, outputs already checked against the oracle.
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,ov", [("tiny", {}), ("dsv3_fwd_bf16w", dict(T=300, H=6))])
def test_bhsd_scales_are_the_head_major_transpose(cuda_device, name, ov):
    w = synth.workload(name, **ov)
    d = helpers.to_dev(synth.make_inputs(w, seed=31), cuda_device)
    args = (d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw = dict(bias=d.get("b"), pos=d["pos"])
    codes, sc = mlaq.fwd(*args, out_mode="mxfp8", **kw)
    codes_h, sc_h = mlaq.fwd(*args, out_mode="mxfp8_bhsd", **kw)
    torch.cuda.synchronize()
    assert tuple(sc_h.shape) == (w.H, w.T, (w.D + 31) // 32)
    assert torch.equal(codes_h, codes)
    assert torch.equal(sc_h, sc.transpose(0, 1).contiguous())


@pytest.mark.parametrize("name,ov", [("tiny", dict(T=130)), ("dsv3_fwd_bf16w", dict(T=300, H=6, bias=True)),
                                     ("dsv3_fwd_bf16w", dict(T=256, H=2, K=128))])
def test_swizzled_bhsd_scales_from_the_epilogue(cuda_device, name, ov):
    """out_mode mxfp8_bhsd_swizzled: the same codes as the other MXFP8 modes,
    and each head's [T, ceil(D/32)] scales in the GEMM's tiled order, i.e.
    the oracle's swizzle of the head-major scales, head after head, with the
    padding rows and columns written as 0 (the buffer starts filled with
    0xEE)."""
    w = synth.workload(name, **ov)
    d = helpers.to_dev(synth.make_inputs(w, seed=32), cuda_device)
    args = (d["x"], d["W"], d["cos"], d["sin"], w.H, w.Dn, w.Dr)
    kw = dict(bias=d.get("b"), pos=d["pos"])
    codes_h, sc_h = mlaq.fwd(*args, out_mode="mxfp8_bhsd", **kw)
    nb = (w.D + 31) // 32
    per_head = int(mlaq.lib().mxfp8_swizzled_scale_bytes(w.T, nb))
    assert per_head == -(-w.T // 128) * 128 * -(-nb // 4) * 4
    buf = torch.full((w.H, per_head), 0xEE, dtype=torch.uint8, device=cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    codes_s, sc_s = mlaq.fwd(*args, out_mode="mxfp8_bhsd_swizzled", q_scales=buf, status=st, **kw)
    mlaq.check_status(st)
    assert sc_s.data_ptr() == buf.data_ptr()
    assert torch.equal(codes_s, codes_h)
    sc_h, sc_s = sc_h.cpu().numpy(), sc_s.cpu().numpy()
    for h in range(w.H):
        assert np.array_equal(sc_s[h], oracle.mxfp8_swizzle_scales(sc_h[h])), h


@pytest.mark.parametrize("rows,cols", [(1, 1), (37, 3), (128, 4), (300, 9), (4096 * 128, 6)])
def test_swizzle_matches_oracle(cuda_device, rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    s = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32).to(torch.uint8)
    out = mlaq.mxfp8_swizzle_scales(s.to(cuda_device))
    torch.cuda.synchronize()
    if rows * cols > 100000:  # the forward's q scales at T=4096: check a slice of whole tiles
        sub = s[:1024].numpy()
        ref = oracle.mxfp8_swizzle_scales(sub)
        assert np.array_equal(out[:ref.size].cpu().numpy(), ref)
        assert out.numel() == ((rows + 127) // 128) * 128 * ((cols + 3) // 4) * 4
    else:
        assert np.array_equal(out.cpu().numpy(), oracle.mxfp8_swizzle_scales(s.numpy()))


@pytest.mark.parametrize("rows,cols,group", [(300, 48, 192), (24576, 48, 192), (77, 9, 96), (1000, 5, 256),
                                            (130, 4, 32), (128, 3, 128)])
def test_grouped_swizzle_matches_oracle(cuda_device, rows, cols, group):
    """Rows in groups of `group`, each group padded to whole 128-row tiles:
    the oracle's plain swizzle applied group by group, concatenated."""
    g = torch.Generator().manual_seed(rows * 7 + cols + group)
    s = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32).to(torch.uint8)
    out = mlaq.mxfp8_swizzle_scales(s.to(cuda_device), group=group).cpu().numpy()
    # every group takes ceil(group/128) row tiles; the oracle's swizzle of a
    # short last group covers fewer, the rest is zero padding
    per = -(-group // 128) * -(-cols // 4) * 512
    blocks = []
    for r0 in range(0, rows, group):
        b = oracle.mxfp8_swizzle_scales(s[r0:r0 + group].numpy())
        blocks.append(np.concatenate([b, np.zeros(per - b.size, np.uint8)]))
    ref = np.concatenate(blocks)
    assert out.size == ref.size == int(mlaq.lib().mxfp8_grouped_scale_bytes(rows, cols, group))
    assert np.array_equal(out, ref)


def test_swizzle_strided_input(cuda_device):
    base = torch.randint(0, 256, (200, 16), dtype=torch.int32).to(torch.uint8)
    view = base.to(cuda_device)[:, 3:10]  # pitch 16, 7 columns
    out = mlaq.mxfp8_swizzle_scales(view)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.mxfp8_swizzle_scales(base[:, 3:10].numpy().copy()))


@pytest.mark.parametrize("D", [128, 48])
def test_kv_quantization_blocks_per_head(cuda_device, D):
    """K or V [T, H, D] quantized with the rowwise helper on [T*H, D]: blocks
    of 32 channels of one head (the last partial when D % 32 != 0)."""
    T, H = 257, 5
    g = torch.Generator().manual_seed(D)
    v = (torch.randn((T, H, D), generator=g) * 3).to(torch.bfloat16)
    codes, sc = mlaq.mxfp8_quantize_rows(v.reshape(T * H, D).to(cuda_device))
    torch.cuda.synchronize()
    rc, rs = oracle.mxfp8_quantize(v.reshape(T * H, D).double().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(sc.cpu().numpy(), rs)
