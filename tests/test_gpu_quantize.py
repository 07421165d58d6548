"""GPU parity of the standalone rowwise MXFP8 quantizer: bit-exact vs the oracle.

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant":
Greptile summary (two-phase MXFP8 quantization helpers) and the review thread
on mxfp8_quantize_only. Codes and scales depend only on the input values, so
the CUDA path must match the oracle byte for byte.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu


def _oracle(t):
    v = t.detach().cpu().double().numpy()
    return oracle.mxfp8_quantize(v)


def _run(inp):
    codes, scales = mlaq.mxfp8_quantize_rows(inp)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("R,C", [(1, 32), (7, 100), (64, 1536), (33, 4000), (3, 5), (128, 24576),
                                 (513, 96),
                                 # rows of C % 32 == 16: each row's last block half full
                                 (5, 48), (9, 1552)])
def test_quantize_matches_oracle(cuda_device, dtype, R, C):
    g = torch.Generator().manual_seed(R * 1000 + C)
    v = torch.randn((R, C), generator=g) * torch.exp2(torch.randint(-20, 20, (R, 1), generator=g).float())
    v = v.to(dtype)
    codes, scales = _run(v.to(cuda_device))
    rc, rs = _oracle(v)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_strided_rows(cuda_device, dtype):
    g = torch.Generator().manual_seed(5)
    base = (torch.randn((40, 200), generator=g) * 3).to(dtype).to(cuda_device)
    for C in (160, 150, 37):
        view = base[:, :C]  # row pitch 200 > C
        codes, scales = _run(view)
        rc, rs = _oracle(view)
        assert np.array_equal(scales, rs) and np.array_equal(codes, rc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_strided_rows_32_byte_pitch(cuda_device, dtype):
    """Rows 32-byte aligned but not contiguous (pitch 192 elements), with
    C % 32 == 0 and C % 32 == 16."""
    g = torch.Generator().manual_seed(6)
    base = (torch.randn((40, 192), generator=g) * 3).to(dtype).to(cuda_device)
    for C in (160, 144):
        view = base[:, :C]
        codes, scales = _run(view)
        rc, rs = _oracle(view)
        assert np.array_equal(scales, rs) and np.array_equal(codes, rc)


def test_quantize_special_values(cuda_device):
    v = torch.zeros((6, 64), dtype=torch.float32)
    v[0] = torch.linspace(-1e-30, 1e-30, 64)                 # tiny: codes round to +-0
    v[1, 3] = float("nan")
    v[2, 40] = float("-inf")
    v[3] = -0.0                                              # signed zeros, scale byte 0
    v[4] = torch.tensor([448.0 * 2 ** 5] + [-3.0e38] + [1.0] * 62)
    v[5] = torch.linspace(-7.0, 7.0, 64) * 2.0 ** -60
    codes, scales = _run(v.to(cuda_device))
    rc, rs = _oracle(v)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


def test_quantize_outliers_and_edges(cuda_device):
    # block maxima exactly on the scale edges 448 * 2^e and just above them
    R = 64
    v = torch.randn((R, 64), generator=torch.Generator().manual_seed(11)).clamp(-1, 1)
    for r in range(R):
        e = r - 32
        v[r, 0] = 448.0 * 2.0 ** e
        v[r, 32] = float(np.nextafter(np.float32(448.0 * 2.0 ** e), np.float32(np.inf)))
    codes, scales = _run(v.to(cuda_device))
    rc, rs = _oracle(v)
    assert np.array_equal(scales, rs) and np.array_equal(codes, rc)
    x = synth.normal_bf16((256, 1536), 1.0, 3, outlier_frac=0.01, outlier_mult=50.0)
    codes, scales = _run(x.to(cuda_device))
    rc, rs = _oracle(x)
    assert np.array_equal(scales, rs) and np.array_equal(codes, rc)


def test_quantize_full_size_bit_exact(cuda_device):
    """[4096, 24576] bf16 activations (the forward's q shape), all elements."""
    x = synth.normal_bf16((4096, 24576), 1.0, 21)
    codes, scales = _run(x.to(cuda_device))
    rc, rs = _oracle(x)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


def test_quantize_weight_shape_bit_exact(cuda_device):
    """[24576, 1536] bf16 (the projection weight quantized for the MXFP8
    weight path, a benchmarked shape), all elements."""
    x = synth.normal_bf16((24576, 1536), 0.02, 22)
    codes, scales = _run(x.to(cuda_device))
    rc, rs = _oracle(x)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


def test_quantize_long_context_shape_sampled(cuda_device):
    """[16384, 24576] bf16 (the long-context q shape, a benchmarked shape):
    every row-block of 128 rows checked on one sampled row, plus the last row."""
    g = torch.Generator().manual_seed(23)
    xd = (torch.randn((16384, 24576), generator=g) * 1.0).to(torch.bfloat16)
    codes, scales = _run(xd.to(cuda_device))
    rows = np.concatenate([np.arange(0, 16384, 128) + np.random.default_rng(4).integers(0, 128, 128), [16383]])
    rc, rs = _oracle(xd[torch.from_numpy(rows)])
    assert np.array_equal(scales[rows], rs)
    assert np.array_equal(codes[rows], rc)


def test_quantize_does_not_touch_input(cuda_device):
    x = synth.normal_bf16((300, 1000), 1.0, 8).to(cuda_device)
    before = x.clone()
    _run(x)
    assert torch.equal(x, before)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C,group", [(4096, 1536, 128), (24576, 1536, 192), (300, 100, 96), (77, 1000, 128),
                                       (64, 40, 256), (130, 64, 32)])
def test_quantize_rows_tiled_scales(cuda_device, dtype, R, C, group):
    """mxfp8_quantize_rows_tiled: the codes of mxfp8_quantize_rows and its
    scales in the grouped tiled order (= mxfp8_swizzle_scales_grouped of the
    row-major scales, padding 0). The buffer starts filled with 0xEE so every
    padding byte must be written."""
    g = torch.Generator().manual_seed(R + C + group)
    x = (torch.randn((R, C), generator=g) * 3.0).to(dtype).to(cuda_device)
    codes, scales = mlaq.mxfp8_quantize_rows(x)
    n = int(mlaq.lib().mxfp8_grouped_scale_bytes(R, (C + 31) // 32, group))
    tiled = torch.full((n,), 0xEE, dtype=torch.uint8, device=cuda_device)
    codes_t, tiled = mlaq.mxfp8_quantize_rows(x, scales=tiled, group=group)
    ref = mlaq.mxfp8_swizzle_scales(scales, group=group)
    torch.cuda.synchronize()
    assert torch.equal(codes_t, codes)
    assert torch.equal(tiled, ref)


def test_quantize_rows_tiled_strided_input(cuda_device):
    base = (torch.randn((200, 80)) * 2.0).to(torch.bfloat16).to(cuda_device)
    view = base[:, 3:67]  # pitch 80, 64 columns, not 16-byte aligned rows
    codes, scales = mlaq.mxfp8_quantize_rows(view)
    codes_t, tiled = mlaq.mxfp8_quantize_rows(view, group=128)
    torch.cuda.synchronize()
    assert torch.equal(codes_t, codes)
    assert torch.equal(tiled, mlaq.mxfp8_swizzle_scales(scales))
