"""GPU parity of the columnwise MXFP8 copy: bit-exact vs the oracle.

TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
Greptile summary: the transpose among the MXFP8 quantization helpers (the
copy along the other axis, for GEMM operands reduced over their rows).
codes_t [C, R] and scales_t [C, ceil(R/32)] must match the oracle byte for
byte, including partial blocks, strided rows and non-finite values.
"""
import numpy as np
import pytest
import torch

import oracle
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu


def _oracle(t):
    return oracle.mxfp8_quantize_columns(t.detach().cpu().double().numpy())


def _run(inp):
    codes, scales = mlaq.mxfp8_quantize_cols(inp)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("R,C", [(32, 1), (100, 7), (1536, 64), (4000, 33), (5, 3), (4096, 1536),
                                 (96, 513), (130, 1025),
                                 # code rows 16- but not 32-byte aligned: 16-byte stores instead of 32
                                 (4016, 64), (48, 300)])
def test_quantize_cols_matches_oracle(cuda_device, dtype, R, C):
    g = torch.Generator().manual_seed(R * 1000 + C + 1)
    v = torch.randn((R, C), generator=g) * torch.exp2(torch.randint(-20, 20, (1, C), generator=g).float())
    v = v.to(dtype)
    codes, scales = _run(v.to(cuda_device))
    rc, rs = _oracle(v)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_cols_strided_and_odd_alignment(cuda_device, dtype):
    g = torch.Generator().manual_seed(6)
    base = (torch.randn((200, 301), generator=g) * 3).to(dtype).to(cuda_device)
    for c0, C in ((0, 160), (0, 150), (1, 37)):  # row pitch 301; an odd start column
        view = base[:, c0:c0 + C]
        codes, scales = _run(view)
        rc, rs = _oracle(view)
        assert np.array_equal(scales, rs) and np.array_equal(codes, rc)


def test_quantize_cols_special_values(cuda_device):
    v = torch.zeros((64, 6), dtype=torch.float32)
    v[:, 0] = torch.linspace(-1e-30, 1e-30, 64)
    v[3, 1] = float("nan")
    v[40, 2] = float("-inf")
    v[:, 3] = -0.0
    v[:, 4] = torch.tensor([448.0 * 2 ** 5] + [-3.0e38] + [1.0] * 62)
    codes, scales = _run(v.to(cuda_device))
    rc, rs = _oracle(v)
    assert np.array_equal(scales, rs) and np.array_equal(codes, rc)


def test_quantize_cols_full_size_sampled(cuda_device):
    """The query-tensor shape [4096, 24576] bf16 (the wgrad operand dq reduced
    over tokens): 64 sampled columns against the oracle, every scale row's
    shape checked."""
    g = torch.Generator().manual_seed(9)
    v = (torch.randn((4096, 24576), generator=g) * 0.01).to(torch.bfloat16)
    codes, scales = mlaq.mxfp8_quantize_cols(v.to(cuda_device))
    torch.cuda.synchronize()
    assert tuple(codes.shape) == (24576, 4096) and tuple(scales.shape) == (24576, 128)
    cols = torch.from_numpy(np.sort(np.random.default_rng(3).choice(24576, 64, replace=False)))
    rc, rs = oracle.mxfp8_quantize_columns(v[:, cols].double().numpy())
    assert np.array_equal(codes[cols.to(cuda_device)].cpu().numpy(), rc)
    assert np.array_equal(scales[cols.to(cuda_device)].cpu().numpy(), rs)


@pytest.mark.parametrize("R,C,group", [(24576, 1536, 192), (4096, 1536, 192), (300, 64, 96), (1000, 40, 128)])
def test_quantize_cols_tiled_scales(cuda_device, R, C, group):
    """mxfp8_quantize_cols_tiled: the codes of mxfp8_quantize_cols and its
    scales in the grouped tiled order (= mxfp8_swizzle_scales_grouped of the
    row-major ones, padding 0; the buffer starts filled with 0xEE)."""
    g = torch.Generator().manual_seed(R + C)
    x = (torch.randn((R, C), generator=g) * 0.05).to(torch.bfloat16).to(cuda_device)
    codes, scales = mlaq.mxfp8_quantize_cols(x)
    n = int(mlaq.lib().mxfp8_grouped_scale_bytes(C, (R + 31) // 32, group))
    buf = torch.full((n,), 0xEE, dtype=torch.uint8, device=cuda_device)
    codes_t, tiled = mlaq.mxfp8_quantize_cols(x, scales=buf, group=group)
    ref = mlaq.mxfp8_swizzle_scales(scales, group=group)
    torch.cuda.synchronize()
    assert torch.equal(codes_t, codes)
    assert torch.equal(tiled, ref)
