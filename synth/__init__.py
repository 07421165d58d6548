"""Seeded synthetic inputs for the fused MLA query up-projection.

This module only *draws* inputs: random normals rounded to their storage
dtype, the per-position cos/sin tables, the position array, and the named
workload shapes. It holds none of the operation's arithmetic (no GEMM, no
rotation, no quantization), so both the CUDA path and the CPU oracle can take
their inputs from here without sharing any of the method.

Shapes follow the DeepSeek-V3 query up-projection that the TransformerEngine
pull request "Add support for fused Q Up-Proj GEMM/RoPE/Quant" targets
(description paragraph: the Q up-proj step of DeepseekV3 training), plus a
tiny correctness shape.

All randomness comes from ``torch.Generator`` seeded per tensor, drawn in
fp32 on the CPU and rounded to bf16 with round-to-nearest-even (torch's
conversion), so the same seed gives the same bytes on every machine.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "workload", "normal_bf16", "rope_table_standard",
    "rope_table_yarn", "positions", "make_inputs", "bf16_bits",
]


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One named problem: shape, value distributions and output modes."""

    name: str
    T: int                    # tokens
    K: int                    # q_lora_rank (forward reduction dim)
    H: int                    # heads
    Dn: int                   # pass-through ("nope") channels per head
    Dr: int                   # rotated channels per head
    bias: bool = False
    x_std: float = 1.0
    w_std: float = 0.02
    b_std: float = 1.0
    dq_std: float = 0.01
    outlier_frac: float = 0.0  # fraction of x elements multiplied by outlier_mult
    outlier_mult: float = 1.0
    table: str = "standard"    # "standard" | "yarn"
    rope_base: float = 10000.0
    seq_len: Optional[int] = None  # positions restart every seq_len tokens (None: pos = t)
    weight_mode: str = "bf16"  # "bf16" | "mxfp8"
    out_modes: tuple = ("mxfp8",)
    passes: tuple = ("fwd",)   # subset of ("fwd", "bwd")
    yarn: dict = field(default_factory=dict)

    @property
    def D(self) -> int:
        return self.Dn + self.Dr

    @property
    def N(self) -> int:
        return self.H * self.D

    @property
    def cs_rows(self) -> int:
        return self.seq_len if self.seq_len is not None else self.T

    def fwd_flop(self) -> int:
        return 2 * self.T * self.K * self.N

    def bwd_flop(self) -> int:
        return 4 * self.T * self.K * self.N


_DSV3 = dict(K=1536, H=128, Dn=128, Dr=64)

WORKLOADS = {
    # tiny correctness shape: one 256-token sequence, q_lora_rank 64, 4 heads of 32+16
    "tiny": Workload("tiny", T=256, K=64, H=4, Dn=32, Dr=16, bias=True,
                     x_std=1.0, w_std=1.0 / 8.0, b_std=1.0, dq_std=1.0,
                     out_modes=("bf16", "mxfp8"), passes=("fwd", "bwd")),
    # DeepSeek-V3 query up-projection forward, bf16 weights, MXFP8 output
    "dsv3_fwd_bf16w": Workload("dsv3_fwd_bf16w", T=4096, **_DSV3, x_std=1.0, w_std=0.02),
    # same shape, MXFP8 weights and activations (1x32 blocks along K), 1% x outliers x50
    "dsv3_fwd_mxfp8w": Workload("dsv3_fwd_mxfp8w", T=4096, **_DSV3, x_std=1.0, w_std=0.02,
                                outlier_frac=0.01, outlier_mult=50.0, weight_mode="mxfp8"),
    # backward at 2 x 4096 tokens, bias on (bias gradient produced)
    "dsv3_bwd": Workload("dsv3_bwd", T=8192, **_DSV3, bias=True, x_std=1.0, w_std=0.02,
                         dq_std=0.01, seq_len=4096, out_modes=(), passes=("bwd",)),
    # long context, 4 x 4096 tokens, YaRN tables, forward + backward
    "dsv3_long_yarn": Workload("dsv3_long_yarn", T=16384, **_DSV3, x_std=1.0, w_std=0.02,
                               dq_std=0.01, seq_len=4096, table="yarn",
                               passes=("fwd", "bwd"),
                               yarn=dict(factor=40.0, original_max_position=4096,
                                         beta_fast=32.0, beta_slow=1.0, mscale=1.0)),
}


def workload(name: str, **overrides) -> Workload:
    """Look up a named workload, optionally overriding fields (e.g. ``T=300``)."""
    return replace(WORKLOADS[name], **overrides)


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------
def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, outlier_frac: float = 0.0,
                outlier_mult: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std) draws (std is a standard deviation), optional outliers,
    rounded to bf16 (RNE). Returns a contiguous CPU bf16 tensor.

    Outliers: each element independently, with probability ``outlier_frac``,
    is multiplied by ``outlier_mult`` before the bf16 rounding."""
    g = _gen(seed)
    v = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * float(std)
    if outlier_frac > 0.0:
        pick = torch.rand(tuple(shape), generator=g, dtype=torch.float32) < outlier_frac
        v = torch.where(pick, v * float(outlier_mult), v)
    return v.to(torch.bfloat16).contiguous()


def normal_f32(shape, std: float, seed: int) -> torch.Tensor:
    g = _gen(seed)
    return (torch.randn(tuple(shape), generator=g, dtype=torch.float32) * float(std)).contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a bf16 tensor (a view, no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def positions(T: int, seq_len: Optional[int] = None) -> torch.Tensor:
    """int32 positions: t, or t mod seq_len for packed equal-length sequences."""
    p = torch.arange(T, dtype=torch.int64)
    if seq_len is not None:
        p = p % int(seq_len)
    return p.to(torch.int32).contiguous()


def _table_from_freqs(rows: int, freqs: np.ndarray, mscale: float = 1.0):
    """cos/sin tables [rows, 2*len(freqs)] fp32; column i and i+len(freqs) share freq i.

    Angles are formed in fp64 and the cos/sin values rounded once to fp32."""
    pos = np.arange(rows, dtype=np.float64)[:, None]
    ang = pos * np.concatenate([freqs, freqs])[None, :]
    cos = (np.cos(ang) * mscale).astype(np.float32)
    sin = (np.sin(ang) * mscale).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(cos)), torch.from_numpy(np.ascontiguousarray(sin))


def rope_table_standard(rows: int, Dr: int, base: float = 10000.0):
    """Standard rotary table: theta_i = base^(-2i/Dr), i < Dr/2."""
    i = np.arange(Dr // 2, dtype=np.float64)
    freqs = base ** (-2.0 * i / Dr)
    return _table_from_freqs(rows, freqs)


def rope_table_yarn(rows: int, Dr: int, base: float = 10000.0, factor: float = 40.0,
                    original_max_position: int = 4096, beta_fast: float = 32.0,
                    beta_slow: float = 1.0, mscale: float = 1.0):
    """YaRN ("NTK-by-parts") context-extended table (Peng et al., 2023).

    Frequencies below the beta_fast correction dimension keep their original
    value, those above the beta_slow one are divided by ``factor``, with a
    linear ramp between; the amplitude is ``mscale``."""
    half = Dr // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / Dr)

    def corr_dim(beta):
        return Dr * math.log(original_max_position / (2.0 * math.pi * beta)) / (2.0 * math.log(base))

    low = max(math.floor(corr_dim(beta_fast)), 0)
    high = min(math.ceil(corr_dim(beta_slow)), half - 1)
    if low == high:
        high += 0.001
    ramp = np.clip((i - low) / (high - low), 0.0, 1.0)
    freqs = inv_freq * (1.0 - ramp) + (inv_freq / factor) * ramp
    return _table_from_freqs(rows, freqs, mscale)


def make_tables(w: Workload):
    if w.table == "yarn":
        return rope_table_yarn(w.cs_rows, w.Dr, w.rope_base, **w.yarn)
    return rope_table_standard(w.cs_rows, w.Dr, w.rope_base)


def make_inputs(w: Workload, seed: int = 0, want=("x", "W", "b", "dq", "tables", "pos")) -> dict:
    """All CPU inputs of a workload, each from its own derived seed.

    Keys: x [T,K] bf16, W [N,K] bf16, b [N] bf16 (None when the workload has no
    bias), dq [T,H,D] bf16, cos/sin [cs_rows, Dr] fp32, pos [T] int32."""
    out = {}
    if "x" in want:
        out["x"] = normal_bf16((w.T, w.K), w.x_std, seed * 1000 + 1,
                               w.outlier_frac, w.outlier_mult)
    if "W" in want:
        out["W"] = normal_bf16((w.N, w.K), w.w_std, seed * 1000 + 2)
    if "b" in want:
        out["b"] = normal_bf16((w.N,), w.b_std, seed * 1000 + 3) if w.bias else None
    if "dq" in want:
        out["dq"] = normal_bf16((w.T, w.H, w.D), w.dq_std, seed * 1000 + 4)
    if "tables" in want:
        out["cos"], out["sin"] = make_tables(w)
    if "pos" in want:
        out["pos"] = positions(w.T, w.seq_len)
    return out
