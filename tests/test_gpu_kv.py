"""GPU parity of the KV-side up-projection with the key's rope part.

Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting upstream
tensor in-place", Solution section: the KV path (the key's rotary kernel)
writes fresh o_key and o_value buffers. Here the up-projection and the key's
rope part are one kernel: kv = c_kv W^T split per head into k_nope and v,
the shared k_pe rotated and written after every head's k_nope.
Tolerance: the bf16 output bound |err| <= 8e-3 |ref| + 2e-3 rms(ref).
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
import synth
import up_proj_gemm_gb300 as mlaq

pytestmark = pytest.mark.gpu


def _inputs(T, K, H, Dn, Dv, Dr, seed, seq_len=None, yarn=False):
    c_kv = synth.normal_bf16((T, K), 1.0, seed)
    W = synth.normal_bf16((H * (Dn + Dv), K), 0.02, seed + 1)
    k_pe = synth.normal_bf16((T, Dr), 1.0, seed + 2)
    rows = 4096 if seq_len else max(T, 1)
    cos, sin = synth.rope_table_yarn(rows, Dr) if yarn else synth.rope_table_standard(rows, Dr)
    pos = synth.positions(T, seq_len)
    return c_kv, W, k_pe, cos, sin, pos


def _check(dev, T, K, H, Dn, Dv, Dr, seed, **kw):
    c_kv, W, k_pe, cos, sin, pos = _inputs(T, K, H, Dn, Dv, Dr, seed, **kw)
    d = [t.to(dev) for t in (c_kv, W, k_pe, cos, sin, pos)]
    keep = [t.clone() for t in d]
    o_key = torch.full((T, H, Dn + Dr), float("nan"), dtype=torch.bfloat16, device=dev)
    o_value = torch.full((T, H, Dv), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mlaq.kv_fwd(d[0], d[1], d[2], d[3], d[4], H, Dn, Dv, Dr, pos=d[5], o_key=o_key, o_value=o_value, status=st)
    torch.cuda.synchronize()
    mlaq.check_status(st)
    rk, rv = oracle.kv_forward(helpers.f64(c_kv), helpers.f64(W), helpers.f64(k_pe), H, Dn, Dv, Dr,
                               cos.numpy(), sin.numpy(), pos.numpy())
    helpers.check_bf16_close(o_key, rk, what="o_key")
    helpers.check_bf16_close(o_value, rv, what="o_value")
    assert all(torch.equal(a, b) for a, b in zip(d, keep)), "an input changed"


@pytest.mark.parametrize("T,K,H,Dn,Dv,Dr", [
    (256, 64, 4, 32, 32, 16),
    (300, 512, 8, 128, 128, 64),     # DeepSeek-V3 head shape, ragged tokens
    (130, 200, 3, 64, 32, 32),       # ragged K
    (1, 64, 2, 0, 64, 64),           # no key channels from the up-projection
])
def test_kv_matches_oracle(cuda_device, T, K, H, Dn, Dv, Dr):
    _check(cuda_device, T, K, H, Dn, Dv, Dr, seed=T + K)


def test_kv_yarn_and_restarting_positions(cuda_device):
    _check(cuda_device, 520, 512, 4, 128, 128, 64, seed=3, seq_len=128, yarn=True)


def test_kv_full_size_sampled(cuda_device):
    """T=4096 at the DeepSeek-V3 KV shape (kv_lora_rank 512, H=128, 128 + 128
    channels per head, Dr=64): 24 sampled tokens against the oracle."""
    T, K, H, Dn, Dv, Dr = 4096, 512, 128, 128, 128, 64
    c_kv, W, k_pe, cos, sin, pos = _inputs(T, K, H, Dn, Dv, Dr, seed=8)
    dev = cuda_device
    o_key, o_value = mlaq.kv_fwd(c_kv.to(dev), W.to(dev), k_pe.to(dev), cos.to(dev), sin.to(dev), H, Dn, Dv, Dr,
                                 pos=pos.to(dev))
    torch.cuda.synchronize()
    toks = torch.from_numpy(np.sort(np.random.default_rng(4).choice(T, 24, replace=False)))
    rk, rv = oracle.kv_forward(helpers.f64(c_kv[toks]), helpers.f64(W), helpers.f64(k_pe[toks]), H, Dn, Dv, Dr,
                               cos.numpy(), sin.numpy(), pos.numpy()[toks.numpy()])
    helpers.check_bf16_close(o_key[toks.to(dev)], rk, what="o_key")
    helpers.check_bf16_close(o_value[toks.to(dev)], rv, what="o_value")


def _kv_sweep(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        Dr = int(rng.choice([16, 32, 64]))
        Dn = 32 * int(rng.integers(0, 5))
        Dv = 32 * int(rng.integers(1, 5))
        if Dn + Dv > 256:
            continue
        out.append((int(rng.integers(1, 500)), 8 * int(rng.integers(1, 80)), int(rng.integers(1, 7)), Dn, Dv, Dr,
                    None if rng.random() < 0.5 else int(rng.integers(16, 300))))
    return out


@pytest.mark.parametrize("T,K,H,Dn,Dv,Dr,seq", _kv_sweep(10, 99))
def test_kv_shape_sweep(cuda_device, T, K, H, Dn, Dv, Dr, seq):
    """Seeded random KV shapes inside the documented limits (Dn, Dv multiples
    of 32 with Dn + Dv <= 256, any K % 8 == 0, ragged T, positions restarting
    or not)."""
    _check(cuda_device, T, K, H, Dn, Dv, Dr, 40 + T, seq_len=seq)
