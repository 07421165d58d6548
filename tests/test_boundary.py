"""The C ABI of libmlaq.so, without a GPU: it loads, exports every symbol that
include/mlaq.h declares, and rejects bad arguments on the host with the
documented status before touching CUDA.

Cases follow the contract of the pages: the cos/sin width guard (Megatron-LM
PR "Fix fused MLA YaRN RoPE query kernel corrupting upstream tensor
in-place", Problem section: an out-of-bounds table read when the table is
narrower than the rotary dim) and no in-place output (same PR).
"""
import ctypes
import os
import re

import pytest
import torch

import up_proj_gemm_gb300 as mlaq
from up_proj_gemm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
S = mlaq.STATUS


@pytest.fixture(scope="module")
def L():
    _build.build()
    return mlaq.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mlaq.h")).read()
    return re.findall(r"MLAQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert set(names) >= {"mla_q_uproj_fwd", "mla_q_uproj_bwd_dgrad", "mla_q_uproj_bwd_wgrad",
                          "mxfp8_quantize_rows", "mla_q_uproj_workspace_size", "mla_status_string",
                          "mla_version"}
    for n in names:
        assert hasattr(L, n), n
    # nothing else is exported
    out = os.popen(f"nm -D --defined-only {mlaq.library_path}").read().split("\n")
    exported = {ln.split()[-1] for ln in out if ln.strip() and " T " in ln}
    assert exported == set(names)


def test_status_strings(L):
    for name, code in S.items():
        assert mlaq.status_string(code) == name
    assert L.mla_version() >= 10000


FAKE = 0x10000  # 64 KiB-aligned fake device addresses: never dereferenced


def p(i):
    return ctypes.c_void_p(FAKE * (i + 1))


def shape(T=256, K=64, H=4, Dn=32, Dr=16, cs_rows=256, cs_width=16):
    return mlaq.Shape(T=T, K=K, H=H, Dn=Dn, Dr=Dr, reserved=0, cs_rows=cs_rows, cs_width=cs_width)


def fwd(L, s, wm=0, om=1, x=p(0), xs=None, W=p(1), ws=None, b=None, cos=p(2), sin=p(3), pos=None,
        q=p(4), qs=p(5), st=None):
    return L.mla_q_uproj_fwd(ctypes.byref(s) if s is not None else None, wm, om, x, xs, W, ws, b, cos,
                             sin, pos, q, qs, st, None)


def test_fwd_valid_args_reach_cuda(L):
    # all host checks pass; without a GPU the first CUDA call fails cleanly
    r = fwd(L, shape())
    assert r in (S["MLA_ERR_CUDA"], S["MLA_OK"])


@pytest.mark.parametrize("kw,code", [
    (dict(s=None), "MLA_ERR_INVALID_ARG"),
    (dict(s=shape(Dr=15)), "MLA_ERR_INVALID_ARG"),          # odd rope dim
    (dict(s=shape(K=0)), "MLA_ERR_INVALID_ARG"),
    (dict(s=shape(H=0)), "MLA_ERR_INVALID_ARG"),
    (dict(s=shape(T=-1)), "MLA_ERR_INVALID_ARG"),
    (dict(x=None), "MLA_ERR_INVALID_ARG"),
    (dict(W=None), "MLA_ERR_INVALID_ARG"),
    (dict(q=None), "MLA_ERR_INVALID_ARG"),
    (dict(qs=None), "MLA_ERR_INVALID_ARG"),                 # MXFP8 out needs scales
    (dict(om=0), "MLA_ERR_INVALID_ARG"),                    # bf16 out must not get scales
    (dict(wm=2), "MLA_ERR_INVALID_ARG"),
    (dict(wm=1), "MLA_ERR_INVALID_ARG"),                    # MXFP8 weights need both scale arrays
    (dict(cos=None), "MLA_ERR_INVALID_ARG"),
    (dict(s=shape(cs_rows=1 << 31)), "MLA_ERR_INVALID_ARG"),  # no int32 position reaches such a row
    (dict(s=shape(cs_width=1 << 40)), "MLA_ERR_INVALID_ARG"),  # table bytes would overflow int64
    (dict(s=shape(H=1 << 26)), "MLA_ERR_INVALID_ARG"),        # N = H * (Dn + Dr) past INT32_MAX
    (dict(s=shape(T=1 << 31, cs_rows=(1 << 31) - 1)), "MLA_ERR_INVALID_ARG"),
    (dict(s=shape(cs_width=15)), "MLA_ERR_ROPE_WIDTH"),     # table narrower than Dr
    (dict(s=shape(cs_width=0)), "MLA_ERR_ROPE_WIDTH"),
    (dict(s=shape(T=300, cs_rows=256)), "MLA_ERR_POS_RANGE"),  # implicit pos = t beyond the table
    (dict(s=shape(Dr=18, cs_width=18)), "MLA_ERR_UNSUPPORTED"),
    (dict(s=shape(Dn=16)), "MLA_ERR_UNSUPPORTED"),
    (dict(s=shape(K=60)), "MLA_ERR_ALIGNMENT"),             # bf16 rows not 16-byte multiples
    (dict(x=ctypes.c_void_p(FAKE + 8)), "MLA_ERR_ALIGNMENT"),
    (dict(q=p(0)), "MLA_ERR_ALIAS"),                        # in-place output
    (dict(q=ctypes.c_void_p(FAKE + 256 * 64 * 2 - 16)), "MLA_ERR_ALIAS"),  # partial overlap with x
    (dict(qs=p(4)), "MLA_ERR_ALIAS"),                       # outputs overlap each other
    (dict(qs=p(3)), "MLA_ERR_ALIAS"),                       # scales written over the sin table
])
def test_fwd_rejects(L, kw, code):
    assert fwd(L, kw.pop("s", shape()), **kw) == S[code]


def test_fwd_mxfp8_weight_checks(L):
    s = shape(K=64)
    assert fwd(L, s, wm=1, xs=p(6), ws=p(7)) == S["MLA_ERR_UNSUPPORTED"]  # K % 128
    s = shape(K=48)
    assert fwd(L, s, wm=1, xs=p(6), ws=p(7)) == S["MLA_ERR_INVALID_ARG"]  # K % 32
    s = shape(K=128)
    r = fwd(L, s, wm=1, xs=ctypes.c_void_p(FAKE * 7 + 2), ws=p(7))
    assert r == S["MLA_ERR_ALIGNMENT"]


def test_fwd_empty_tokens_is_noop(L):
    assert fwd(L, shape(T=0)) == S["MLA_OK"]


def _bwd(L, which, s, dq=p(0), op=p(1), cos=p(2), sin=p(3), pos=None, out=p(4), db=None, ws=None,
         wsb=0, rope=None):
    if which == "dgrad":
        return L.mla_q_uproj_bwd_dgrad(ctypes.byref(s), dq, op, cos, sin, pos, out, rope, ws, wsb, None,
                                       None)
    return L.mla_q_uproj_bwd_wgrad(ctypes.byref(s), dq, rope, op, cos, sin, pos, out, db, ws, wsb, None,
                                   None)


@pytest.mark.parametrize("which", ["dgrad", "wgrad"])
def test_bwd_rejects(L, which):
    assert _bwd(L, which, shape(cs_width=8)) == S["MLA_ERR_ROPE_WIDTH"]
    assert _bwd(L, which, shape(), dq=None) == S["MLA_ERR_INVALID_ARG"]
    assert _bwd(L, which, shape(), out=p(0)) == S["MLA_ERR_ALIAS"]
    assert _bwd(L, which, shape(), out=p(1)) == S["MLA_ERR_ALIAS"]
    assert _bwd(L, which, shape(Dn=24)) == S["MLA_ERR_UNSUPPORTED"]   # Dn % Dr
    assert _bwd(L, which, shape(K=36)) == S["MLA_ERR_ALIGNMENT"]
    assert _bwd(L, which, shape(T=257)) == S["MLA_ERR_POS_RANGE"]
    assert _bwd(L, which, shape()) in (S["MLA_ERR_CUDA"], S["MLA_OK"])


def test_noalloc_dgrad_returns_the_same_codes(L):
    """mla_q_uproj_bwd_dgrad_noalloc runs the allocating entry point's
    argument checks before anything else: the same status for every bad
    argument (narrow table, null pointer, overlap, unsupported split, odd K,
    implicit positions past the table, misaligned rope buffer) and for a good
    one on a machine without a GPU."""
    def noalloc(s, dq=p(0), W=p(1), cos=p(2), sin=p(3), pos=None, dx=p(4), rope=None):
        return L.mla_q_uproj_bwd_dgrad_noalloc(ctypes.byref(s), dq, W, cos, sin, pos, dx, rope, None, None)
    cases = [dict(s=shape(cs_width=8)), dict(s=shape(), dq=None), dict(s=shape(), dx=p(0)),
             dict(s=shape(), dx=p(1)), dict(s=shape(Dn=24)), dict(s=shape(K=36)), dict(s=shape(T=257)),
             dict(s=shape(Dr=3)), dict(s=shape(), rope=p(0)), dict(s=shape(), rope=ctypes.c_void_p(FAKE * 9 + 8)),
             dict(s=shape())]
    for c in cases:
        kw = {k: v for k, v in c.items() if k != "s"}
        ref = _bwd(L, "dgrad", c["s"], dq=kw.get("dq", p(0)), op=kw.get("W", p(1)), out=kw.get("dx", p(4)),
                   rope=kw.get("rope"))
        assert noalloc(c["s"], **kw) == ref, c


def test_rope_table_pack_rejects(L):
    pk = L.mla_rope_table_pack
    assert L.mla_rope_table_packed_bytes(100, 64) == 100 * 32 * 16
    assert L.mla_rope_table_packed_bytes(100, 63) == 0
    assert pk(10, 8, 16, p(0), p(1), p(2), None) == S["MLA_ERR_ROPE_WIDTH"]   # narrower than Dr
    assert pk(10, 16, 15, p(0), p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]  # odd Dr
    assert pk(-1, 16, 16, p(0), p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert pk(10, 16, 16, None, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert pk(10, 16, 16, p(0), p(1), ctypes.c_void_p(FAKE * 2 + 4), None) == S["MLA_ERR_ALIGNMENT"]
    assert pk(10, 16, 16, p(0), p(1), p(0), None) == S["MLA_ERR_ALIAS"]        # over cos
    assert pk(0, 16, 16, None, None, None, None) == S["MLA_OK"]                 # nothing to pack
    assert pk(10, 16, 16, p(0), p(1), p(2), None) in (S["MLA_ERR_CUDA"], S["MLA_OK"])


def test_fwd_packed_checks(L):
    def fp(s, packed=p(2), q=p(5), qs=p(6), pos=None):
        return L.mla_q_uproj_fwd_packed(ctypes.byref(s), 0, 1, p(0), None, p(1), None, None, packed, pos,
                                        q, qs, None, None)
    assert fp(shape(cs_width=8)) == S["MLA_ERR_ROPE_WIDTH"]
    assert fp(shape(), packed=None) == S["MLA_ERR_INVALID_ARG"]
    assert fp(shape(), packed=ctypes.c_void_p(FAKE * 2 + 4)) == S["MLA_ERR_ALIGNMENT"]  # needs 16 bytes
    assert fp(shape(), q=p(2)) == S["MLA_ERR_ALIAS"]            # q over the packed table
    assert fp(shape(T=257)) == S["MLA_ERR_POS_RANGE"]
    assert fp(shape()) in (S["MLA_ERR_CUDA"], S["MLA_OK"])


def test_rope_buffer_checks(L):
    # dgrad writes dq_pre_rope (an output): it may overlap nothing
    ok = (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert _bwd(L, "dgrad", shape(), rope=p(8)) in ok
    assert _bwd(L, "dgrad", shape(), rope=p(0)) == S["MLA_ERR_ALIAS"]   # over dq
    assert _bwd(L, "dgrad", shape(), rope=p(4)) == S["MLA_ERR_ALIAS"]   # over dx
    assert _bwd(L, "dgrad", shape(), rope=ctypes.c_void_p(FAKE * 9 + 8)) == S["MLA_ERR_ALIGNMENT"]
    # wgrad reads it (an input): it may share bytes with other inputs, not with dW
    assert _bwd(L, "wgrad", shape(), rope=p(8)) in ok
    assert _bwd(L, "wgrad", shape(), rope=p(4)) == S["MLA_ERR_ALIAS"]   # under dW
    assert _bwd(L, "wgrad", shape(), rope=ctypes.c_void_p(FAKE * 9 + 8)) == S["MLA_ERR_ALIGNMENT"]


def test_wgrad_bias_alias(L):
    assert _bwd(L, "wgrad", shape(), db=p(0)) == S["MLA_ERR_ALIAS"]
    assert _bwd(L, "wgrad", shape(), db=p(4)) == S["MLA_ERR_ALIAS"]


def test_workspace_size(L):
    s = shape()
    for which in (0, 1, 2):
        assert L.mla_q_uproj_workspace_size(ctypes.byref(s), which) == 0
    assert L.mla_q_uproj_workspace_size(ctypes.byref(shape(Dr=3)), 0) == 0


def test_quantize_rejects(L):
    q = L.mxfp8_quantize_rows
    assert q(4, 64, 0, p(0), 32, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]   # ld < C
    assert q(4, 64, 5, p(0), 64, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert q(4, 64, 0, None, 64, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert q(0, 64, 0, None, 64, None, None, None) == S["MLA_OK"]
    assert q(4, 64, 0, ctypes.c_void_p(FAKE + 2), 64, p(1), p(2), None) == S["MLA_ERR_ALIGNMENT"]
    assert q(4, 64, 0, p(0), 64, ctypes.c_void_p(FAKE + 100), p(2), None) == S["MLA_ERR_ALIAS"]
    assert q(4, 64, 0, p(0), 64, p(1), p(1), None) == S["MLA_ERR_ALIAS"]


def test_quantize_cols_rejects(L):
    q = L.mxfp8_quantize_cols
    assert q(64, 4, 0, p(0), 2, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]   # ld < C
    assert q(64, 4, 7, p(0), 4, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert q(64, 4, 0, None, 4, p(1), p(2), None) == S["MLA_ERR_INVALID_ARG"]
    assert q(0, 4, 0, None, 4, None, None, None) == S["MLA_OK"]
    assert q(64, 4, 0, ctypes.c_void_p(FAKE + 2), 4, p(1), p(2), None) == S["MLA_ERR_ALIGNMENT"]
    assert q(64, 4, 0, p(0), 4, ctypes.c_void_p(FAKE + 100), p(2), None) == S["MLA_ERR_ALIAS"]
    assert q(64, 4, 0, p(0), 4, p(1), p(1), None) == S["MLA_ERR_ALIAS"]


def test_swizzle_rejects(L):
    z = L.mxfp8_swizzle_scales
    assert L.mxfp8_swizzled_scale_bytes(130, 5) == 2 * 128 * 8
    assert L.mxfp8_swizzled_scale_bytes(0, 5) == 0
    assert z(10, 4, p(0), 2, p(1), None) == S["MLA_ERR_INVALID_ARG"]          # ld < cols
    assert z(10, 4, None, 4, p(1), None) == S["MLA_ERR_INVALID_ARG"]
    assert z(0, 4, None, 4, None, None) == S["MLA_OK"]
    assert z(10, 4, p(0), 4, ctypes.c_void_p(FAKE * 2 + 8), None) == S["MLA_ERR_ALIGNMENT"]
    assert z(10, 4, p(0), 4, p(0), None) == S["MLA_ERR_ALIAS"]


def test_fwd_accepts_bhsd_scale_modes(L):
    assert fwd(L, shape(), om=2, qs=p(9)) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert fwd(L, shape(), om=3, qs=p(9)) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert fwd(L, shape(), om=4, qs=p(9)) == S["MLA_ERR_INVALID_ARG"]


def test_fwd_swizzled_scales_extent_in_alias_check(L):
    """With swizzled scales q_scales_out spans H tiles of 128 rows per head
    (here 4 x 1024 bytes, against 2048 for the dense [T, H, 2] order): a
    buffer ending 3072 bytes before cos overlaps it only in the swizzled mode."""
    assert L.mxfp8_swizzled_scale_bytes(256, 2) == 1024
    qs = ctypes.c_void_p(FAKE * 3 - 3072)  # cos is at FAKE * 3
    assert fwd(L, shape(), om=1, qs=qs) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert fwd(L, shape(), om=3, qs=qs) == S["MLA_ERR_ALIAS"]


def _kv(L, T=256, K=64, H=4, Dn=32, Dv=32, Dr=16, cs_rows=256, cs_width=16, c=p(0), W=p(1), kp=p(2),
        cos=p(3), sin=p(4), pos=None, ok=p(5), ov=p(8)):
    s = mlaq.KvShape(T=T, K=K, H=H, Dn=Dn, Dv=Dv, Dr=Dr, cs_rows=cs_rows, cs_width=cs_width)
    return L.mla_kv_uproj_fwd(ctypes.byref(s), c, W, kp, cos, sin, pos, ok, ov, None, None)


def test_kv_rejects(L):
    assert _kv(L) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert _kv(L, cs_width=8) == S["MLA_ERR_ROPE_WIDTH"]
    assert _kv(L, T=300) == S["MLA_ERR_POS_RANGE"]
    assert _kv(L, Dv=40) == S["MLA_ERR_UNSUPPORTED"]
    assert _kv(L, Dn=160, Dv=128) == S["MLA_ERR_UNSUPPORTED"]      # more than 256 channels per head
    assert _kv(L, Dr=24, cs_width=24) == S["MLA_ERR_UNSUPPORTED"]
    assert _kv(L, K=36) == S["MLA_ERR_ALIGNMENT"]
    assert _kv(L, ok=p(0)) == S["MLA_ERR_ALIAS"]                   # key over c_kv
    assert _kv(L, ov=p(5)) == S["MLA_ERR_ALIAS"]                   # value over key
    assert _kv(L, c=None) == S["MLA_ERR_INVALID_ARG"]
    assert _kv(L, cs_rows=1 << 31) == S["MLA_ERR_INVALID_ARG"]
    assert _kv(L, cs_width=1 << 40) == S["MLA_ERR_INVALID_ARG"]
    assert _kv(L, T=0, c=None) == S["MLA_OK"]


def _mx_shape(**kw):
    base = dict(T=64, K=64, H=4, Dn=32, Dr=32, cs_rows=64, cs_width=32)
    base.update(kw)
    return shape(**base)


def _bmx(L, s, dq=p(0), W=p(1), x=p(2), cos=p(3), sin=p(4), pos=None, dx=p(5), dW=p(6), db=p(7), ws=p(40),
         ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = L.mla_q_uproj_workspace_size(ctypes.byref(s), 3)
    return L.mla_q_uproj_bwd_mxfp8(ctypes.byref(s), dq, W, x, cos, sin, pos, dx, dW, db, ws, ws_bytes, None,
                                   None)


def test_bwd_mxfp8_rejects(L):
    ok = (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert _bmx(L, _mx_shape()) in ok
    assert _bmx(L, _mx_shape(Dr=16, cs_width=16)) == S["MLA_ERR_UNSUPPORTED"]   # D % 32: blocks span heads
    assert _bmx(L, _mx_shape(H=1)) == S["MLA_ERR_UNSUPPORTED"]                  # N = 64: not a 128 multiple
    assert _bmx(L, _mx_shape(K=48)) == S["MLA_ERR_UNSUPPORTED"]                 # K % 32
    assert _bmx(L, _mx_shape(cs_width=16)) == S["MLA_ERR_ROPE_WIDTH"]
    assert _bmx(L, _mx_shape(T=65)) == S["MLA_ERR_POS_RANGE"]
    assert _bmx(L, _mx_shape(), dx=None, dW=None, db=None) == S["MLA_ERR_INVALID_ARG"]
    assert _bmx(L, _mx_shape(), W=None) == S["MLA_ERR_INVALID_ARG"]              # dx needs W
    assert _bmx(L, _mx_shape(), x=None) == S["MLA_ERR_INVALID_ARG"]              # dW needs x
    assert _bmx(L, _mx_shape(), dq=None) == S["MLA_ERR_INVALID_ARG"]
    assert _bmx(L, _mx_shape(), W=None, dx=None) in ok
    assert _bmx(L, _mx_shape(), x=None, dW=None) in ok
    assert _bmx(L, _mx_shape(), ws_bytes=1024) == S["MLA_ERR_WORKSPACE"]
    assert _bmx(L, _mx_shape(), ws=None) == S["MLA_ERR_WORKSPACE"]
    assert _bmx(L, _mx_shape(), dx=p(0)) == S["MLA_ERR_ALIAS"]                   # dx over dq
    assert _bmx(L, _mx_shape(), db=p(6)) == S["MLA_ERR_ALIAS"]                   # db over dW
    assert _bmx(L, _mx_shape(), ws=p(1)) == S["MLA_ERR_ALIAS"]                   # workspace over W
    assert _bmx(L, _mx_shape(), ws=p(1), x=p(30), dx=None, W=None) in ok        # W unused without dx
    assert _bmx(L, _mx_shape(), dW=ctypes.c_void_p(FAKE * 7 + 8)) == S["MLA_ERR_ALIGNMENT"]
    assert _bmx(L, _mx_shape(), ws=ctypes.c_void_p(FAKE * 41 + 8)) == S["MLA_ERR_ALIGNMENT"]
    assert _bmx(L, _mx_shape(T=0), dq=None, ws=None, ws_bytes=0) in ok          # writes dW = 0, db = 0
    assert _bmx(L, _mx_shape(T=0), dq=None, W=None, x=None, ws=None, ws_bytes=0) in ok  # empty inputs


def test_bwd_mxfp8_layout(L):
    """The workspace regions are disjoint, 256-byte aligned, in order, and as
    large as their operands; the token axis is padded to 128."""
    for T, K, H, Dn, Dr in ((64, 64, 4, 32, 32), (200, 96, 2, 64, 64), (1, 32, 2, 32, 32),
                            (4096, 1536, 128, 128, 64)):
        N = H * (Dn + Dr)
        lay = mlaq.bwd_mxfp8_layout(T, K, H, Dn, Dr, max(T, 1), Dr)
        Tp, G = lay["t_pad"], lay["b_group"]
        assert Tp % 128 == 0 and Tp - 128 < T <= Tp
        assert K % G == 0 and G % 32 == 0 and G <= 192
        bsz = lambda cols: K // G * -(-G // 128) * -(-cols // 4) * 512   # B: groups padded to 128 rows
        sizes = [("qa", T * N), ("qa_scales", Tp * N // 32), ("qb", N * Tp), ("qb_scales", N * Tp // 32),
                 ("wt", K * N), ("wt_scales", bsz(N // 32)), ("xt", K * Tp), ("xt_scales", bsz(Tp // 32)),
                 ("db_partials", 4 * N * ((T + 31) // 32))]
        end = 0
        for name, size in sizes:
            assert lay[name] % 256 == 0 and lay[name] >= end, name
            end = lay[name] + size
        assert lay["total"] >= end
        assert lay["total"] == mlaq.workspace_size(T, K, H, Dn, Dr, max(T, 1), Dr, 3)
    assert mlaq.workspace_size(0, 64, 4, 32, 32, 1, 32, 3) == 0
    assert mlaq.workspace_size(64, 64, 4, 32, 32, 64, 32, 4) == 0


def test_autograd_face_has_no_cpu_path():
    from up_proj_gemm_gb300.autograd import q_up_proj
    x = torch.zeros((4, 8), dtype=torch.bfloat16, requires_grad=True)
    W = torch.zeros((12, 8), dtype=torch.bfloat16, requires_grad=True)
    cs = torch.zeros((4, 4), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        q_up_proj(x, W, cs, cs, 1, 8, 4)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mlaq, "_lib", None)
    monkeypatch.setattr(mlaq, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no non-CUDA fallback"):
        mlaq.lib()


def test_wait_selftest_flag_rejects(L):
    f = L.mla_wait_selftest_flag
    assert f(0, 50_000_000, None, None) == S["MLA_ERR_INVALID_ARG"]                      # no status word
    assert f(0, 50_000_000, ctypes.c_void_p(FAKE + 2), None) == S["MLA_ERR_INVALID_ARG"]  # misaligned
    assert f(0, 999_999, p(0), None) == S["MLA_ERR_INVALID_ARG"]                          # limit below 1 ms
    assert f(0, 1_000_000_001, p(0), None) == S["MLA_ERR_INVALID_ARG"]                    # above 1 s


def test_wait_selftest_rejects(L):
    """mla_wait_selftest checks its arguments before any launch."""
    bad = S["MLA_ERR_INVALID_ARG"]
    assert L.mla_wait_selftest(0, 50_000_000, None, None) == bad            # status required
    assert L.mla_wait_selftest(0, 50_000_000, ctypes.c_void_p(FAKE + 2), None) == bad  # misaligned
    assert L.mla_wait_selftest(0, 999_999, p(0), None) == bad               # limit below 1 ms
    assert L.mla_wait_selftest(1, 1_000_000_001, p(0), None) == bad         # limit above 1 s


def test_w_scale_group_and_grouped_bytes(L):
    """The W scale group for MLA_WEIGHT_MXFP8_TILED is the forward's channel
    tile with MXFP8 weights: 192 (one head) at the DeepSeek-V3 shape."""
    assert L.mla_q_uproj_w_scale_group(ctypes.byref(shape(T=4096, K=1536, H=128, Dn=128, Dr=64,
                                                          cs_rows=4096, cs_width=64))) == 192
    assert L.mla_q_uproj_w_scale_group(ctypes.byref(shape())) == 192   # 4 heads of 48
    assert L.mla_q_uproj_w_scale_group(ctypes.byref(shape(Dr=3))) == 0
    gb = L.mxfp8_grouped_scale_bytes
    assert gb(300, 48, 192) == 2 * 2 * 12 * 512          # 2 groups x 2 row tiles x 12 column tiles
    assert gb(300, 48, 128) == L.mxfp8_swizzled_scale_bytes(300, 48)
    assert gb(0, 48, 192) == 0 and gb(10, 48, 0) == 0
    z = L.mxfp8_swizzle_scales_grouped
    assert z(10, 4, 0, p(0), 4, p(1), None) == S["MLA_ERR_INVALID_ARG"]
    assert z(10, 4, 96, p(0), 2, p(1), None) == S["MLA_ERR_INVALID_ARG"]
    assert z(10, 4, 96, p(0), 4, ctypes.c_void_p(FAKE * 2 + 8), None) == S["MLA_ERR_ALIGNMENT"]
    assert z(0, 4, 96, None, 4, None, None) == S["MLA_OK"]


def test_fwd_tiled_scales_checks(L):
    """weight_mode MLA_WEIGHT_MXFP8_TILED: scales required, 16-byte aligned,
    and their tiled extents enter the overlap check."""
    s = shape(K=128)
    mx = dict(wm=2, xs=p(6), ws=p(7))
    assert fwd(L, s, **mx) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert fwd(L, s, wm=2, xs=None, ws=p(7)) == S["MLA_ERR_INVALID_ARG"]
    assert fwd(L, s, wm=2, xs=ctypes.c_void_p(FAKE * 7 + 4), ws=p(7)) == S["MLA_ERR_ALIGNMENT"]
    assert fwd(L, s, wm=3, xs=p(6), ws=p(7)) == S["MLA_ERR_INVALID_ARG"]
    # W's tiled scales: 192 rows -> 1 group x 2 row tiles x 1 column tile = 1024 bytes, against
    # 192 x 4 = 768 dense: a buffer starting 896 bytes before q overlaps it only when tiled
    assert L.mxfp8_grouped_scale_bytes(192, 4, 192) == 1024
    ws = ctypes.c_void_p(FAKE * 5 - 896)  # q is at FAKE * 5
    assert fwd(L, s, wm=1, xs=p(6), ws=ws) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert fwd(L, s, wm=2, xs=p(6), ws=ws) == S["MLA_ERR_ALIAS"]


def test_quantize_rows_tiled_checks(L):
    q = L.mxfp8_quantize_rows_tiled
    assert q(10, 64, 1, p(0), 64, p(1), p(2), 0, None) == S["MLA_ERR_INVALID_ARG"]     # group <= 0
    assert q(10, 64, 2, p(0), 64, p(1), p(2), 128, None) == S["MLA_ERR_INVALID_ARG"]   # dtype
    assert q(0, 64, 1, None, 64, None, None, 128, None) == S["MLA_OK"]
    # 10 rows x 2 blocks tile to 512 bytes (128 rows x 4 columns): a scale buffer
    # starting 256 bytes before the input overlaps it only in the tiled order
    sc = ctypes.c_void_p(FAKE - 256)  # the input is at FAKE
    assert L.mxfp8_quantize_rows(10, 64, 1, p(0), 64, p(1), sc, None) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    assert q(10, 64, 1, p(0), 64, p(1), sc, 128, None) == S["MLA_ERR_ALIAS"]


def test_bwd_mxfp8_prepared_checks(L):
    """mla_q_uproj_bwd_mxfp8_prepared: the prepared copy is wt and its scales
    together, 16-byte aligned, and required when dx is asked for."""
    s = shape(T=64, K=64, H=2, Dn=32, Dr=32, cs_rows=64, cs_width=32)
    need = L.mla_q_uproj_workspace_size(ctypes.byref(s), 3)
    f = L.mla_q_uproj_bwd_mxfp8_prepared
    ws = p(20)
    args = lambda wt, wts, dx=p(9): (ctypes.byref(s), p(0), wt, wts, p(2), p(3), p(4), None, dx, p(10), p(11),
                                     ws, need, None, None)
    assert f(*args(p(1), None)) == S["MLA_ERR_INVALID_ARG"]                 # scales missing
    assert f(*args(None, None)) == S["MLA_ERR_INVALID_ARG"]                 # dx without W's copy
    assert f(*args(ctypes.c_void_p(FAKE * 2 + 8), p(12))) == S["MLA_ERR_ALIGNMENT"]
    assert f(*args(p(1), p(12))) in (S["MLA_ERR_CUDA"], S["MLA_OK"])
    q = L.mxfp8_quantize_cols_tiled
    assert q(64, 32, 1, p(0), 32, p(1), p(2), 0, None) == S["MLA_ERR_INVALID_ARG"]
    assert q(0, 32, 1, None, 32, None, None, 128, None) == S["MLA_OK"]


def test_public_names_are_exported():
    """Every public function and structure of the binding is in __all__."""
    import inspect
    public = {n for n, o in vars(mlaq).items() if not n.startswith("_")
              and (inspect.isfunction(o) or inspect.isclass(o)) and o.__module__ == mlaq.__name__}
    assert public <= set(mlaq.__all__), sorted(public - set(mlaq.__all__))
    assert all(hasattr(mlaq, n) for n in mlaq.__all__)
