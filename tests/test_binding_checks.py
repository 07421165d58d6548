"""Host-side argument checks of the Python binding, without a GPU.

The C ABI receives bare pointers and cannot see how large a buffer is, so
the binding checks every extent a kernel reads or writes before it calls the
library. Here each binding runs on CPU tensors that report themselves as CUDA
tensors, with a recording stand-in for the library's compute entry points
(the host-only size queries run in the real library):
- the call patterns used on the GPU (outputs allocated by the binding or
  passed in, views into larger buffers, tiled scales, the prepared weight
  copy) reach the C call;
- every mis-sized, mistyped or mismatched buffer is refused with an
  exception before any C compute call.
"""
import contextlib

import pytest
import torch

import up_proj_gemm_gb300 as mlaq
from up_proj_gemm_gb300 import _build

COMPUTE = {
    "mla_q_uproj_fwd", "mla_q_uproj_bwd_dgrad", "mla_q_uproj_bwd_wgrad", "mla_q_uproj_bwd_mxfp8",
    "mla_q_uproj_bwd_mxfp8_prepared", "mla_kv_uproj_fwd", "mxfp8_quantize_rows", "mxfp8_quantize_cols",
    "mxfp8_quantize_rows_tiled", "mxfp8_quantize_cols_tiled", "mxfp8_swizzle_scales",
    "mxfp8_swizzle_scales_grouped", "mla_wait_selftest",
}
bf16, f32, u8, i32 = torch.bfloat16, torch.float32, torch.uint8, torch.int32


@pytest.fixture(scope="module")
def built():
    _build.build()
    return mlaq.lib()


@pytest.fixture
def calls(built, monkeypatch):
    """Record compute calls instead of making them; CPU tensors pass as CUDA."""
    log = []
    real = mlaq._call

    def call(fn, what, *args):
        if what in COMPUTE:
            log.append(what)
            return
        real(fn, what, *args)

    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda t: True))
    monkeypatch.setattr(mlaq, "_call", call)
    monkeypatch.setattr(mlaq, "_stream", lambda device, stream: None)
    monkeypatch.setattr(torch.cuda, "device", lambda d: contextlib.nullcontext())
    return log


def _q(T=130, K=64, H=4, Dn=32, Dr=16, rows=None):
    """Inputs of the query path: x, W, b, dq, cos, sin, pos, status."""
    N = H * (Dn + Dr)
    rows = rows or T
    return dict(T=T, K=K, H=H, Dn=Dn, Dr=Dr, N=N, x=torch.zeros((T, K), dtype=bf16),
                W=torch.zeros((N, K), dtype=bf16), b=torch.zeros((N,), dtype=bf16),
                dq=torch.zeros((T, H, Dn + Dr), dtype=bf16), cos=torch.zeros((rows, Dr), dtype=f32),
                sin=torch.zeros((rows, Dr), dtype=f32), pos=torch.zeros((T,), dtype=i32),
                st=torch.zeros((1,), dtype=i32))


def test_fwd_valid_patterns(calls):
    s = _q()
    T, H, D, N = s["T"], s["H"], s["Dn"] + s["Dr"], s["N"]
    args = (s["x"], s["W"], s["cos"], s["sin"], H, s["Dn"], s["Dr"])
    kw = dict(bias=s["b"], pos=s["pos"], status=s["st"])
    q, sc = mlaq.fwd(*args, out_mode="mxfp8", **kw)
    assert q.shape == (T, H, D) and q.dtype == u8 and sc.shape == (T, H, 2)
    assert mlaq.fwd(*args, out_mode="bf16", **kw).dtype == bf16
    assert mlaq.fwd(*args, out_mode="mxfp8_bhsd", **kw)[1].shape == (H, T, 2)
    per_head = int(mlaq.lib().mxfp8_swizzled_scale_bytes(T, 2))
    assert mlaq.fwd(*args, out_mode="mxfp8_bhsd_swizzled", **kw)[1].shape == (H, per_head)
    # caller buffers, as views into larger allocations
    qbuf, sbuf = torch.zeros(T * N + 64, dtype=u8), torch.zeros(T * H * 2 + 64, dtype=u8)
    q2, s2 = mlaq.fwd(*args, out_mode="mxfp8", q_out=qbuf[32:32 + T * N].view(T, H, D),
                      q_scales=sbuf[32:32 + T * H * 2].view(T, H, 2), **kw)
    assert q2.data_ptr() == qbuf.data_ptr() + 32 and s2.data_ptr() == sbuf.data_ptr() + 32
    assert calls == ["mla_q_uproj_fwd"] * 5


def test_fwd_mxfp8_weight_patterns(calls):
    T, K, H, Dn, Dr = 77, 256, 6, 32, 16
    N = H * (Dn + Dr)
    x, W = torch.zeros((T, K), dtype=u8), torch.zeros((N, K), dtype=u8)
    xs, ws = torch.zeros((T, K // 32), dtype=u8), torch.zeros((N, K // 32), dtype=u8)
    cos = torch.zeros((T, Dr), dtype=f32)
    args = (x, W, cos, cos.clone(), H, Dn, Dr)
    mlaq.fwd(*args, weight_mode="mxfp8", x_scales=xs, w_scales=ws)
    G = mlaq.w_scale_group(T, K, H, Dn, Dr, T, Dr)
    assert G > 0
    xst = mlaq.mxfp8_swizzle_scales(xs)
    wst = mlaq.mxfp8_swizzle_scales(ws, group=G)
    assert wst.numel() == int(mlaq.lib().mxfp8_grouped_scale_bytes(N, K // 32, G))
    mlaq.fwd(*args, weight_mode="mxfp8_tiled", x_scales=xst, w_scales=wst)
    c, t = mlaq.mxfp8_quantize_rows(torch.zeros((N, K), dtype=bf16), group=G)
    assert c.shape == (N, K) and t.numel() == wst.numel()
    mlaq.fwd(*args, weight_mode="mxfp8_tiled", x_scales=xst, w_scales=t)
    assert calls == ["mla_q_uproj_fwd", "mxfp8_swizzle_scales", "mxfp8_swizzle_scales_grouped",
                     "mla_q_uproj_fwd", "mxfp8_quantize_rows_tiled", "mla_q_uproj_fwd"]


def test_bwd_valid_patterns(calls):
    s = _q()
    T, K, H, N = s["T"], s["K"], s["H"], s["N"]
    rope = torch.zeros((T, H, s["Dr"]), dtype=bf16)
    dx = mlaq.bwd_dgrad(s["dq"], s["W"], s["cos"], s["sin"], H, s["Dn"], s["Dr"], pos=s["pos"],
                        status=s["st"], dq_pre_rope=rope)
    assert dx.shape == (T, K)
    dW, db = mlaq.bwd_wgrad(s["dq"], s["x"], s["cos"], s["sin"], H, s["Dn"], s["Dr"], pos=s["pos"],
                            status=s["st"], dq_pre_rope=rope)
    assert dW.shape == (N, K) and db.shape == (N,)
    _, none = mlaq.bwd_wgrad(s["dq"], s["x"], s["cos"], s["sin"], H, s["Dn"], s["Dr"], db=None,
                             dW=torch.zeros((N, K), dtype=bf16))
    assert none is None
    dxb = torch.zeros(T * K + 16, dtype=bf16)
    mlaq.bwd_dgrad(s["dq"], s["W"], s["cos"], s["sin"], H, s["Dn"], s["Dr"], dx=dxb[8:8 + T * K].view(T, K),
                   workspace=torch.zeros(1 << 16, dtype=u8))
    assert calls == ["mla_q_uproj_bwd_dgrad", "mla_q_uproj_bwd_wgrad", "mla_q_uproj_bwd_wgrad",
                     "mla_q_uproj_bwd_dgrad"]


def test_bwd_mxfp8_valid_patterns(calls):
    s = _q(T=200, K=96, H=2, Dn=64, Dr=64)
    T, K, H, N = s["T"], s["K"], s["H"], s["N"]
    a = (s["dq"], s["W"], s["x"], s["cos"], s["sin"], H, s["Dn"], s["Dr"])
    dx, dW, db = mlaq.bwd_mxfp8(*a, pos=s["pos"], status=s["st"])
    assert (dx.shape, dW.shape, db.shape) == ((T, K), (N, K), (N,))
    # one output at a time; x alone gives K for db
    mlaq.bwd_mxfp8(s["dq"], s["W"], None, *a[3:], dx=torch.zeros((T, K), dtype=bf16), dW=None, db=None)
    mlaq.bwd_mxfp8(s["dq"], None, s["x"], *a[3:], dx=None, dW=torch.zeros((N, K), dtype=bf16), db=None)
    mlaq.bwd_mxfp8(s["dq"], None, s["x"], *a[3:], dx=None, dW=None, db=torch.zeros((N,), dtype=bf16))
    wt, wts = mlaq.bwd_mxfp8_prepare_weight(s["W"], T, H, s["Dn"], s["Dr"], s["cos"])
    assert wt.shape == (K, N)
    mlaq.bwd_mxfp8(s["dq"], None, s["x"], *a[3:], pos=s["pos"], prepared=(wt, wts))
    assert calls == ["mla_q_uproj_bwd_mxfp8"] * 4 + ["mxfp8_quantize_cols_tiled",
                                                     "mla_q_uproj_bwd_mxfp8_prepared"]


def test_kv_and_quantizer_valid_patterns(calls):
    T, K, H, Dn, Dv, Dr = 96, 64, 2, 32, 32, 16
    c_kv, W = torch.zeros((T, K), dtype=bf16), torch.zeros((H * (Dn + Dv), K), dtype=bf16)
    k_pe, cos = torch.zeros((T, 1, Dr), dtype=bf16), torch.zeros((T, Dr), dtype=f32)
    ok, ov = mlaq.kv_fwd(c_kv, W, k_pe, cos, cos.clone(), H, Dn, Dv, Dr)
    assert ok.shape == (T, H, Dn + Dr) and ov.shape == (T, H, Dv)
    mlaq.kv_fwd(c_kv, W, k_pe, cos, cos.clone(), H, Dn, Dv, Dr, o_key=ok, o_value=ov)
    x = torch.zeros((300, 64), dtype=f32)
    c, sc = mlaq.mxfp8_quantize_rows(x)
    assert c.shape == (300, 64) and sc.shape == (300, 2)
    c, sc = mlaq.mxfp8_quantize_cols(x)
    assert c.shape == (64, 300) and sc.shape == (64, 10)
    n = int(mlaq.lib().mxfp8_grouped_scale_bytes(64, 10, 96))
    mlaq.mxfp8_quantize_cols(x, scales=torch.zeros(n, dtype=u8), group=96)
    assert calls == ["mla_kv_uproj_fwd"] * 2 + ["mxfp8_quantize_rows", "mxfp8_quantize_cols",
                                                "mxfp8_quantize_cols_tiled"]


def _z(shape, dtype=bf16):
    return torch.zeros(shape, dtype=dtype)


def _bad_cases():
    """(what is wrong, call) pairs; each call gets a fresh valid set of inputs."""
    def fwd(s, **over):
        kw = dict(bias=s["b"], pos=s["pos"], status=s["st"], out_mode="mxfp8")
        kw.update(over)
        a = [s["x"], s["W"], s["cos"], s["sin"], s["H"], s["Dn"], s["Dr"]]
        for i, k in enumerate(("x", "W", "cos", "sin")):
            if k in kw:
                a[i] = kw.pop(k)
        return lambda: mlaq.fwd(*a, **kw)

    def dgrad(s, **over):
        kw = dict(pos=s["pos"])
        kw.update(over)
        W, sin = kw.pop("W", s["W"]), kw.pop("sin", s["sin"])
        return lambda: mlaq.bwd_dgrad(s["dq"], W, s["cos"], sin, s["H"], s["Dn"], s["Dr"], **kw)

    def wgrad(s, **over):
        kw = dict(pos=s["pos"])
        kw.update(over)
        dq = kw.pop("dq", s["dq"])
        return lambda: mlaq.bwd_wgrad(dq, s["x"], s["cos"], s["sin"], s["H"], s["Dn"], s["Dr"], **kw)

    def mx(s, **over):
        kw = dict(pos=s["pos"])
        kw.update(over)
        W, x = kw.pop("W", s["W"]), kw.pop("x", s["x"])
        return lambda: mlaq.bwd_mxfp8(s["dq"], W, x, s["cos"], s["sin"], s["H"], s["Dn"], s["Dr"], **kw)

    T, K, N, H = 130, 64, 192, 4
    return [
        ("W", "fwd: W rows != H * (Dn + Dr)", lambda s: fwd(s, W=_z((N - 48, K)))),
        ("W", "fwd: W dtype", lambda s: fwd(s, W=_z((N, K), f32))),
        ("bias", "fwd: bias length", lambda s: fwd(s, bias=_z((N - 1,)))),
        ("pos", "fwd: pos length", lambda s: fwd(s, pos=_z((T - 1,), i32))),
        ("sin", "fwd: sin shape != cos shape", lambda s: fwd(s, sin=_z((T, 8), f32))),
        ("status", "fwd: empty status", lambda s: fwd(s, status=_z((0,), i32))),
        ("q_out", "fwd: q_out too small", lambda s: fwd(s, q_out=_z((T - 1, H, 48), u8))),
        ("q_out", "fwd: q_out bf16 for mxfp8", lambda s: fwd(s, q_out=_z((T, H, 48)))),
        ("q_scales", "fwd: q_scales token-major for head-major",
         lambda s: fwd(s, out_mode="mxfp8_bhsd_swizzled", q_scales=_z((T, H, 2), u8))),
        ("x_scales", "fwd: x_scales rows", lambda s: fwd(s, x=_z((T, 256), u8), W=_z((N, 256), u8),
                                                           weight_mode="mxfp8", x_scales=_z((T - 1, 8), u8),
                                                           w_scales=_z((N, 8), u8))),
        ("w_scales", "fwd: tiled w_scales short", lambda s: fwd(s, x=_z((T, 256), u8), W=_z((N, 256), u8),
                                                              weight_mode="mxfp8_tiled",
                                                              x_scales=_z((1 << 16,), u8),
                                                              w_scales=_z((512,), u8))),
        ("W", "dgrad: W rows != H * (Dn + Dr)", lambda s: dgrad(s, W=_z((N + 48, K)))),
        ("sin", "dgrad: sin shape", lambda s: dgrad(s, sin=_z((T + 1, 16), f32))),
        ("dx", "dgrad: dx size", lambda s: dgrad(s, dx=_z((T, K + 1)))),
        ("dq_pre_rope", "dgrad: rope buffer size", lambda s: dgrad(s, dq_pre_rope=_z((T, H, 8)))),
        ("workspace", "dgrad: workspace dtype", lambda s: dgrad(s, workspace=_z((1024,), f32))),
        ("dq", "wgrad: dq size", lambda s: wgrad(s, dq=_z((T, H, 47)))),
        ("dW", "wgrad: dW size", lambda s: wgrad(s, dW=_z((N, K - 1)))),
        ("db", "wgrad: db size", lambda s: wgrad(s, db=_z((N + 1,)))),
        ("pos", "wgrad: pos dtype", lambda s: wgrad(s, pos=_z((T,), torch.int64))),
        ("x", "bwd_mxfp8: x rows", lambda s: mx(s, x=_z((T + 1, K)))),
        ("W", "bwd_mxfp8: W rows", lambda s: mx(s, W=_z((N - 64, K)))),
        ("x", "bwd_mxfp8: x columns != W columns", lambda s: mx(s, W=_z((N, K + 32)))),
        ("db", "bwd_mxfp8: db size", lambda s: mx(s, db=_z((N - 1,)))),
        ("dW", "bwd_mxfp8: dW size", lambda s: mx(s, dW=_z((N, K, 2)))),
        ("wt", "bwd_mxfp8: prepared copy not [K, N]",
         lambda s: mx(s, W=None, prepared=(_z((K, N - 32), u8), _z((1 << 16,), u8)))),
        ("wt_scales", "bwd_mxfp8: prepared scales short",
         lambda s: mx(s, W=None, prepared=(_z((K, N), u8), _z((16,), u8)))),
        ("either", "bwd_mxfp8: both W and the prepared copy",
         lambda s: mx(s, prepared=(_z((K, N), u8), _z((1 << 16,), u8)))),
    ]


@pytest.mark.parametrize("name,what,make", _bad_cases(), ids=[c[1] for c in _bad_cases()])
def test_mis_sized_buffers_are_refused(calls, name, what, make):
    call = make(_q())
    with pytest.raises((ValueError, TypeError), match=name):
        call()
    assert calls == [], f"{what}: reached {calls}"


@pytest.mark.parametrize("what,call", [
    ("kv o_key", lambda: mlaq.kv_fwd(_z((8, 64)), _z((128, 64)), _z((8, 16)), _z((8, 16), f32),
                                     _z((8, 16), f32), 2, 32, 32, 16, o_key=_z((8, 2, 47)))),
    ("kv k_pe", lambda: mlaq.kv_fwd(_z((8, 64)), _z((128, 64)), _z((8, 15)), _z((8, 16), f32),
                                    _z((8, 16), f32), 2, 32, 32, 16)),
    ("rows codes", lambda: mlaq.mxfp8_quantize_rows(_z((40, 64), f32), codes=_z((40, 63), u8))),
    ("rows scales", lambda: mlaq.mxfp8_quantize_rows(_z((40, 64), f32), scales=_z((40, 3), u8))),
    ("rows tiled scales", lambda: mlaq.mxfp8_quantize_rows(_z((40, 64), f32), scales=_z((100,), u8), group=128)),
    ("cols codes", lambda: mlaq.mxfp8_quantize_cols(_z((40, 64), f32), codes=_z((40, 64, 2), u8))),
    ("cols scales", lambda: mlaq.mxfp8_quantize_cols(_z((40, 64), f32), scales=_z((64, 1), u8))),
    ("swizzle out", lambda: mlaq.mxfp8_swizzle_scales(_z((40, 2), u8), out=_z((100,), u8))),
])
def test_kv_and_quantizer_refusals(calls, what, call):
    with pytest.raises(ValueError):
        call()
    assert calls == []


@pytest.mark.parametrize("grads,expect", [
    ("xwb", ["mla_q_uproj_fwd", "mla_q_uproj_bwd_dgrad", "mla_q_uproj_bwd_wgrad"]),
    ("x", ["mla_q_uproj_fwd", "mla_q_uproj_bwd_dgrad"]),
    ("w", ["mla_q_uproj_fwd", "mla_q_uproj_bwd_wgrad"]),
])
def test_autograd_calls_only_the_needed_passes(calls, monkeypatch, grads, expect):
    """The autograd face computes only what autograd asks for: dgrad for x,
    one wgrad call for W and b, and dgrad hands the rotated rope channels to
    wgrad when both run."""
    from up_proj_gemm_gb300 import autograd
    seen = {}
    real_wgrad = autograd.bwd_wgrad

    def wgrad(*a, **k):
        seen["rope"] = k.get("dq_pre_rope")
        return real_wgrad(*a, **k)

    monkeypatch.setattr(autograd, "bwd_wgrad", wgrad)
    s = _q()
    x = s["x"].clone().requires_grad_("x" in grads)
    W = s["W"].clone().requires_grad_("w" in grads)
    b = s["b"].clone().requires_grad_("b" in grads)
    q = autograd.q_up_proj(x, W, s["cos"], s["sin"], s["H"], s["Dn"], s["Dr"], bias=b, pos=s["pos"])
    assert q.shape == (s["T"], s["H"], s["Dn"] + s["Dr"])
    q.backward(torch.zeros_like(q))
    assert calls == expect
    assert (x.grad is not None) == ("x" in grads) and (W.grad is not None) == ("w" in grads)
    assert (b.grad is not None) == ("b" in grads)
    if grads == "xwb":
        assert seen["rope"] is not None and seen["rope"].shape == (s["T"], s["H"], s["Dr"])
    elif "rope" in seen:
        assert seen["rope"] is None
