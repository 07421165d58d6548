"""GB300 (sm_103a) fused MLA query up-projection: Python binding of libmlaq.so.

The functions here only marshal torch tensors (device memory, the current
stream) into the C ABI declared in ``include/mlaq.h``; every step of the
computation runs in the library's CUDA kernels. There is no fallback: when
``libmlaq.so`` is missing or the call is rejected, an exception is raised.

Forward (TransformerEngine PR "Add support for fused Q Up-Proj
GEMM/RoPE/Quant"): ``q = RoPE(x W^T + b)``, optionally MXFP8.
Backward (TransformerEngine PR "Add a backwards linear function to be used
with the fused mla q up-proj"): inverse RoPE on dq fused into dgrad and
wgrad, plus the bias gradient.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "MlaError", "lib", "library_path", "fwd", "bwd_dgrad", "bwd_wgrad", "mxfp8_quantize_rows",
    "mxfp8_quantize_cols", "mxfp8_swizzle_scales", "kv_fwd", "rope_table_pack", "bwd_mxfp8", "bwd_mxfp8_layout",
    "bwd_mxfp8_operands", "bwd_mxfp8_prepare_weight", "w_scale_group", "wait_selftest", "wait_selftest_flag",
    "workspace_size", "status_string", "check_status", "Shape", "KvShape", "Mxfp8BwdLayout", "STATUS",
    "WEIGHT_MODES", "OUT_MODES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmlaq.so")

STATUS = {
    "MLA_OK": 0, "MLA_ERR_INVALID_ARG": 1, "MLA_ERR_ROPE_WIDTH": 2, "MLA_ERR_ALIGNMENT": 3,
    "MLA_ERR_ALIAS": 4, "MLA_ERR_UNSUPPORTED": 5, "MLA_ERR_CUDA": 6, "MLA_ERR_TIMEOUT": 7,
    "MLA_ERR_POS_RANGE": 8, "MLA_ERR_WORKSPACE": 9,
}
WEIGHT_MODES = {"bf16": 0, "mxfp8": 1, "mxfp8_tiled": 2}
OUT_MODES = {"bf16": 0, "mxfp8": 1, "mxfp8_bhsd": 2, "mxfp8_bhsd_swizzled": 3}


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("K", ctypes.c_int64), ("H", ctypes.c_int32),
                ("Dn", ctypes.c_int32), ("Dr", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cs_rows", ctypes.c_int64), ("cs_width", ctypes.c_int64)]


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
class KvShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("K", ctypes.c_int64), ("H", ctypes.c_int32), ("Dn", ctypes.c_int32),
                ("Dv", ctypes.c_int32), ("Dr", ctypes.c_int32), ("cs_rows", ctypes.c_int64),
                ("cs_width", ctypes.c_int64)]


class Mxfp8BwdLayout(ctypes.Structure):
    _fields_ = [("t_pad", ctypes.c_int64), ("b_group", ctypes.c_int64)] + [(n, ctypes.c_size_t) for n in (
        "qa", "qa_scales", "qb", "qb_scales", "wt", "wt_scales", "xt", "xt_scales", "db_partials", "total")]


_int = ctypes.c_int
_SIGS = {
    "mla_q_uproj_fwd": (_int, [ctypes.POINTER(Shape), _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _vp]),
    "mla_q_uproj_fwd_packed": (_int, [ctypes.POINTER(Shape), _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp]),
    "mla_rope_table_pack": (_int, [_i64, _i64, _int, _vp, _vp, _vp, _vp]),
    "mla_rope_table_packed_bytes": (ctypes.c_size_t, [_i64, _int]),
    "mla_q_uproj_bwd_dgrad": (_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_size_t, _vp, _vp]),
    "mla_q_uproj_bwd_wgrad": (_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_size_t, _vp, _vp]),
    "mla_q_uproj_bwd_dgrad_noalloc": (_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                             _vp, _vp]),
    "mxfp8_quantize_rows": (_int, [_i64, _i64, _int, _vp, _i64, _vp, _vp, _vp]),
    "mxfp8_quantize_cols": (_int, [_i64, _i64, _int, _vp, _i64, _vp, _vp, _vp]),
    "mxfp8_swizzle_scales": (_int, [_i64, _i64, _vp, _i64, _vp, _vp]),
    "mla_kv_uproj_fwd": (_int, [ctypes.POINTER(KvShape)] + [_vp] * 10),
    "mla_q_uproj_bwd_mxfp8": (_int, [ctypes.POINTER(Shape)] + [_vp] * 10 + [ctypes.c_size_t, _vp, _vp]),
    "mla_q_uproj_bwd_mxfp8_prepared": (_int, [ctypes.POINTER(Shape)] + [_vp] * 11 + [ctypes.c_size_t, _vp, _vp]),
    "mxfp8_quantize_cols_tiled": (_int, [_i64, _i64, _int, _vp, _i64, _vp, _vp, _i64, _vp]),
    "mla_q_uproj_bwd_mxfp8_layout": (_int, [ctypes.POINTER(Shape), ctypes.POINTER(Mxfp8BwdLayout)]),
    "mxfp8_swizzled_scale_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "mxfp8_quantize_rows_tiled": (_int, [_i64, _i64, _int, _vp, _i64, _vp, _vp, _i64, _vp]),
    "mxfp8_grouped_scale_bytes": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "mxfp8_swizzle_scales_grouped": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _vp]),
    "mla_q_uproj_w_scale_group": (ctypes.c_int64, [ctypes.POINTER(Shape)]),
    "mla_q_uproj_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Shape), _int]),
    "mla_wait_selftest": (_int, [_int, ctypes.c_uint64, _vp, _vp]),
    "mla_wait_selftest_flag": (_int, [_int, ctypes.c_uint64, _vp, _vp]),
    "mla_status_string": (ctypes.c_char_p, [_int]),
    "mla_version": (_int, []),
}


def lib() -> ctypes.CDLL:
    """The loaded libmlaq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"{library_path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                    f"g.build()\"` (nvcc, sm_103a). There is no non-CUDA fallback.")
            l = ctypes.CDLL(library_path)
            for name, (res, args) in _SIGS.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def wait_selftest(arrive: bool, limit_ms: float, status: torch.Tensor, stream=None) -> None:
    """Run the bounded-wait self-test (mla_wait_selftest) on the status
    tensor's device: with arrive=False a device wait gives up after limit_ms
    and MLA_ERR_TIMEOUT lands in ``status``; with arrive=True nothing does."""
    _need(status, "status", torch.int32, min_numel=1)
    _call(lib().mla_wait_selftest, "mla_wait_selftest", int(bool(arrive)), int(round(limit_ms * 1e6)),
          _ptr(status), _stream(status.device, stream))


def wait_selftest_flag(set_flag: bool, limit_ms: float, status: torch.Tensor, stream=None) -> None:
    """Run the flag-wait self-test (mla_wait_selftest_flag): with
    set_flag=False a device wait on a flag nothing raises gives up after
    limit_ms and MLA_ERR_TIMEOUT lands in ``status``."""
    _need(status, "status", torch.int32, min_numel=1)
    _call(lib().mla_wait_selftest_flag, "mla_wait_selftest_flag", int(bool(set_flag)), int(round(limit_ms * 1e6)),
          _ptr(status), _stream(status.device, stream))


def status_string(code: int) -> str:
    return lib().mla_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None, ndim=None, shape=None, numel=None, min_numel=None):
    """Check a tensor argument. The C ABI receives bare pointers, so every
    extent a kernel reads or writes is checked here: type, dtype, rank and
    size first, then device and layout."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} must hold at least {min_numel} elements, got {t.numel()}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cols(t):
    """Last extent of a tensor argument (None when it has none), read before
    `_need` has checked it."""
    return t.shape[-1] if isinstance(t, torch.Tensor) and t.dim() > 0 else None


def _tables(cos, sin, dev, T, pos):
    """The rotary tables (fp32 [rows, width], same shape) and positions (int32 [T])."""
    _need(cos, "cos", torch.float32, dev, ndim=2)
    _need(sin, "sin", torch.float32, dev, shape=cos.shape)
    if pos is not None:
        _need(pos, "pos", torch.int32, dev, shape=(T,))


def _status(status, dev):
    """The optional device status word (int32, at least one element)."""
    if status is not None:
        _need(status, "status", torch.int32, dev, min_numel=1)


def _shape(T, K, H, Dn, Dr, cos):
    return Shape(T=int(T), K=int(K), H=int(H), Dn=int(Dn), Dr=int(Dr), reserved=0,
                 cs_rows=int(cos.shape[0]), cs_width=int(cos.shape[1]))


def _call(fn, what, *args):
    st = fn(*args)
    if st != 0:
        raise MlaError(st, what)


def check_status(status: torch.Tensor, what: str = "device status") -> None:
    """Synchronize on the status word written by the kernels; raise if set."""
    v = int(status.item())
    if v != 0:
        raise MlaError(v, what)


def workspace_size(T, K, H, Dn, Dr, cs_rows, cs_width, which: int) -> int:
    s = Shape(T=T, K=K, H=H, Dn=Dn, Dr=Dr, reserved=0, cs_rows=cs_rows, cs_width=cs_width)
    return int(lib().mla_q_uproj_workspace_size(ctypes.byref(s), int(which)))


def rope_table_pack(cos, sin, Dr, out=None, stream=None):
    """The rotary table in the forward's packed layout (mla_rope_table_pack):
    float32 [Dr/2, rows, 4], entry [i, p] = (cos[p, i], sin[p, i],
    cos[p, i + Dr/2], sin[p, i + Dr/2]). Pack once, pass as ``rope_packed``."""
    dev = cos.device
    _need(cos, "cos", torch.float32, dev, ndim=2)
    _need(sin, "sin", torch.float32, dev, shape=cos.shape)
    rows, width = cos.shape
    if out is None:
        out = torch.empty((Dr // 2, rows, 4), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev, numel=rows * (Dr // 2) * 4)
    _call(lib().mla_rope_table_pack, "mla_rope_table_pack", int(rows), int(width), int(Dr), _ptr(cos), _ptr(sin),
          _ptr(out), _stream(dev, stream))
    return out


def fwd(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None, weight_mode="bf16", out_mode="mxfp8",
        x_scales=None, w_scales=None, q_out=None, q_scales=None, status=None, stream=None, rope_packed=None):
    """Fused forward. Returns q [T, H, D] (bf16 or uint8 E4M3 codes), plus the
    scales uint8 [T, H, ceil(D/32)] when out_mode is "mxfp8", or head-major
    [H, T, ceil(D/32)] when it is "mxfp8_bhsd", or [H, S] when it is
    "mxfp8_bhsd_swizzled": each head's scales in the block-scaled GEMM's
    tiled order (S = mxfp8_swizzled_scale_bytes(T, ceil(D/32)))

    weight_mode "bf16": x [T, K] bf16, W [N, K] bf16.
    weight_mode "mxfp8": x, W uint8 E4M3 codes with x_scales [T, K/32],
    w_scales [N, K/32] uint8 E8M0.
    weight_mode "mxfp8_tiled": the same codes with the scales already tiled:
    x_scales = mxfp8_swizzle_scales(x scales), w_scales =
    mxfp8_swizzle_scales(W scales, group=w_scale_group(...)) (flat uint8).

    rope_packed: the table packed by rope_table_pack(cos, sin, Dr); cos and
    sin are then only read for their shape (same results, bit for bit)."""
    wm, om = WEIGHT_MODES[weight_mode], OUT_MODES[out_mode]
    in_dtype = torch.uint8 if wm else torch.bfloat16
    dev = x.device
    _need(x, "x", in_dtype, ndim=2)
    T, K = x.shape
    D = Dn + Dr
    N = H * D
    _need(W, "W", in_dtype, dev, shape=(N, K))
    _tables(cos, sin, dev, T, pos)
    if rope_packed is not None:
        _need(rope_packed, "rope_packed", torch.float32, dev, numel=cos.shape[0] * (Dr // 2) * 4)
    _status(status, dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, dev, shape=(N,))
    if wm == 1:  # [rows, K/32] scales (K not a multiple of 32 is refused by the library)
        kb = (K + 31) // 32
        _need(x_scales, "x_scales", torch.uint8, dev, shape=(T, kb))
        _need(w_scales, "w_scales", torch.uint8, dev, shape=(N, kb))
    elif wm == 2:  # flat buffers in the tiled order: x in 128-row groups, W in the kernel's column tiles
        kb = K // 32
        G = w_scale_group(T, K, H, Dn, Dr, cos.shape[0], cos.shape[1])
        _need(x_scales, "x_scales", torch.uint8, dev, ndim=1,
              min_numel=int(lib().mxfp8_grouped_scale_bytes(T, kb, 128)))
        _need(w_scales, "w_scales", torch.uint8, dev, ndim=1,
              min_numel=int(lib().mxfp8_grouped_scale_bytes(N, kb, G)) if G else None)
    nb = (D + 31) // 32
    if out_mode == "mxfp8_bhsd_swizzled":
        sshape = (H, int(lib().mxfp8_swizzled_scale_bytes(T, nb)))
    elif out_mode == "mxfp8_bhsd":
        sshape = (H, T, nb)
    else:
        sshape = (T, H, nb)
    q_dtype = torch.uint8 if om else torch.bfloat16
    if q_out is None:
        q_out = torch.empty((T, H, D), dtype=q_dtype, device=dev)
    _need(q_out, "q_out", q_dtype, dev, numel=T * N)
    if om and q_scales is None:
        q_scales = torch.empty(sshape, dtype=torch.uint8, device=dev)
    if om:
        _need(q_scales, "q_scales", torch.uint8, dev, numel=math.prod(sshape))
    s = _shape(T, K, H, Dn, Dr, cos)
    if rope_packed is not None:
        _call(lib().mla_q_uproj_fwd_packed, "mla_q_uproj_fwd_packed", ctypes.byref(s), wm, om, _ptr(x),
              _ptr(x_scales), _ptr(W), _ptr(w_scales), _ptr(bias), _ptr(rope_packed), _ptr(pos),
              _ptr(q_out), _ptr(q_scales if om else None), _ptr(status), _stream(dev, stream))
    else:
        _call(lib().mla_q_uproj_fwd, "mla_q_uproj_fwd", ctypes.byref(s), wm, om, _ptr(x),
              _ptr(x_scales), _ptr(W), _ptr(w_scales), _ptr(bias), _ptr(cos), _ptr(sin), _ptr(pos),
              _ptr(q_out), _ptr(q_scales if om else None), _ptr(status), _stream(dev, stream))
    return (q_out, q_scales) if om else q_out


def _rope_buf(t, T, H, Dr, dev):
    """The optional rope hand-off buffer: contiguous bf16 holding T * H * Dr."""
    if t is not None:
        _need(t, "dq_pre_rope", torch.bfloat16, dev, numel=T * H * Dr)
    return t


def bwd_dgrad(dq, W, cos, sin, H, Dn, Dr, pos=None, dx=None, status=None, stream=None, workspace=None,
              dq_pre_rope=None):
    """dx [T, K] bf16 = (inverse-RoPE dq) W.

    dgrad may need a device workspace: ``workspace_size(..., which=1)``
    bytes select its fastest path (allocated here unless passed in), at
    least ``which=4`` bytes a slower one that needs less. ``dq_pre_rope`` (a [T, H, Dr] bf16 tensor, or
    None) receives the rotated rope channels, for bwd_wgrad."""
    dev = dq.device
    T = dq.shape[0] if isinstance(dq, torch.Tensor) and dq.dim() > 0 else 0
    N = H * (Dn + Dr)
    K = _cols(W)
    _need(dq, "dq", torch.bfloat16, numel=T * N)
    _need(W, "W", torch.bfloat16, dev, ndim=2, shape=(N, K))
    _tables(cos, sin, dev, T, pos)
    _status(status, dev)
    if dx is None:
        dx = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    _need(dx, "dx", torch.bfloat16, dev, numel=T * K)
    _rope_buf(dq_pre_rope, T, H, Dr, dev)
    s = _shape(T, K, H, Dn, Dr, cos)
    with torch.cuda.device(dev):
        need = int(lib().mla_q_uproj_workspace_size(ctypes.byref(s), 1))
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev, ndim=1)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call(lib().mla_q_uproj_bwd_dgrad, "mla_q_uproj_bwd_dgrad", ctypes.byref(s), _ptr(dq), _ptr(W),
          _ptr(cos), _ptr(sin), _ptr(pos), _ptr(dx), _ptr(dq_pre_rope), _ptr(workspace), ws_bytes,
          _ptr(status), _stream(dev, stream))
    return dx


def bwd_wgrad(dq, x, cos, sin, H, Dn, Dr, pos=None, dW=None, db=True, status=None, stream=None,
              dq_pre_rope=None):
    """dW [N, K] bf16 = (inverse-RoPE dq)^T x and db [N] bf16 = its token sum.

    db=True allocates the bias gradient, db=None/False skips it, or pass a
    tensor. ``dq_pre_rope``: None, or the buffer bwd_dgrad filled from the
    same dq (its rope tiles are then read instead of rotated again).
    Returns (dW, db-or-None)."""
    dev = dq.device
    _need(x, "x", torch.bfloat16, dev, ndim=2)
    T, K = x.shape
    N = H * (Dn + Dr)
    _need(dq, "dq", torch.bfloat16, numel=T * N)
    _tables(cos, sin, dev, T, pos)
    _status(status, dev)
    if dW is None:
        dW = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    _need(dW, "dW", torch.bfloat16, dev, numel=N * K)
    if db is True:
        db = torch.empty((N,), dtype=torch.bfloat16, device=dev)
    elif db is False:
        db = None
    if db is not None:
        _need(db, "db", torch.bfloat16, dev, numel=N)
    _rope_buf(dq_pre_rope, T, H, Dr, dev)
    s = _shape(T, K, H, Dn, Dr, cos)
    _call(lib().mla_q_uproj_bwd_wgrad, "mla_q_uproj_bwd_wgrad", ctypes.byref(s), _ptr(dq),
          _ptr(dq_pre_rope), _ptr(x), _ptr(cos), _ptr(sin), _ptr(pos), _ptr(dW), _ptr(db), None, 0,
          _ptr(status), _stream(dev, stream))
    return dW, db


def bwd_mxfp8_layout(T, K, H, Dn, Dr, cs_rows, cs_width) -> dict:
    """Byte offsets of the MXFP8 backward's workspace regions (and ``t_pad``,
    ``total``) as ``mla_q_uproj_bwd_mxfp8_layout`` reports them."""
    s = Shape(T=T, K=K, H=H, Dn=Dn, Dr=Dr, reserved=0, cs_rows=cs_rows, cs_width=cs_width)
    out = Mxfp8BwdLayout()
    _call(lib().mla_q_uproj_bwd_mxfp8_layout, "mla_q_uproj_bwd_mxfp8_layout", ctypes.byref(s),
          ctypes.byref(out))
    return {name: int(getattr(out, name)) for name, _ in Mxfp8BwdLayout._fields_}


def bwd_mxfp8_operands(workspace, T, K, H, Dn, Dr, cs_rows, cs_width) -> dict:
    """uint8 views of the quantized operands a bwd_mxfp8 call left in
    ``workspace``: codes qa [T, N], qb [N, t_pad], wt [K, N], xt [K, t_pad]
    (t_pad = T rounded up to 128) and the flat scale arrays qa_s, qb_s,
    wt_s, xt_s in the GEMMs' tiled order (see mla_mxfp8_bwd_layout), plus
    ``t_pad`` and ``b_group``."""
    L = bwd_mxfp8_layout(T, K, H, Dn, Dr, cs_rows, cs_width)
    N = H * (Dn + Dr)
    Tp, G = L["t_pad"], L["b_group"]

    def view(off, rows, cols):
        return workspace[off:off + rows * cols].view(rows, cols)

    def tiled(off, rows, cols, g):
        n = -(-rows // g) * -(-g // 128) * -(-cols // 4) * 512
        return workspace[off:off + n]

    return dict(qa=view(L["qa"], T, N), qa_s=tiled(L["qa_scales"], Tp, N // 32, 128),
                qb=view(L["qb"], N, Tp), qb_s=tiled(L["qb_scales"], N, Tp // 32, 128),
                wt=view(L["wt"], K, N), wt_s=tiled(L["wt_scales"], K, N // 32, G),
                xt=view(L["xt"], K, Tp), xt_s=tiled(L["xt_scales"], K, Tp // 32, G), t_pad=Tp, b_group=G)


def bwd_mxfp8(dq, W, x, cos, sin, H, Dn, Dr, pos=None, dx=True, dW=True, db=True, status=None, stream=None,
              workspace=None, prepared=None):
    """Backward with MXFP8 tensor-core GEMMs (``mla_q_uproj_bwd_mxfp8``):
    dx [T, K], dW [N, K], db [N] (bf16) from dq [T, H, D] bf16.

    Each of dx / dW / db: True allocates it, False/None skips it, or pass a
    tensor. W [N, K] is needed for dx, x [T, K] for dW (else may be None).
    ``prepared``: W's columnwise MXFP8 copy from ``bwd_mxfp8_prepare_weight``
    (then W must be None; ``mla_q_uproj_bwd_mxfp8_prepared``, same results).
    The workspace (``workspace_size(..., which=3)`` bytes, uint8) is
    allocated unless passed; afterwards it holds the quantized operands
    (``bwd_mxfp8_operands``). Returns (dx, dW, db), None where skipped."""
    dev = dq.device
    T = dq.shape[0] if isinstance(dq, torch.Tensor) and dq.dim() > 0 else 0
    N = H * (Dn + Dr)
    _need(dq, "dq", torch.bfloat16, numel=T * N)
    _tables(cos, sin, dev, T, pos)
    _status(status, dev)
    want_dx = dx is not None and dx is not False
    want_dw = dW is not None and dW is not False
    if prepared is not None:
        if W is not None:
            raise ValueError("pass either W or its prepared copy, not both")
        wt, wt_s = prepared
        K = wt.shape[0] if isinstance(wt, torch.Tensor) and wt.dim() == 2 else None
        _need(wt, "wt", torch.uint8, dev, ndim=2, shape=(K, N))
        G = bwd_mxfp8_layout(max(int(T), 1), K, H, Dn, Dr, cos.shape[0], cos.shape[1])["b_group"]
        _need(wt_s, "wt_scales", torch.uint8, dev, ndim=1,
              min_numel=int(lib().mxfp8_grouped_scale_bytes(K, N // 32, G)))
    elif want_dx:
        K = _cols(W)
        _need(W, "W", torch.bfloat16, dev, ndim=2, shape=(N, K))
    elif x is not None:
        K = _cols(x)
    else:
        raise ValueError("need W (for dx) or x (for dW) to know K")
    if want_dw or x is not None:
        _need(x, "x", torch.bfloat16, dev, ndim=2, shape=(T, K))
    outs = {}
    for name, t, shape in (("dx", dx, (T, K)), ("dW", dW, (N, K)), ("db", db, (N,))):
        if t is True:
            t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        elif t is False:
            t = None
        if t is not None:
            _need(t, name, torch.bfloat16, dev, numel=math.prod(shape))
        outs[name] = t
    dx, dW, db = outs["dx"], outs["dW"], outs["db"]
    s = _shape(T, K, H, Dn, Dr, cos)
    need = int(lib().mla_q_uproj_workspace_size(ctypes.byref(s), 3))
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev, ndim=1)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if prepared is not None:
        _call(lib().mla_q_uproj_bwd_mxfp8_prepared, "mla_q_uproj_bwd_mxfp8_prepared", ctypes.byref(s), _ptr(dq),
              _ptr(prepared[0]), _ptr(prepared[1]), _ptr(x) if want_dw else None, _ptr(cos), _ptr(sin),
              _ptr(pos), _ptr(dx), _ptr(dW), _ptr(db), _ptr(workspace), ws_bytes, _ptr(status),
              _stream(dev, stream))
    else:
        _call(lib().mla_q_uproj_bwd_mxfp8, "mla_q_uproj_bwd_mxfp8", ctypes.byref(s), _ptr(dq),
              _ptr(W) if want_dx else None, _ptr(x) if want_dw else None, _ptr(cos), _ptr(sin), _ptr(pos),
              _ptr(dx), _ptr(dW), _ptr(db), _ptr(workspace), ws_bytes, _ptr(status), _stream(dev, stream))
    return dx, dW, db


def bwd_mxfp8_prepare_weight(W, T, H, Dn, Dr, cos, stream=None):
    """W [N, K] bf16 -> (wt [K, N] E4M3 codes, wt_scales flat, in the GEMM's
    tiled order): the copy ``bwd_mxfp8(..., prepared=...)`` takes in place of
    W, to quantize a weight once for several backward calls."""
    _need(W, "W", torch.bfloat16, ndim=2)
    N, K = W.shape
    G = bwd_mxfp8_layout(max(int(T), 1), K, H, Dn, Dr, cos.shape[0], cos.shape[1])["b_group"]
    return mxfp8_quantize_cols(W, group=G, stream=stream)


def mxfp8_quantize_rows(inp, codes=None, scales=None, stream=None, group=None):
    """Rowwise MXFP8 of a 2-D fp32/bf16 CUDA tensor -> (codes uint8 [R, C], scales uint8 [R, ceil(C/32)]).

    A row pitch larger than C is taken from ``inp.stride(0)`` (the tensor must
    have unit inner stride). With ``group``, the scales come back flat in the
    block-scaled GEMM's tiled order with row groups of that size
    (mxfp8_quantize_rows_tiled)."""
    if inp.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("input must be float32 or bfloat16")
    if not inp.is_cuda or inp.dim() != 2 or inp.stride(1) != 1:
        raise ValueError("input must be a 2-D CUDA tensor with unit inner stride")
    R, C = inp.shape
    ld_in = int(inp.stride(0)) if R > 1 else int(C)
    dev = inp.device
    if codes is None:
        codes = torch.empty((R, C), dtype=torch.uint8, device=dev)
    _need(codes, "codes", torch.uint8, dev, numel=R * C)
    dt = 0 if inp.dtype == torch.float32 else 1
    if group is not None:
        n = int(lib().mxfp8_grouped_scale_bytes(R, (C + 31) // 32, int(group)))
        if scales is None:
            scales = torch.empty((n,), dtype=torch.uint8, device=dev)
        _need(scales, "scales", torch.uint8, dev, numel=n)
        _call(lib().mxfp8_quantize_rows_tiled, "mxfp8_quantize_rows_tiled", R, C, dt, _ptr(inp), ld_in,
              _ptr(codes), _ptr(scales), int(group), _stream(dev, stream))
        return codes, scales
    if scales is None:
        scales = torch.empty((R, (C + 31) // 32), dtype=torch.uint8, device=dev)
    _need(scales, "scales", torch.uint8, dev, numel=R * ((C + 31) // 32))
    _call(lib().mxfp8_quantize_rows, "mxfp8_quantize_rows", R, C, dt, _ptr(inp), ld_in, _ptr(codes),
          _ptr(scales), _stream(dev, stream))
    return codes, scales


def mxfp8_quantize_cols(inp, codes=None, scales=None, stream=None, group=None):
    """Columnwise MXFP8 of a 2-D fp32/bf16 CUDA tensor [R, C], i.e. the rowwise
    quantization of its transpose -> (codes uint8 [C, R], scales uint8
    [C, ceil(R/32)]). A row pitch larger than C is taken from ``inp.stride(0)``.
    With ``group``, the scales come back flat in the block-scaled GEMM's tiled
    order with row groups of that size (mxfp8_quantize_cols_tiled)."""
    if inp.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("input must be float32 or bfloat16")
    if not inp.is_cuda or inp.dim() != 2 or inp.stride(1) != 1:
        raise ValueError("input must be a 2-D CUDA tensor with unit inner stride")
    R, C = inp.shape
    ld_in = int(inp.stride(0)) if R > 1 else int(C)
    dev = inp.device
    if codes is None:
        codes = torch.empty((C, R), dtype=torch.uint8, device=dev)
    _need(codes, "codes", torch.uint8, dev, numel=R * C)
    dt = 0 if inp.dtype == torch.float32 else 1
    if group is not None:
        n = int(lib().mxfp8_grouped_scale_bytes(C, (R + 31) // 32, int(group)))
        if scales is None:
            scales = torch.empty((n,), dtype=torch.uint8, device=dev)
        _need(scales, "scales", torch.uint8, dev, numel=n)
        _call(lib().mxfp8_quantize_cols_tiled, "mxfp8_quantize_cols_tiled", R, C, dt, _ptr(inp), ld_in,
              _ptr(codes), _ptr(scales), int(group), _stream(dev, stream))
        return codes, scales
    if scales is None:
        scales = torch.empty((C, (R + 31) // 32), dtype=torch.uint8, device=dev)
    _need(scales, "scales", torch.uint8, dev, numel=C * ((R + 31) // 32))
    _call(lib().mxfp8_quantize_cols, "mxfp8_quantize_cols", R, C, dt, _ptr(inp), ld_in, _ptr(codes),
          _ptr(scales), _stream(dev, stream))
    return codes, scales


def mxfp8_swizzle_scales(scales, out=None, stream=None, group=128):
    """Row-major E8M0 scales [rows, cols] (uint8 CUDA tensor, unit inner
    stride) -> the 128 x 4 tiled order of block-scaled GEMMs, as a flat uint8
    tensor of mxfp8_grouped_scale_bytes(rows, cols, group) bytes; rows in
    groups of `group`, each padded to whole 128-row tiles (group 128: the
    plain swizzle, mxfp8_swizzle_scales)."""
    if scales.dtype != torch.uint8 or not scales.is_cuda or scales.dim() != 2 or scales.stride(1) != 1:
        raise ValueError("scales must be a 2-D uint8 CUDA tensor with unit inner stride")
    rows, cols = scales.shape
    n = int(lib().mxfp8_grouped_scale_bytes(rows, cols, group))
    if out is None:
        out = torch.empty((n,), dtype=torch.uint8, device=scales.device)
    _need(out, "out", torch.uint8, scales.device, numel=n)
    ld = int(scales.stride(0)) if rows > 1 else int(cols)
    if group == 128:
        _call(lib().mxfp8_swizzle_scales, "mxfp8_swizzle_scales", rows, cols, _ptr(scales), ld, _ptr(out),
              _stream(scales.device, stream))
    else:
        _call(lib().mxfp8_swizzle_scales_grouped, "mxfp8_swizzle_scales_grouped", rows, cols, int(group),
              _ptr(scales), ld, _ptr(out), _stream(scales.device, stream))
    return out


def w_scale_group(T, K, H, Dn, Dr, cs_rows, cs_width) -> int:
    """Row group of W's tiled scales for weight_mode "mxfp8_tiled" (0: none)."""
    s = Shape(T=T, K=K, H=H, Dn=Dn, Dr=Dr, reserved=0, cs_rows=cs_rows, cs_width=cs_width)
    return int(lib().mla_q_uproj_w_scale_group(ctypes.byref(s)))


def kv_fwd(c_kv, W, k_pe, cos, sin, H, Dn, Dv, Dr, pos=None, o_key=None, o_value=None, status=None, stream=None):
    """KV side: kv = c_kv W^T split per head -> (o_key [T, H, Dn + Dr] bf16 with
    the rotated shared k_pe after each head's Dn channels, o_value [T, H, Dv] bf16)."""
    dev = c_kv.device
    _need(c_kv, "c_kv", torch.bfloat16, ndim=2)
    T, K = c_kv.shape
    _need(W, "W", torch.bfloat16, dev, shape=(H * (Dn + Dv), K))
    _need(k_pe, "k_pe", torch.bfloat16, dev, numel=T * Dr)
    _tables(cos, sin, dev, T, pos)
    _status(status, dev)
    if o_key is None:
        o_key = torch.empty((T, H, Dn + Dr), dtype=torch.bfloat16, device=dev)
    if o_value is None:
        o_value = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    _need(o_key, "o_key", torch.bfloat16, dev, numel=T * H * (Dn + Dr))
    _need(o_value, "o_value", torch.bfloat16, dev, numel=T * H * Dv)
    s = KvShape(T=T, K=K, H=H, Dn=Dn, Dv=Dv, Dr=Dr, cs_rows=cos.shape[0], cs_width=cos.shape[1])
    _call(lib().mla_kv_uproj_fwd, "mla_kv_uproj_fwd", ctypes.byref(s), _ptr(c_kv), _ptr(W), _ptr(k_pe),
          _ptr(cos), _ptr(sin), _ptr(pos), _ptr(o_key), _ptr(o_value), _ptr(status), _stream(dev, stream))
    return o_key, o_value
