"""Python face of the fp64 CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package. It shares no code with
the CUDA path (``up_proj_gemm_gb300``) and never imports it; the CUDA path
never imports this.

The C library is built on first use (``gcc -O2 -fopenmp -ffp-contract=off``);
``build()`` compiles it explicitly. Every function here only marshals numpy
arrays into the C routines and composes them in the order the method runs:
decode -> linear (+bias) -> RoPE -> (MXFP8 quantize) for the forward, RoPE
backward -> dgrad / wgrad / bgrad for the backward.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_ARG = 1
ERR_ROPE_WIDTH = 2
ERR_POS_RANGE = 8


class OracleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"oracle {what}: status {status}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (no-op when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.POINTER
_d = _P(ctypes.c_double)
_f = _P(ctypes.c_float)
_u8 = _P(ctypes.c_uint8)
_u16 = _P(ctypes.c_uint16)
_i32 = _P(ctypes.c_int32)
_i64p = _P(ctypes.c_int64)
_i64 = ctypes.c_int64
_i32v = ctypes.c_int32


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            sig = {
                "oracle_num_threads": (ctypes.c_int, []),
                "oracle_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "oracle_decode_bf16": (None, [_i64, _u16, _d]),
                "oracle_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "oracle_e8m0_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "oracle_mxfp8_dequantize": (None, [_i64, _i64, _u8, _u8, _d]),
                "oracle_e8m0_exponent": (ctypes.c_int, [ctypes.c_double]),
                "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "oracle_mxfp8_quantize": (None, [_i64, _i64, _d, _i64, _u8, _u8]),
                "oracle_linear": (None, [_i64, _i64, _i64, _d, _d, _d, _d]),
                "oracle_rope_fwd": (ctypes.c_int, [_i64, _i32v, _i32v, _i32v, _d, _f, _f, _i64,
                                                    _i64, _i32, _d]),
                "oracle_rope_bwd": (ctypes.c_int, [_i64, _i32v, _i32v, _i32v, _d, _f, _f, _i64,
                                                    _i64, _i32, _d]),
                "oracle_dgrad": (None, [_i64, _i64, _i64, _d, _d, _d]),
                "oracle_wgrad": (None, [_i64, _i64, _i64, _d, _d, _i64p, _i64, _d]),
                "oracle_bgrad": (None, [_i64, _i64, _d, _d]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle's row-parallel loops use."""
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------- scalars
def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e8m0_exponent(amax: float) -> int:
    return int(_load().oracle_e8m0_exponent(float(amax)))


def e8m0_decode(byte: int) -> float:
    return _load().oracle_e8m0_decode(int(byte))


# ------------------------------------------------------------------ arrays
def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_decode_bf16(b.size, _ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double))
    return out


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes [R, C] uint8 and scales [R, ceil(C/32)] uint8 -> float64 [R, C]."""
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    R, C = c.shape
    assert s.shape == (R, (C + 31) // 32)
    out = np.empty((R, C), np.float64)
    _load().oracle_mxfp8_dequantize(R, C, _ptr(c, ctypes.c_uint8), _ptr(s, ctypes.c_uint8),
                                    _ptr(out, ctypes.c_double))
    return out


def mxfp8_quantize(values: np.ndarray):
    """Rowwise MXFP8 of a 2-D float64 array -> (codes uint8 [R, C], scales uint8 [R, nb])."""
    v = _c(values, np.float64)
    R, C = v.shape
    nb = (C + 31) // 32
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R, nb), np.uint8)
    _load().oracle_mxfp8_quantize(R, C, _ptr(v, ctypes.c_double), C, _ptr(codes, ctypes.c_uint8),
                                  _ptr(scales, ctypes.c_uint8))
    return codes, scales


def mxfp8_quantize_columns(values: np.ndarray):
    """Columnwise MXFP8 of a 2-D float64 array [R, C]: blocks of 32 consecutive
    rows of each column, i.e. the rowwise quantization of the transpose ->
    (codes uint8 [C, R], scales uint8 [C, ceil(R/32)]). TransformerEngine PR
    "Add support for fused Q Up-Proj GEMM/RoPE/Quant", Greptile summary (the
    transpose among the MXFP8 quantization helpers)."""
    return mxfp8_quantize(np.ascontiguousarray(np.asarray(values, np.float64).T))


def mxfp8_swizzle_scales(scales: np.ndarray) -> np.ndarray:
    """Row-major E8M0 scales [rows, cols] -> the tiled order of block-scaled
    GEMMs (TransformerEngine PR "Add support for fused Q Up-Proj
    GEMM/RoPE/Quant": the GEMM scale swizzle): tiles of 128 rows x 4 columns,
    512 bytes each, tile (i, j) at (i * ceil(cols/4) + j) * 512; inside, row r
    and column c at (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4); padding 0.
    Written out element by element from that definition."""
    rows, cols = scales.shape
    tiles_c = (cols + 3) // 4
    out = np.zeros(((rows + 127) // 128) * 128 * tiles_c * 4, np.uint8)
    for r in range(rows):
        for c in range(cols):
            tile = (r // 128) * tiles_c + c // 4
            out[tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)] = scales[r, c]
    return out


def linear(x: np.ndarray, W: np.ndarray, b=None) -> np.ndarray:
    """y = x W^T (+ b) in fp64; x [T, K], W [N, K], b [N]."""
    x = _c(x, np.float64)
    W = _c(W, np.float64)
    T, K = x.shape
    N, K2 = W.shape
    assert K == K2
    bb = None if b is None else _c(b, np.float64)
    y = np.empty((T, N), np.float64)
    _load().oracle_linear(T, K, N, _ptr(x, ctypes.c_double), _ptr(W, ctypes.c_double),
                          _ptr(bb, ctypes.c_double), _ptr(y, ctypes.c_double))
    return y


def _rope(fn, y, H, Dn, Dr, cos, sin, pos):
    y = _c(y, np.float64)
    T = y.shape[0]
    assert y.size == T * H * (Dn + Dr)
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    assert cos.shape == sin.shape and cos.ndim == 2
    cs_rows, cs_width = cos.shape
    p = None if pos is None else _c(pos, np.int32)
    out = np.empty((T, H, Dn + Dr), np.float64)
    st = fn(T, H, Dn, Dr, _ptr(y, ctypes.c_double), _ptr(cos, ctypes.c_float),
            _ptr(sin, ctypes.c_float), cs_rows, cs_width, _ptr(p, ctypes.c_int32),
            _ptr(out, ctypes.c_double))
    if st != OK:
        raise OracleError(st, fn.__name__)
    return out


def rope_fwd(y, H, Dn, Dr, cos, sin, pos=None) -> np.ndarray:
    """Rotate-half RoPE on y [T, H*(Dn+Dr)] -> q [T, H, Dn+Dr] (fresh array)."""
    return _rope(_load().oracle_rope_fwd, y, H, Dn, Dr, cos, sin, pos)


def rope_bwd(dq, H, Dn, Dr, cos, sin, pos=None) -> np.ndarray:
    """Transpose of the RoPE Jacobian applied to dq [T, H, Dn+Dr] -> dq_pre."""
    return _rope(_load().oracle_rope_bwd, dq, H, Dn, Dr, cos, sin, pos)


def backward_mxfp8(dq, x, W, H, Dn, Dr, cos, sin, pos=None):
    """MXFP8 backward (the low-precision backward beyond the fused bf16 one;
    TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant"
    names the MXFP8 quantization helpers it would use, the rowwise copy and
    its transpose; the pages give no formula, so this is the plain reading):
    dq_pre = the exact (fp64) RoPE backward of dq (rope_bwd); every GEMM
    operand quantized along its reduction dimension with the MXFP8 rule:
    dgrad's along the channels (rowwise MXFP8 of dq_pre [T, N], columnwise
    of W [N, K]), wgrad's along the tokens (columnwise MXFP8 of dq_pre and of
    x [T, K]); dx, dW = exact products of the dequantized operands; db = the
    token sum of dq_pre.
    Returns dict(dx, dW, db, dq_pre, qa, qa_s, qb, qb_s, wt, wt_s, xt, xt_s)."""
    T = dq.shape[0]
    dqp = rope_bwd(dq, H, Dn, Dr, cos, sin, pos).reshape(T, -1)
    qa, qa_s = mxfp8_quantize(dqp)                 # [T, N], blocks along N
    qb, qb_s = mxfp8_quantize_columns(dqp)         # [N, T], blocks along T
    wt, wt_s = mxfp8_quantize_columns(W)           # [K, N], blocks along N
    xt, xt_s = mxfp8_quantize_columns(x)           # [K, T], blocks along T
    A = mxfp8_dequantize(qa, qa_s)
    B = mxfp8_dequantize(wt, wt_s)
    dx = A @ B.T
    dW = mxfp8_dequantize(qb, qb_s) @ mxfp8_dequantize(xt, xt_s).T
    return dict(dx=dx, dW=dW, db=dqp.sum(axis=0), dq_pre=dqp, qa=qa, qa_s=qa_s, qb=qb, qb_s=qb_s, wt=wt,
                wt_s=wt_s, xt=xt, xt_s=xt_s)


def kv_forward(c_kv, W, k_pe, H, Dn, Dv, Dr, cos, sin, pos=None):
    """The KV side of the attention block (Megatron-LM PR "Fix fused MLA YaRN
    RoPE query kernel corrupting upstream tensor in-place", Solution section:
    the KV path writes fresh o_key and o_value buffers; the pages give no
    formula, this is the plain MLA reading): kv = c_kv W^T as [T, H, Dn + Dv];
    o_key [T, H, Dn + Dr] = the first Dn channels of each head followed by the
    shared k_pe [T, Dr] rotated by rotate-half RoPE (same table and positions
    as the query), the same for every head; o_value [T, H, Dv] = the last Dv
    channels of each head. All float64 in, float64 out."""
    c_kv = np.asarray(c_kv, np.float64)
    T = c_kv.shape[0]
    kv = linear(c_kv, W).reshape(T, H, Dn + Dv)
    kr = rope_fwd(np.asarray(k_pe, np.float64).reshape(T, Dr), 1, 0, Dr, cos, sin, pos).reshape(T, 1, Dr)
    o_key = np.concatenate([kv[:, :, :Dn], np.broadcast_to(kr, (T, H, Dr))], axis=2)
    return o_key, np.ascontiguousarray(kv[:, :, Dn:])


def dgrad(dq_pre: np.ndarray, W: np.ndarray) -> np.ndarray:
    """dx = dq_pre W; dq_pre [T, N], W [N, K] -> [T, K]."""
    g = _c(dq_pre.reshape(dq_pre.shape[0], -1), np.float64)
    W = _c(W, np.float64)
    T, N = g.shape
    N2, K = W.shape
    assert N == N2
    dx = np.empty((T, K), np.float64)
    _load().oracle_dgrad(T, K, N, _ptr(g, ctypes.c_double), _ptr(W, ctypes.c_double),
                         _ptr(dx, ctypes.c_double))
    return dx


def wgrad(dq_pre: np.ndarray, x: np.ndarray, rows=None) -> np.ndarray:
    """dW = dq_pre^T x; dq_pre [T, N], x [T, K] -> [N, K] (or only ``rows``)."""
    g = _c(dq_pre.reshape(dq_pre.shape[0], -1), np.float64)
    x = _c(x, np.float64)
    T, N = g.shape
    T2, K = x.shape
    assert T == T2
    r = None if rows is None else _c(rows, np.int64)
    nrows = N if r is None else r.size
    dW = np.empty((nrows, K), np.float64)
    _load().oracle_wgrad(T, K, N, _ptr(g, ctypes.c_double), _ptr(x, ctypes.c_double),
                         _ptr(r, ctypes.c_int64), nrows, _ptr(dW, ctypes.c_double))
    return dW


def bgrad(dq_pre: np.ndarray) -> np.ndarray:
    """db = sum over tokens of dq_pre [T, N] -> [N]."""
    g = _c(dq_pre.reshape(dq_pre.shape[0], -1), np.float64)
    T, N = g.shape
    db = np.empty((N,), np.float64)
    _load().oracle_bgrad(T, N, _ptr(g, ctypes.c_double), _ptr(db, ctypes.c_double))
    return db


# ------------------------------------------------------------- composites
def forward(x, W, H, Dn, Dr, cos, sin, pos=None, b=None, quantize=False):
    """Full forward on fp64 operands: linear (+bias) -> RoPE [-> MXFP8].

    x [T, K], W [N, K], b [N] or None (all float64, already decoded).
    Returns q [T, H, D] float64, and with ``quantize`` also (codes [T, H, D],
    scales [T, H, ceil(D/32)]) from quantizing each head's D channels."""
    y = linear(x, W, b)
    q = rope_fwd(y, H, Dn, Dr, cos, sin, pos)
    if not quantize:
        return q
    T, D = q.shape[0], Dn + Dr
    codes, scales = mxfp8_quantize(q.reshape(T * H, D))
    return q, codes.reshape(T, H, D), scales.reshape(T, H, -1)


def backward(dq, x, W, H, Dn, Dr, cos, sin, pos=None, want=("dx", "dW", "db"), wgrad_rows=None):
    """RoPE backward then the linear backward, all fp64.

    dq [T, H, D], x [T, K], W [N, K] float64. Returns a dict with the requested
    gradients (dW restricted to ``wgrad_rows`` when given) and dq_pre."""
    dq_pre = rope_bwd(dq, H, Dn, Dr, cos, sin, pos).reshape(dq.shape[0], -1)
    out = {"dq_pre": dq_pre}
    if "dx" in want:
        out["dx"] = dgrad(dq_pre, W)
    if "dW" in want:
        out["dW"] = wgrad(dq_pre, x, wgrad_rows)
    if "db" in want:
        out["db"] = bgrad(dq_pre)
    return out
