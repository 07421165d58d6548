"""The C oracle under AddressSanitizer and UndefinedBehaviorSanitizer: a copy
of oracle.c built with -fsanitize=address,undefined (UB aborts) runs every
exported routine on small ragged inputs, including partial MXFP8 blocks,
non-finite values, positions restarting, a wide cos/sin table, and
out-of-range or narrow-table arguments it must reject. A memory error or
undefined behaviour fails the child process. CPU only.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
sys.path.insert(0, __ROOT__)
import oracle
oracle._LIB_PATH = __LIB__
rng = np.random.default_rng(0)

def table(rows, width):
    ang = np.arange(rows)[:, None] * (10000.0 ** (-np.arange(width) / width))[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)

# quantizer: partial blocks, zeros, NaN/Inf, rows and columns
v = rng.standard_normal((7, 70)) * 4.0
v[1, 3] = np.nan
v[2, 40] = -np.inf
v[3, :] = 0.0
c, s = oracle.mxfp8_quantize(v)
oracle.mxfp8_dequantize(c, s)
oracle.mxfp8_quantize_columns(v)
oracle.mxfp8_swizzle_scales(s)
for code in range(256):
    oracle.e4m3_decode(code)
    oracle.e8m0_decode(code)
oracle.e8m0_exponent(0.0)
oracle.e4m3_encode(-0.0)

# forward / backward at ragged shapes, with and without bias, pos restarting
for T, K, H, Dn, Dr in [(37, 24, 3, 32, 16), (5, 8, 2, 0, 64), (19, 40, 1, 64, 32)]:
    D = Dn + Dr
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((H * D, K)) * 0.1
    b = rng.standard_normal(H * D)
    dq = rng.standard_normal((T, H, D))
    cos, sin = table(11, Dr + 4)
    pos = (np.arange(T) % 11).astype(np.int32)
    oracle.forward(x, W, H, Dn, Dr, cos, sin, pos, b, quantize=True)
    oracle.forward(x, W, H, Dn, Dr, cos, sin, pos, None, quantize=False)
    oracle.backward(dq, x, W, H, Dn, Dr, cos, sin, pos)
    if Dr in (32, 64) and D % 32 == 0:
        oracle.backward_mxfp8(dq, x, W, H, Dn, Dr, cos, sin, pos)
    # rejections: a position past the table, a table narrower than Dr
    for bad in (lambda: oracle.forward(x, W, H, Dn, Dr, cos, sin, pos + 11),
                lambda: oracle.forward(x, W, H, Dn, Dr, cos[:, :Dr - 2], sin[:, :Dr - 2], pos)):
        try:
            bad()
        except (oracle.OracleError, ValueError, AssertionError):
            pass
        else:
            raise SystemExit("a bad argument was not rejected")

# KV side
c_kv = rng.standard_normal((13, 16))
Wkv = rng.standard_normal((2 * (32 + 32), 16)) * 0.1
k_pe = rng.standard_normal((13, 16))
cos, sin = table(13, 16)
oracle.kv_forward(c_kv, Wkv, k_pe, 2, 32, 32, 16, cos, sin)
# the sanitized build is the one loaded, with the ASan runtime in the process
assert oracle._lib._name == __LIB__, oracle._lib._name
maps = open("/proc/self/maps").read()
assert "libasan" in maps and "liboracle_san" in maps
print("sanitized oracle ok")
'''


def test_oracle_under_asan_ubsan(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    asan = subprocess.run([gcc, "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.exists(asan):
        pytest.skip("no AddressSanitizer runtime")
    lib = tmp_path / "liboracle_san.so"
    subprocess.run([gcc, "-O1", "-g", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer",
                    "-o", str(lib), os.path.join(ROOT, "oracle", "oracle.c"), "-lm"], check=True)
    env = dict(os.environ, LD_PRELOAD=asan, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1", OMP_NUM_THREADS="2")
    code = CHILD.replace("__ROOT__", repr(ROOT)).replace("__LIB__", repr(str(lib)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0 and "sanitized oracle ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
    assert "runtime error" not in r.stderr, r.stderr[-4000:]
