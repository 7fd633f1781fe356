"""CPU oracle for GGUF Q4_K / Q6_K / Q8_0 / IQ4_XS x Q8 integer matmul (ctypes over plain C).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. The
CUDA library and its Python binding never import it, and it imports nothing
from them.

The arithmetic lives in ``oracle.c`` (scalar loops, exact int64 sub-block
sums, fp64 combine; the Q8 quantizer in fp32 exactly as written). This module
only compiles that file with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

Q4K_BYTES = 144
Q6K_BYTES = 210
Q8_0_BYTES = 34
IQ4XS_BYTES = 136

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, no FP contraction,
    pthreads for sharing output rows among threads, see set_threads)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    deps = [_SRC, os.path.join(_HERE, "oracle.h")]
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(d) for d in deps)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c99", "-Wall", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def set_threads(n: int) -> int:
    """Threads the matmul routines may use (output rows are shared out; every
    output is still computed by one thread in the same order, so results do
    not depend on it). Returns the count in use."""
    return int(_load().oracle_set_threads(int(n)))


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_quantize_q8.argtypes = [P, I, I, P, P, P]
    lib.oracle_silu_mul.argtypes = [P, P, I, P]
    lib.oracle_q4k_fields.argtypes = [P, P, P, P, P, P]
    lib.oracle_q4k_fields.restype = None
    lib.oracle_q6k_fields.argtypes = [P, P, P, P]
    lib.oracle_q6k_fields.restype = None
    lib.oracle_q8_0_fields.argtypes = [P, P, P]
    lib.oracle_q8_0_fields.restype = None
    lib.oracle_dequant_q8_0.argtypes = [P, I, I, P]
    lib.oracle_iq4xs_fields.argtypes = [P, P, P, P, P]
    lib.oracle_iq4xs_fields.restype = None
    lib.oracle_dequant_iq4xs.argtypes = [P, P, I, I, P]
    lib.oracle_matmul_iq4xs_q8.argtypes = [P, P, P, P, I, I, I, P, P, P]
    lib.oracle_matmul_q8_0_q8.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.oracle_dequant_q4k.argtypes = [P, I, I, P]
    lib.oracle_dequant_q6k.argtypes = [P, I, I, P]
    lib.oracle_dequant_q8.argtypes = [P, P, I, I, P]
    lib.oracle_matmul_q4k_q8.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.oracle_matmul_q6k_q8.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.oracle_gemv_f64.argtypes = [P, P, I, I, I, P]
    lib.oracle_set_threads.argtypes = [I]
    lib.oracle_set_threads.restype = I
    for name in ("oracle_quantize_q8", "oracle_dequant_q4k", "oracle_dequant_q6k",
                 "oracle_dequant_q8", "oracle_matmul_q4k_q8", "oracle_matmul_q6k_q8",
                 "oracle_gemv_f64", "oracle_dequant_q8_0", "oracle_matmul_q8_0_q8",
                 "oracle_dequant_iq4xs", "oracle_matmul_iq4xs_q8", "oracle_silu_mul"):
        getattr(lib, name).restype = ctypes.c_int
    lib.oracle_set_threads(1)
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle: bad shape for {what}")


def half_to_double(h: int) -> float:
    return _load().oracle_half_to_double(int(h) & 0xFFFF)


def quantize_q8(x: np.ndarray):
    """Q8 activation quantization of fp32 x [M][K] -> (qs int8, d8 f32, s8 f32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    qs = np.zeros((M, K), np.int8)
    d8 = np.zeros((M, K // 32), np.float32)
    s8 = np.zeros((M, K // 32), np.float32)
    _check(_load().oracle_quantize_q8(_p(x), M, K, _p(qs), _p(d8), _p(s8)), "quantize_q8")
    return qs, d8, s8


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u = g / (1 + e^-g) * u in fp64, from fp32 g and u of one shape."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    assert g.shape == u.shape
    h = np.zeros(g.shape, np.float64)
    _check(_load().oracle_silu_mul(_p(g), _p(u), g.size, _p(h)), "silu_mul")
    return h


def q4k_fields(blk: np.ndarray):
    """Decoded fields of one 144-byte Q4_K super-block: (d, dmin, sc[8], m[8], q[256])."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == Q4K_BYTES
    d = ctypes.c_double()
    dmin = ctypes.c_double()
    sc = np.zeros(8, np.int32)
    mn = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_q4k_fields(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return d.value, dmin.value, sc, mn, q


def q6k_fields(blk: np.ndarray):
    """Decoded fields of one 210-byte Q6_K super-block: (d, s[16], q[256])."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == Q6K_BYTES
    d = ctypes.c_double()
    s = np.zeros(16, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_q6k_fields(_p(blk), ctypes.byref(d), _p(s), _p(q))
    return d.value, s, q


def q8_0_fields(blk: np.ndarray):
    """Decoded fields of one 34-byte Q8_0 block: (d, q[32])."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == Q8_0_BYTES
    d = ctypes.c_double()
    q = np.zeros(32, np.int32)
    _load().oracle_q8_0_fields(_p(blk), ctypes.byref(d), _p(q))
    return d.value, q


def _codebook(codebook) -> np.ndarray:
    cb = np.ascontiguousarray(codebook, dtype=np.int8)
    assert cb.shape == (16,), "an IQ4_XS codebook is 16 int8 values"
    return cb


def iq4xs_fields(blk: np.ndarray, codebook):
    """Decoded fields of one 136-byte IQ4_XS super-block: (d, ls[8], v[256]),
    v the codebook value of each weight's index."""
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size == IQ4XS_BYTES
    cb = _codebook(codebook)
    d = ctypes.c_double()
    ls = np.zeros(8, np.int32)
    v = np.zeros(256, np.int32)
    _load().oracle_iq4xs_fields(_p(blk), _p(cb), ctypes.byref(d), _p(ls), _p(v))
    return d.value, ls, v


def _weight_shape(W: np.ndarray, K: int, nbytes: int):
    W = np.ascontiguousarray(W, dtype=np.uint8)
    nsb = K // 256
    assert K % 256 == 0 and W.size % (nsb * nbytes) == 0
    return W, W.size // (nsb * nbytes)


def dequant_q4k(W: np.ndarray, K: int) -> np.ndarray:
    W, N = _weight_shape(W, K, Q4K_BYTES)
    w = np.zeros((N, K), np.float64)
    _check(_load().oracle_dequant_q4k(_p(W), N, K, _p(w)), "dequant_q4k")
    return w


def dequant_q6k(W: np.ndarray, K: int) -> np.ndarray:
    W, N = _weight_shape(W, K, Q6K_BYTES)
    w = np.zeros((N, K), np.float64)
    _check(_load().oracle_dequant_q6k(_p(W), N, K, _p(w)), "dequant_q6k")
    return w


def dequant_q8_0(W: np.ndarray, K: int) -> np.ndarray:
    W, N = _weight_shape(W, K, 8 * Q8_0_BYTES)
    w = np.zeros((N, K), np.float64)
    _check(_load().oracle_dequant_q8_0(_p(W), N, K, _p(w)), "dequant_q8_0")
    return w


def dequant_iq4xs(W: np.ndarray, K: int, codebook) -> np.ndarray:
    W, N = _weight_shape(W, K, IQ4XS_BYTES)
    cb = _codebook(codebook)
    w = np.zeros((N, K), np.float64)
    _check(_load().oracle_dequant_iq4xs(_p(W), _p(cb), N, K, _p(w)), "dequant_iq4xs")
    return w


def dequant_q8(qs: np.ndarray, d8: np.ndarray) -> np.ndarray:
    qs = np.ascontiguousarray(qs, dtype=np.int8)
    d8 = np.ascontiguousarray(d8, dtype=np.float32)
    M, K = qs.shape
    xhat = np.zeros((M, K), np.float64)
    _check(_load().oracle_dequant_q8(_p(qs), _p(d8), M, K, _p(xhat)), "dequant_q8")
    return xhat


def _matmul(fn, W, qs, d8, K, nbytes, want_isum, isum_per_row):
    W, N = _weight_shape(W, K, nbytes)
    qs = np.ascontiguousarray(qs, dtype=np.int8)
    d8 = np.ascontiguousarray(d8, dtype=np.float32)
    M = qs.shape[0]
    assert qs.shape == (M, K) and d8.shape == (M, K // 32)
    y = np.zeros((M, N), np.float64)
    ab = np.zeros((M, N), np.float64)
    isum = np.zeros((M, N, isum_per_row), np.int32) if want_isum else None
    rc = fn(_p(W), _p(qs), _p(d8), M, N, K, _p(y), _p(ab),
            _p(isum) if want_isum else None)
    _check(rc, "matmul")
    return y, ab, isum


def matmul_q4k_q8(W, qs, d8, K, want_isum=False):
    """Integer route: y [M][N] (double), sum|terms| [M][N], isums [M][N][K/32] or None."""
    return _matmul(_load().oracle_matmul_q4k_q8, W, qs, d8, K, Q4K_BYTES, want_isum, K // 32)


def matmul_q6k_q8(W, qs, d8, K, want_isum=False):
    """Integer route: y [M][N] (double), sum|terms| [M][N], isums [M][N][K/16] or None."""
    return _matmul(_load().oracle_matmul_q6k_q8, W, qs, d8, K, Q6K_BYTES, want_isum, K // 16)


def matmul_q8_0_q8(W, qs, d8, K, want_isum=False):
    """Integer route: y [M][N] (double), sum|terms| [M][N], isums [M][N][K/32] or None."""
    return _matmul(_load().oracle_matmul_q8_0_q8, W, qs, d8, K, 8 * Q8_0_BYTES, want_isum, K // 32)


def matmul_iq4xs_q8(W, qs, d8, K, codebook, want_isum=False):
    """Integer route: y [M][N] (double), sum|terms| [M][N], isums [M][N][K/32] or None."""
    cb = _codebook(codebook)
    fn = _load().oracle_matmul_iq4xs_q8

    def call(Wp, qp, dp, M, N, K_, yp, ap, ip):
        return fn(Wp, _p(cb), qp, dp, M, N, K_, yp, ap, ip)
    return _matmul(call, W, qs, d8, K, IQ4XS_BYTES, want_isum, K // 32)


def gemv_f64(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Plain definition y[m][n] = sum_k w[n][k] * x[m][k] in double."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    N, K = w.shape
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    _check(_load().oracle_gemv_f64(_p(w), _p(x), M, N, K, _p(y)), "gemv_f64")
    return y


def matmul(qtype: int, W, qs, d8, K, want_isum=False, codebook=None):
    """Dispatch on the GGUF type id (8 = Q8_0, 12 = Q4_K, 14 = Q6_K,
    23 = IQ4_XS, which needs its codebook)."""
    if qtype == 8:
        return matmul_q8_0_q8(W, qs, d8, K, want_isum)
    if qtype == 12:
        return matmul_q4k_q8(W, qs, d8, K, want_isum)
    if qtype == 14:
        return matmul_q6k_q8(W, qs, d8, K, want_isum)
    if qtype == 23:
        return matmul_iq4xs_q8(W, qs, d8, K, codebook, want_isum)
    raise ValueError(f"unsupported type {qtype}")
