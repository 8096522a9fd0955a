"""W12 oracle — TEST INFRASTRUCTURE ONLY.

Plain scalar C (``w12_oracle.c``) behind ctypes.  Only ``tests/``, the smoke
check and the benchmark's CPU-baseline leg may import this package; the product
library never does, and the two share no code.  See ``w12_oracle.h`` for what
each routine computes and which passages of the SpecPilot pages it follows
("StargazerX0/SpecPilot" §What it is; "SpecPilot" §Differentiation; "SpecPilot:
an agent doubled speculative decoding speed, and the 10.87x needs context" §The
mechanisms it found).

Parity status: encode/decode and the fp64 GEMM are pinned by the CPU tests
(exhaustive BF16 round trip, a hand-worked 2x2 blob, a hand-worked blob whose
escape bytes and segment headers are listed by hand, table-optimality and
escape-mass invariants, size closed form, normal-CDF escape rate, numpy
float64 matmul, one-hot and small-integer exact products); the Q8 copy and
its fp64 product by hand-worked rows and products.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w12_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_w12.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP for the baseline GEMM); return the .so path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "w12_oracle.h"))
    ):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-fPIC", "-shared", "-fopenmp",
         _SRC, "-o", tmp, "-lm"],
        check=True,
    )
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_q8_size.argtypes = [i64, i64]
    lib.oracle_q8_size.restype = i64
    lib.oracle_q8_encode.argtypes = [u16p, i64, i64, u8p, i64]
    lib.oracle_q8_encode.restype = i64
    lib.oracle_q8_decode.argtypes = [u8p, i64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int8)]
    lib.oracle_q8_decode.restype = ctypes.c_int
    lib.oracle_w12_size.argtypes = [u16p, i64, i64]
    lib.oracle_w12_size.restype = i64
    lib.oracle_w12_encode.argtypes = [u16p, i64, i64, u8p, i64]
    lib.oracle_w12_encode.restype = i64
    lib.oracle_w12_decode.argtypes = [u8p, i64, u16p]
    lib.oracle_w12_decode.restype = ctypes.c_int
    lib.oracle_w12_dims.argtypes = [u8p, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.oracle_w12_dims.restype = ctypes.c_int
    lib.oracle_gemm_f64.argtypes = [u16p, u16p, i64, i64, i64, f64p]
    lib.oracle_gemm_f64.restype = None
    lib.oracle_w12_gemm_f64.argtypes = [u16p, u8p, i64, i64, f64p, ctypes.c_int]
    lib.oracle_w12_gemm_f64.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = [ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _u16(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _u8(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _as_u16(w) -> np.ndarray:
    w = np.ascontiguousarray(w)
    if w.dtype != np.uint16:
        raise TypeError("oracle expects BF16 bit patterns as uint16")
    return w


def encoded_size(w: np.ndarray) -> int:
    w = _as_u16(w)
    n, k = w.shape
    size = _load().oracle_w12_size(_u16(w), n, k)
    if size < 0:
        raise ValueError("bad shape")
    return int(size)


def encode(w: np.ndarray) -> np.ndarray:
    """W12 v1 blob of the N x K BF16 matrix ``w`` (uint16 bit patterns)."""
    w = _as_u16(w)
    n, k = w.shape
    size = encoded_size(w)
    blob = np.empty(size, dtype=np.uint8)
    got = _load().oracle_w12_encode(_u16(w), n, k, _u8(blob), size)
    if got != size:
        raise RuntimeError("oracle encode failed")
    return blob


def dims(blob: np.ndarray) -> tuple[int, int]:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    n, k = ctypes.c_int64(), ctypes.c_int64()
    if _load().oracle_w12_dims(_u8(blob), blob.size, ctypes.byref(n), ctypes.byref(k)) != 0:
        raise ValueError("malformed W12 blob")
    return n.value, k.value


def decode(blob: np.ndarray) -> np.ndarray:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    n, k = dims(blob)
    out = np.empty((n, k), dtype=np.uint16)
    if _load().oracle_w12_decode(_u8(blob), blob.size, _u16(out)) != 0:
        raise ValueError("malformed W12 blob")
    return out


def gemm_f64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[M,N] = x[M,K] . w[N,K]^T in float64 over BF16 bit patterns."""
    x = _as_u16(x)
    w = _as_u16(w)
    m, k = x.shape
    n, k2 = w.shape
    if k != k2:
        raise ValueError("K mismatch")
    y = np.empty((m, n), dtype=np.float64)
    _load().oracle_gemm_f64(_u16(x), _u16(w), m, n, k, y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return y


def argmax_f64(x: np.ndarray, w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """LM-head argmax ("SpecPilot: an agent doubled speculative decoding
    speed, and the 10.87x needs context", §The mechanisms it found): per token
    m, the row n with the largest logit sum_k x[m,k] * W[n,k] (fp64, from
    gemm_f64), ties to the smallest n, a NaN logit ranking as -infinity.
    Returns (indices [M], logits [M, N])."""
    y = gemm_f64(x, w)
    ranked = np.where(np.isnan(y), -np.inf, y)
    return np.argmax(ranked, axis=1).astype(np.int64), y


def w12_gemm_f64(x: np.ndarray, blob: np.ndarray, threads: int = 0) -> np.ndarray:
    """fp64 GEMM over the weights a blob holds (decode, then dot products)."""
    x = _as_u16(x)
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    n, k = dims(blob)
    m = x.shape[0]
    if x.shape[1] != k:
        raise ValueError("K mismatch")
    y = np.empty((m, n), dtype=np.float64)
    rc = _load().oracle_w12_gemm_f64(_u16(x), _u8(blob), blob.size, m,
                                     y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), threads)
    if rc != 0:
        raise ValueError("malformed W12 blob")
    return y


def q8_encode(w: np.ndarray) -> np.ndarray:
    """Q8 v1 blob (INT8 per-row copy) of the N x K BF16 bit patterns."""
    w = _as_u16(w)
    n, k = w.shape
    size = int(_load().oracle_q8_size(n, k))
    blob = np.empty(size, dtype=np.uint8)
    if _load().oracle_q8_encode(_u16(w), n, k, _u8(blob), size) != size:
        raise ValueError("bad arguments or a non-finite weight")
    return blob


def q8_decode(blob: np.ndarray, n: int, k: int) -> tuple[np.ndarray, np.ndarray]:
    """(scales float32 [N], q int8 [N, K]) held by a Q8 blob."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    s = np.empty(n, dtype=np.float32)
    q = np.empty((n, k), dtype=np.int8)
    rc = _load().oracle_q8_decode(_u8(blob), blob.size, s.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                  q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)))
    if rc != 0:
        raise ValueError("malformed Q8 blob")
    return s, q


def q8_gemm_f64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[m, n] = s[n] * sum_k x[m, k] * q[n, k] in float64, (s, q) the
    oracle's own Q8 copy of w."""
    x = _as_u16(x)
    w = _as_u16(w)
    s, q = q8_decode(q8_encode(w), w.shape[0], w.shape[1])
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return (xf @ q.astype(np.float64).T) * s.astype(np.float64)[None, :]


def max_threads(threads: int = 0) -> int:
    return int(_load().oracle_max_threads(threads))
