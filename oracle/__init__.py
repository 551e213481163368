"""CPU oracle for C = A . B^T in fp64 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under ``skinny_gemv_gb300``
never does, and the two share no code: the oracle is the plain C file
``gemm_ref.c`` (fp64 sums over k in increasing order of exactly decoded bf16
inputs), built with gcc into ``oracle/_build/libgemm_ref.so``.

Functions
---------
gemm(A, B)                    full fp64 reference, shape (M, N)
gemm_sampled(A, B, rows, cols) the same sum at the intersections rows x cols
silu(x)                        x * sigmoid(x) = x / (1 + exp(-x)), fp64
swiglu(A, Wg, Wu)              silu(A . Wg^T) * (A . Wu^T), fp64 (gated MLP)
gemm_residual(A, B, R)         A . B^T + R, fp64 (a projection with its residual add)
build()                        compile the C oracle (idempotent)

A and B are uint16 arrays of bf16 bit patterns, A[M, lda] and B[N, ldb]; the
first K columns of each row are the operands (K defaults to A.shape[1]).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libgemm_ref.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc -O2 (no fast-math: sums keep their order)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
                               "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm_f64.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_gemm_f64.restype = ctypes.c_int
        lib.oracle_gemm_sampled_f64.argtypes = [p, p, p, p, i64, p, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_gemm_sampled_f64.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16 and x.ndim == 2, (x.dtype, x.shape)
    return x


def gemm(A: np.ndarray, B: np.ndarray, K: int | None = None, threads: int | None = None,
         return_threads: bool = False):
    """fp64 C[M, N] = sum_k A[m, k] B[n, k] over the first K columns."""
    A, B = _u16(A), _u16(B)
    K = A.shape[1] if K is None else K
    M, N = A.shape[0], B.shape[0]
    C = np.zeros((M, N), dtype=np.float64)
    used = _load().oracle_gemm_f64(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K,
                                   A.shape[1], B.shape[1], N, threads or default_threads())
    if used < 0:
        raise ValueError("oracle_gemm_f64: bad arguments")
    return (C, used) if return_threads else C


def gemm_sampled(A: np.ndarray, B: np.ndarray, rows, cols, K: int | None = None,
                 threads: int | None = None, return_threads: bool = False):
    """fp64 out[i, c] = sum_k A[rows[i], k] B[cols[c], k]."""
    A, B = _u16(A), _u16(B)
    K = A.shape[1] if K is None else K
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < A.shape[0])
    assert cols.size == 0 or (cols.min() >= 0 and cols.max() < B.shape[0])
    out = np.zeros((rows.size, cols.size), dtype=np.float64)
    used = _load().oracle_gemm_sampled_f64(A.ctypes.data, B.ctypes.data, out.ctypes.data,
                                           rows.ctypes.data, rows.size, cols.ctypes.data, cols.size,
                                           K, A.shape[1], B.shape[1], threads or default_threads())
    if used < 0:
        raise ValueError("oracle_gemm_sampled_f64: bad arguments")
    return (out, used) if return_threads else out


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU (the swish with unit slope) in fp64: x * sigmoid(x), written as
    x / (1 + exp(-x)).  For x far below zero exp(-x) overflows to inf and the
    quotient is the correct limit, -0 or 0."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(A: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, K: int | None = None,
           threads: int | None = None) -> np.ndarray:
    """The gated MLP's first half: silu(A . Wg^T) * (A . Wu^T), each product an
    fp64 gemm() of the same inputs, the SiLU and the product in fp64 (no
    rounding to bf16).  Wg and Wu are [N, K] bf16 bit patterns."""
    g = gemm(A, Wg, K=K, threads=threads)
    u = gemm(A, Wu, K=K, threads=threads)
    return silu(g) * u


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 values of bf16 bit patterns: the pattern is the high half of the
    fp32 with the same value."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_residual(A: np.ndarray, B: np.ndarray, R: np.ndarray, K: int | None = None,
                  threads: int | None = None) -> np.ndarray:
    """A projection with its residual added: gemm(A, B) + R in fp64, R an [M, N]
    (or wider-pitched [M, ldr]) array of bf16 bit patterns (first N columns)."""
    C = gemm(A, B, K=K, threads=threads)
    return C + _bf16_to_f64(R)[:, :C.shape[1]]
