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
e2m1_value(codes)              fp64 values of E2M1 (FP4) codes
e4m3_value(codes)              fp64 values of E4M3 (FP8) codes
nvfp4_dequant(P, S, K)         packed FP4 rows times their 16-element block scales, fp64
gemm_nvfp4(A, SFA, B, SFB, K)  alpha * dequant(A) . dequant(B)^T in fp64 (NVFP4 GEMM)
gemm_nvfp4_sampled(...)        the same at chosen rows x columns
attention(Q, K, V, ...)        softmax(scale Q K^T, causal mask) V per head, fp64, with
                               the log-sum-exp of each row's scores
attention_combine(parts)       merges attention over disjoint key ranges by their
                               log-sum-exps (the split-KV combine step)
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


# ------------------------------------------------------------------ NVFP4
# The dense W4A4 GEMM of the gemm3 benchmarks page ("Implementations": packed
# NVFP4 operands, E4M3 scales over 16-element blocks, alpha): each element is an
# E2M1 code times the E4M3 scale of its block, and the GEMM is the plain sum of
# their products, here in fp64 after decoding every code exactly.

def e2m1_value(codes) -> np.ndarray:
    """E2M1 (FP4): bit 3 sign, bits 2-1 exponent e (bias 1), bit 0 mantissa m.
    e = 0 is subnormal, m * 2**-1; otherwise (1 + m/2) * 2**(e - 1).  There is no
    infinity or NaN: the largest magnitude is 6."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def e4m3_value(codes) -> np.ndarray:
    """E4M3 (FP8, the variant with no infinities): bit 7 sign, bits 6-3 exponent e
    (bias 7), bits 2-0 mantissa m.  e = 0 is subnormal, (m/8) * 2**-6; e = 15 with
    m = 7 is NaN; otherwise (1 + m/8) * 2**(e - 7), up to 448."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def nvfp4_unpack(packed: np.ndarray, K: int) -> np.ndarray:
    """E2M1 codes [rows, K] of packed rows: element k is in byte k // 2, the low
    nibble for even k and the high nibble for odd k."""
    b = np.ascontiguousarray(packed, dtype=np.uint8)[:, :K // 2].astype(np.int64)
    out = np.empty((b.shape[0], K), dtype=np.int64)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def nvfp4_dequant(packed: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    """fp64 values x[r, k] = e2m1(code[r, k]) * e4m3(scale[r, k // 16]); `scales` is
    plain row-major, one code per 16 elements (first K // 16 columns)."""
    assert K % 16 == 0
    v = e2m1_value(nvfp4_unpack(packed, K))
    s = e4m3_value(np.asarray(scales)[:, :K // 16])
    return v * np.repeat(s, 16, axis=1)


def gemm_nvfp4(A: np.ndarray, SFA: np.ndarray, B: np.ndarray, SFB: np.ndarray, K: int,
               alpha: float = 1.0) -> np.ndarray:
    """C[m, n] = alpha * sum_k a[m, k] sa[m, k // 16] b[n, k] sb[n, k // 16] in fp64,
    not rounded to fp16.  A [M, >= K/2] and B [N, >= K/2] are packed codes, SFA and
    SFB plain row-major scale codes.  The sum over k is numpy's fp64 matmul of the
    decoded values (every product is exact in fp64)."""
    return float(alpha) * (nvfp4_dequant(A, SFA, K) @ nvfp4_dequant(B, SFB, K).T)


def gemm_nvfp4_sampled(A, SFA, B, SFB, rows, cols, K: int, alpha: float = 1.0) -> np.ndarray:
    """gemm_nvfp4 at the intersections rows x cols only."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a = nvfp4_dequant(np.asarray(A)[rows], np.asarray(SFA)[rows], K)
    b = nvfp4_dequant(np.asarray(B)[cols], np.asarray(SFB)[cols], K)
    return float(alpha) * (a @ b.T)


# Scaled dot-product attention of one decoder layer, the fused kernel the
# spark-kernels page builds ("attention": flash attention with the online
# softmax, causal tiles above the diagonal skipped, a split-KV schedule merged
# by a combine step, and a short-query tile for decode).  The oracle is the
# definition written out, per (batch, head), in fp64:
#
#   s[i, j] = scale * sum_d q[i, d] k[j, d]          for visible keys j
#   p[i, j] = exp(s[i, j] - max_j s[i, j]),  l[i] = sum_j p[i, j]
#   o[i, :] = sum_j p[i, j] v[j, :] / l[i],  lse[i] = log(l[i]) + max_j s[i, j]
#
# Key j is visible to query i when j < Sk and, if causal, j <= i + (Sk - Sq): the
# queries are the last Sq positions of a sequence whose first Sk positions are the
# keys (a decode step against a cache when Sq < Sk; the usual lower triangle when
# Sq = Sk).  A query with no visible key gets o = 0 and lse = -inf.  Grouped
# query heads share key/value heads: query head h reads key/value head
# h // (H // Hkv).

def _bf16_tensor(x: np.ndarray) -> np.ndarray:
    """fp64 values of a bf16 bit-pattern array of any shape."""
    return (np.asarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, causal: bool = False,
              scale: float | None = None, return_lse: bool = False):
    """Attention of Q [B, Sq, H, D] against K, V [B, Sk, Hkv, D] (bf16 bit patterns
    as uint16, or float arrays taken as exact values); returns fp64 O [B, Sq, H, D]
    and, with return_lse, the fp64 log-sum-exp [B, H, Sq] of each row's scaled
    scores.  scale defaults to 1 / sqrt(D)."""
    def val(x):
        x = np.asarray(x)
        return _bf16_tensor(x) if x.dtype == np.uint16 else x.astype(np.float64)
    q, k, v = val(Q), val(K), val(V)
    Bt, Sq, H, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    assert k.shape == (Bt, Sk, Hkv, D) and v.shape == k.shape and H % Hkv == 0
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    group = H // Hkv
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    visible = np.ones((Sq, Sk), dtype=bool) if not causal else (j <= i + (Sk - Sq))
    O = np.zeros((Bt, Sq, H, D))
    lse = np.full((Bt, H, Sq), -np.inf)
    for b in range(Bt):
        for h in range(H):
            kh = h // group
            s = sc * (q[b, :, h, :] @ k[b, :, kh, :].T)
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            rows = np.isfinite(m[:, 0])
            p = np.where(visible, np.exp(s - np.where(rows[:, None], m, 0.0)), 0.0)
            l = p.sum(axis=1)
            o = p @ v[b, :, kh, :]
            O[b, rows, h, :] = o[rows] / l[rows, None]
            lse[b, h, rows] = np.log(l[rows]) + m[rows, 0]
    return (O, lse) if return_lse else O


def attention_combine(parts) -> tuple[np.ndarray, np.ndarray]:
    """Merges attention results over disjoint key ranges: parts is a sequence of
    (O_p [B, Sq, H, D], lse_p [B, H, Sq]).  With L = log(sum_p exp(lse_p)), the
    result is O = sum_p exp(lse_p - L) O_p and L itself; a part with lse = -inf
    (no visible key) has weight 0."""
    Os = [np.asarray(o, dtype=np.float64) for o, _ in parts]
    Ls = [np.asarray(l, dtype=np.float64) for _, l in parts]
    m = np.max(np.stack(Ls), axis=0)
    finite = np.isfinite(m)
    m0 = np.where(finite, m, 0.0)
    w = [np.where(np.isfinite(l), np.exp(l - m0), 0.0) for l in Ls]
    tot = np.sum(np.stack(w), axis=0)
    L = np.where(finite, np.log(np.where(finite, tot, 1.0)) + m0, -np.inf)
    O = np.zeros_like(Os[0])
    for o, wi in zip(Os, w):
        # weights [B, H, Sq] -> [B, Sq, H, 1]
        wt = np.where(finite, wi / np.where(finite, tot, 1.0), 0.0)
        O += o * np.transpose(wt, (0, 2, 1))[..., None]
    return O, L
