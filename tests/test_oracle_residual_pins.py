"""Pins for oracle.gemm_residual = A . B^T + R (the down projection with its
residual add, the second fused MLP epilogue of the pages' "next" steps).

- zero weights give exactly R's values, decoded independently here from the
  bf16 layout (sign, 8 exponent bits, 7 fraction bits);
- a zero residual gives exactly oracle.gemm (itself pinned);
- the residual enters linearly: R2 - R1 shifts the output by exactly that
  difference when both are small integers;
- a residual read from a wider row pitch uses only its first N columns.
A dropped residual, a residual added twice, a transposed residual or a wrong
decode each fail one of these."""
import numpy as np

import oracle
import synthetic as syn


def _bf16_value(bits: int) -> float:
    sign = -1.0 if bits & 0x8000 else 1.0
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0:
        return sign * f * 2.0 ** -133
    return sign * (1.0 + f / 128.0) * 2.0 ** (e - 127)


def test_zero_weights_give_the_residual():
    M, N, K = 5, 7, 16
    A = syn.matrix(M, K, "normal:1", 601)
    B = np.zeros((N, K), dtype=np.uint16)
    R = syn.matrix(M, N, "normal:3", 602)
    want = np.array([[_bf16_value(int(b)) for b in row] for row in R])
    np.testing.assert_array_equal(oracle.gemm_residual(A, B, R), want)


def test_zero_residual_is_the_gemm():
    M, N, K = 6, 9, 40
    A = syn.matrix(M, K, "normal:1", 611)
    B = syn.matrix(N, K, "normal:0.1", 612)
    np.testing.assert_array_equal(oracle.gemm_residual(A, B, np.zeros((M, N), np.uint16)), oracle.gemm(A, B))


def test_residual_enters_linearly():
    M, N, K = 4, 6, 24
    A = syn.small_int_matrix(M, K, -2, 2, 621)
    B = syn.small_int_matrix(N, K, -2, 2, 622)
    R1 = syn.small_int_matrix(M, N, -50, 50, 623)
    R2 = syn.small_int_matrix(M, N, -50, 50, 624)
    d = oracle.gemm_residual(A, B, R2) - oracle.gemm_residual(A, B, R1)
    want = np.array([[_bf16_value(int(b)) for b in row] for row in R2]) - \
        np.array([[_bf16_value(int(b)) for b in row] for row in R1])
    np.testing.assert_array_equal(d, want)


def test_padded_residual_and_no_transpose():
    M, N, K = 3, 5, 8
    A = syn.matrix(M, K, "normal:1", 631)
    B = syn.matrix(N, K, "normal:1", 632)
    R = syn.matrix(M, N, "normal:1", 633, ld=16)
    got = oracle.gemm_residual(A, B, R)
    assert got.shape == (M, N)
    np.testing.assert_array_equal(got - oracle.gemm(A, B),
                                  np.array([[_bf16_value(int(b)) for b in row[:N]] for row in R]))
