"""Pins for the fp64 CPU oracle, each independent of the oracle's own code.

The oracle computes ref[m, n] = sum_k A[m, k] B[n, k] in fp64 (spark-kernels,
"how things are measured": a CPU double-precision reference; UwULLM kernel-dev,
section 6: fp64 references for GEMMs).  The pages print no worked GEMM example,
so the pins are the mathematics: exact rational brute force, identity and
permutation operands, one-hot rows, linearity, the transpose identity, a
library fp64 matmul, padding that must never be read, and the sampled mode
against the full one.  Each is chosen so that a dropped term, a wrong index or
stride, a transposed operand or a wrong bf16 decode fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic as syn


def _bf16_value_exact(bits: int) -> Fraction:
    """Exact value of a bf16 bit pattern from the IEEE-754 binary16-brain layout:
    1 sign bit, 8 exponent bits (bias 127), 7 fraction bits."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(f, 1 << 7) * Fraction(1, 1 << 126)
    mant = Fraction(128 + f, 128)
    return sign * mant * (Fraction(2) ** (e - 127))


def _rand(shape, seed, dist="uniform"):
    return syn.matrix(shape[0], shape[1], dist, seed)


def test_bf16_decode_known_patterns():
    # 1.0, -2.0, 1 + 2^-7, 0.5, the smallest normal, a subnormal, -0
    pats = np.array([[0x3F80, 0xC000, 0x3F81, 0x3F00, 0x0080, 0x0001, 0x8000]], dtype=np.uint16)
    one = np.array([[0x3F80]], dtype=np.uint16)
    # C[0, n] = pats[n] * 1.0 reads each pattern back through the oracle
    got = oracle.gemm(one, pats.T.copy())[0]
    want = [float(_bf16_value_exact(int(p))) for p in pats[0]]
    assert got.tolist() == want
    assert want[:4] == [1.0, -2.0, 1.0 + 2.0 ** -7, 0.5]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 4), (5, 7, 8), (8, 8, 8), (3, 1, 6)])
def test_bruteforce_exact_rational(M, N, K):
    A = _rand((M, K), 11 + M)
    B = _rand((N, K), 21 + N)
    ref = oracle.gemm(A, B)
    for m in range(M):
        for n in range(N):
            terms = [_bf16_value_exact(int(A[m, k])) * _bf16_value_exact(int(B[n, k]))
                     for k in range(K)]
            exact = sum(terms, Fraction(0))
            # fp64 summation of K exact products: |err| <= K * 2^-53 * sum |terms|
            bound = float(K * sum(abs(t) for t in terms)) * 2.0 ** -53
            assert abs(ref[m, n] - float(exact)) <= bound + 1e-300


def test_small_integers_exact():
    # integer operands: every partial sum is an integer far below 2^53, so exact
    A = syn.small_int_matrix(9, 40, -4, 4, 3)
    B = syn.small_int_matrix(6, 40, -4, 4, 4)
    Ai = syn.bf16_bits_to_f32(A).astype(np.int64)
    Bi = syn.bf16_bits_to_f32(B).astype(np.int64)
    want = Ai @ Bi.T  # integer arithmetic: exact
    assert np.array_equal(oracle.gemm(A, B), want.astype(np.float64))


def test_identity_gives_A():
    K = 24
    A = _rand((7, K), 5)
    eye = syn.f64_to_bf16_bits(np.eye(K))
    got = oracle.gemm(A, eye)
    assert np.array_equal(got, syn.bf16_bits_to_f32(A).astype(np.float64))


def test_permutation_permutes_columns():
    K = 16
    A = _rand((5, K), 6)
    perm = np.array([3, 0, 15, 7, 7, 1, 12])  # rows of B = unit vectors e_perm
    P = np.zeros((perm.size, K))
    P[np.arange(perm.size), perm] = 1.0
    got = oracle.gemm(A, syn.f64_to_bf16_bits(P))
    want = syn.bf16_bits_to_f32(A).astype(np.float64)[:, perm]
    assert np.array_equal(got, want)


def test_one_hot_rows_select_B_columns():
    K = 32
    B = _rand((9, K), 8)
    hot = np.array([0, 31, 4])
    H = np.zeros((hot.size, K))
    H[np.arange(hot.size), hot] = 1.0
    got = oracle.gemm(syn.f64_to_bf16_bits(H), B)
    want = syn.bf16_bits_to_f32(B).astype(np.float64)[:, hot].T
    assert np.array_equal(got, want)


def test_closed_form_constant_operands():
    # A = 1.5 everywhere, B[n, :] = 2^-n: ref[m, n] = K * 1.5 * 2^-n exactly
    M, N, K = 3, 5, 100
    A = syn.f64_to_bf16_bits(np.full((M, K), 1.5))
    B = syn.f64_to_bf16_bits(np.repeat(2.0 ** -np.arange(N), K).reshape(N, K))
    want = np.tile(K * 1.5 * 2.0 ** -np.arange(N), (M, 1))
    assert np.array_equal(oracle.gemm(A, B), want)


def test_alternating_signs_cancel_in_order():
    # A[m,k] = (-1)^k, B = 1: even K sums to exactly 0, odd K to exactly 1
    for K in (10, 11):
        A = syn.f64_to_bf16_bits((-1.0) ** np.arange(K)[None, :])
        B = syn.f64_to_bf16_bits(np.ones((2, K)))
        assert oracle.gemm(A, B).tolist() == [[float(K % 2)] * 2]


def test_transpose_identity_bitwise():
    # (A B^T)^T = B A^T: the same products in the same k order, so bit-equal
    A = _rand((13, 37), 31)
    B = _rand((11, 37), 32)
    assert np.array_equal(oracle.gemm(A, B).T, oracle.gemm(B, A))


def test_linearity_in_A_and_B():
    rng_a1, rng_a2, rng_b1, rng_b2 = (_rand((6, 50), s, "normal:1") for s in (41, 42, 43, 44))
    # exact small-integer coefficients keep the combinations exactly representable
    f = syn.bf16_bits_to_f32
    a1, a2 = f(rng_a1).astype(np.float64), f(rng_a2).astype(np.float64)
    b1, b2 = f(rng_b1).astype(np.float64), f(rng_b2).astype(np.float64)
    # 2*a1 is exact in bf16; a1 + a2 is not, so check linearity on each term
    two_a1 = syn.f64_to_bf16_bits(2.0 * a1)
    assert np.array_equal(oracle.gemm(two_a1, rng_b1), 2.0 * oracle.gemm(rng_a1, rng_b1))
    neg_b2 = syn.f64_to_bf16_bits(-b2)
    assert np.array_equal(oracle.gemm(rng_a2, neg_b2), -oracle.gemm(rng_a2, rng_b2))
    # additivity over a split of the k range: [A1 | A2] [B1 | B2]^T = A1 B1^T + A2 B2^T
    A = np.concatenate([rng_a1, rng_a2], axis=1)
    B = np.concatenate([rng_b1[:6], rng_b2[:6]], axis=1)
    lhs = oracle.gemm(A, B)
    rhs = oracle.gemm(rng_a1, rng_b1[:6]) + oracle.gemm(rng_a2, rng_b2[:6])
    scale = np.abs(a1) @ np.abs(b1[:6]).T + np.abs(a2) @ np.abs(b2[:6]).T
    assert np.all(np.abs(lhs - rhs) <= 100 * 2.0 ** -53 * scale)
    # additivity in A: rows stacked give stacked results
    assert np.array_equal(oracle.gemm(np.concatenate([rng_a1, rng_a2]), rng_b1),
                          np.concatenate([oracle.gemm(rng_a1, rng_b1), oracle.gemm(rng_a2, rng_b1)]))


def test_matches_numpy_fp64_matmul():
    M, N, K = 192, 160, 256
    A = _rand((M, K), 51)
    B = _rand((N, K), 52)
    a = syn.bf16_bits_to_f32(A).astype(np.float64)
    b = syn.bf16_bits_to_f32(B).astype(np.float64)
    want = a @ b.T
    got = oracle.gemm(A, B)
    scale = np.abs(a) @ np.abs(b).T
    assert np.all(np.abs(got - want) <= 2 * K * 2.0 ** -53 * scale)
    assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


def test_leading_dimensions_never_read_padding():
    M, N, K = 4, 6, 20
    A = syn.matrix(M, K, "uniform", 61, ld=K + 13)  # padding = NaN patterns
    B = syn.matrix(N, K, "uniform", 62, ld=K + 5)
    got = oracle.gemm(A, B, K=K)
    assert np.isfinite(got).all()
    assert np.array_equal(got, oracle.gemm(A[:, :K].copy(), B[:, :K].copy()))


def test_sampled_equals_full_bitwise():
    M, N, K = 40, 50, 64
    A = _rand((M, K), 71)
    B = _rand((N, K), 72)
    rows = syn.sample_indices(M, 9, 1)
    cols = syn.sample_indices(N, 7, 2)
    full = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm_sampled(A, B, rows, cols), full[np.ix_(rows, cols)])


def test_threads_do_not_change_bits():
    A = _rand((33, 70), 81)
    B = _rand((17, 70), 82)
    assert np.array_equal(oracle.gemm(A, B, threads=1), oracle.gemm(A, B, threads=5))


def test_empty_and_zero_k():
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((4, 0), dtype=np.uint16)
    assert np.array_equal(oracle.gemm(A, B), np.zeros((3, 4)))
    assert oracle.gemm(np.zeros((0, 5), np.uint16), np.zeros((2, 5), np.uint16)).shape == (0, 2)


def test_transposed_operand_would_fail():
    # a non-square case where using B[k, n] instead of B[n, k] changes the answer
    A = _rand((2, 3), 91)
    B = _rand((3, 3), 92)
    good = oracle.gemm(A, B)
    wrong = oracle.gemm(A, B.T.copy())
    assert not np.array_equal(good, wrong)
