"""Pins for the gated-MLP oracle, oracle.swiglu = silu(A . Wg^T) * (A . Wu^T).

The pages' fused MLP epilogue (spark-kernels, "the bf16 gemm" and its fused
MLP numbers) computes the SwiGLU of the gate and up projections in one pass.
The pins are mathematics the oracle's own code does not restate:
- sigmoid(ln 3) = 3/4 and sigmoid(0) = 1/2 exactly, so silu(+-ln 3) and
  silu(0) have closed forms;
- silu(g) - silu(-g) = g for every g, so negating the gate weights (exact in
  bf16) changes the output by exactly (A . Wg^T) * (A . Wu^T), the product of
  two independently pinned GEMMs;
- scaling the up weights by 2 (exact) scales the output by 2; zero gate weights
  give exactly 0; silu(g) * g >= 0 when the gate and up weights are the same;
- the limits silu(x) -> x (x -> +inf) and -> 0 (x -> -inf) without NaN.
A dropped SiLU, a sigmoid in its place, a wrong sign inside the exponential,
or the gate and up operands exchanged each fail at least one of these.
"""
import math

import numpy as np

import oracle
import synthetic as syn


def test_silu_closed_forms():
    ln3 = math.log(3.0)
    x = np.array([0.0, ln3, -ln3, 2 * math.log(2.0)])
    got = oracle.silu(x)
    # sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4, sigmoid(-ln 3) = 1/4, sigmoid(ln 4) = 4/5
    want = np.array([0.0, 0.75 * ln3, -0.25 * ln3, 0.8 * 2 * math.log(2.0)])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)


def test_silu_limits_and_no_nan():
    got = oracle.silu(np.array([50.0, -50.0, -1000.0, 1000.0]))
    assert got[0] == 50.0 and got[3] == 1000.0          # sigmoid rounds to 1 in fp64
    assert -1e-19 < got[1] < 0.0                           # -50 e^-50 ~ -9.6e-21
    assert got[2] == 0.0 and np.all(np.isfinite(got))     # the -inf limit, as -0


def _neg(bits):
    return bits ^ np.uint16(0x8000)


def test_negated_gate_changes_output_by_the_product():
    M, N, K = 7, 11, 96
    A = syn.matrix(M, K, "normal:1", 501)
    Wg = syn.matrix(N, K, "normal:0.2", 502)
    Wu = syn.matrix(N, K, "normal:0.2", 503)
    d = oracle.swiglu(A, Wg, Wu) - oracle.swiglu(A, _neg(Wg), Wu)
    prod = oracle.gemm(A, Wg) * oracle.gemm(A, Wu)
    np.testing.assert_allclose(d, prod, rtol=1e-12, atol=1e-14)


def test_scaling_up_weights_and_zero_gate():
    M, N, K = 5, 9, 64
    A = syn.matrix(M, K, "normal:1", 511)
    Wg = syn.matrix(N, K, "normal:0.2", 512)
    Wu = syn.matrix(N, K, "normal:0.2", 513)
    Wu2 = syn.f64_to_bf16_bits(2.0 * syn.bf16_bits_to_f32(Wu).astype(np.float64))
    np.testing.assert_array_equal(oracle.swiglu(A, Wg, Wu2), 2.0 * oracle.swiglu(A, Wg, Wu))
    zero = np.zeros_like(Wg)
    assert np.all(oracle.swiglu(A, zero, Wu) == 0.0)
    # the up product is not the gate: zero up weights give 0 whatever the gate
    assert np.all(oracle.swiglu(A, Wg, np.zeros_like(Wu)) == 0.0)


def test_same_weights_are_never_negative():
    M, N, K = 6, 8, 48
    A = syn.matrix(M, K, "normal:1", 521)
    W = syn.matrix(N, K, "normal:0.3", 522)
    out = oracle.swiglu(A, W, W)          # silu(g) * g = g^2 sigmoid(g) >= 0
    assert np.all(out >= 0.0)
    assert np.count_nonzero(out) == out.size


def test_swapped_operands_would_fail():
    # exchanging gate and up is caught: silu(g) u != silu(u) g for these inputs
    M, N, K = 4, 6, 32
    A = syn.matrix(M, K, "normal:1", 531)
    Wg = syn.matrix(N, K, "normal:0.3", 532)
    Wu = syn.matrix(N, K, "normal:0.3", 533)
    assert not np.allclose(oracle.swiglu(A, Wg, Wu), oracle.swiglu(A, Wu, Wg))
