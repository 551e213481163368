"""Pins of the fp64 attention oracle (oracle.attention, oracle.attention_combine)
to facts that do not come from the oracle itself: closed forms (uniform weights
when every score is equal, the two-key logistic weights, log n for the
log-sum-exp of n equal scores), the one-visible-key case, invariances of the
softmax (a common shift of a row's scores, a joint permutation of keys and
values), linearity in V, the grouped-head mapping, the causal rule on a prefix,
and the split-KV merge identity.  A dropped scale, a transposed operand, a wrong
mask offset or a wrong head mapping fails at least one of them.

The operation is the attention of the spark-kernels page ("attention": flash
attention with the online softmax, causal tiles skipped above the diagonal,
split-KV tails merged by a combine step, short-query tiles for decode).
"""
import math

import numpy as np
import pytest

import oracle


def rnd(rng, *shape):
    return rng.standard_normal(shape)


def visible_counts(Sq, Sk, causal):
    if not causal:
        return np.full(Sq, Sk)
    return np.clip(np.arange(Sq) + (Sk - Sq) + 1, 0, Sk)


@pytest.mark.parametrize("Sq,Sk,causal", [(6, 6, True), (3, 9, True), (5, 5, False), (9, 4, True), (1, 12, True)])
def test_zero_queries_average_visible_values(Sq, Sk, causal):
    rng = np.random.default_rng(1)
    B, H, D = 2, 3, 8
    Q = np.zeros((B, Sq, H, D))
    K = rnd(rng, B, Sk, H, D)
    V = rnd(rng, B, Sk, H, D)
    O, lse = oracle.attention(Q, K, V, causal=causal, return_lse=True)
    n = visible_counts(Sq, Sk, causal)
    for i in range(Sq):
        if n[i] == 0:  # no visible key: zero output, lse = -inf
            assert np.all(O[:, i] == 0) and np.all(np.isneginf(lse[:, :, i]))
            continue
        want = V[:, : n[i]].mean(axis=1)  # [B, H, D]
        np.testing.assert_allclose(O[:, i], want, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n[i]), rtol=0, atol=1e-13)


def test_equal_keys_give_uniform_weights():
    rng = np.random.default_rng(2)
    B, Sq, Sk, H, D = 1, 4, 7, 2, 16
    Q = rnd(rng, B, Sq, H, D)
    K = np.broadcast_to(rnd(rng, B, 1, H, D), (B, Sk, H, D)).copy()
    V = rnd(rng, B, Sk, H, D)
    O = oracle.attention(Q, K, V)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=1, keepdims=True), O.shape), atol=1e-13)


def test_two_keys_logistic_weights():
    # o = sigma(s0 - s1) v0 + sigma(s1 - s0) v1 with sigma(x) = (1 + tanh(x / 2)) / 2
    rng = np.random.default_rng(3)
    D = 8
    Q = rnd(rng, 1, 3, 1, D)
    K = rnd(rng, 1, 2, 1, D)
    V = rnd(rng, 1, 2, 1, D)
    scale = 0.7
    O = oracle.attention(Q, K, V, scale=scale)
    for i in range(3):
        s0 = scale * float(Q[0, i, 0] @ K[0, 0, 0])
        s1 = scale * float(Q[0, i, 0] @ K[0, 1, 0])
        w0 = 0.5 * (1.0 + math.tanh((s0 - s1) / 2.0))
        want = w0 * V[0, 0, 0] + (1.0 - w0) * V[0, 1, 0]
        np.testing.assert_allclose(O[0, i, 0], want, rtol=1e-13, atol=1e-14)


def test_default_scale_is_inverse_sqrt_d():
    rng = np.random.default_rng(4)
    D = 32
    Q, K, V = rnd(rng, 1, 2, 1, D), rnd(rng, 1, 5, 1, D), rnd(rng, 1, 5, 1, D)
    np.testing.assert_allclose(oracle.attention(Q, K, V), oracle.attention(Q, K, V, scale=1 / math.sqrt(D)),
                               rtol=0, atol=0)
    # doubling the scale equals doubling the queries
    np.testing.assert_allclose(oracle.attention(Q, K, V, scale=2 / math.sqrt(D)), oracle.attention(2 * Q, K, V),
                               atol=1e-13)


def test_first_causal_row_is_first_value():
    rng = np.random.default_rng(5)
    Q, K, V = rnd(rng, 2, 6, 4, 8), rnd(rng, 2, 6, 4, 8), rnd(rng, 2, 6, 4, 8)
    O = oracle.attention(Q, K, V, causal=True)
    np.testing.assert_array_equal(O[:, 0], V[:, 0])


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(6)
    D, Sk = 8, 10
    K = rnd(rng, 1, Sk, 1, D) * 0.01
    K[0, 7, 0, 0] = 1.0
    Q = np.zeros((1, 1, 1, D))
    Q[0, 0, 0, 0] = 400.0  # score gap ~ 400 / sqrt(8) > 140: other weights < e^-140
    V = rnd(rng, 1, Sk, 1, D)
    O = oracle.attention(Q, K, V)
    np.testing.assert_allclose(O[0, 0, 0], V[0, 7, 0], rtol=1e-12, atol=1e-14)


def test_common_score_shift_changes_nothing():
    # an extra dimension with q = c and k = 1 adds c * scale to every score of a row
    rng = np.random.default_rng(7)
    B, Sq, Sk, H, D = 1, 5, 9, 2, 8
    Q, K, V = rnd(rng, B, Sq, H, D), rnd(rng, B, Sk, H, D), rnd(rng, B, Sk, H, D)
    Q2 = np.concatenate([Q, np.full((B, Sq, H, 1), 37.0)], axis=3)
    K2 = np.concatenate([K, np.ones((B, Sk, H, 1))], axis=3)
    V2 = np.concatenate([V, np.zeros((B, Sk, H, 1))], axis=3)
    sc = 1 / math.sqrt(D)
    O1, l1 = oracle.attention(Q, K, V, causal=True, scale=sc, return_lse=True)
    O2, l2 = oracle.attention(Q2, K2, V2, causal=True, scale=sc, return_lse=True)
    np.testing.assert_allclose(O2[..., :D], O1, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + 37.0 * sc, atol=1e-12)


def test_joint_key_permutation_invariance():
    rng = np.random.default_rng(8)
    Q, K, V = rnd(rng, 2, 4, 2, 16), rnd(rng, 2, 11, 2, 16), rnd(rng, 2, 11, 2, 16)
    perm = rng.permutation(11)
    np.testing.assert_allclose(oracle.attention(Q, K[:, perm], V[:, perm]), oracle.attention(Q, K, V), atol=1e-13)
    # permuting queries permutes the rows of the output
    qp = rng.permutation(4)
    np.testing.assert_allclose(oracle.attention(Q[:, qp], K, V), oracle.attention(Q, K, V)[:, qp], atol=1e-13)


def test_linear_in_values():
    rng = np.random.default_rng(9)
    Q, K = rnd(rng, 1, 6, 2, 8), rnd(rng, 1, 6, 2, 8)
    V1, V2 = rnd(rng, 1, 6, 2, 8), rnd(rng, 1, 6, 2, 8)
    lhs = oracle.attention(Q, K, V1 + 2.5 * V2, causal=True)
    rhs = oracle.attention(Q, K, V1, causal=True) + 2.5 * oracle.attention(Q, K, V2, causal=True)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)


def test_grouped_heads_equal_repeated_kv_heads():
    rng = np.random.default_rng(10)
    B, Sq, Sk, H, Hkv, D = 2, 5, 7, 6, 2, 8
    Q, K, V = rnd(rng, B, Sq, H, D), rnd(rng, B, Sk, Hkv, D), rnd(rng, B, Sk, Hkv, D)
    rep = H // Hkv
    Kr, Vr = np.repeat(K, rep, axis=2), np.repeat(V, rep, axis=2)
    np.testing.assert_allclose(oracle.attention(Q, K, V, causal=True), oracle.attention(Q, Kr, Vr, causal=True),
                               atol=1e-14)
    # and head h really reads kv head h // rep: swapping the kv heads moves the result
    Ks, Vs = K[:, :, ::-1], V[:, :, ::-1]
    O = oracle.attention(Q, Ks, Vs)
    O_ref = oracle.attention(Q, K, V)
    np.testing.assert_allclose(O[:, :, :rep], oracle.attention(Q[:, :, :rep], K[:, :, 1:2], V[:, :, 1:2]), atol=1e-13)
    assert not np.allclose(O, O_ref)


def test_causal_row_is_noncausal_attention_over_its_prefix():
    rng = np.random.default_rng(11)
    Sq, Sk = 4, 10
    Q, K, V = rnd(rng, 1, Sq, 1, 8), rnd(rng, 1, Sk, 1, 8), rnd(rng, 1, Sk, 1, 8)
    O = oracle.attention(Q, K, V, causal=True)
    for i in range(Sq):
        n = i + Sk - Sq + 1
        want = oracle.attention(Q[:, i:i + 1], K[:, :n], V[:, :n])
        np.testing.assert_allclose(O[:, i:i + 1], want, atol=1e-14)


@pytest.mark.parametrize("splits", [[0, 5, 13], [0, 1, 2, 13], [0, 12, 13]])
def test_split_keys_merge_to_full_attention(splits):
    rng = np.random.default_rng(12)
    B, Sq, Sk, H, D = 1, 3, 13, 2, 8
    Q, K, V = rnd(rng, B, Sq, H, D), rnd(rng, B, Sk, H, D), rnd(rng, B, Sk, H, D)
    full, lse = oracle.attention(Q, K, V, return_lse=True)
    parts = [oracle.attention(Q, K[:, a:b], V[:, a:b], return_lse=True) for a, b in zip(splits[:-1], splits[1:])]
    O, L = oracle.attention_combine(parts)
    np.testing.assert_allclose(O, full, atol=1e-13)
    np.testing.assert_allclose(L, lse, atol=1e-13)


def test_bf16_inputs_decode_exactly():
    # bf16 bit patterns of small integers: 0x3F80 = 1.0, 0x4000 = 2.0, 0xC040 = -3.0
    Q = np.array([[[[0x3F80, 0x4000]]]], dtype=np.uint16)
    K = np.array([[[[0x3F80, 0x0000]], [[0x0000, 0xC040]]]], dtype=np.uint16)  # [1, 2, 1, 2]
    V = np.array([[[[0x4000, 0x0000]], [[0x0000, 0x3F80]]]], dtype=np.uint16)
    O = oracle.attention(Q, K, V, scale=1.0)
    s0, s1 = 1.0, -6.0
    w0 = 0.5 * (1.0 + math.tanh((s0 - s1) / 2.0))
    np.testing.assert_allclose(O[0, 0, 0], [2.0 * w0, 1.0 - w0], rtol=0, atol=1e-15)
