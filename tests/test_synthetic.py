"""The seeded input generators: determinism, distributions and bf16 rounding."""
import numpy as np
import pytest
import torch

import synthetic as syn


def test_splitmix64_reference_values():
    # splitmix64 of the stream started at seed 0: the published generator's first
    # outputs (Steele, Lea, Flood, "Fast splittable pseudorandom number generators").
    got = syn.splitmix64(0, 0, 3).tolist()
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_slices_match_full_stream():
    full = syn.splitmix64(123, 0, 1000)
    assert np.array_equal(syn.splitmix64(123, 400, 100), full[400:500])
    n_full = syn.normal(5, 1000, 1.0)
    assert np.array_equal(syn.normal(5, 200, 1.0, start=300), n_full[300:500])


def test_matrix_chunking_is_invisible():
    a = syn.matrix(5, 7, "normal:0.02", 9)
    flat = syn.f64_to_bf16_bits(syn.normal(9, 35, 0.02))
    assert np.array_equal(a.reshape(-1), flat)


def test_distribution_moments():
    u = syn.uniform_pm1(1, 200000)
    assert u.min() >= -1 and u.max() < 1
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    z = syn.normal(2, 200000, 0.02)
    assert abs(z.mean()) < 2e-4 and abs(z.std() - 0.02) < 2e-4


def test_rne_matches_torch_on_fp32_values():
    x = np.random.default_rng(0).standard_normal(200000).astype(np.float32)
    ours = syn.f64_to_bf16_bits(x.astype(np.float64))
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


@pytest.mark.parametrize("value,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),            # tie, even neighbour below
    (1.0 + 3 * 2.0 ** -8, 0x3F82),        # tie, even neighbour above
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above the tie: rounds up
    (-(1.0 + 2.0 ** -8), 0xBF80),
    (0.0, 0x0000),
])
def test_rne_ties_from_fp64(value, bits):
    # a tie in fp64 that an fp32 detour would not see: 1 + 2^-8 + 2^-40 rounds up
    assert int(syn.f64_to_bf16_bits(np.array([value]))[0]) == bits


def test_workload_table():
    w = syn.WORKLOADS
    assert (w["sq4096"].M, w["sq4096"].N, w["sq4096"].K) == (4096, 4096, 4096)
    assert (w["mlp_up"].N, w["mlp_up"].K) == (11008, 4096)
    assert (w["mlp_down"].N, w["mlp_down"].K) == (4096, 11008)
    dec = [x for x in w.values() if x.name.startswith("dec")]
    assert sorted({x.M for x in dec}) == [1, 2, 16, 64] and len(dec) == 8
    assert len({x.cfg for x in w.values()}) == len(w)
    # decode traffic per the scope table: 90.21 MB at M = 1
    assert abs(w["dec1_up"].decode_bytes / 1e6 - 90.21) < 0.01


def test_sample_indices():
    s = syn.sample_indices(16384, 128, 7)
    assert s.size == 128 and np.all(np.diff(s) > 0) and s[-1] < 16384
    assert np.array_equal(s, syn.sample_indices(16384, 128, 7))


def test_matrix_rows_equal_the_full_matrix_rows():
    for dist in ("uniform", "normal:0.02"):
        full = syn.matrix(37, 50, dist, 99)
        idx = np.array([0, 3, 17, 36])
        assert np.array_equal(syn.matrix_rows(idx, 50, dist, 99), full[idx])
