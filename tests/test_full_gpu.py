"""Parity at the workloads' full sizes, through gemm_bf16 exactly as bench.py calls it.

4096^3 and the 7B-model MLP projections are checked element by element against
the full fp64 oracle.  8192^3 and 16384^3 are checked on the intersections of
128 seeded rows and 128 seeded columns (gemm3 benchmarks page, "Correctness": a
128 x 128 sample of row/column intersections), plus two properties that hold at
any size and cover every tile: scaling A by 2 and negating B are exact in bf16
and in fp32 accumulation, so the outputs must be exactly 2C and -C.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import skinny_gemv_gb300 as sg  # noqa: E402


def _gemm(A, B):
    C = sg.gemm_bf16(A, B)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("name", ["sq4096", "mlp_up", "mlp_down"])
def test_full_oracle(name):
    w = syn.WORKLOADS[name]
    A_bits, B_bits = w.a(), w.b()
    C = _gemm(to_device(A_bits), to_device(B_bits))
    stats = assert_close(to_bits(C), oracle.gemm(A_bits, B_bits), w.K, name)
    assert stats["n"] == w.M * w.N


@pytest.mark.parametrize("name", ["sq8192", "sq16384"])
def test_sampled_oracle_and_exact_identities(name):
    w = syn.WORKLOADS[name]
    A_bits, B_bits = w.a(), w.b()
    A, B = to_device(A_bits), to_device(B_bits)
    C = _gemm(A, B)
    rows = syn.sample_indices(w.M, 128, 1)
    cols = syn.sample_indices(w.N, 128, 2)
    got = to_bits(C)[np.ix_(rows, cols)]
    assert_close(got, oracle.gemm_sampled(A_bits, B_bits, rows, cols), w.K, name + " sampled")
    assert torch.isfinite(C.float()).all()
    # every tile: C(2A, B) == 2 C(A, B) and C(A, -B) == -C(A, B), bit for bit
    C2 = _gemm(A * 2, B)
    assert torch.equal(C2, C * 2)
    del C2
    Cn = _gemm(A, -B)
    assert torch.equal(Cn, -C)
