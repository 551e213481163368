"""Roofline microbenchmarks and the device query run and give plausible numbers
(the bench divides by them, so a broken one would mislead every fraction)."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


def test_device_query():
    d = sg.device_query()
    assert (d["cc_major"], d["cc_minor"]) == (10, 3)
    assert d["sm_count"] >= 100 and d["smem_optin_bytes"] >= 200 * 1024
    assert d["l2_bytes"] >= 64 << 20


def test_tcgen05_peak_is_plausible():
    tflops, mhz = sg.bench_tcgen05_peak(200000)
    # nominal dense bf16 is 2.25 PFLOP/s; a loop that reached far less or more is broken
    assert 800 < tflops < 3000, tflops
    assert 500 < mhz < 2300, mhz


def test_copy_and_read_roofs():
    n = 1 << 29  # 1 GiB
    src = torch.ones(n, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    copy = sg.bench_copy(dst, src, reps=5)
    read = sg.bench_read(src, sink, reps=5)
    assert 2000 < copy < 12000, copy
    assert 2000 < read < 12000, read
