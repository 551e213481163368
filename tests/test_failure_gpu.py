"""Bounded waits: a launch whose wait can never complete gives up, records the
timeout, unwinds and exits, and the GPU stays usable.

The failure is made on the host: sg_debug_inject_missing_tx makes the next
GEMM launch expect more TMA bytes on its first stage than its copies deliver,
so the MMA issuer's barrier wait runs out (a flag that nothing sets).  Nothing
traps, faults or hangs; the kernel's own wait bound ends it.
"""
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402

DEFAULT_TIMEOUT_NS = 2_000_000_000


@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
def test_missing_copy_times_out_and_gpu_recovers(path):
    M, N, K = 512, 512, 512
    A_bits = syn.matrix(M, K, "uniform", 201)
    B_bits = syn.matrix(N, K, "uniform", 202)
    A, B = to_device(A_bits), to_device(B_bits)
    lib = sg.load()
    st, _ = sg.check_device_errors()
    assert st == sg.SG_OK
    try:
        sg.set_wait_timeout_ns(20_000_000)  # 20 ms per wait
        lib.sg_debug_inject_missing_tx(4096)
        C = sg.gemm_bf16(A, B, path=path)
        st, detail = sg.check_device_errors()
        assert st == sg.SG_ERR_TIMEOUT, (st, detail)
        assert detail[0] in (1, 2, 3, 4, 5), detail  # a recorded wait code
        # the error word was cleared: the next check is clean
        assert sg.check_device_errors()[0] == sg.SG_OK
    finally:
        lib.sg_debug_inject_missing_tx(0)
        sg.set_wait_timeout_ns(DEFAULT_TIMEOUT_NS)
    # the context is still usable and results are correct again
    C = sg.gemm_bf16(A, B, path=path)
    torch.cuda.synchronize()
    assert sg.check_device_errors()[0] == sg.SG_OK
    assert_close(to_bits(C), oracle.gemm(A_bits, B_bits), K, "after recovery")
