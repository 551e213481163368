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


def _inject_and_recover(run, check):
    """Runs `run` with a missing-byte injection and a 20 ms wait bound: the launch
    must report SG_ERR_TIMEOUT; then `run` again without it, and `check` it."""
    lib = sg.load()
    assert sg.check_device_errors()[0] == sg.SG_OK
    try:
        sg.set_wait_timeout_ns(20_000_000)
        lib.sg_debug_inject_missing_tx(4096)
        run()
        st, detail = sg.check_device_errors()
        assert st == sg.SG_ERR_TIMEOUT, (st, detail)
        assert detail[0] in (1, 2, 3, 4, 5), detail
        assert sg.check_device_errors()[0] == sg.SG_OK
    finally:
        lib.sg_debug_inject_missing_tx(0)
        sg.set_wait_timeout_ns(DEFAULT_TIMEOUT_NS)
    out = run()
    torch.cuda.synchronize()
    assert sg.check_device_errors()[0] == sg.SG_OK
    check(out)


@pytest.mark.parametrize("Sq,Sk", [(300, 300), (1, 1000)])  # one tile per CTA; key splits and the combine
def test_attention_missing_copy_times_out_and_recovers(Sq, Sk):
    import numpy as np
    H = 2
    Qb = syn.matrix(Sq, H * 128, "normal", 211).reshape(1, Sq, H, 128)
    Kb = syn.matrix(Sk, H * 128, "normal", 212).reshape(1, Sk, H, 128)
    Vb = syn.matrix(Sk, H * 128, "normal", 213).reshape(1, Sk, H, 128)
    dev = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in (Qb, Kb, Vb)]

    def check(O):
        got = oracle._bf16_tensor(O.cpu().view(torch.int16).numpy().view(np.uint16))
        ref = oracle.attention(Qb, Kb, Vb, causal=True)
        W = oracle.attention(Qb, Kb, np.abs(oracle._bf16_tensor(Vb)), causal=True)
        assert np.all(np.abs(got - ref) <= 4e-3 * (np.abs(ref) + W))

    # the tcgen05 kernel, whose copies the injection withholds (the decode kernel
    # that attention_bf16 would pick for Sq = 1 has no waits to time out)
    _inject_and_recover(lambda: sg.attention_bf16(*dev, causal=True, path=sg.PATH_TENSOR_CORE), check)


def test_nvfp4_missing_copy_times_out_and_recovers():
    import numpy as np
    M, N, K = 256, 512, 512
    A, B = syn.nvfp4_codes(M, K, 221), syn.nvfp4_codes(N, K, 222)
    SA, SB = syn.nvfp4_scales(M, K, 223), syn.nvfp4_scales(N, K, 224)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    SAd = sg.nvfp4_pack_scales(torch.from_numpy(SA).cuda(), K)
    SBd = sg.nvfp4_pack_scales(torch.from_numpy(SB).cuda(), K)

    def check(C):
        ref = oracle.gemm_nvfp4(A, SA, B, SB, K)
        got = C.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-2 * np.abs(ref).max())

    _inject_and_recover(lambda: sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K, path=sg.PATH_GEMM), check)
