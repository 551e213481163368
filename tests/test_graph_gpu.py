"""Calls are graph-capturable: they enqueue only on the caller's stream ("The
kernels that were there", "The bench that lied": a launch on the wrong stream
records nothing and the replay returns stale output)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


@pytest.mark.parametrize("M,N,K,fn", [(2048, 2048, 2048, "gemm"), (1000, 520, 1000, "gemm"),
                                      (2, 4096, 11008, "gemv"), (16, 4096, 11008, "gemv"),
                                      (64, 11008, 4096, "gemm")])
def test_capture_and_replay(M, N, K, fn):
    A_bits = syn.matrix(M, K, "normal:1", 51)
    B_bits = syn.matrix(N, K, "normal:0.02", 52)
    A, B = to_device(A_bits), to_device(B_bits)
    ld = -(-N // 8) * 8
    Cbuf = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")
    C = Cbuf[:, :N]
    call = (lambda: sg.gemm_bf16(A, B, C)) if fn == "gemm" else (lambda: sg.gemv_bf16(A, B, C))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()  # warm-up outside capture (workspace allocation)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    Cbuf.view(torch.int16).fill_(0x7FC0)  # NaN sentinels: a replay that records nothing shows
    torch.cuda.synchronize()
    ref = oracle.gemm(A_bits, B_bits)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert_close(to_bits(C), ref, K, f"replay {fn} {M}x{N}x{K}")
        Cbuf.view(torch.int16).fill_(0x7FC0)
