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


def _capture(call):
    """Runs `call` once outside capture (first-call set-up), then captures it."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    return g


@pytest.mark.parametrize("B,Sq,Sk,H,causal,path", [(1, 300, 300, 4, True, sg.PATH_AUTO),
                                                   (1, 1, 2000, 8, True, sg.PATH_AUTO),
                                                   (1, 1, 2000, 8, True, sg.PATH_TENSOR_CORE)])
def test_attention_capture_and_replay(B, Sq, Sk, H, causal, path):
    """Prefill, and the key-split decode step on the CUDA-core decode kernel (AUTO)
    and on the tcgen05 kernel, each with the combine kernel."""
    Qb = syn.matrix(B * Sq, H * 128, "normal", 61).reshape(B, Sq, H, 128)
    Kb = syn.matrix(B * Sk, H * 128, "normal", 62).reshape(B, Sk, H, 128)
    Vb = syn.matrix(B * Sk, H * 128, "normal", 63).reshape(B, Sk, H, 128)
    dev = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in (Qb, Kb, Vb)]
    O = torch.empty((B, Sq, H, 128), dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: sg.attention_bf16(*dev, O=O, causal=causal, path=path))
    ref = oracle.attention(Qb, Kb, Vb, causal=causal)
    W = oracle.attention(Qb, Kb, np.abs(oracle._bf16_tensor(Vb)), causal=causal)
    for _ in range(2):
        O.view(torch.int16).fill_(0x7FC0)
        g.replay()
        torch.cuda.synchronize()
        got = oracle._bf16_tensor(O.cpu().view(torch.int16).numpy().view(np.uint16))
        assert np.all(np.abs(got - ref) <= 4e-3 * (np.abs(ref) + W)), "replayed attention"


def test_nvfp4_capture_and_replay():
    M, N, K = 512, 768, 1024
    A, B = syn.nvfp4_codes(M, K, 71), syn.nvfp4_codes(N, K, 72)
    SA, SB = syn.nvfp4_scales(M, K, 73), syn.nvfp4_scales(N, K, 74)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    SAd = sg.nvfp4_pack_scales(torch.from_numpy(SA).cuda(), K)
    SBd = sg.nvfp4_pack_scales(torch.from_numpy(SB).cuda(), K)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    g = _capture(lambda: sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K, C=C))
    C.fill_(float("nan"))
    torch.cuda.synchronize()
    direct = sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K).clone()
    C.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), direct.view(torch.int16))  # deterministic kernel: same bits
