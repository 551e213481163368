"""Parity of the fused gate/up projection with its SwiGLU epilogue,
gemm_bf16_swiglu: C = silu(A . Wg^T) * (A . Wu^T), against the fp64 oracle
(oracle.swiglu), within the GEMM parity tolerance (tests/_parity.py).  The fp32
accumulators, the fp32 SiLU and product and the bf16 rounding of the output
keep the GPU's error near the output rounding; the tolerance is the GEMM's.

Covers tiles with ragged M, N and K, leading dimensions wider than the rows,
Stream-K tiles (whose partial sums the fixup warps combine before the gate),
the 7B-model gate/up shape on sampled rows and columns, determinism, K = 0 and
argument errors."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


def _run(A_bits, G_bits, U_bits, M, N, K, path=sg.PATH_AUTO):
    A = to_device(A_bits, K)
    Wg = to_device(G_bits, K)
    Wu = to_device(U_bits, K)
    ld = -(-N // 8) * 8
    Cfull = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")
    sg.gemm_bf16_swiglu(A, Wg, Wu, Cfull[:, :N], path=path)
    torch.cuda.synchronize()
    return to_bits(Cfull)[:, :N]


def _inputs(M, N, K, seed, ld=None):
    A = syn.matrix(M, K, "normal:1", seed, ld=ld)
    G = syn.matrix(N, K, "normal:0.05", seed + 1, ld=ld)
    U = syn.matrix(N, K, "normal:0.05", seed + 2, ld=ld)
    return A, G, U


GEMM_PATHS = [sg.PATH_GEMM, sg.PATH_GEMM_PAIR]


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 512), (200, 300, 192), (130, 257, 128),
                                   (65, 1000, 1024), (1000, 96, 4104), (520, 640, 256)])
def test_full_oracle(M, N, K, path):
    A, G, U = _inputs(M, N, K, 700 + M + N)
    assert_close(_run(A, G, U, M, N, K, path=path), oracle.swiglu(A, G, U), K, f"swiglu {M}x{N}x{K} path {path}")


@pytest.mark.parametrize("path", GEMM_PATHS)
def test_padded_leading_dimensions(path):
    M, N, K = 300, 140, 200
    A, G, U = _inputs(M, N, K, 801, ld=216)
    assert_close(_run(A, G, U, M, N, K, path=path), oracle.swiglu(A, G, U, K=K), K, "padded")


@pytest.mark.parametrize("path", GEMM_PATHS)
def test_stream_k_tiles_are_gated_after_the_sum(path):
    # 2048 x 4096 x 4096: 512 tiles of 128 x 128 (256 of 256 x 128 on pairs) over
    # the SMs leave a Stream-K remainder; each split tile's gate and up sums are
    # combined by the fixup warps before the SiLU.
    M, N, K = 2048, 4096, 4096
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info = sg.plan_swiglu(M, N, K, sms, path)
    assert info["sk_tiles"] > 0
    A, G, U = _inputs(M, N, K, 811)
    got = _run(A, G, U, M, N, K, path=path)
    rows = syn.sample_indices(M, 256, 3)
    ref = oracle.silu(oracle.gemm(A[rows], G)) * oracle.gemm(A[rows], U)
    assert_close(got[rows], ref, K, "stream-k")


def test_mlp_gate_up_shape_sampled():
    # the 7B model's gate/up projection: M = 4096 tokens, K = 4096, N = 11008
    w = syn.WORKLOADS["mlp_up"]
    A = w.a()
    G = w.b()
    U = syn.matrix(w.N, w.K, w.dist_b, w.seed_b + 77)
    got = _run(A, G, U, w.M, w.N, w.K)
    rows = syn.sample_indices(w.M, 128, 5)
    cols = syn.sample_indices(w.N, 128, 6)
    g = oracle.gemm_sampled(A, G, rows, cols)
    u = oracle.gemm_sampled(A, U, rows, cols)
    assert_close(got[np.ix_(rows, cols)], oracle.silu(g) * u, w.K, "mlp gate/up sampled")


def test_deterministic():
    M, N, K = 1024, 2048, 2048
    A, G, U = (to_device(x) for x in _inputs(M, N, K, 821))
    C1 = sg.gemm_bf16_swiglu(A, G, U)
    for _ in range(2):
        C2 = sg.gemm_bf16_swiglu(A, G, U)
        torch.cuda.synchronize()
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 13])
@pytest.mark.parametrize("N,K", [(300, 1000), (4096, 11008), (1000, 4104)])
def test_cuda_core_path(M, N, K):
    # the decode path for M <= 2 (and, chosen explicitly, any M <= 64): each CTA
    # streams the gate and up rows of its outputs once for all M activation rows
    A, G, U = _inputs(M, N, K, 900 + M + N)
    ref = oracle.swiglu(A, G, U)
    assert_close(_run(A, G, U, M, N, K, path=sg.PATH_CUDA_CORE), ref, K, f"cuda core M={M}")
    if M <= 2:
        assert_close(_run(A, G, U, M, N, K), ref, K, f"auto M={M}")


@pytest.mark.parametrize("M", [3, 9, 16, 17, 33, 64])
@pytest.mark.parametrize("N,K", [(300, 1000), (11008, 4096), (4096, 11008), (640, 8192)])
def test_tensor_core_path(M, N, K):
    # the decode path for 3 <= M <= 64: two MMAs per k slice fill a gate and an up
    # accumulator side by side in TMEM; split pieces are summed before the gate
    A, G, U = _inputs(M, N, K, 950 + M + N)
    ref = oracle.swiglu(A, G, U)
    assert_close(_run(A, G, U, M, N, K, path=sg.PATH_TENSOR_CORE), ref, K, f"tensor core M={M}")
    assert_close(_run(A, G, U, M, N, K), ref, K, f"auto M={M}")


def test_tensor_core_path_persistent_and_deterministic():
    # more 64-output tiles than resident CTAs: the persistent schedule
    M, N, K = 16, 24000, 320
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sg.plan_swiglu(M, N, K, sms, sg.PATH_TENSOR_CORE)["split_k"] == 0
    A, G, U = _inputs(M, N, K, 971)
    got = _run(A, G, U, M, N, K, path=sg.PATH_TENSOR_CORE)
    assert_close(got, oracle.swiglu(A, G, U), K, "persistent")
    assert np.array_equal(got, _run(A, G, U, M, N, K, path=sg.PATH_TENSOR_CORE))


def test_zero_k_and_errors():
    A = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")[:, :0]   # K = 0, rows 16-byte aligned
    W = torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    C = torch.full((4, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    sg.gemm_bf16_swiglu(A, W, W, C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0
    A = torch.randn(64, 64, device="cuda").bfloat16()
    W = torch.randn(64, 64, device="cuda").bfloat16()
    lib = sg.load()
    st = lib.gemm_bf16_swiglu(A.data_ptr(), W.data_ptr(), None, torch.empty_like(A).data_ptr(), 64, 64, 64,
                              64, 64, 64, None)
    assert st == sg.SG_ERR_INVALID_ARG
    st = lib.gemm_bf16_swiglu(A.data_ptr(), W.data_ptr(), W.data_ptr() + 2, torch.empty_like(A).data_ptr(),
                              64, 64, 64, 64, 64, 64, None)
    assert st == sg.SG_ERR_MISALIGNED


@pytest.mark.parametrize("g", [g for g in syn.GATED_WORKLOADS.values() if g.base.M <= 64], ids=lambda g: g.name)
def test_decode_gated_workloads(g):
    # the bench's gated decode rows: M = 1, 2, 16, 64 against 11008 x 4096 gate and up weights
    w = g.base
    A, G, U = w.a(), w.b(), g.up()
    assert_close(_run(A, G, U, w.M, w.N, w.K), oracle.swiglu(A, G, U), w.K, g.name)
