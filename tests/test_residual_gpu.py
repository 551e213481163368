"""Parity of the projection with its residual add, gemm_bf16_residual:
C = A . B^T + R, against the fp64 oracle (oracle.gemm_residual) within the
GEMM parity tolerance (tests/_parity.py), on every kernel (CUDA-core and tcgen05 skinny paths,
both GEMMs), ragged shapes, a padded residual, Stream-K tiles, in place (R = C),
the 7B-model down projection, K = 0 and argument errors."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


def _inputs(M, N, K, seed, ldr=None):
    A = syn.matrix(M, K, "normal:1", seed)
    B = syn.matrix(N, K, "normal:0.05", seed + 1)
    R = syn.matrix(M, N, "normal:1", seed + 2, ld=ldr or -(-N // 8) * 8)  # rows 16-byte aligned
    return A, B, R


def _run(A_bits, B_bits, R_bits, M, N, K, path=sg.PATH_AUTO, inplace=False):
    A, B = to_device(A_bits, K), to_device(B_bits, K)
    Rd = to_device(R_bits, N)
    if inplace:
        C = Rd
    else:
        ld = -(-N // 8) * 8
        C = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")[:, :N]
    sg.gemm_bf16_residual(A, B, Rd, C, path=path)
    torch.cuda.synchronize()
    st, detail = sg.check_device_errors()  # no bounded wait in any role ran out
    assert st == sg.SG_OK, detail
    return to_bits(C)


@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 192), (130, 257, 136), (520, 640, 512)])
def test_gemm_paths(M, N, K, path):
    A, B, R = _inputs(M, N, K, 1100 + M + N)
    assert_close(_run(A, B, R, M, N, K, path), oracle.gemm_residual(A, B, R), K, f"gemm {path}")


@pytest.mark.parametrize("path", [sg.PATH_CUDA_CORE, sg.PATH_TENSOR_CORE])
@pytest.mark.parametrize("M", [1, 2, 5, 16, 33, 64])
@pytest.mark.parametrize("N,K", [(300, 1000), (4096, 11008), (11008, 4096)])
def test_skinny_paths(M, N, K, path):
    A, B, R = _inputs(M, N, K, 1200 + M + N)
    assert_close(_run(A, B, R, M, N, K, path), oracle.gemm_residual(A, B, R), K, f"skinny {path} M={M}")


def test_padded_residual_and_in_place():
    M, N, K = 300, 140, 200
    A, B, R = _inputs(M, N, K, 1301, ldr=152)
    ref = oracle.gemm_residual(A, B, R)
    assert_close(_run(A, B, R, M, N, K)[:, :N], ref, K, "padded R")
    assert_close(_run(A, B, R, M, N, K, inplace=True)[:, :N], ref, K, "in place")
    assert_close(_run(A[:16], B, R[:16], 16, N, K, inplace=True)[:, :N], ref[:16], K, "skinny in place")


def test_narrow_stream_k_tiles():
    # 128 x 128 single-CTA tiles split along K: the residual is added once, after the partials
    M, N, K = 384, 512, 8192
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info = sg.plan(M, N, K, sms, sg.PATH_GEMM)
    assert info["tile_n"] == 128 and info["sk_tiles"] > 0, info
    A, B, R = _inputs(M, N, K, 1331)
    assert_close(_run(A, B, R, M, N, K, sg.PATH_GEMM), oracle.gemm_residual(A, B, R), K, "narrow stream-k residual")


@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
def test_stream_k_tiles(path):
    M, N, K = 4096, 4096, 4096
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sg.plan(M, N, K, sms, path)["sk_tiles"] > 0
    A, B, R = _inputs(M, N, K, 1311)
    got = _run(A, B, R, M, N, K, path)
    rows = syn.sample_indices(M, 128, 7)
    cols = syn.sample_indices(N, 128, 8)
    ref = oracle.gemm_sampled(A, B, rows, cols) + oracle._bf16_to_f64(R)[np.ix_(rows, cols)]
    assert_close(got[np.ix_(rows, cols)], ref, K, "stream-k residual")


def test_mlp_down_projection():
    w = syn.WORKLOADS["mlp_down"]
    A, B = w.a(), w.b()
    R = syn.matrix(w.M, w.N, "normal:1", 1321)  # N = 4096: rows already aligned
    got = _run(A, B, R, w.M, w.N, w.K)
    rows = syn.sample_indices(w.M, 128, 9)
    cols = syn.sample_indices(w.N, 128, 10)
    ref = oracle.gemm_sampled(A, B, rows, cols) + oracle._bf16_to_f64(R)[np.ix_(rows, cols)]
    assert_close(got[np.ix_(rows, cols)], ref, w.K, "mlp down + residual")


def test_zero_k_and_errors():
    A = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    B = torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    R = torch.randn(4, 16, device="cuda").bfloat16()
    C = sg.gemm_bf16_residual(A, B, R)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), R.view(torch.int16))
    lib = sg.load()
    A = torch.randn(64, 64, device="cuda").bfloat16()
    C = torch.empty_like(A)
    assert lib.gemm_bf16_residual(A.data_ptr(), A.data_ptr(), None, C.data_ptr(), 64, 64, 64, 64, 64, 64, 64,
                                  None) == sg.SG_ERR_INVALID_ARG
    assert lib.gemm_bf16_residual(A.data_ptr(), A.data_ptr(), C.data_ptr() + 2, C.data_ptr(), 64, 64, 64, 64, 64,
                                  64, 64, None) == sg.SG_ERR_MISALIGNED
    assert lib.gemm_bf16_residual(A.data_ptr(), A.data_ptr(), C.data_ptr(), C.data_ptr(), 64, 64, 64, 64, 64,
                                  72, 64, None) == sg.SG_ERR_INVALID_ARG
