"""Parity of the skinny path (gemv_bf16, 1 <= M <= 64) against the fp64 oracle,
for both kernels: the CUDA-core weight stream and the tcgen05 kernel with the
weight rows on the MMA's M side, plus the decode workloads of the pages
(M = 1, 2, 16, 64 against the 7B-model 4096 x 11008 and 11008 x 4096 weights)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, assert_exact, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402

PATHS = [sg.PATH_CUDA_CORE, sg.PATH_TENSOR_CORE]


def _gemv(A_bits, B_bits, M, N, K, path, entry="gemv"):
    A = to_device(A_bits, K)
    B = to_device(B_bits, K)
    ld = -(-N // 8) * 8
    Cfull = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")
    C = Cfull[:, :N]
    if entry == "gemv":
        sg.gemv_bf16(A, B, C, path=path)
    else:
        sg.gemm_bf16(A, B, C)
    torch.cuda.synchronize()
    return to_bits(Cfull)[:, :N]


@pytest.mark.parametrize("path", PATHS)
def test_every_m_from_1_to_64(path):
    N, K = 300, 1000
    B = syn.matrix(N, K, "normal:0.02", 101)
    A_all = syn.matrix(64, K, "normal:1", 102)
    ref_all = oracle.gemm(A_all, B)
    for M in range(1, 65):
        got = _gemv(A_all[:M].copy(), B, M, N, K, path)
        assert_close(got, ref_all[:M], K, f"path {path} M={M}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (2, 257, 512), (5, 1000, 2048), (8, 64, 4096),
                                   (16, 300, 256), (33, 130, 128), (64, 520, 192)])
def test_exact_integers(path, M, N, K):
    A = syn.small_int_matrix(M, K, -1, 1, 7000 + M)
    B = syn.small_int_matrix(N, K, -1, 1, 8000 + N)
    assert_exact(_gemv(A, B, M, N, K, path), oracle.gemm(A, B), f"path {path} {M}x{N}x{K}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (3, 7, 24), (2, 33, 4104), (7, 4095, 136), (40, 129, 72)])
def test_ragged(path, M, N, K):
    A = syn.matrix(M, K, "normal:1", 9000 + M)
    B = syn.matrix(N, K, "normal:0.02", 9100 + N)
    assert_close(_gemv(A, B, M, N, K, path), oracle.gemm(A, B), K, f"ragged path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_k_not_multiple_of_8(path):
    # K = 20 with a padded pitch of 24: the CUDA-core kernel's scalar K tail and
    # the tensor path's zero-filled last stage both see the ragged end.
    M, N, K = 3, 77, 20
    A = syn.matrix(M, K, "normal:1", 31, ld=24)
    B = syn.matrix(N, K, "normal:0.02", 32, ld=24)
    Ad = to_device(A)[:, :K]
    Bd = to_device(B)[:, :K]
    C = torch.empty((M, 80), dtype=torch.bfloat16, device="cuda")[:, :N]
    sg.gemv_bf16(Ad, Bd, C, path=path)
    torch.cuda.synchronize()
    assert_close(to_bits(C), oracle.gemm(A, B, K=K), K, "K=20")


DECODE = [w for w in syn.WORKLOADS.values() if w.name.startswith("dec")]


@pytest.mark.parametrize("w", DECODE, ids=lambda w: w.name)
def test_decode_workloads(w):
    A, B = w.a(), w.b()
    ref = oracle.gemm(A, B)
    assert_close(_gemv(A, B, w.M, w.N, w.K, sg.PATH_AUTO), ref, w.K, w.name + " gemv")
    assert_close(_gemv(A, B, w.M, w.N, w.K, None, entry="gemm"), ref, w.K, w.name + " gemm")
    other = sg.PATH_TENSOR_CORE if w.M <= 2 else sg.PATH_CUDA_CORE
    assert_close(_gemv(A, B, w.M, w.N, w.K, other), ref, w.K, w.name + f" path {other}")


@pytest.mark.parametrize("path", PATHS)
def test_deterministic_split_k(path):
    # 4096 x 11008 weights: few row groups, so the K split and its fixup run.
    M, N, K = 2, 4096, 11008
    A = to_device(syn.matrix(M, K, "normal:1", 41))
    B = to_device(syn.matrix(N, K, "normal:0.02", 42))
    C1 = sg.gemv_bf16(A, B, path=path)
    for _ in range(3):
        C2 = sg.gemv_bf16(A, B, path=path)
        torch.cuda.synchronize()
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("M,N", [(16, 40000), (64, 40000)])
def test_tensor_core_persistent_schedule(M, N):
    # More weight tiles than resident CTAs (two per SM): the tensor-core kernel
    # walks its tiles persistently with a Stream-K remainder instead of cutting
    # each tile into k pieces.
    K = 320
    info = sg.plan(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count, sg.PATH_TENSOR_CORE)
    assert info["split_k"] == 0
    A = syn.matrix(M, K, "normal:1", 51)
    B = syn.matrix(N, K, "normal:0.02", 52)
    assert_close(_gemv(A, B, M, N, K, sg.PATH_TENSOR_CORE), oracle.gemm(A, B), K, f"persistent M={M} N={N}")


@pytest.mark.parametrize("M", [16, 64])
def test_tensor_core_split_pieces(M):
    # Few weight tiles and a long K: each tile is cut into several k pieces whose
    # fp32 partials the last arriving piece sums in k order (bit-identical reruns).
    N, K = 640, 8192
    info = sg.plan(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count, sg.PATH_TENSOR_CORE)
    assert info["split_k"] > 1
    A = syn.matrix(M, K, "normal:1", 61)
    B = syn.matrix(N, K, "normal:0.02", 62)
    got = _gemv(A, B, M, N, K, sg.PATH_TENSOR_CORE)
    assert_close(got, oracle.gemm(A, B), K, f"split M={M}")
    assert np.array_equal(got, _gemv(A, B, M, N, K, sg.PATH_TENSOR_CORE))
