"""Parity of gemv_bf16_batched: several weight matrices against the same
activations in one launch, against the fp64 oracle per matrix (tests/_parity.py
tolerance), on both skinny kernels: Q/K/V-like equal shapes, unequal and ragged
N (so CUDA-core row blocks and tcgen05 tiles meet matrix boundaries), a split K,
matrices with no rows, determinism, and argument errors."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402

PATHS = [sg.PATH_CUDA_CORE, sg.PATH_TENSOR_CORE]


def _case(M, Ns, K, seed):
    A = syn.matrix(M, K, "normal:1", seed)
    Bs = [syn.matrix(N, K, "normal:0.02", seed + 1 + i) for i, N in enumerate(Ns)]
    return A, Bs


def _run(A, Bs, K, path):
    Ad = to_device(A, K)
    outs = sg.gemv_bf16_batched(Ad, [to_device(B, K) for B in Bs], path=path)
    torch.cuda.synchronize()
    return [to_bits(C) for C in outs]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 2, 7, 16, 64])
@pytest.mark.parametrize("Ns,K", [([4096, 4096, 4096], 4096), ([1000, 37, 4100, 64], 2048),
                                  ([11008, 300], 1024), ([129, 65, 63, 1, 200, 64, 127, 300], 520)])
def test_batched_matches_each_product(M, Ns, K, path):
    A, Bs = _case(M, Ns, K, 1400 + M + len(Ns))
    got = _run(A, Bs, K, path)
    for i, (B, C) in enumerate(zip(Bs, got)):
        assert_close(C[:, :B.shape[0]], oracle.gemm(A, B), K, f"path {path} M={M} matrix {i}")


@pytest.mark.parametrize("path", PATHS)
def test_split_k_and_determinism(path):
    M, Ns, K = 2, [512, 700], 11008   # few rows: the CUDA-core kernel splits K
    A, Bs = _case(M, Ns, K, 1451)
    g1 = _run(A, Bs, K, path)
    for B, C in zip(Bs, g1):
        assert_close(C[:, :B.shape[0]], oracle.gemm(A, B), K, "split")
    g2 = _run(A, Bs, K, path)
    assert all(np.array_equal(x, y) for x, y in zip(g1, g2))


def test_empty_matrices_and_errors():
    A = torch.randn(4, 64, device="cuda").bfloat16()
    B0 = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    B1 = torch.randn(32, 64, device="cuda").bfloat16()
    C0, C1 = sg.gemv_bf16_batched(A, [B0, B1])
    torch.cuda.synchronize()
    ref = A.float() @ B1.float().t()
    assert C0.shape == (4, 0)
    assert torch.allclose(C1.float(), ref, rtol=1e-2, atol=1e-1)
    with pytest.raises(sg.SgError):
        sg.gemv_bf16_batched(A, [B1] * 9)   # more than 8 matrices
    with pytest.raises(sg.SgError):
        sg.gemv_bf16_batched(torch.randn(65, 64, device="cuda").bfloat16(), [B1])   # M > 64


@pytest.mark.parametrize("w", list(syn.BATCHED_WORKLOADS.values()), ids=lambda w: w.name)
def test_qkv_workloads(w):
    # the bench's Q/K/V rows: three 4096 x 4096 weights, M = 1, 16, 64
    A, Bs = w.a(), w.bs()
    got = _run(A, Bs, w.K, sg.PATH_AUTO)
    for i, (B, C) in enumerate(zip(Bs, got)):
        assert_close(C, oracle.gemm(A, B), w.K, f"{w.name} matrix {i}")
