"""gemv_bf16_noalloc: the skinny GEMV for callers that cannot allocate device memory.

Callers whose device memory is owned by their own pool allocator, plug-ins whose
host framework forbids raw cudaMalloc, and code that cannot take cudaMalloc's
implicit synchronisation use this entry point.  Its split-K scratch is a fixed
array in the library's device image instead of a workspace allocated on first use.
These tests call it through the C ABI and check its output against the existing
gemv_bf16_path(..., SG_PATH_CUDA_CORE) entry point, with the tolerance of the
other parity tests, on two calls in a row (the second call finds the first
call's scratch contents).  The file is named to be collected last.
"""
import numpy as np
import pytest

import synthetic as syn
from _parity import assert_close, bf16_f64, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


def _call(fn, A, B, C, M, N, K, *extra):
    s = torch.cuda.current_stream().cuda_stream
    return fn(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, A.stride(0), B.stride(0), C.stride(0),
              *extra, s)


@pytest.mark.parametrize("M,N,K", [
    (2, 4096, 11008),   # few row groups: K is split, partials and counters live in the array
    (19, 300, 2048),    # three 8-row blocks, each with its own K split
    (1, 11008, 4096),   # enough row groups: no split
    (8, 40, 8192),      # one row group, eight K slices
])
def test_noalloc_matches_gemv_on_two_calls(M, N, K):
    lib = sg.load()
    A = to_device(syn.matrix(M, K, "normal:1", 301 + M))
    B = to_device(syn.matrix(N, K, "normal:0.02", 302 + N))
    ld = -(-N // 8) * 8
    C_ref = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")[:, :N]
    assert _call(lib.gemv_bf16_path, A, B, C_ref, M, N, K, sg.PATH_CUDA_CORE) == sg.SG_OK
    torch.cuda.synchronize()
    ref = bf16_f64(to_bits(C_ref))
    for _ in range(2):
        C = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :N]
        assert _call(lib.gemv_bf16_noalloc, A, B, C, M, N, K) == sg.SG_OK
        torch.cuda.synchronize()
        assert_close(to_bits(C), ref, K, f"noalloc {M}x{N}x{K}")


def test_noalloc_rejects_sizes_beyond_its_limits():
    lib = sg.load()
    buf = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gemv_bf16_noalloc(p, p, p, 65, 8, 64, 64, 64, 64, s) == sg.SG_ERR_INVALID_ARG
    assert lib.gemv_bf16_noalloc(p, p, p, 4, 8, 64, 56, 64, 64, s) == sg.SG_ERR_INVALID_ARG
    assert lib.gemv_bf16_noalloc(p + 2, p, p, 4, 8, 64, 64, 64, 64, s) == sg.SG_ERR_MISALIGNED
