"""gemv_bf16_noalloc: the skinny GEMV for callers that cannot allocate device memory.

Callers whose device memory is owned by their own pool allocator, plug-ins whose
host framework forbids raw cudaMalloc, and code that cannot take cudaMalloc's
implicit synchronisation use this entry point.  Its split-K scratch is a fixed
array in the library's device image instead of a workspace allocated on first use.

Each test calls it through the C ABI twice in a row (the second call finds the
first call's scratch contents) and checks every call
  * against the fp64 oracle with the parity tolerance of the other GEMM tests, and
  * bit for bit against the existing gemv_bf16_path(..., SG_PATH_CUDA_CORE) entry:
    the same kernel with the same plan must give the same bits.
The cases that are meant to use the array are checked to plan a K split (through
sg_plan), one of them with the largest partial-sum footprint the planner makes and
one with the largest number of K slices.  The file is named to be collected last.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


def _call(fn, A, B, C, M, N, K, *extra):
    s = torch.cuda.current_stream().cuda_stream
    return fn(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, A.stride(0), B.stride(0), C.stride(0),
              *extra, s)


def _splits(M, N, K):
    """The K split of each 8-row block of the CUDA-core plan on this device."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return [sg.plan(min(8, M - m0), N, K, sms, sg.PATH_CUDA_CORE)["split_k"] for m0 in range(0, M, 8)]


@pytest.mark.parametrize("M,N,K,split", [
    (1, 11008, 4096, False),   # enough row blocks for every SM: no split, the array is not touched
    (2, 128, 11008, True),     # 128 rows: K split three ways, partials and counters in the array
    (19, 300, 2048, True),     # three 8-row blocks, each with its own K split
    (8, 40, 8192, True),       # one row block, eight K slices
    (8, 303, 8192, True),      # the largest partial-sum footprint: 2 slices x 8 rows x 303 columns
    (8, 8, 40960, True),       # the most K slices: 38
])
def test_noalloc_matches_oracle_and_gemv_on_two_calls(M, N, K, split):
    lib = sg.load()
    splits = _splits(M, N, K)
    assert (max(splits) > 1) == split, splits
    A_bits = syn.matrix(M, K, "normal:1", 301 + M)
    B_bits = syn.matrix(N, K, "normal:0.02", 302 + N)
    A, B = to_device(A_bits), to_device(B_bits)
    ref = oracle.gemm(A_bits, B_bits)
    ld = -(-N // 8) * 8
    C_ref = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")[:, :N]
    assert _call(lib.gemv_bf16_path, A, B, C_ref, M, N, K, sg.PATH_CUDA_CORE) == sg.SG_OK
    torch.cuda.synchronize()
    want = to_bits(C_ref)
    for call in range(2):
        C = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :N]
        assert _call(lib.gemv_bf16_noalloc, A, B, C, M, N, K) == sg.SG_OK
        torch.cuda.synchronize()
        got = to_bits(C)
        assert_close(got, ref, K, f"noalloc {M}x{N}x{K} call {call}")
        assert np.array_equal(got, want), f"noalloc {M}x{N}x{K} call {call}: differs from gemv_bf16_path"


def test_noalloc_rejects_sizes_beyond_its_limits():
    lib = sg.load()
    buf = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gemv_bf16_noalloc(p, p, p, 65, 8, 64, 64, 64, 64, s) == sg.SG_ERR_INVALID_ARG
    assert lib.gemv_bf16_noalloc(p, p, p, 4, 8, 64, 56, 64, 64, s) == sg.SG_ERR_INVALID_ARG
    assert lib.gemv_bf16_noalloc(p + 2, p, p, 4, 8, 64, 64, 64, 64, s) == sg.SG_ERR_MISALIGNED
