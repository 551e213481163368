"""Parity of the tcgen05 GEMM (gemm_bf16, M > 64) against the fp64 oracle.

Exactness probes use small-integer operands: every partial sum is an integer
below 2^24 (exact in fp32) and |C| <= 256 (exact in bf16), so any layout,
swizzle, descriptor or scheduling mistake shows as a bit difference that a
tolerance could hide.  Tolerance cases use the seeded uniform / normal inputs
of the pages' workloads, with ragged edges in M, N and K and padded strides.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from _parity import assert_close, assert_exact, bf16_f64, to_bits, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402


GEMM_PATHS = [sg.PATH_GEMM, sg.PATH_GEMM_PAIR]


def _run(A_bits, B_bits, M, N, K, ldc=None, fill=None, path=sg.PATH_AUTO):
    A = to_device(A_bits, K)
    B = to_device(B_bits, K)
    ldc = -(-N // 8) * 8 if ldc is None else ldc  # 16-byte row pitch
    Cfull = torch.empty((M, ldc), dtype=torch.bfloat16, device="cuda")
    if fill is not None:
        Cfull.view(torch.int16).fill_(fill)
    C = Cfull[:, :N]
    sg.gemm_bf16(A, B, C, path=path)
    torch.cuda.synchronize()
    st, detail = sg.check_device_errors()  # no bounded wait in any role ran out
    assert st == sg.SG_OK, detail
    return to_bits(Cfull)[:, :N]


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 256), (200, 300, 192), (130, 257, 128),
                                   (1024, 768, 256), (300, 1000, 64), (512, 256, 1024)])
def test_exact_integers_pm1(M, N, K, path):
    A = syn.small_int_matrix(M, K, -1, 1, 1000 + M)
    B = syn.small_int_matrix(N, K, -1, 1, 2000 + N)
    assert_exact(_run(A, B, M, N, K, path=path), oracle.gemm(A, B), f"pm1 {M}x{N}x{K} path {path}")


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("M,N,K", [(192, 320, 16), (129, 129, 8)])
def test_exact_integers_pm4(M, N, K, path):
    A = syn.small_int_matrix(M, K, -4, 4, 3000 + M)
    B = syn.small_int_matrix(N, K, -4, 4, 4000 + N)
    assert_exact(_run(A, B, M, N, K, path=path), oracle.gemm(A, B), f"pm4 {M}x{N}x{K} path {path}")


def test_identity_and_permutation():
    M, K = 300, 512
    A = syn.matrix(M, K, "uniform", 77)
    eye = syn.f64_to_bf16_bits(np.eye(K))
    assert_exact(_run(A, eye, M, K, K), bf16_f64(A), "identity")
    perm = np.random.default_rng(5).permutation(K)[:384]
    P = np.zeros((perm.size, K))
    P[np.arange(perm.size), perm] = 1.0
    assert_exact(_run(A, syn.f64_to_bf16_bits(P), M, perm.size, K), bf16_f64(A)[:, perm], "permutation")


def test_one_hot_rows_select_weight_columns():
    M, N, K = 256, 384, 320
    B = syn.matrix(N, K, "normal:0.02", 78)
    hot = np.random.default_rng(6).integers(0, K, size=M)
    H = np.zeros((M, K))
    H[np.arange(M), hot] = 1.0
    assert_exact(_run(syn.f64_to_bf16_bits(H), B, M, N, K), bf16_f64(B)[:, hot].T, "one-hot")


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("M,N,K", [
    (65, 1, 8), (65, 8, 16), (127, 9, 24), (129, 255, 72), (200, 257, 4104), (513, 1000, 200),
    (1000, 520, 1000), (64 + 128 * 3, 256 * 2 + 8, 64 * 5 + 8), (2500, 1300, 704),
])
def test_ragged_shapes(M, N, K, path):
    A = syn.matrix(M, K, "uniform", 5000 + M)
    B = syn.matrix(N, K, "uniform", 6000 + N)
    assert_close(_run(A, B, M, N, K, path=path), oracle.gemm(A, B), K, f"ragged {M}x{N}x{K} path {path}")


def test_padded_strides_and_guard_band():
    M, N, K = 300, 200, 136
    lda, ldb, ldc = K + 24, K + 8, N + 40
    A = syn.matrix(M, K, "uniform", 11, ld=lda)  # NaN patterns in the padding
    B = syn.matrix(N, K, "uniform", 12, ld=ldb)
    Ad = to_device(A)[:, :K]
    Bd = to_device(B)[:, :K]
    sentinel = 0x7FC1
    Cbuf = torch.full((M + 4, ldc), 0, dtype=torch.int16, device="cuda")
    Cbuf.fill_(sentinel)
    C = Cbuf.view(torch.bfloat16)[:M, :N]
    sg.gemm_bf16(Ad, Bd, C)
    torch.cuda.synchronize()
    out = Cbuf.cpu().numpy().view(np.uint16)
    assert_close(out[:M, :N], oracle.gemm(A, B, K=K), K, "padded")
    assert np.all(out[:M, N:] == sentinel), "C padding columns were written"
    assert np.all(out[M:, :] == sentinel), "rows after C were written"


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("name", ["sq512", "sq2048"])
def test_workload_full_oracle(name, path):
    w = syn.WORKLOADS[name]
    A, B = w.a(), w.b()
    assert_close(_run(A, B, w.M, w.N, w.K, path=path), oracle.gemm(A, B), w.K, f"{name} path {path}")


@pytest.mark.parametrize("path", GEMM_PATHS)
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (1000, 3000, 1000), (384, 512, 8192), (4096, 4096, 1024)])
def test_deterministic_across_runs(M, N, K, path):
    A = to_device(syn.matrix(M, K, "uniform", 90))
    B = to_device(syn.matrix(N, K, "uniform", 91))
    C1 = sg.gemm_bf16(A, B, path=path)
    C2 = torch.empty_like(C1)
    for _ in range(3):
        sg.gemm_bf16(A, B, C2, path=path)
        torch.cuda.synchronize()
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(128, 4096, 4096), (384, 512, 8192), (300, 1000, 2048)])
def test_narrow_tiles_with_stream_k(M, N, K):
    # 128 x 128 single-CTA tiles, chosen automatically when they fit in one wave;
    # these shapes also split K, so Stream-K partials of the narrow tiles are summed
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info = sg.plan(M, N, K, sms, sg.PATH_AUTO)
    assert info["path"] == sg.PATH_GEMM and info["tile_n"] == 128 and info["sk_tiles"] > 0, info
    A = syn.matrix(M, K, "normal:1", 7000 + M)
    B = syn.matrix(N, K, "normal:0.02", 7100 + N)
    got = _run(A, B, M, N, K)
    assert_close(got, oracle.gemm(A, B), K, f"narrow {M}x{N}x{K}")
    again = _run(A, B, M, N, K)
    assert np.array_equal(got, again), "narrow tiles: not the same bits on a rerun"


def test_zero_k_and_empty():
    s = torch.cuda.current_stream().cuda_stream
    C = torch.full((100, 72), 3.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")
    # K = 0: an empty sum, so C := 0 (lda = ldb = 0 satisfy ld >= K)
    assert sg.gemm_bf16_ptr(dummy.data_ptr(), dummy.data_ptr(), C.data_ptr(), 100, 72, 0, 0, 0, 72, s) == sg.SG_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(C.float()).item() == 0
    # M = 0 or N = 0: nothing is written
    C.fill_(3.0)
    assert sg.gemm_bf16_ptr(dummy.data_ptr(), dummy.data_ptr(), C.data_ptr(), 0, 72, 8, 8, 8, 72, s) == sg.SG_OK
    assert sg.gemm_bf16_ptr(dummy.data_ptr(), dummy.data_ptr(), C.data_ptr(), 100, 0, 8, 8, 8, 72, s) == sg.SG_OK
    torch.cuda.synchronize()
    assert torch.all(C.float() == 3.0)


def test_misaligned_device_pointers_rejected():
    buf = torch.zeros((256, 72), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    p = buf.data_ptr()
    assert sg.gemm_bf16_ptr(p + 2, p, p, 100, 64, 64, 64, 64, 64, s) == sg.SG_ERR_MISALIGNED
    assert sg.gemv_bf16_ptr(p, p + 8, p, 4, 64, 64, 64, 64, 64, s) == sg.SG_ERR_MISALIGNED
