"""Parity of the NVFP4 block-scaled GEMM (gemm_nvfp4) against the fp64 oracle.

Tolerance: per element |gpu - ref| <= 1e-2 |ref| + 2e-3 sqrt(K) s and, over the
compared set, ||gpu - ref||_F / ||ref||_F <= 4e-3, where s is the rms of the
elementwise products a[m,k] sa b[n,k] sb (1 for the bf16 GEMM's unit-scale
inputs; the NVFP4 operands reach 6 x 1.875).  The fp16 rounding of the output is
at most 2^-11 |ref|; every product is exact in fp32, so fp32 accumulation of K of
them adds far less.  A stricter check counts the elements that differ from the
oracle rounded to fp16 by more than one fp16 step.

Exactness probes use single-block operands whose sums are exact in fp32 and fp16,
so a wrong scale column, atom byte or nibble shows as a bit difference.
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402

REL_TOL = 1e-2
ABS_TOL_PER_SQRT_K = 2e-3
FRO_TOL = 4e-3


def atoms_numpy(plain: np.ndarray, rows: int, K: int) -> np.ndarray:
    """The scale-atom layout, restated: atom (R, c) at (R * kc + c) * 512, row r of
    the atom's 128 and block j of its 4 at byte (r % 32) * 16 + (r // 32) * 4 + j."""
    kc = -(-K // 64)
    rb = -(-rows // 128)
    out = np.zeros(rb * kc * 512, dtype=np.uint8)
    for r in range(rows):
        for blk in range(K // 16):
            R, rr, c, j = r // 128, r % 128, blk // 4, blk % 4
            out[(R * kc + c) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + j] = plain[r, blk]
    return out


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(A, SA, B, SB, M, N, K, alpha=1.0, ldc=None, lda=None, ldb=None, path=0):
    """Packs the scales with the library and runs gemm_nvfp4; returns fp64 [M, N].
    Row pitches default to K/2 rounded up to 16 bytes (the TMA stride rule)."""
    pitch = -(-(K // 2) // 16) * 16
    lda = pitch if lda is None and pitch != A.shape[1] else lda
    ldb = pitch if ldb is None and pitch != B.shape[1] else ldb
    Ad = dev(A if lda is None else np.pad(A, ((0, 0), (0, lda - A.shape[1])), constant_values=0xFF))[:, :K // 2]
    Bd = dev(B if ldb is None else np.pad(B, ((0, 0), (0, ldb - B.shape[1])), constant_values=0xFF))[:, :K // 2]
    SAd = sg.nvfp4_pack_scales(dev(SA), K)
    SBd = sg.nvfp4_pack_scales(dev(SB), K)
    ldc = -(-N // 8) * 8 if ldc is None else ldc
    Cfull = torch.full((M, ldc), float("nan"), dtype=torch.float16, device="cuda")
    C = Cfull[:, :N]
    sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K, C=C, alpha=alpha, path=path)
    torch.cuda.synchronize()
    st, detail = sg.check_device_errors()
    assert st == 0, detail
    out = Cfull.cpu().numpy()
    if ldc > N:  # padding columns untouched
        assert np.isnan(out[:, N:]).all()
    return out[:, :N].astype(np.float64)


def product_rms(A, SA, B, SB, K):
    a = oracle.nvfp4_dequant(A, SA, K)
    b = oracle.nvfp4_dequant(B, SB, K)
    return math.sqrt(float(np.mean(a * a)) * float(np.mean(b * b)))


def assert_close(got, ref, K, s, label=""):
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    d = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref) + ABS_TOL_PER_SQRT_K * math.sqrt(max(K, 1)) * s
    n_over = int(np.count_nonzero(d > bound))
    fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    # one fp16 step at |ref| (subnormal spacing below 2^-14)
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))), -14) - 10)
    n_far = int(np.count_nonzero(np.abs(got - ref.astype(np.float16).astype(np.float64)) > step))
    assert n_over == 0, f"{label}: {n_over} elements over the bound (max |d| {d.max():.3g})"
    assert fro <= FRO_TOL, f"{label}: relative Frobenius error {fro:.3g}"
    assert n_far <= max(1, got.size // 1000), f"{label}: {n_far} elements more than one fp16 step from the oracle"


def test_pack_scales_matches_layout():
    for rows, K in [(1, 16), (128, 256), (300, 1040), (129, 64)]:
        plain = syn.nvfp4_scales(rows, K, 7 + rows)
        got = sg.nvfp4_pack_scales(dev(plain), K).cpu().numpy()
        assert got.size >= sg.nvfp4_scale_bytes(rows, K)
        assert np.array_equal(got[:sg.nvfp4_scale_bytes(rows, K)], atoms_numpy(plain, rows, K)), (rows, K)


def test_pack_scales_pitch():
    plain = syn.nvfp4_scales(200, 512, 9, ld=48)  # 32 blocks in a 48-byte pitch
    got = sg.nvfp4_pack_scales(dev(plain)[:, :32], 512).cpu().numpy()
    assert np.array_equal(got, atoms_numpy(plain, 200, 512))


def _single_block(M, N, K, m_blk, seed):
    """Operands that are zero except k-block m_blk, where A's codes are +-1 and B's
    small: sums of at most 16 products, exact in fp32 and fp16."""
    A = np.zeros((M, K // 2), dtype=np.uint8)
    B = np.zeros((N, K // 2), dtype=np.uint8)
    rng = np.random.default_rng(seed)
    lo = 8 * m_blk
    A[:, lo:lo + 8] = rng.choice([0x22, 0x2A, 0xA2, 0xAA, 0x20, 0x02], size=(M, 8))  # +-1 / 0 pairs
    B[:, lo:lo + 8] = rng.integers(0, 256, size=(N, 8), dtype=np.uint8)
    # scales 0.5 or 1: every sum is a multiple of 1/8 below 96, exact in fp16
    SA = rng.choice(np.array([0x30, 0x38], dtype=np.uint8), size=(M, K // 16))
    SB = rng.choice(np.array([0x30, 0x38], dtype=np.uint8), size=(N, K // 16))
    return A, SA, B, SB


PATHS = [sg.PATH_GEMM, sg.PATH_GEMM_PAIR]  # one CTA per 128 x 256 tile; CTA pairs per 256 x 256 tile


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K,blk", [(128, 256, 256, 0), (128, 256, 256, 7), (130, 300, 512, 21),
                                       (256, 512, 1024, 63), (77, 129, 64, 3), (300, 260, 1040, 64),
                                       (512, 256, 256, 2), (700, 520, 768, 40)])
def test_exact_single_block(M, N, K, blk, path):
    A, SA, B, SB = _single_block(M, N, K, blk, 100 + blk)
    ref = oracle.gemm_nvfp4(A, SA, B, SB, K)
    assert np.array_equal(ref.astype(np.float16).astype(np.float64), ref)  # exact in fp16
    got = run(A, SA, B, SB, M, N, K, path=path)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:3].tolist()}"


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (512, 512, 512), (300, 500, 1040), (1, 256, 4096),
                                   (129, 1, 256), (1000, 700, 2048), (256, 1024, 16), (640, 640, 4096)])
@pytest.mark.parametrize("path", PATHS)
def test_parity_seeded(M, N, K, path):
    A, B = syn.nvfp4_codes(M, K, 1000 + M), syn.nvfp4_codes(N, K, 2000 + N)
    SA, SB = syn.nvfp4_scales(M, K, 3000 + M), syn.nvfp4_scales(N, K, 4000 + N)
    ref = oracle.gemm_nvfp4(A, SA, B, SB, K)
    got = run(A, SA, B, SB, M, N, K, path=path)
    assert_close(got, ref, K, product_rms(A, SA, B, SB, K), f"{M}x{N}x{K} path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_alpha_and_pitches(path):
    M, N, K = 300, 300, 768
    A, B = syn.nvfp4_codes(M, K, 11), syn.nvfp4_codes(N, K, 12)
    SA, SB = syn.nvfp4_scales(M, K, 13), syn.nvfp4_scales(N, K, 14)
    ref = oracle.gemm_nvfp4(A, SA, B, SB, K, alpha=-0.375)
    got = run(A, SA, B, SB, M, N, K, alpha=-0.375, ldc=320, lda=400, ldb=416, path=path)
    assert_close(got, ref, K, 0.375 * product_rms(A, SA, B, SB, K), "alpha, pitches")


def test_zero_k_and_empty():
    C = torch.full((4, 8), 7.0, dtype=torch.float16, device="cuda")
    z = torch.zeros((4, 0), dtype=torch.uint8, device="cuda")
    s = torch.zeros(16, dtype=torch.uint8, device="cuda")
    sg.gemm_nvfp4(z, s, torch.zeros((8, 0), dtype=torch.uint8, device="cuda"), s, K=0, C=C)
    torch.cuda.synchronize()
    assert (C == 0).all()


@pytest.mark.parametrize("path", PATHS)
def test_deterministic(path):
    M, N, K = 700, 900, 2048
    A, B = syn.nvfp4_codes(M, K, 21), syn.nvfp4_codes(N, K, 22)
    SA, SB = syn.nvfp4_scales(M, K, 23), syn.nvfp4_scales(N, K, 24)
    Ad, Bd = dev(A), dev(B)
    SAd, SBd = sg.nvfp4_pack_scales(dev(SA), K), sg.nvfp4_pack_scales(dev(SB), K)
    c1 = sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K, path=path).clone()
    c2 = sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=K, path=path)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("name", ["fp4_sq512", "fp4_sq4096"])
def test_workload_sampled(name):
    """The bench's workloads, checked at 128 x 128 sampled intersections (the gemm3
    benchmarks page's sampled correctness check)."""
    w = syn.NVFP4_WORKLOADS[name]
    A, B, SA, SB = w.a(), w.b(), w.sfa(), w.sfb()
    Ad, Bd = dev(A), dev(B)
    SAd, SBd = sg.nvfp4_pack_scales(dev(SA), w.K), sg.nvfp4_pack_scales(dev(SB), w.K)
    C = sg.gemm_nvfp4(Ad, SAd, Bd, SBd, K=w.K, alpha=w.alpha)
    torch.cuda.synchronize()
    rows = syn.sample_indices(w.M, 128, 90 + w.cfg)
    cols = syn.sample_indices(w.N, 128, 91 + w.cfg)
    got = C.cpu().numpy().astype(np.float64)[np.ix_(rows, cols)]
    ref = oracle.gemm_nvfp4_sampled(A, SA, B, SB, rows, cols, w.K, alpha=w.alpha)
    assert_close(got, ref, w.K, product_rms(A[rows], SA[rows], B[cols], SB[cols], w.K), name)
