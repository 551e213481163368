"""Pins of the NVFP4 oracle (oracle.gemm_nvfp4) to things other than itself.

* E4M3: every one of the 256 codes against PyTorch's float8_e4m3fn conversion (an
  independent library decoder), plus the format's landmarks (1.0, 448, the
  smallest normal and subnormal, NaN).
* E2M1: the eight magnitudes of the FP4 format (0, 0.5, 1, 1.5, 2, 3, 4, 6, the
  value set of the OCP microscaling formats' FP4 type) and the sign bit.
* Packing: element k in byte k // 2, low nibble first (the layout the library
  documents).
* The GEMM: reduces exactly to the pinned bf16 oracle (oracle.gemm, the C code)
  on pre-multiplied values, which are exact in bf16 (2 + 4 significant bits); and
  equals an exact rational brute force on a tiny case.  A dropped scale, a wrong
  block index (k % 16 for k // 16), swapped nibbles or a transposed operand each
  fail one of these.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
# bf16 bit patterns of those magnitudes (sign: 0x8000), written from the bf16
# format: 1.0 = 0x3F80, each power of two adds 0x0080, a half-step mantissa 0x0040.
E2M1_BF16 = [0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0]


def torch_e4m3(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_value(codes), torch_e4m3(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_e4m3_landmarks():
    v = oracle.e4m3_value([0x38, 0x7E, 0x08, 0x01, 0x30, 0x40, 0x00, 0x80, 0x7F, 0xFF])
    assert list(v[:6]) == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 0.5, 2.0]
    assert v[6] == 0.0 and v[7] == 0.0 and np.signbit(v[7])
    assert np.isnan(v[8]) and np.isnan(v[9])
    finite = oracle.e4m3_value(np.arange(0x00, 0x7F))
    assert np.all(np.diff(finite) > 0)


def test_e2m1_values_and_sign():
    v = oracle.e2m1_value(np.arange(16))
    assert list(v[:8]) == E2M1_MAGNITUDES
    assert list(-v[8:]) == E2M1_MAGNITUDES
    assert np.signbit(v[8])  # code 8 is -0


def test_unpack_low_nibble_first():
    packed = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert oracle.nvfp4_unpack(packed, 4).tolist() == [[1, 2, 7, 15]]


def _premultiplied_bf16(packed: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    """bf16 bits of e2m1 * e4m3 from the tables above and torch's E4M3 decoder."""
    b = packed[:, :K // 2].astype(np.int64)
    codes = np.empty((b.shape[0], K), dtype=np.int64)
    codes[:, 0::2], codes[:, 1::2] = b & 0xF, b >> 4
    mag_bits = np.array(E2M1_BF16, dtype=np.uint32)[codes & 7]
    val = (mag_bits << 16).view(np.float32).astype(np.float64)
    val = np.where(codes & 8, -val, val)
    sc = np.repeat(torch_e4m3(scales[:, :K // 16]), 16, axis=1)
    prod = (val * sc).astype(np.float32)
    assert np.array_equal(prod.astype(np.float64), val * sc)  # exact in fp32
    bits = prod.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)  # and in bf16
    return (bits >> 16).astype(np.uint16)


@pytest.mark.parametrize("M,N,K", [(5, 7, 64), (33, 17, 256), (3, 130, 1040)])
def test_reduces_to_bf16_oracle(M, N, K):
    A, B = synthetic.nvfp4_codes(M, K, 11), synthetic.nvfp4_codes(N, K, 12)
    SA, SB = synthetic.nvfp4_scales(M, K, 13), synthetic.nvfp4_scales(N, K, 14)
    ref = oracle.gemm(_premultiplied_bf16(A, SA, K), _premultiplied_bf16(B, SB, K))
    got = oracle.gemm_nvfp4(A, SA, B, SB, K)
    assert np.array_equal(got, ref)


def test_unit_scales_reduce_to_plain_fp4_gemm():
    M, N, K = 9, 11, 96
    A, B = synthetic.nvfp4_codes(M, K, 21), synthetic.nvfp4_codes(N, K, 22)
    one = lambda r: np.full((r, K // 16), 0x38, dtype=np.uint8)
    ref = oracle.gemm(_premultiplied_bf16(A, one(M), K), _premultiplied_bf16(B, one(N), K))
    assert np.array_equal(oracle.gemm_nvfp4(A, one(M), B, one(N), K), ref)


def test_exact_rational_brute_force():
    M, N, K = 2, 3, 48
    A, B = synthetic.nvfp4_codes(M, K, 31), synthetic.nvfp4_codes(N, K, 32)
    SA, SB = synthetic.nvfp4_scales(M, K, 33), synthetic.nvfp4_scales(N, K, 34)
    mags = [Fraction(x) for x in (0, Fraction(1, 2), 1, Fraction(3, 2), 2, 3, 4, 6)]

    def elem(packed, r, k):
        c = (int(packed[r, k // 2]) >> (4 * (k % 2))) & 0xF
        return -mags[c & 7] if c & 8 else mags[c & 7]

    def scale(codes, r, blk):
        c = int(codes[r, blk])
        e, m = (c >> 3) & 0xF, c & 7
        return Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)

    got = oracle.gemm_nvfp4(A, SA, B, SB, K, alpha=0.75)
    for m in range(M):
        for n in range(N):
            s = sum(elem(A, m, k) * scale(SA, m, k // 16) * elem(B, n, k) * scale(SB, n, k // 16) for k in range(K))
            assert Fraction(got[m, n]) == Fraction(3, 4) * s


def test_one_block_scale_moves_one_block():
    # doubling the scale of block j of row m changes C[m, :] by exactly that
    # block's contribution
    M, N, K = 4, 5, 128
    A, B = synthetic.nvfp4_codes(M, K, 41), synthetic.nvfp4_codes(N, K, 42)
    SA, SB = synthetic.nvfp4_scales(M, K, 43), synthetic.nvfp4_scales(N, K, 44)
    base = oracle.gemm_nvfp4(A, SA, B, SB, K)
    SA2 = SA.copy()
    SA2[2, 5] += 8  # exponent + 1: the scale doubles (0x28..0x3F stays below 0x7F)
    moved = oracle.gemm_nvfp4(A, SA2, B, SB, K)
    blk = slice(16 * 5, 16 * 6)
    a = oracle.nvfp4_dequant(A, SA, K)[2, blk]
    b = oracle.nvfp4_dequant(B, SB, K)[:, blk]
    assert np.array_equal(np.delete(moved, 2, axis=0), np.delete(base, 2, axis=0))
    assert np.allclose(moved[2] - base[2], b @ a, rtol=0, atol=1e-12)


def test_sampled_equals_full():
    M, N, K = 40, 50, 160
    A, B = synthetic.nvfp4_codes(M, K, 51), synthetic.nvfp4_codes(N, K, 52)
    SA, SB = synthetic.nvfp4_scales(M, K, 53), synthetic.nvfp4_scales(N, K, 54)
    rows, cols = np.array([0, 7, 39]), np.array([3, 49])
    full = oracle.gemm_nvfp4(A, SA, B, SB, K, alpha=1.5)
    assert np.array_equal(oracle.gemm_nvfp4_sampled(A, SA, B, SB, rows, cols, K, alpha=1.5), full[np.ix_(rows, cols)])


def test_synthetic_scales_in_range():
    s = synthetic.nvfp4_scales(64, 1024, 5)
    assert s.min() >= synthetic.NVFP4_SCALE_LO and s.max() <= synthetic.NVFP4_SCALE_HI
    assert np.all(np.isfinite(oracle.e4m3_value(s)))
