"""Seeded synthetic inputs shared by the CUDA tests, the bench and the oracle tests.

This module only *draws* operands: it holds none of the GEMM's arithmetic.  Every
tensor is produced on the host from a counter-based generator, so the same
(seed, index) always gives the same bf16 bit pattern on any machine.

Generator (the pages fix none; this is the plain reading used throughout):
  * splitmix64 in counter form: x_i = mix(seed + (i + 1) * 0x9E3779B97F4A7C15);
  * uniform[-1, 1):      u = (x >> 11) * 2**-53,  v = 2u - 1;
  * normal(0, sigma):    Box-Muller on two consecutive draws of the stream;
  * rounding to bf16:    round-to-nearest-even straight from the fp64 value
    (no intermediate fp32 rounding), with no NaN/Inf possible by construction.

Workloads (the shapes of the pages' benchmarks: square cubes, 7B-model MLP
projections, decode batches) are listed in ``WORKLOADS``.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

SEED_A_BASE = 0x5EED0001
SEED_B_BASE = 0x5EED1001


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``count`` 64-bit words x_start .. x_{start+count-1} of the stream."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """fp64 values in [0, 1) with 53 random bits."""
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_pm1(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Elements start .. start+count-1 of the uniform[-1, 1) stream."""
    return uniform01(seed, start, count) * 2.0 - 1.0


def normal(seed: int, count: int, sigma: float, start: int = 0) -> np.ndarray:
    """Box-Muller: draws 2i and 2i+1 give the i-th pair (cos, sin) of variates.

    Element e is the (e % 2)-th member of pair e // 2, so any even ``start``
    yields exactly the slice of the full stream.
    """
    assert start % 2 == 0
    npairs = (count + 1) // 2
    u = uniform01(seed, start, 2 * npairs).reshape(npairs, 2)
    u1 = 1.0 - u[:, 0]  # (0, 1]: log is finite
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u[:, 1]
    z = np.empty((npairs, 2), dtype=np.float64)
    z[:, 0] = r * np.cos(t)
    z[:, 1] = r * np.sin(t)
    return z.reshape(-1)[:count] * sigma


def draws(dist: str, seed: int, start: int, count: int) -> np.ndarray:
    """fp64 draws for element indices [start, start + count) of one tensor."""
    if dist == "uniform":
        return uniform_pm1(seed, count, start)
    if dist.startswith("normal"):
        sigma = float(dist.split(":")[1]) if ":" in dist else 1.0
        return normal(seed, count, sigma, start)
    raise ValueError(dist)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to the nearest bf16 (ties to even); returns uint16 bit patterns.

    bf16 keeps 8 significant bits, so an fp64 significand (53 bits) is rounded at
    bit 45.  Values here are finite and far above the bf16 subnormal range, or zero.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bias = np.uint64((1 << 44) - 1) + lsb
    with np.errstate(over="ignore"):
        rounded = ((bits + bias) >> np.uint64(45)) << np.uint64(45)
    f32 = rounded.view(np.float64).astype(np.float32)  # exact: fits in 8 bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def matrix(rows: int, cols: int, dist: str, seed: int, ld: int | None = None,
           pad_value: int = 0xFFFF) -> np.ndarray:
    """A rows x ld uint16 matrix whose first ``cols`` columns hold bf16 draws.

    Element (r, c) is draw number r*cols + c of the stream, so the values do not
    depend on ``ld``; padding columns hold ``pad_value`` (a NaN pattern by default,
    so a kernel that reads padding shows it).
    """
    ld = cols if ld is None else ld
    assert ld >= cols
    core = np.empty((rows, cols), dtype=np.uint16)
    step = max(2, (1 << 24) // max(cols, 1) // 2 * 2)  # rows per chunk (even)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        v = draws(dist, seed, r0 * cols, (r1 - r0) * cols)
        core[r0:r1] = f64_to_bf16_bits(v).reshape(r1 - r0, cols)
    if ld == cols:
        return core
    out = np.full((rows, ld), pad_value, dtype=np.uint16)
    out[:, :cols] = core
    return out


def matrix_rows(row_idx, cols: int, dist: str, seed: int) -> np.ndarray:
    """Rows ``row_idx`` of ``matrix(rows, cols, dist, seed)`` without drawing the
    others (element (r, c) is draw r*cols + c; ``cols`` even for normal draws)."""
    row_idx = np.asarray(row_idx, dtype=np.int64)
    out = np.empty((row_idx.size, cols), dtype=np.uint16)
    for i, r in enumerate(row_idx):
        out[i] = f64_to_bf16_bits(draws(dist, seed, int(r) * cols, cols))
    return out


def small_int_matrix(rows: int, cols: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Integers in [lo, hi] stored as bf16 (exact for |v| <= 256)."""
    u = uniform01(seed, 0, rows * cols)
    v = np.floor(u * (hi - lo + 1)).astype(np.int64) + lo
    return f64_to_bf16_bits(v.astype(np.float64)).reshape(rows, cols)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic GEMM problem C[M,N] = A[M,K] . B[N,K]^T."""
    name: str
    M: int
    N: int
    K: int
    dist_a: str
    dist_b: str
    cfg: int  # seed offset
    oracle: str  # "full" or "sampled"

    @property
    def seed_a(self) -> int:
        return SEED_A_BASE + self.cfg

    @property
    def seed_b(self) -> int:
        return SEED_B_BASE + self.cfg

    def a(self) -> np.ndarray:
        return matrix(self.M, self.K, self.dist_a, self.seed_a)

    def b(self) -> np.ndarray:
        return matrix(self.N, self.K, self.dist_b, self.seed_b)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def decode_bytes(self) -> int:
        """Bytes a skinny GEMM must move at least once: weights, activations, output."""
        return 2 * (self.N * self.K + self.M * self.K + self.M * self.N)


def _decode(m: int, n: int, k: int, cfg: int) -> Workload:
    tag = "up" if n > k else "down"
    return Workload(f"dec{m}_{tag}", m, n, k, "normal:1", "normal:0.02", cfg, "full")


WORKLOADS = {w.name: w for w in [
    Workload("sq512", 512, 512, 512, "uniform", "uniform", 0, "full"),
    Workload("sq2048", 2048, 2048, 2048, "uniform", "uniform", 1, "full"),
    Workload("sq4096", 4096, 4096, 4096, "uniform", "uniform", 2, "full"),
    Workload("mlp_up", 4096, 11008, 4096, "normal:1", "normal:0.02", 3, "full"),
    Workload("mlp_down", 4096, 4096, 11008, "normal:1", "normal:0.02", 4, "full"),
    _decode(1, 11008, 4096, 5), _decode(2, 11008, 4096, 6),
    _decode(16, 11008, 4096, 7), _decode(64, 11008, 4096, 8),
    _decode(1, 4096, 11008, 9), _decode(2, 4096, 11008, 10),
    _decode(16, 4096, 11008, 11), _decode(64, 4096, 11008, 12),
    Workload("sq8192", 8192, 8192, 8192, "uniform", "uniform", 13, "sampled"),
    Workload("sq16384", 16384, 16384, 16384, "uniform", "uniform", 14, "sampled"),
]}


@dataclasses.dataclass(frozen=True)
class GatedWorkload:
    """One synthetic gated projection C = silu(A . Wg^T) * (A . Wu^T): the Llama
    MLP's gate and up weights [N, K] share a shape and a distribution."""
    base: Workload   # A and the gate weights Wg (its B)

    @property
    def name(self) -> str:
        return "swiglu_" + self.base.name

    def up(self) -> np.ndarray:
        return matrix(self.base.N, self.base.K, self.base.dist_b, self.base.seed_b + 1000)

    @property
    def flops(self) -> int:
        return 2 * self.base.flops

    @property
    def decode_bytes(self) -> int:
        b = self.base
        return 2 * (2 * b.N * b.K + b.M * b.K + b.M * b.N)


GATED_WORKLOADS = {g.name: g for g in [GatedWorkload(WORKLOADS[n]) for n in
                                       ("mlp_up", "dec1_up", "dec2_up", "dec16_up", "dec64_up")]}


@dataclasses.dataclass(frozen=True)
class ResidualWorkload:
    """One synthetic projection with its residual added, C = A . B^T + R: the
    Llama MLP's down projection onto the residual stream R ~ N(0, 1), [M, N]."""
    base: Workload

    @property
    def name(self) -> str:
        return "resid_" + self.base.name

    def r(self) -> np.ndarray:
        return matrix(self.base.M, self.base.N, "normal:1", self.base.seed_a + 2000)

    @property
    def flops(self) -> int:
        return self.base.flops

    @property
    def decode_bytes(self) -> int:
        b = self.base
        return 2 * (b.N * b.K + b.M * b.K + 2 * b.M * b.N)


RESIDUAL_WORKLOADS = {r.name: r for r in [ResidualWorkload(WORKLOADS[n]) for n in
                                          ("mlp_down", "dec1_down", "dec16_down", "dec64_down")]}


@dataclasses.dataclass(frozen=True)
class BatchedWorkload:
    """Several weight matrices read against the same activations in one launch:
    the Llama attention's Q, K and V projections (three 4096 x 4096 weights) for
    M decode tokens."""
    name: str
    M: int
    Ns: tuple
    K: int
    cfg: int

    def a(self) -> np.ndarray:
        return matrix(self.M, self.K, "normal:1", SEED_A_BASE + self.cfg)

    def bs(self) -> list:
        return [matrix(n, self.K, "normal:0.02", SEED_B_BASE + self.cfg + 100 * i) for i, n in enumerate(self.Ns)]

    @property
    def decode_bytes(self) -> int:
        n = sum(self.Ns)
        return 2 * (n * self.K + self.M * self.K + self.M * n)


BATCHED_WORKLOADS = {w.name: w for w in [BatchedWorkload(f"qkv_dec{m}", m, (4096, 4096, 4096), 4096, 40 + m)
                                         for m in (1, 16, 64)]}


def sample_indices(extent: int, count: int, seed: int) -> np.ndarray:
    """A sorted, seeded choice of ``count`` distinct indices in [0, extent)."""
    if count >= extent:
        return np.arange(extent, dtype=np.int64)
    keys = splitmix64(seed, 0, extent)
    return np.sort(np.argsort(keys, kind="stable")[:count]).astype(np.int64)


# ------------------------------------------------------------------ NVFP4 inputs
# Packed FP4 operands and their E4M3 block scales, drawn as raw codes: every byte
# of a packed row is uniform over 0..255 (two uniform E2M1 codes, signed zeros
# included), every scale code uniform over 0x28..0x3F (E4M3 values 0.25 .. 1.875),
# so sums over K = 4096 stay far inside the fp16 output range.  The pages give no
# distribution for their NVFP4 operands; this is the plain reading.
NVFP4_SCALE_LO = 0x28
NVFP4_SCALE_HI = 0x3F


def nvfp4_codes(rows: int, K: int, seed: int, ld: int | None = None) -> np.ndarray:
    """rows x ld bytes: the first K/2 of each row hold K packed E2M1 codes; padding
    bytes are 0xFF (a pair of -6 codes, so a kernel that reads padding shows it)."""
    assert K % 2 == 0
    ld = K // 2 if ld is None else ld
    assert ld >= K // 2
    core = (splitmix64(seed, 0, rows * (K // 2)) >> np.uint64(56)).astype(np.uint8).reshape(rows, K // 2)
    if ld == K // 2:
        return core
    out = np.full((rows, ld), 0xFF, dtype=np.uint8)
    out[:, :K // 2] = core
    return out


def nvfp4_scales(rows: int, K: int, seed: int, ld: int | None = None) -> np.ndarray:
    """rows x ld plain row-major E4M3 scale codes, one per 16 elements of K."""
    assert K % 16 == 0
    nblk = K // 16
    ld = nblk if ld is None else ld
    span = NVFP4_SCALE_HI - NVFP4_SCALE_LO + 1
    u = splitmix64(seed, 1 << 40, rows * nblk) >> np.uint64(32)
    core = (NVFP4_SCALE_LO + (u % np.uint64(span))).astype(np.uint8).reshape(rows, nblk)
    out = np.zeros((rows, ld), dtype=np.uint8)
    out[:, :nblk] = core
    return out


@dataclasses.dataclass(frozen=True)
class Nvfp4Workload:
    """C[M,N] = alpha (A . SFA) . (B . SFB)^T with packed NVFP4 operands, E4M3
    scales over 16-element blocks and FP16 output: the square shapes of the gemm3
    benchmarks page (4096^3 .. 32768^3) and a small one the oracle finishes fast."""
    name: str
    M: int
    N: int
    K: int
    cfg: int
    alpha: float = 1.0

    def a(self) -> np.ndarray:
        return nvfp4_codes(self.M, self.K, SEED_A_BASE + self.cfg)

    def b(self) -> np.ndarray:
        return nvfp4_codes(self.N, self.K, SEED_B_BASE + self.cfg)

    def sfa(self) -> np.ndarray:
        return nvfp4_scales(self.M, self.K, SEED_A_BASE + 500 + self.cfg)

    def sfb(self) -> np.ndarray:
        return nvfp4_scales(self.N, self.K, SEED_B_BASE + 500 + self.cfg)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


NVFP4_WORKLOADS = {w.name: w for w in [
    Nvfp4Workload("fp4_sq512", 512, 512, 512, 60),
    Nvfp4Workload("fp4_sq4096", 4096, 4096, 4096, 61),
    Nvfp4Workload("fp4_sq8192", 8192, 8192, 8192, 62),
    Nvfp4Workload("fp4_sq16384", 16384, 16384, 16384, 63),
]}


@dataclasses.dataclass(frozen=True)
class AttentionWorkload:
    """Attention of one decoder layer: Q [B, Sq, H, 128] against K, V [B, Sk, Hkv,
    128], all N(0, 1) rounded to bf16 (query/key/value activations of unit scale),
    token-major with heads x head_dim contiguous.  The spark-kernels page's shapes:
    4096 tokens and 32 heads of 128, causal and not, and one decode query against
    a 4096-token cache."""
    name: str
    B: int
    Sq: int
    Sk: int
    H: int
    Hkv: int
    causal: bool
    cfg: int
    D: int = 128

    def _t(self, S: int, heads: int, seed: int) -> np.ndarray:
        return matrix(self.B * S, heads * self.D, "normal", seed).reshape(self.B, S, heads, self.D)

    def q(self) -> np.ndarray:
        return self._t(self.Sq, self.H, SEED_A_BASE + 700 + self.cfg)

    def k(self) -> np.ndarray:
        return self._t(self.Sk, self.Hkv, SEED_B_BASE + 700 + self.cfg)

    def v(self) -> np.ndarray:
        return self._t(self.Sk, self.Hkv, SEED_B_BASE + 800 + self.cfg)

    @property
    def flops(self) -> int:
        """4 B H D x (visible query-key pairs): two products of 2 FLOP per pair and
        dimension (the causal count is the halved one the page quotes)."""
        if self.causal:
            pairs = sum(min(self.Sk, i + (self.Sk - self.Sq) + 1) for i in range(self.Sq))
        else:
            pairs = self.Sq * self.Sk
        return 4 * self.B * self.H * self.D * pairs

    @property
    def kv_bytes(self) -> int:
        return 2 * 2 * self.B * self.Sk * self.Hkv * self.D


ATTENTION_WORKLOADS = {w.name: w for w in [
    AttentionWorkload("attn_small", 2, 300, 300, 4, 4, True, 70),
    AttentionWorkload("attn_causal_4096", 1, 4096, 4096, 32, 32, True, 71),
    AttentionWorkload("attn_4096", 1, 4096, 4096, 32, 32, False, 72),
    AttentionWorkload("attn_decode_4096", 1, 1, 4096, 32, 32, True, 73),
]}
