"""Parity of the fused attention kernels (attention_bf16: the tcgen05 kernel and the
CUDA-core decode kernel) against the fp64 oracle.

Tolerance, per element: |gpu - ref| <= 4e-3 |ref| + 4e-3 W, where W is the
attention of |V| (the weighted mean of the visible |v_j|).  The kernel rounds the
softmax weights to bf16 for the P V product (relative error <= 2^-9 per weight;
the normalisation uses the same rounded weights, so the output moves by at most
2^-9 (W + |O|)) and rounds O to bf16 (2^-9 |O|); fp32 scores, exp2 and
accumulation add far less.  The CUDA-core decode kernel keeps the weights in
fp32, so the same bound holds for it with margin.  Over the compared set the
relative Frobenius error must stay <= 1e-2.

Layout probes use inputs whose results are exact or nearly so: zero queries (every
visible key weighs the same, so O is the mean of the visible values), and
one-hot queries against one-hot keys (one key dominates by e^-64 or more), which
pin the Q K^T operand layout, the V operand (read MN-major), the causal offset,
the grouped-head mapping and the row stores.
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import skinny_gemv_gb300 as sg  # noqa: E402

REL_TOL = 4e-3
W_TOL = 4e-3
FRO_TOL = 1e-2
D = 128


def to_dev(bits: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def from_dev(t) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16(x: np.ndarray) -> np.ndarray:
    return syn.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def run(Qb, Kb, Vb, causal, scale=None, O=None, path=sg.PATH_AUTO):
    O = sg.attention_bf16(to_dev(Qb), to_dev(Kb), to_dev(Vb), O=O, causal=causal, scale=scale, path=path)
    torch.cuda.synchronize()
    st, detail = sg.check_device_errors()
    assert st == 0, detail
    return oracle._bf16_tensor(from_dev(O))


def assert_close(got, Qb, Kb, Vb, causal, scale=None, label=""):
    ref = oracle.attention(Qb, Kb, Vb, causal=causal, scale=scale)
    W = oracle.attention(Qb, Kb, np.abs(oracle._bf16_tensor(Vb)), causal=causal, scale=scale)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    d = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref) + W_TOL * W
    n_over = int(np.count_nonzero(d > bound))
    fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    assert n_over == 0, f"{label}: {n_over} elements over the bound (max |d| {d.max():.3g})"
    assert fro <= FRO_TOL, f"{label}: relative Frobenius error {fro:.3g}"
    return fro


def seeded(B, S, H, seed):
    return syn.matrix(B * S, H * D, "normal", seed).reshape(B, S, H, D)


@pytest.mark.parametrize("Sq,Sk,causal", [(128, 128, True), (300, 300, True), (200, 333, False), (5, 260, True),
                                          (130, 70, True), (1, 1, True), (2, 700, True), (1, 4096, False)])
def test_zero_queries_average_values(Sq, Sk, causal):
    rng = np.random.default_rng(Sq * 1000 + Sk)
    B, H = 2, 2
    Qb = np.zeros((B, Sq, H, D), dtype=np.uint16)
    Kb = bf16(rng.standard_normal((B, Sk, H, D)))
    Vb = bf16(rng.integers(-8, 9, size=(B, Sk, H, D)).astype(np.float64))
    # H = Hkv: one query row per kv head and query, so the decode kernel takes Sq <= 4
    paths = [sg.PATH_TENSOR_CORE] + ([sg.PATH_CUDA_CORE] if Sq <= 4 else [])
    for path in paths:
        _zero_queries_check(run(Qb, Kb, Vb, causal, path=path), Qb, Kb, Vb, causal)


def _zero_queries_check(got, Qb, Kb, Vb, causal):
    ref = oracle.attention(Qb, Kb, Vb, causal=causal)
    # every weight is exactly 1: O is the mean of small integers, rounded to bf16 (one
    # bf16 step); a key split merges per-split means with fp32 weights from
    # exp2/log2 approximations, which moves a result by ~1e-6 at most
    want = oracle._bf16_tensor(bf16(ref))
    step = np.abs(want) * 2.0 ** -7 + 1e-5
    assert np.all(np.abs(got - want) <= step), f"max |d| {np.abs(got - want).max()}"


@pytest.mark.parametrize("Sk", [128, 256, 200])
def test_one_hot_scores_select_one_value(Sk):
    # query i has 64 at coordinate c_i; key j is e_{j mod 128} (negated past the
    # first block), so with scale 1 key c_i wins by 64 over every other key.
    rng = np.random.default_rng(7)
    B, Sq, H = 1, 128, 2
    perm = rng.permutation(128)
    Q = np.zeros((B, Sq, H, D))
    for i in range(Sq):
        Q[0, i, :, perm[i]] = 64.0
    K = np.zeros((B, Sk, H, D))
    for j in range(Sk):
        K[0, j, :, j % 128] = 1.0 if j < 128 else -1.0
    V = rng.integers(-100, 101, size=(B, Sk, H, D)).astype(np.float64)
    Qb, Kb, Vb = bf16(Q), bf16(K), bf16(V)
    got = run(Qb, Kb, Vb, causal=False, scale=1.0)
    want = np.stack([V[0, perm[i]] for i in range(Sq)])[None]
    np.testing.assert_allclose(got, want, rtol=2.0 ** -8, atol=1e-6)


def test_grouped_heads_read_their_kv_head():
    rng = np.random.default_rng(8)
    B, Sq, Sk, H, Hkv = 1, 64, 130, 6, 2
    Qb = np.zeros((B, Sq, H, D), dtype=np.uint16)
    Kb = bf16(rng.standard_normal((B, Sk, Hkv, D)))
    Vb = bf16(np.broadcast_to(np.arange(Hkv, dtype=np.float64)[None, None, :, None] * 10 + 1.0, (B, Sk, Hkv, D)))
    got = run(Qb, Kb, Vb, causal=False)
    for h in range(H):
        assert np.all(got[:, :, h] == 10.0 * (h // (H // Hkv)) + 1.0), h


def test_grouped_heads_decode_kernel():
    # one query per head, four query heads per kv head: the decode kernel's rows
    rng = np.random.default_rng(18)
    B, Sq, Sk, H, Hkv = 2, 1, 130, 8, 2
    Qb = bf16(rng.standard_normal((B, Sq, H, D)))
    Kb = bf16(rng.standard_normal((B, Sk, Hkv, D)))
    Vb = bf16(np.broadcast_to(np.arange(Hkv, dtype=np.float64)[None, None, :, None] * 10 + 1.0, (B, Sk, Hkv, D)))
    got = run(Qb, Kb, Vb, causal=True, path=sg.PATH_CUDA_CORE)
    for h in range(H):
        assert np.all(got[:, :, h] == 10.0 * (h // (H // Hkv)) + 1.0), h


DECODE_CASES = [
    (1, 1, 4096, 32, 32, True),   # the decode workload's shape
    (2, 1, 777, 8, 2, True),      # grouped heads: four query rows per kv head
    (3, 2, 300, 4, 4, True),      # two queries: the first sees one key fewer
    (1, 4, 129, 2, 2, True),      # four causal queries
    (2, 3, 50, 1, 1, False),      # three rows, few keys
    (1, 1, 31, 4, 2, True),       # fewer keys than one step of the kernel
    (1, 3, 2, 2, 2, True),        # more queries than keys: the first row sees nothing
]


@pytest.mark.parametrize("B,Sq,Sk,H,Hkv,causal", DECODE_CASES)
def test_decode_kernel_parity(B, Sq, Sk, H, Hkv, causal):
    # both kernels on the decode shapes (AUTO takes the CUDA-core one)
    seed = 9500 + B * 131 + Sq * 7 + Sk
    Qb, Kb, Vb = seeded(B, Sq, H, seed), seeded(B, Sk, Hkv, seed + 1), seeded(B, Sk, Hkv, seed + 2)
    for path in (sg.PATH_CUDA_CORE, sg.PATH_TENSOR_CORE, sg.PATH_AUTO):
        got = run(Qb, Kb, Vb, causal, path=path)
        assert_close(got, Qb, Kb, Vb, causal, label=f"path {path} {(B, Sq, Sk, H, Hkv, causal)}")
        if causal and Sq > Sk:
            assert np.all(got[:, : Sq - Sk] == 0.0)


def test_decode_kernel_rejects_many_rows():
    Q = torch.zeros((1, 5, 2, D), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((1, 9, 2, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        sg.attention_bf16(Q, K, K, causal=True, path=sg.PATH_CUDA_CORE)


@pytest.mark.parametrize("B,Sq,Sk,H,Hkv,causal", [
    (1, 256, 256, 2, 2, True),
    (1, 256, 256, 2, 2, False),
    (2, 200, 333, 4, 2, True),
    (2, 200, 333, 4, 4, False),
    (1, 1, 1000, 4, 1, True),     # one decode query against a cache
    (3, 17, 17, 2, 1, True),      # batches inside one tile
    (1, 300, 129, 2, 2, True),    # more queries than keys: the first rows see nothing
])
def test_parity_seeded(B, Sq, Sk, H, Hkv, causal):
    seed = 9000 + B * 131 + Sq * 7 + Sk
    Qb, Kb, Vb = seeded(B, Sq, H, seed), seeded(B, Sk, Hkv, seed + 1), seeded(B, Sk, Hkv, seed + 2)
    got = run(Qb, Kb, Vb, causal)
    assert_close(got, Qb, Kb, Vb, causal, label=f"{(B, Sq, Sk, H, Hkv, causal)}")
    if causal and Sq > Sk:
        assert np.all(got[:, : Sq - Sk] == 0.0)


def test_scale_and_pitches():
    rng = np.random.default_rng(10)
    B, Sq, Sk, H = 1, 150, 190, 2
    Qb, Kb, Vb = (bf16(rng.standard_normal((B, S, H, D))) for S in (Sq, Sk, Sk))
    # padded token rows: views of wider buffers, NaN padding that must not be read
    def padded(x, extra):
        buf = torch.full((x.shape[0], x.shape[1], (H * D + extra)), float("nan"), dtype=torch.bfloat16, device="cuda")
        buf[:, :, :H * D] = to_dev(x).reshape(x.shape[0], x.shape[1], H * D)
        return buf[:, :, :H * D].unflatten(2, (H, D))
    Qd, Kd, Vd = padded(Qb, 8), padded(Kb, 64), padded(Vb, 16)
    Obuf = torch.full((B, Sq, H * D + 24), float("nan"), dtype=torch.bfloat16, device="cuda")
    Od = Obuf[:, :, :H * D].unflatten(2, (H, D))
    sg.attention_bf16(Qd, Kd, Vd, O=Od, causal=True, scale=0.05)
    torch.cuda.synchronize()
    got = oracle._bf16_tensor(from_dev(Od.contiguous()))
    assert_close(got, Qb, Kb, Vb, True, scale=0.05, label="pitched")
    assert torch.isnan(Obuf[:, :, H * D:]).all(), "padding columns of O were written"


def test_empty_and_zero_keys():
    Q = torch.zeros((1, 4, 2, D), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((1, 0, 2, D), dtype=torch.bfloat16, device="cuda")
    O = torch.full((1, 4, 2, D), 7.0, dtype=torch.bfloat16, device="cuda")
    sg.attention_bf16(Q, K, K, O=O)
    torch.cuda.synchronize()
    assert (O == 0).all()
    E = torch.zeros((1, 0, 2, D), dtype=torch.bfloat16, device="cuda")
    sg.attention_bf16(E, Q, Q, O=E.clone())  # no queries: no work


def test_deterministic():
    Qb, Kb, Vb = seeded(1, 300, 2, 77), seeded(1, 300, 2, 78), seeded(1, 300, 2, 79)
    a = run(Qb, Kb, Vb, True)
    b = run(Qb, Kb, Vb, True)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["attn_causal_4096", "attn_4096", "attn_decode_4096"])
def test_workload_sampled(name):
    """The full-size workloads, checked on sampled (head, query) rows: row i of a
    causal launch against the oracle over its key prefix."""
    w = syn.ATTENTION_WORKLOADS[name]
    Qb, Kb, Vb = w.q(), w.k(), w.v()
    O = sg.attention_bf16(to_dev(Qb), to_dev(Kb), to_dev(Vb), causal=w.causal)
    torch.cuda.synchronize()
    got = oracle._bf16_tensor(from_dev(O))
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, w.Sq - 1], rng.integers(0, w.Sq, size=6)]))
    heads = np.unique(np.concatenate([[0, w.H - 1], rng.integers(0, w.H, size=2)]))
    for i in rows:
        n = w.Sk if not w.causal else i + (w.Sk - w.Sq) + 1
        sub = (slice(None), slice(i, i + 1), heads)
        kv = (slice(None), slice(0, n), heads // (w.H // w.Hkv))
        assert_close(got[sub], Qb[sub], Kb[kv], Vb[kv], False, label=f"{name} row {i}")


@pytest.mark.parametrize("scale", [-0.08, 0.0, 0.3])
def test_negative_zero_and_large_scales(scale):
    Qb, Kb, Vb = seeded(1, 200, 2, 500), seeded(1, 260, 2, 501), seeded(1, 260, 2, 502)
    got = run(Qb, Kb, Vb, True, scale=scale)
    assert_close(got, Qb, Kb, Vb, True, scale=scale, label=f"scale {scale}")


def test_decode_kernel_pitches_scales_and_reruns():
    # the decode kernel (three query rows per kv head) on NaN-padded token rows:
    # padding must be neither read nor written; any finite scale; identical reruns
    rng = np.random.default_rng(11)
    B, Sq, Sk, H, Hkv = 2, 1, 190, 6, 2
    Qb = bf16(rng.standard_normal((B, Sq, H, D)))
    Kb, Vb = (bf16(rng.standard_normal((B, Sk, Hkv, D))) for _ in range(2))

    def padded(x, heads, extra):
        buf = torch.full((x.shape[0], x.shape[1], heads * D + extra), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        buf[:, :, :heads * D] = to_dev(x).reshape(x.shape[0], x.shape[1], heads * D)
        return buf[:, :, :heads * D].unflatten(2, (heads, D))
    Qd, Kd, Vd = padded(Qb, H, 8), padded(Kb, Hkv, 64), padded(Vb, Hkv, 16)
    for scale in (0.05, -0.08, 0.0, 0.3):
        Obuf = torch.full((B, Sq, H * D + 24), float("nan"), dtype=torch.bfloat16, device="cuda")
        Od = Obuf[:, :, :H * D].unflatten(2, (H, D))
        sg.attention_bf16(Qd, Kd, Vd, O=Od, causal=True, scale=scale, path=sg.PATH_CUDA_CORE)
        torch.cuda.synchronize()
        got = oracle._bf16_tensor(from_dev(Od.contiguous()))
        assert_close(got, Qb, Kb, Vb, True, scale=scale, label=f"decode kernel, pitched, scale {scale}")
        assert torch.isnan(Obuf[:, :, H * D:]).all(), "padding columns of O were written"
        again = sg.attention_bf16(Qd, Kd, Vd, causal=True, scale=scale, path=sg.PATH_CUDA_CORE)
        torch.cuda.synchronize()
        assert torch.equal(again.view(torch.int16), Od.contiguous().view(torch.int16)), "rerun differs"
