"""The C-ABI library on the host (no GPU needed): it loads, exports every symbol
the header declares, rejects bad arguments before touching CUDA, and its launch
planner produces schedules that cover every (tile, k-step) exactly once."""
import ctypes
import os

import numpy as np
import pytest

import skinny_gemv_gb300 as sg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    sg._build.build()
    return sg.load()


def test_exports_every_declared_symbol(lib):
    names = sg.declared_symbols()
    assert len(names) >= 14
    for n in ["gemm_bf16", "gemv_bf16", "gemv_bf16_path", "sg_status_string", "sg_last_cuda_error",
              "sg_check_device_errors", "sg_plan", "sg_bench_tcgen05_peak", "sg_bench_copy",
              "sg_bench_read", "sg_device_query"]:
        assert n in names
    exported = set()
    import subprocess
    out = subprocess.check_output(["nm", "-D", "--defined-only", sg.library_path()]).decode()
    for line in out.splitlines():
        parts = line.split()
        if len(parts) == 3 and parts[1] == "T":
            exported.add(parts[2])
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)
        # every entry point has a full ctypes prototype: without one, ctypes would
        # pass 64-bit pointers and sizes as 32-bit ints
        assert getattr(lib, n).argtypes is not None, f"{n} has no argtypes"
        assert getattr(lib, n).restype is not None or n in ("sg_set_wait_timeout_ns",
                                                            "sg_debug_inject_missing_tx"), n


def test_status_strings(lib):
    for code in range(7):
        s = lib.sg_status_string(code).decode()
        assert s.startswith("SG_")
    assert lib.sg_status_string(99).decode() == "unknown sg_status"


@pytest.mark.parametrize("args,code", [
    # (A, B, C, M, N, K, lda, ldb, ldc)
    ((16, 16, 16, -1, 8, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),
    ((16, 16, 16, 8, -1, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),
    ((16, 16, 16, 8, 8, -8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),
    ((0, 16, 16, 8, 8, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),       # null A
    ((16, 0, 16, 8, 8, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),       # null B
    ((16, 16, 0, 8, 8, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),       # null C
    ((16, 16, 16, 8, 8, 16, 8, 16, 8), sg.SG_ERR_INVALID_ARG),    # lda < K
    ((16, 16, 16, 8, 8, 16, 16, 8, 8), sg.SG_ERR_INVALID_ARG),    # ldb < K
    ((16, 16, 16, 8, 16, 8, 8, 8, 8), sg.SG_ERR_INVALID_ARG),     # ldc < N
    ((18, 16, 16, 8, 8, 8, 8, 8, 8), sg.SG_ERR_MISALIGNED),       # A not 16-B aligned
    ((16, 24, 16, 8, 8, 8, 8, 8, 8), sg.SG_ERR_MISALIGNED),       # B not 16-B aligned
    ((16, 16, 16, 8, 8, 12, 12, 16, 8), sg.SG_ERR_MISALIGNED),    # lda % 8
    ((16, 16, 16, 8, 8, 8, 8, 8, 12), sg.SG_ERR_MISALIGNED),      # ldc % 8
])
def test_argument_errors_before_any_cuda_call(lib, args, code):
    assert lib.gemm_bf16(*args, None) == code
    assert lib.gemv_bf16(*args, None) == code


def test_empty_problems_are_noops(lib):
    # M = 0 or N = 0: nothing to do, no CUDA call, even with null pointers
    assert lib.gemm_bf16(None, None, None, 0, 8, 8, 8, 8, 8, None) == sg.SG_OK
    assert lib.gemm_bf16(None, None, None, 8, 0, 8, 8, 8, 8, None) == sg.SG_OK
    assert lib.gemv_bf16(None, None, None, 0, 8, 8, 8, 8, 8, None) == sg.SG_OK


def test_gemv_rejects_large_m_and_bad_path(lib):
    assert lib.gemv_bf16(16, 16, 16, 65, 8, 8, 8, 8, 8, None) == sg.SG_ERR_INVALID_ARG
    assert lib.gemv_bf16_path(16, 16, 16, 4, 8, 8, 8, 8, 8, 7, None) == sg.SG_ERR_INVALID_ARG
    assert lib.gemm_bf16_path(16, 16, 16, 4, 8, 8, 8, 8, 8, 5, None) == sg.SG_ERR_INVALID_ARG
    assert lib.gemm_bf16_path(16, 16, 16, 65, 8, 8, 8, 8, 8, sg.PATH_CUDA_CORE, None) == sg.SG_ERR_INVALID_ARG


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split(None, 4))
    return rows


def test_wave_efficiency_matches_printed_values(lib):
    rows = _golden_rows("wave_efficiency.txt")
    assert len(rows) >= 5
    for ctas, slots, want, tol, *_ in rows:
        got = sg.wave_efficiency(int(ctas), int(slots))
        assert abs(got - float(want)) <= float(tol), (ctas, slots, got, want)
    # the two-factor product the page prints: 86.1% x 95.7% = 82.4%
    assert abs(sg.wave_efficiency(1024, 170) * 0.957 - 0.824) < 0.001


def test_waves_of_the_rtx5090_example():
    for tiles, slots, waves in (r[:3] for r in _golden_rows("waves.txt")):
        assert round(int(tiles) / int(slots), 2) == float(waves)
    # tiles of a 4096^2 output in 128 x 128 tiles
    assert (4096 // 128) ** 2 == 1024


def _check_plan_coverage(info):
    items = sg.plan_items(info)
    T = info["tiles_m"] * info["tiles_n"]
    KS = info["k_steps"]
    cover = np.zeros((T, KS), dtype=np.int32)
    pieces = {}
    # split mode (the swapped skinny plans, and GEMM plans below one wave): every
    # tile cut into split_k pieces, one per CTA
    split_mode = info["path"] in (sg.PATH_TENSOR_CORE, sg.PATH_GEMM, sg.PATH_GEMM_PAIR) and info["split_k"] > 0
    for cta, row in enumerate(items):
        assert len(row) >= 1, f"CTA {cta} has no work"
        n_sk = sum(1 for it in row if it[0] < info["sk_tiles"])
        # Stream-K pieces (tiles [0, sk_tiles)) come first, then whole tiles
        assert all(it[0] < info["sk_tiles"] for it in row[:n_sk])
        for idx, (tile, k0, k1, piece, npieces, slot, sk, tm, tn) in enumerate(row):
            assert 0 <= tile < T and 0 <= k0 < k1 <= KS
            assert 0 <= tm < info["tiles_m"] and 0 <= tn < info["tiles_n"]
            cover[tile, k0:k1] += 1
            if npieces > 1:
                if split_mode:  # one piece per CTA, its own slot
                    assert slot == cta and len(row) == 1
                else:
                    assert slot in (2 * cta, 2 * cta + 1)
                    # slot 0 of a CTA is its first Stream-K item, slot 1 its last
                    assert (slot == 2 * cta) == (idx == 0)
                    assert idx in (0, n_sk - 1)
                pieces.setdefault(tile, []).append((k0, k1, piece, npieces, cta, slot))
            else:
                assert (k0, k1) == (0, KS) and slot == -1
    assert np.all(cover == 1), "every (tile, k-step) exactly once"
    # (tile row, tile col) is a bijection of tile indices
    coords = {(it[7], it[8]) for row in items for it in row}
    assert len(coords) == T
    for tile, ps in pieces.items():
        ps.sort()
        n = ps[0][3]
        assert len(ps) == n and [p[2] for p in ps] == list(range(n))
        assert ps[0][0] == 0 and ps[-1][1] == KS
        assert all(ps[i][1] == ps[i + 1][0] for i in range(n - 1))
        assert [p[4] for p in ps] == list(range(ps[0][4], ps[0][4] + n)), "consecutive CTAs"
        assert len({p[5] for p in ps}) == n
    return items


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (2048, 2048, 2048), (512, 512, 512),
                                   (4096, 11008, 4096), (4096, 4096, 11008), (8192, 8192, 8192),
                                   (65, 257, 4104), (1000, 3000, 200), (129, 8, 64),
                                   # below one wave: narrow tiles, K split into equal pieces
                                   (128, 4096, 4096), (384, 512, 8192), (300, 1000, 2048), (256, 256, 65536)])
@pytest.mark.parametrize("sms", [148, 152, 170])
@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
def test_gemm_plan_covers_every_unit_once(lib, M, N, K, sms, path):
    info = sg.plan(M, N, K, sms, path)
    pair = path == sg.PATH_GEMM_PAIR
    assert info["path"] == path and info["cluster_size"] == (2 if pair else 1)
    tm = 256 if pair else 128
    units = sms // 2 if pair else sms
    # single-CTA tiles are 128 wide when the 128 x 128 tiles fit in one wave
    tn = 128 if not pair and -(-M // 128) * -(-N // 128) <= sms else 256
    assert info["tile_m"] == tm and info["tile_n"] == tn and info["tile_k"] == 64
    assert info["stages"] == (6 if pair or tn == 128 else 4)
    assert info["tiles_m"] == -(-M // tm) and info["tiles_n"] == -(-N // tn)
    assert info["grid"] <= units
    T = info["tiles_m"] * info["tiles_n"]
    assert info["dp_tiles"] + info["sk_tiles"] == T
    if info["split_k"] > 0:  # below one wave: every tile in split_k equal pieces, at most 8
        assert T < units and 2 <= info["split_k"] <= 8 and info["grid"] == T * info["split_k"]
    if T >= units and T % units:
        rem, KS = T % units, info["k_steps"]
        if (units - rem) * KS <= 24 * units:
            assert info["sk_tiles"] == 0  # quantisation costs less than a fixup
        elif rem * KS >= 16 * units:
            assert info["sk_tiles"] == rem  # Stream-K over the remainder
        else:
            assert info["sk_tiles"] == rem + units  # thin remainder: plus the last wave
    _check_plan_coverage(info)


def test_auto_gemm_kernel_choice(lib):
    # 128 x 128 single-CTA tiles wherever they fit in one wave of SMs
    for M, N in [(128, 4096), (255, 4096), (256, 4096), (512, 4096), (512, 512), (1536, 1536), (128, 19456)]:
        info = sg.plan(M, N, 4096, 152, 0)
        assert info["path"] == sg.PATH_GEMM and info["tile_n"] == 128, (M, N)
    # past one wave: 128 x 256 single tiles below M = 256, CTA pairs from there
    assert sg.plan(128, 32768, 4096, 152, 0)["path"] == sg.PATH_GEMM
    assert sg.plan(128, 32768, 4096, 152, 0)["tile_n"] == 256
    assert sg.plan(255, 32768, 4096, 152, 0)["path"] == sg.PATH_GEMM
    assert sg.plan(256, 32768, 4096, 152, 0)["path"] == sg.PATH_GEMM_PAIR
    assert sg.plan(4096, 4096, 4096, 152, 0)["grid"] == 76
    # pair tiles short of a wave at <= 32 k-steps, 128 x 256 single tiles within one: single
    for M, N, K in [(2048, 2048, 2048), (1792, 1792, 1792), (1024, 4096, 2048)]:
        info = sg.plan(M, N, K, 152, 0)
        assert info["path"] == sg.PATH_GEMM and info["tile_n"] == 256, (M, N, K)
    assert sg.plan(1024, 4096, 4096, 152, 0)["path"] == sg.PATH_GEMM_PAIR  # 64 k-steps: pairs
    assert sg.plan(2048, 4096, 2048, 152, 0)["path"] == sg.PATH_GEMM_PAIR  # a full wave of pairs
    # the rules follow the SM count: 1536^3 is 144 tiles of 128 x 128, more than 132
    # SMs, so 128 x 256 single tiles (36 pair tiles are short of 66 clusters)
    info = sg.plan(1536, 1536, 1536, 132, 0)
    assert info["path"] == sg.PATH_GEMM and info["tile_n"] == 256


@pytest.mark.parametrize("M", [1, 2, 9, 16, 17, 33, 64])
@pytest.mark.parametrize("N,K", [(11008, 4096), (4096, 11008), (300, 700), (128, 64), (32000, 4096)])
def test_skinny_tensor_core_plan(lib, M, N, K):
    info = sg.plan(M, N, K, 152, sg.PATH_TENSOR_CORE)
    assert info["path"] == sg.PATH_TENSOR_CORE
    assert info["tile_n"] == (16 if M <= 16 else 32 if M <= 32 else 64)
    rows = 128 if M <= 16 else 64  # wider weight tiles (fewer thin MMAs) up to 16 activation rows
    assert info["tile_m"] == rows and info["tiles_n"] == 1 and info["tiles_m"] == -(-N // rows)
    assert info["ctas_per_sm"] == 2 and info["tile_k"] == (128 if rows == 64 else 64)
    assert info["k_steps"] == -(-K // info["tile_k"])
    items = _check_plan_coverage(info)
    T, KS = info["tiles_m"], info["k_steps"]
    if T <= 304:
        # split mode: S equal k pieces per tile (each at least 512 of K), one resident CTA each
        S = max(1, min(304 // T, KS // (512 // info["tile_k"])))
        assert info["split_k"] == S and info["grid"] == T * S <= 304
        sizes = [k1 - k0 for row in items for (_, k0, k1, *_) in row]
        assert max(sizes) - min(sizes) <= 1
    else:
        assert info["split_k"] == 0 and info["grid"] == 304
        if T % 304:
            assert info["sk_tiles"] == T % 304  # only the remainder is split
    # the weights are read once: each weight tile's k-steps are covered exactly once
    assert sum(k1 - k0 for row in items for (_, k0, k1, *_) in row) == info["tiles_m"] * info["k_steps"]
    # early L2 reads of the first 8 k-steps only when the grid fills 70% of the slots
    assert info["prefetch_steps"] == (8 if info["grid"] * 10 >= 7 * 304 else 0)


def test_prefetch_only_on_skinny_paths(lib):
    assert sg.plan(4096, 4096, 4096, 152, 0)["prefetch_steps"] == 0
    assert sg.plan(128, 4096, 4096, 152, 0)["prefetch_steps"] == 0
    assert sg.plan(64, 11008, 4096, 152, 0)["prefetch_steps"] == 0  # 172 CTAs on 304 slots
    assert sg.plan(64, 4096, 11008, 152, 0)["prefetch_steps"] == 8  # 64 tiles x 4 pieces
    assert sg.plan(16, 11008, 4096, 152, 0)["prefetch_steps"] == 8  # 86 tiles x 3 pieces
    assert sg.plan(1, 11008, 4096, 152, 0)["prefetch_steps"] == 1


def test_auto_path_choice(lib):
    assert sg.plan(1, 4096, 4096, 152, 0)["path"] == sg.PATH_CUDA_CORE
    assert sg.plan(2, 4096, 4096, 152, 0)["path"] == sg.PATH_CUDA_CORE
    assert sg.plan(3, 4096, 4096, 152, 0)["path"] == sg.PATH_TENSOR_CORE
    assert sg.plan(9, 4096, 4096, 152, 0)["path"] == sg.PATH_TENSOR_CORE
    assert sg.plan(64, 4096, 4096, 152, 0)["path"] == sg.PATH_TENSOR_CORE
    assert sg.plan(65, 4096, 4096, 152, 0)["path"] == sg.PATH_GEMM


@pytest.mark.parametrize("N,K", [(11008, 4096), (4096, 11008), (256, 8192), (100, 24), (1 << 20, 64)])
def test_cuda_core_plan(lib, N, K):
    info = sg.plan(2, N, K, 152, sg.PATH_CUDA_CORE)
    blocks = info["tiles_m"]
    # two CTAs per SM unless there are fewer rows; at most 256 rows per CTA
    assert blocks == max(min(N, 304), -(-N // 256))
    assert info["rows_per_cta"] == -(-N // blocks) <= 256
    k_slice = info["k_steps"]
    assert k_slice % 8 == 0 and info["split_k"] == -(-K // k_slice)
    assert info["grid"] == blocks * info["split_k"]
    if blocks >= 304:
        assert info["split_k"] == 1
    assert info["prefetch_steps"] == (1 if info["grid"] * 10 >= 7 * 304 else 0)
    # every row belongs to exactly one block: [b*N/blocks, (b+1)*N/blocks)
    bounds = [(b * N) // blocks for b in range(blocks + 1)]
    assert bounds[0] == 0 and bounds[-1] == N and all(x < y for x, y in zip(bounds, bounds[1:]))


def _header_define(name):
    with open(os.path.join(os.path.dirname(GOLDEN), "..", "include", "skinny_gemm.h")) as f:
        for line in f:
            if line.startswith(f"#define {name} "):
                return eval(line.split(None, 2)[2].replace("u", ""))  # "(1u << 20)" / "4096u"
    raise KeyError(name)


@pytest.mark.parametrize("sms", [152, 148, 160, 132])
def test_cuda_core_split_fits_the_noalloc_array(lib, sms):
    # gemv_bf16_noalloc keeps the CUDA-core kernel's split-K partials and counters
    # in a fixed array.  The planner splits K only when there are fewer than
    # 2 x SMs row blocks (N < 2 SMs), with at most ceil(2 SMs / N) slices, so the
    # partials stay below (2 SMs / N + 1) * 8 rows * N * 4 B < 128 * SMs bytes and
    # the counters at N < 2 SMs: far inside the array for any of these parts.
    part_bytes = _header_define("SG_NOALLOC_PARTIAL_BYTES")
    counters = _header_define("SG_NOALLOC_COUNTERS")
    assert part_bytes == 1 << 20 and counters == 4096
    worst = 0
    for M in range(1, 9):
        for N in list(range(1, 2 * sms + 2)) + [4096, 11008]:
            for K in (2048, 11008, 1 << 16, 1 << 22):
                info = sg.plan(M, N, K, sms, sg.PATH_CUDA_CORE)
                if info["split_k"] > 1:
                    assert N < 2 * sms
                    need = info["split_k"] * M * N * 4
                    worst = max(worst, need)
                    assert need < 128 * sms <= part_bytes, (M, N, K, info)
                    assert info["tiles_m"] <= counters, (M, N, K, info)
    assert worst > 0  # some plans do split


def test_plan_rejects_bad_arguments(lib):
    out = sg.PlanInfo()
    assert lib.sg_plan(-1, 8, 8, 152, 0, ctypes.byref(out)) == sg.SG_ERR_INVALID_ARG
    assert lib.sg_plan(8, 8, 8, 0, 0, ctypes.byref(out)) == sg.SG_ERR_INVALID_ARG
    assert lib.sg_plan(65, 8, 8, 152, sg.PATH_CUDA_CORE, ctypes.byref(out)) == sg.SG_ERR_INVALID_ARG


@pytest.mark.parametrize("M,N,K", [(4096, 11008, 4096), (2048, 4096, 4096), (128, 128, 64), (1000, 3000, 200),
                                   (16, 11008, 4096), (130, 257, 128)])
@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
def test_swiglu_plan_covers_every_unit_once(lib, M, N, K, path):
    info = sg.plan_swiglu(M, N, K, 152, path)
    tm = 256 if path == sg.PATH_GEMM_PAIR else 128
    assert info["path"] == path and info["tile_m"] == tm and info["tile_n"] == 128
    assert info["tiles_m"] == -(-M // tm) and info["tiles_n"] == -(-N // 128)
    items = _check_plan_coverage(info)
    # no CTA gets more Stream-K pieces than the fixup warps take
    assert max(sum(1 for it in row if it[4] > 1) for row in items) <= 4


def test_swiglu_path_choice(lib):
    assert sg.plan_swiglu(1, 11008, 4096, 152)["path"] == sg.PATH_CUDA_CORE
    assert sg.plan_swiglu(2, 11008, 4096, 152)["path"] == sg.PATH_CUDA_CORE
    info = sg.plan_swiglu(16, 11008, 4096, 152)
    assert info["path"] == sg.PATH_TENSOR_CORE and info["tile_m"] == 64 and info["tile_k"] == 64
    assert info["grid"] == 172 and info["split_k"] == 1
    assert sg.plan_swiglu(64, 4096, 11008, 152)["split_k"] == 4
    assert sg.plan_swiglu(65, 4096, 4096, 152)["path"] == sg.PATH_GEMM
    assert sg.plan_swiglu(256, 4096, 4096, 152)["path"] == sg.PATH_GEMM_PAIR
    out = sg.PlanInfo()
    assert lib.sg_plan_swiglu(65, 8, 8, 152, sg.PATH_TENSOR_CORE, ctypes.byref(out)) == sg.SG_ERR_INVALID_ARG
    assert lib.sg_plan_swiglu(8, 8, 8, 152, 7, ctypes.byref(out)) == sg.SG_ERR_INVALID_ARG


# ------------------------------------------------------------------ NVFP4
@pytest.mark.parametrize("args,code", [
    # (A, SFA, B, SFB, C, M, N, K, lda, ldb, ldc)
    ((16, 16, 16, 16, 16, 8, 8, 24, 16, 16, 8), sg.SG_ERR_INVALID_ARG),   # K % 16
    ((16, 16, 16, 16, 16, -1, 8, 32, 16, 16, 8), sg.SG_ERR_INVALID_ARG),  # negative M
    ((16, 16, 16, 16, 0, 8, 8, 32, 16, 16, 8), sg.SG_ERR_INVALID_ARG),    # null C
    ((16, 0, 16, 16, 16, 8, 8, 32, 16, 16, 8), sg.SG_ERR_INVALID_ARG),    # null SFA
    ((16, 16, 16, 16, 16, 8, 8, 64, 16, 32, 8), sg.SG_ERR_INVALID_ARG),   # lda < K/2
    ((16, 16, 16, 16, 16, 8, 16, 32, 16, 16, 8), sg.SG_ERR_INVALID_ARG),  # ldc < N
    ((24, 16, 16, 16, 16, 8, 8, 32, 16, 16, 8), sg.SG_ERR_MISALIGNED),    # A
    ((16, 20, 16, 16, 16, 8, 8, 32, 16, 16, 8), sg.SG_ERR_MISALIGNED),    # SFA
    ((16, 16, 16, 16, 16, 8, 8, 32, 24, 16, 8), sg.SG_ERR_MISALIGNED),    # lda % 16
    ((16, 16, 16, 16, 16, 8, 8, 32, 16, 16, 12), sg.SG_ERR_MISALIGNED),   # ldc % 8
])
def test_nvfp4_argument_errors_before_any_cuda_call(lib, args, code):
    assert lib.gemm_nvfp4(*args, 1.0, None) == code


def test_nvfp4_empty_is_noop(lib):
    assert lib.gemm_nvfp4(None, None, None, None, None, 0, 8, 32, 16, 16, 8, 1.0, None) == sg.SG_OK
    assert lib.gemm_nvfp4(None, None, None, None, None, 8, 0, 32, 16, 16, 8, 1.0, None) == sg.SG_OK
    assert lib.nvfp4_pack_scales(None, 0, 64, 4, None, None) == sg.SG_OK
    assert lib.nvfp4_pack_scales(None, 8, 24, 4, None, None) == sg.SG_ERR_INVALID_ARG  # K % 16
    assert lib.nvfp4_pack_scales(None, 8, 64, 3, None, None) == sg.SG_ERR_INVALID_ARG  # ld < K/16


def test_nvfp4_scale_bytes(lib):
    assert sg.nvfp4_scale_bytes(1, 16) == 512
    assert sg.nvfp4_scale_bytes(128, 64) == 512
    assert sg.nvfp4_scale_bytes(129, 64) == 1024
    assert sg.nvfp4_scale_bytes(4096, 4096) == 32 * 64 * 512
    assert sg.nvfp4_scale_bytes(300, 1040) == 3 * 17 * 512
    assert sg.nvfp4_scale_bytes(0, 64) == 0 and sg.nvfp4_scale_bytes(-1, 64) == -1


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 8192, 8192), (300, 500, 1040), (1, 1, 16),
                                   (128, 256, 256), (16384, 16384, 16384)])
@pytest.mark.parametrize("path", [sg.PATH_GEMM, sg.PATH_GEMM_PAIR])
def test_nvfp4_plan_covers_every_tile_once(lib, M, N, K, path):
    info = sg.plan_nvfp4(M, N, K, 152, path)
    pair = path == sg.PATH_GEMM_PAIR
    tm = 256 if pair else 128
    assert (info["tile_m"], info["tile_n"], info["tile_k"]) == (tm, 256, 256)
    assert info["cluster_size"] == (2 if pair else 1)
    assert info["tiles_m"] == -(-M // tm) and info["tiles_n"] == -(-N // 256) and info["k_steps"] == -(-K // 256)
    T = info["tiles_m"] * info["tiles_n"]
    units = 76 if pair else 152
    assert info["grid"] == min(T, units) and info["sk_tiles"] == 0 and info["dp_tiles"] == T
    items = _check_plan_coverage(info)
    assert all(k0 == 0 and k1 == info["k_steps"] for row in items for (_, k0, k1, *_) in row)


def test_nvfp4_auto_path_is_the_one_cta_kernel(lib):
    assert sg.plan_nvfp4(255, 4096, 4096, 152)["path"] == sg.PATH_GEMM
    assert sg.plan_nvfp4(8192, 8192, 8192, 152)["path"] == sg.PATH_GEMM
    assert sg.plan_nvfp4(8192, 64, 64, 152, sg.PATH_GEMM_PAIR)["path"] == sg.PATH_GEMM_PAIR
    with pytest.raises(sg.SgError):
        sg.plan_nvfp4(256, 256, 256, 152, sg.PATH_CUDA_CORE)
    assert lib.gemm_nvfp4_path(16, 16, 16, 16, 16, 8, 8, 32, 16, 16, 8, 1.0, sg.PATH_CUDA_CORE, None) == \
        sg.SG_ERR_INVALID_ARG


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("args,code", [
    # (Q, K, V, O, batch, seq_q, seq_k, heads, kv_heads, head_dim, ldq, ldk, ldv, ldo, causal, scale)
    ((16, 16, 16, 16, 1, 8, 8, 2, 2, 64, 128, 128, 128, 128, 1, 0.1), sg.SG_ERR_INVALID_ARG),   # head_dim != 128
    ((16, 16, 16, 16, 1, 8, 8, 3, 2, 128, 384, 256, 256, 384, 1, 0.1), sg.SG_ERR_INVALID_ARG),  # heads % kv_heads
    ((16, 16, 16, 16, -1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1), sg.SG_ERR_INVALID_ARG),  # negative batch
    ((16, 16, 16, 0, 1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1), sg.SG_ERR_INVALID_ARG),    # null O
    ((16, 0, 16, 16, 1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1), sg.SG_ERR_INVALID_ARG),    # null K
    ((16, 16, 16, 16, 1, 8, 8, 2, 2, 128, 255, 256, 256, 256, 1, 0.1), sg.SG_ERR_INVALID_ARG),  # short ldq
    ((16, 16, 16, 16, 1, 8, 8, 2, 1, 128, 256, 127, 128, 256, 1, 0.1), sg.SG_ERR_INVALID_ARG),  # short ldk
    ((16, 16, 16, 16, 1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, float("inf")), sg.SG_ERR_INVALID_ARG),
    ((24, 16, 16, 16, 1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1), sg.SG_ERR_MISALIGNED),   # Q
    ((16, 16, 16, 16, 1, 8, 8, 2, 2, 128, 260, 256, 256, 256, 1, 0.1), sg.SG_ERR_MISALIGNED),   # ldq % 8
    ((16, 16, 16, 16, 1, 8, 8, 2, 2, 128, 256, 256, 256, 260, 1, 0.1), sg.SG_ERR_MISALIGNED),   # ldo % 8
])
def test_attention_argument_errors_before_any_cuda_call(lib, args, code):
    assert lib.attention_bf16(*args[:14], args[14], args[15], None) == code


def test_attention_path_errors_before_any_cuda_call(lib):
    # (Q, K, V, O, batch, seq_q, seq_k, heads, kv_heads, head_dim, ldq, ldk, ldv, ldo, causal, scale, path)
    ok = (16, 16, 16, 16, 1, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1)
    for bad_path in (sg.PATH_GEMM, sg.PATH_GEMM_PAIR, 7, -1):
        assert lib.attention_bf16_path(*ok, bad_path, None) == sg.SG_ERR_INVALID_ARG
    # the decode kernel holds at most four query rows per kv head: 8 queries x 1 head
    assert lib.attention_bf16_path(*ok, sg.PATH_CUDA_CORE, None) == sg.SG_ERR_INVALID_ARG
    # 1 query x 8 heads per kv head (grouped): 8 rows
    grouped = (16, 16, 16, 16, 1, 1, 8, 8, 1, 128, 1024, 128, 128, 1024, 1, 0.1)
    assert lib.attention_bf16_path(*grouped, sg.PATH_CUDA_CORE, None) == sg.SG_ERR_INVALID_ARG


def test_attention_empty_is_noop(lib):
    # no batch, no queries or no heads: nothing to do, nothing dereferenced
    assert lib.attention_bf16(None, None, None, None, 0, 8, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1, None) == sg.SG_OK
    assert lib.attention_bf16(None, None, None, None, 1, 0, 8, 2, 2, 128, 256, 256, 256, 256, 1, 0.1, None) == sg.SG_OK
    assert lib.attention_bf16(None, None, None, None, 1, 8, 8, 0, 0, 128, 256, 256, 256, 256, 1, 0.1, None) == sg.SG_OK


class _Rows:
    """A stand-in for a [B, S, heads, 128] bf16 CUDA tensor: the binding's token
    pitch logic reads only its shape and strides."""

    def __init__(self, shape, strides):
        import torch
        self.shape, self._strides, self.dtype, self.is_cuda = shape, strides, torch.bfloat16, True

    def dim(self):
        return 4

    def stride(self, i):
        return self._strides[i]

    def data_ptr(self):
        return 0


def test_attention_token_pitch():
    H, D = 6, 128
    # one token per sequence: the rows are the batches, whatever the size-1 stride says
    assert sg._tokens_heads(_Rows((2, 1, H, D), (776, 768, 128, 1)), "Q") == (0, 776)
    assert sg._tokens_heads(_Rows((2, 5, H, D), (5 * 776, 776, 128, 1)), "Q") == (0, 776)
    assert sg._tokens_heads(_Rows((1, 1, H, D), (768, 768, 128, 1)), "Q") == (0, 768)
    with pytest.raises(ValueError):  # broadcast rows
        sg._tokens_heads(_Rows((1, 5, H, D), (0, 0, 128, 1)), "K")
    with pytest.raises(ValueError):  # batches that are not whole runs of rows
        sg._tokens_heads(_Rows((2, 5, H, D), (776, 776, 128, 1)), "K")
    with pytest.raises(ValueError):  # heads not dense
        sg._tokens_heads(_Rows((1, 5, H, D), (5 * 1024, 1024, 136, 1)), "V")
