"""bench.py host logic without a GPU: the printed formulas against the pages'
numbers, the max-over-ranks timing with two gloo ranks, and the reference arm's
rank handling."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_tflops_formula_matches_printed_table():
    # gemm3 benchmarks page, "Library comparison" + "Throughput and precision":
    # 2*M*N*K / (latency_us * 1e6) TFLOP/s; 4096^3 at 22.05 us and 8192^3 at 119.15 us.
    assert round(bench.tflops(4096, 4096, 4096, 22.05e-6)) == 6233
    assert round(bench.tflops(8192, 8192, 8192, 119.15e-6)) == 9228
    assert round(bench.tflops(16384, 16384, 16384, 960.30e-6)) == 9160


def test_decode_bytes():
    # a 4096 x 4096 bf16 weight is 32 MiB (spark-kernels, "1024 cubed and the decode shapes")
    assert bench.decode_bytes(1, 4096, 4096) - 2 * (4096 + 4096) == 32 * 2**20
    assert bench.decode_bytes(64, 11008, 4096) == 2 * (11008 * 4096 + 64 * 4096 + 64 * 11008)


def test_rotation_spans_four_l2():
    l2 = 129 * 2**20
    n = bench.rotation_count(64 * 2**20, l2)
    assert n * 64 * 2**20 >= 4 * l2


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist = bench.init_dist(world)
    bench.barrier(dist)
    q.put((rank, bench.max_over_ranks(dist, 10.0 + rank)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOPS" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_rows_only_rejects_unknown_workloads():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--rows-only", "no_such_workload"])
    with pytest.raises(SystemExit):
        bench.main(["--rows-only", "dec16_up", "--entry", "no_such_entry"])


def test_tensor_peak_follows_the_timed_region():
    import bench
    peaks = {"bf16_tflops": 1883.7, "bf16_tflops_sustained": 1707.5, "hbm_gbs": 6769.4}
    assert bench.tensor_peak(peaks, 10.0) == (1883.7, "bf16_tflops")
    assert bench.tensor_peak(peaks, 400.0) == (1707.5, "bf16_tflops_sustained")
    assert bench.tensor_peak({"bf16_tflops": 1.0, "bf16_tflops_sustained": None}, 400.0) == (1.0, "bf16_tflops")


def test_summary_fits_the_tail_of_the_line():
    # The bench line ends with a compact digest of every config (graph and
    # single-launch times, throughput, fraction of the roof, oracle seconds), so a
    # reader that keeps only the last ~1.5 KB of the line still has all of them.
    rows = []
    for n in bench.SUMMARY_WORKLOADS:
        r = {"workload": n, "entry": "gemm_bf16", "us": 12345.678, "single_us": 12399.1}
        if n.startswith("dec"):
            r.update(gbs=6123.456, frac_of_hbm=0.904567)
        else:
            r.update(tflops=1888.888, frac_of_peak=0.99999)
        rows.append(r)
    orows = [{"workload": n, "s": 1.0, "full_s_extrapolated": 123456.789} for n in bench.SUMMARY_WORKLOADS]
    s = bench.summary(rows, orows)
    assert all(n in s for n in bench.SUMMARY_WORKLOADS)
    text = json.dumps({"summary": s})
    assert len(text) < 1400, len(text)


def test_kernel_hash_ignores_comments_not_code():
    src = 'int a = 1; // note\n/* block */ asm("x // y"); char q = \'"\';\n'
    assert bench.strip_c_comments(src) == 'int a = 1; asm("x // y"); char q = \'"\';'
    assert bench.strip_c_comments(src.replace("// note", "// other words")) == bench.strip_c_comments(src)
    assert bench.strip_c_comments(src.replace("a = 1", "a = 2")) != bench.strip_c_comments(src)
