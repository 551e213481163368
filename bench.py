#!/usr/bin/env python3
"""Benchmark of the bf16 GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

One step is one gemm_bf16 call on the headline workload: C = A . B^T with
M = N = K = 4096, A and B uniform[-1, 1] rounded to bf16 from the seeded
generator (fp32 accumulation, bf16 output).  The timed region runs exactly K
steps back to back on one stream, inputs already resident in HBM; the inputs
rotate over enough copies (each at its own address) that the working set is
several times the L2, so no step reads its operands from L2 left by the one
before.  The JSON line (printed by rank 0) carries:

  value / ms_per_step  whole-job TFLOP/s (2*M*N*K per step, all ranks) over the
                       max-over-ranks time of the K steps
  roofline             the GEMM kernel's achieved TFLOP/s (CUDA-event time of
                       the K back-to-back launches / K) against the measured
                       bf16 peak
  e2e                  the same metric with host buffers: each step copies A and
                       B from pinned host memory, calls gemm_bf16 and copies C back;
                       consecutive steps overlap (uploads of A and B, GEMM and
                       download on four streams, two sets of device buffers)
  cpu_baseline         the fp64 oracle on a bounded row sample, on the host cores
  rows                 every bf16 config (512^3 ... 16384^3, the 7B MLP
                       projections, the decode shapes M = 1, 2, 16, 64 on every
                       skinny entry) and the fused, batched, NVFP4 and attention
                       workloads: per-launch graph-replay median over 8 rounds
                       of 50-launch graphs, arm order rotated and reversed
                       between rounds (cuBLAS through torch.matmul is an
                       arm, for context), single-launch median of 100, wave
                       efficiency of the plan
  microbench           the measured tcgen05 peak / copy / read roofs
  oracle_rows          the fp64 oracle's seconds per config (full up to the MLP
                       shapes; sampled 128 x 128 and extrapolated beyond)
  clocks               nvidia-smi SM clock samples taken during the timed region
  summary              (last, compact) per config: graph and single-launch us,
                       throughput, fraction of the measured roof; oracle seconds

--impl reference times the oracle itself (the reference arm): each step is the
fp64 oracle on a 64-row sample of the same 4096^3 workload, on the host cores.

With N > 1 (torchrun) every rank runs an independent replica on its own GPU:
the problem does not need to be sharded, and no data moves between ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOPS and % of measured tcgen05 peak; decode GB/s and % of HBM roof (1×GB300)"
HEADLINE = "sq4096"
REF_ROWS_PER_STEP = 64
CPU_SAMPLE_ROWS = 2048
PROFILES = os.path.join(ROOT, "profiles")


def tflops(M: int, N: int, K: int, seconds: float) -> float:
    """Dense throughput with the requested dims: 2*M*N*K / time (gemm3 benchmarks page,
    "Throughput and precision")."""
    return 2.0 * M * N * K / seconds / 1e12


def decode_bytes(M: int, N: int, K: int) -> int:
    """Bytes a skinny GEMM must move once: bf16 weights, activations and output."""
    return 2 * (N * K + M * K + M * N)


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    """Max of a float over all ranks (control plane only; gloo)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None, interval_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", str(interval_ms)]
        if device_id:
            self.cmd += ["-i", device_id]
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)  # let the first samples arrive
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self) -> dict:
        sms, maxes, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms), "power_w_max": max(power) if power else None}


def device_id_for_smi(torch, dev: int) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- helpers
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# A back-to-back run longer than this settles under the 1.4 kW power cap (the
# SM clock drops from 2070 MHz to ~1870 MHz within ~40 ms of dense GEMMs), so its
# tensor roof is the sustained cuBLAS figure; shorter runs use the burst figure.
SUSTAINED_AFTER_MS = 50.0
# Nominal dense tensor rates per GB300: FP4 13.5 PFLOP/s against bf16 2.25.
FP4_PER_BF16 = 6.0


def tensor_peak(peaks: dict, timed_ms: float):
    """The measured bf16 tensor roof that matches a timed region of timed_ms."""
    if timed_ms > SUSTAINED_AFTER_MS and peaks.get("bf16_tflops_sustained"):
        return peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"
    return peaks["bf16_tflops"], "bf16_tflops"


# The sources that define the headline GEMM kernel (its translation unit and the
# headers it includes); recorded DRAM traffic is valid while these are unchanged.
GEMM_KERNEL_SOURCES = ("sg_gemm_tcgen05.cu", "sg_internal.h", "sg_ptx.cuh", "sg_sched.cuh")


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments, whitespace runs collapsed (string and
    character literals kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the GEMM kernel's sources, comments and layout aside: a recorded
    traffic figure stays valid across comment edits, not across code changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_gemv_gb300", "csrc")
    for name in GEMM_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{workload}")
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def host_bits_to_device(torch, bits, device):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def copies(t, n: int):
    return [t] + [t.clone() for _ in range(n - 1)]


def rotation_count(bytes_per_set: int, l2: int) -> int:
    """Input sets needed so that the rotation spans at least four L2 capacities."""
    return max(2, math.ceil(4 * l2 / max(bytes_per_set, 1)) + 1)


def build_graphs(torch, stream, fns, steps: int, graph_chunk: int = 500, offset: int = 0):
    """Captures fns[(offset + i) % len(fns)] for i < steps into CUDA graphs of at
    most graph_chunk launches each (one launch per step)."""
    graphs = []
    for c0 in range(0, steps, graph_chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(c0, min(steps, c0 + graph_chunk)):
                fns[(offset + i) % len(fns)]()
        graphs.append(g)
    stream.synchronize()
    return graphs


def time_launches(torch, stream, fns, steps: int, warmup: int, graph_chunk: int = 500):
    """Runs fns[i % len(fns)] `warmup` times eagerly, then captures the `steps`
    timed calls into CUDA graphs (at most graph_chunk launches each) and replays
    them back to back on `stream`, bracketed by CUDA events on that stream.
    Graph replay keeps host launch overhead out of the device timeline, so
    short kernels are timed as they run back to back.  Returns total ms."""
    for i in range(warmup):
        fns[i % len(fns)]()
    stream.synchronize()
    graphs = build_graphs(torch, stream, fns, steps, graph_chunk, offset=warmup)
    # The first replay of a new graph also uploads it to the device; replay each
    # once untimed so the timed replay measures the launches alone.
    replay_ms(torch, stream, graphs)
    return replay_ms(torch, stream, graphs)


def replay_ms(torch, stream, graphs) -> float:
    """Replays the graphs back to back on `stream` (CUDAGraph.replay launches on
    the current stream, so `stream` is made current) and returns the CUDA-event
    time on that stream, in ms."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for g in graphs:
            g.replay()
        t1.record(stream)
    t1.synchronize()
    return t0.elapsed_time(t1)


# ---------------------------------------------------------------- the reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import synthetic as syn
    import oracle
    w = syn.WORKLOADS[HEADLINE]
    A = w.a()
    B = w.b()
    threads = oracle.default_threads()
    rows_per = REF_ROWS_PER_STEP
    used = threads

    def step(i):
        nonlocal used
        r0 = (i * rows_per) % w.M
        _, used = oracle.gemm(A[r0:r0 + rows_per], B, threads=threads, return_threads=True)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t
    value = tflops(rows_per, w.N, w.K, dt / args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded uniform[-1,1] -> bf16)",
        "config": {"workload": f"{HEADLINE}: bf16 GEMM C[4096,4096] = A[4096,4096] . B[4096,4096]^T",
                   "sample": f"{rows_per} rows of C per step (all 4096 columns, full K)"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": used, "kind": "oracle",
                         "sample": f"{rows_per} x 4096 outputs of the 4096^3 GEMM per step, fp64"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import skinny_gemv_gb300 as sg
    import synthetic as syn

    dist = init_dist(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    sg.load()
    info = sg.device_query()
    l2 = info["l2_bytes"]
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device)
    w = syn.WORKLOADS[HEADLINE]
    M, N, K = w.M, w.N, w.K

    with torch.cuda.stream(stream):
        A0 = host_bits_to_device(torch, w.a(), device)
        B0 = host_bits_to_device(torch, w.b(), device)
        nrot = rotation_count(A0.numel() * 2 + B0.numel() * 2, l2)
        As, Bs = copies(A0, nrot), copies(B0, nrot)
        Cs = [torch.empty((M, N), dtype=torch.bfloat16, device=device) for _ in range(nrot)]
    stream.synchronize()
    fns = [(lambda a=a, b=b, c=c: sg.gemm_bf16(a, b, c, stream=stream)) for a, b, c in zip(As, Bs, Cs)]

    check = None
    if not args.no_check:
        check = sanity_gate(torch, sg, w, As[0], Bs[0], Cs[0], stream)

    sampler = ClockSampler(device_id_for_smi(torch, local))
    barrier(dist)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        fns[i % nrot]()
    torch.cuda.synchronize()
    barrier(dist)
    graphs = build_graphs(torch, stream, fns, args.steps)
    # One untimed replay first: the first replay of a new graph also uploads it,
    # and once took 0.8 s for 30 launches on an otherwise idle GPU.
    replay_ms(torch, stream, graphs)
    with sampler:
        torch.cuda.synchronize()
        total_ms = replay_ms(torch, stream, graphs)
        torch.cuda.synchronize()
    barrier(dist)
    st, detail = sg.check_device_errors(stream)
    if st != sg.SG_OK:
        raise RuntimeError(f"device error {st} {detail}")

    local_ms = total_ms
    total_ms = max_over_ranks(dist, total_ms)
    value = tflops(M, N, K, total_ms / 1e3 / args.steps) * world
    kernel_ms = local_ms / args.steps  # mean launch duration, back to back
    achieved = tflops(M, N, K, kernel_ms / 1e3)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(torch, sg, w, A0, B0, stream, args, dist, world)

    rows = []
    micro = {}
    cpu = None
    oracle_rows = []
    if rank == 0 and not args.quick:
        rows = measure_rows(torch, sg, syn, stream, l2, peaks, args)
        micro = measure_micro(torch, sg, stream)
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(syn, w)
        if not args.quick:
            oracle_rows = oracle_table(syn)

    if rank != 0:
        return 0
    plan = sg.plan(M, N, K, info["sm_count"], 0)
    peak, peak_key = tensor_peak(peaks, total_ms)
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 uniform[-1,1] rounded to bf16)",
        "config": {
            "workload": f"{HEADLINE}: bf16 GEMM C[4096,4096] = A[4096,4096] . B[4096,4096]^T, fp32 accumulate, bf16 out",
            "M": M, "N": N, "K": K, "accumulate": "f32",
            "l2": f"inputs larger than L2: {nrot} rotating copies of A, B, C "
                  f"({nrot * 3 * M * K * 2 / 2**20:.0f} MiB vs {l2 / 2**20:.0f} MiB L2), no flush",
            "tile": f"{plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']}",
            "ctas": plan["grid"] * plan["cluster_size"], "cluster": plan["cluster_size"],
            "dp_tiles": plan["dp_tiles"], "sk_tiles": plan["sk_tiles"],
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        },
        "roofline": {
            "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "suspect": achieved > 1.15 * max(peak, micro.get("tcgen05_peak_tflops", 0) if micro else 0),
            "traffic": recorded_traffic("tc_gemm_kernel", HEADLINE),
            "kernel": ("tc_gemm_kernel<256,6,pair>" if plan["path"] == sg.PATH_GEMM_PAIR
                       else "tc_gemm_kernel<256,4,single>"), "kernel_ms": kernel_ms,
            "peak_source": (f"MEASURED_PEAKS.json {peak_key} ({peaks['source']}; cuBLAS 8192^3, "
                            f"{'back to back for 4 s under the power cap' if peak_key.endswith('sustained') else 'burst'}"
                            f"): the timed region ran {total_ms:.0f} ms of back-to-back launches"),
            "frac_of_burst": achieved / peaks["bf16_tflops"],
            "algorithmic": f"2*M*N*K = {2 * M * N * K / 1e9:.1f} GFLOP per launch",
        },
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": args.steps,
        "correctness": check,
        "rows": rows,
        "microbench": micro,
        "oracle_rows": oracle_rows,
    }
    if micro:
        # against the card's own tcgen05 loop (the metric's "measured tcgen05 peak"),
        # with the clock each was measured at
        line["roofline"]["frac_of_tcgen05_loop"] = achieved / micro["tcgen05_peak_tflops"]
        line["roofline"]["tcgen05_loop"] = {"tflops": micro["tcgen05_peak_tflops"],
                                            "sm_mhz": micro["tcgen05_peak_sm_mhz"],
                                            "timed_region_sm_mhz": clocks.get("sm_mhz")}
    if rows:
        line["summary"] = summary(rows, oracle_rows)
    print(json.dumps(line), flush=True)
    return 0


def sanity_gate(torch, sg, w, A, B, C, stream):
    """Guards the timing against a broken build: 256 sampled rows of the headline
    output must agree with an fp32 matmul of the same rows on the device, within
    the parity tests' tolerance.  (Parity proper is the test suite's job.)"""
    sg.gemm_bf16(A, B, C, stream=stream)
    stream.synchronize()
    g = torch.Generator(device="cpu")
    g.manual_seed(1)
    rows = torch.randperm(w.M, generator=g)[:256].to(A.device)
    ref = (A[rows].float() @ B.float().t()).double()
    got = C[rows].double()
    diff = (got - ref).abs()
    bound = 1e-2 * ref.abs() + 2e-3 * math.sqrt(w.K)
    n_over = int((diff > bound).sum().item())
    rel_fro = float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref))
    if n_over or rel_fro > 4e-3 or not torch.isfinite(got).all():
        raise RuntimeError(f"headline output fails the sanity gate: n_over={n_over} rel_fro={rel_fro}")
    return {"vs": "device fp32 matmul, 256 sampled rows", "max_abs": float(diff.max().item()),
            "rel_fro": rel_fro, "n_over": n_over}


def measure_e2e(torch, sg, w, A0, B0, stream, args, dist, world):
    """Host buffers in, host buffer out: every step copies A and B from pinned
    memory to the device, runs gemm_bf16 and copies C back into pinned memory.
    Steps are pipelined as a serving loop would run them: step i's uploads (A and
    B on two streams), its GEMM (the bench stream) and its download (a fourth
    stream) each
    wait only for what they need, over two sets of device buffers, so step i + 1's
    uploads overlap step i's GEMM and download.  The timed region runs from before
    the first upload to after the last download."""
    M, N, K = w.M, w.N, w.K
    hA = A0.cpu().pin_memory()
    hB = B0.cpu().pin_memory()
    hC = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dA = [torch.empty_like(A0) for _ in range(2)]
    dB = [torch.empty_like(B0) for _ in range(2)]
    dC = [torch.empty((M, N), dtype=torch.bfloat16, device=A0.device) for _ in range(2)]
    up = torch.cuda.Stream(A0.device)
    up2 = torch.cuda.Stream(A0.device)  # A and B upload side by side (two copy engines)
    down = torch.cuda.Stream(A0.device)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("up", "up2", "gemm", "down")}
    used = [False, False]

    def step(i):
        b = i % 2
        if used[b]:  # buffer set b: its previous GEMM read dA/dB, its previous download read dC
            up.wait_event(ev["gemm"][b])
            up2.wait_event(ev["gemm"][b])
        with torch.cuda.stream(up):
            dA[b].copy_(hA, non_blocking=True)
        with torch.cuda.stream(up2):
            dB[b].copy_(hB, non_blocking=True)
        ev["up"][b].record(up)
        ev["up2"][b].record(up2)
        stream.wait_event(ev["up"][b])
        stream.wait_event(ev["up2"][b])
        if used[b]:
            stream.wait_event(ev["down"][b])
        sg.gemm_bf16(dA[b], dB[b], dC[b], stream=stream)
        ev["gemm"][b].record(stream)
        down.wait_event(ev["gemm"][b])
        with torch.cuda.stream(down):
            hC[b].copy_(dC[b], non_blocking=True)
        ev["down"][b].record(down)
        used[b] = True

    steps = max(3, min(args.steps, 50))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    barrier(dist)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    up.wait_event(t0)
    up2.wait_event(t0)
    down.wait_event(t0)
    for i in range(steps):
        step(3 + i)
    stream.wait_event(ev["down"][(3 + steps - 1) % 2])
    t1.record(stream)
    t1.synchronize()
    ms = max_over_ranks(dist, t0.elapsed_time(t1)) / steps
    return {"value": tflops(M, N, K, ms / 1e3) * world, "unit": "TFLOPS", "ms_per_step": ms,
            "steps": steps, "h2d_bytes_per_step": 2 * (M * K + N * K), "d2h_bytes_per_step": 2 * M * N,
            "pipelined": "uploads (A, B), GEMM and download of consecutive steps overlap on four streams"}


ENTRIES = {"auto": None, "cuda_core": 1, "tensor_core": 2}

# Rows' timing protocol (gemm3 benchmarks page, "Methodology"; spark-kernels, "how
# things are measured"): every arm of a workload (our entries, and cuBLAS through
# torch.matmul for context) is captured as one CUDA graph of ROUND_LAUNCHES
# launches over the rotating inputs (the page's 50 timed replays per round);
# ROUNDS rounds replay the arms in an order rotated, and reversed every other
# round, and each arm's per-launch time is the median over the rounds.  Beside it,
# SINGLE_LAUNCHES launches are timed one by one (events around each) and their
# median is the single-launch time, which includes the launch gap.
ROUNDS = 8
ROUND_LAUNCHES = 50
SINGLE_LAUNCHES = 100
COOL_DOWN_S = 1.0  # idle before each compute-bound row


def time_arms(torch, stream, arms, warmup: int = 5, rounds: int = ROUNDS, per_round: int = ROUND_LAUNCHES,
              singles: int = SINGLE_LAUNCHES):
    """arms: list of (label, fns), each fns a list of zero-argument launches on
    `stream` (called in rotation).  Returns {label: {"graph_us", "single_us",
    "graph_ms_total"}}: the median per-launch time of graph replay over `rounds`
    rounds in rotated arm order, and the median of `singles` one-launch event
    timings."""
    graphs = {}
    for label, fns in arms:
        for i in range(warmup):
            fns[i % len(fns)]()
        stream.synchronize()
        graphs[label] = build_graphs(torch, stream, fns, per_round, offset=warmup)
        replay_ms(torch, stream, graphs[label])  # uploads the graph
    per = {label: [] for label, _ in arms}
    labels = [label for label, _ in arms]
    for r in range(rounds):
        k = r % len(labels)
        order = labels[k:] + labels[:k]
        if r % 2:
            order.reverse()
        for label in order:
            per[label].append(replay_ms(torch, stream, graphs[label]) / per_round)
    out = {}
    for label, fns in arms:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(singles)]
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(ev):
                e0.record(stream)
                fns[i % len(fns)]()
                e1.record(stream)
        stream.synchronize()
        single = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        out[label] = {"graph_us": statistics.median(per[label]) * 1e3, "single_us": single * 1e3,
                      "graph_ms_total": sum(per[label]) * per_round}
    del graphs
    return out


def _tensor_row(row, flops, t, peaks):
    row["tflops"] = flops / (row["us"] / 1e6) / 1e12
    rpeak, rkey = tensor_peak(peaks, t["graph_ms_total"])
    row["frac_of_peak"] = row["tflops"] / rpeak
    row["peak"] = rkey


def _hbm_row(row, byts, peaks):
    row["gbs"] = byts / (row["us"] / 1e6) / 1e9
    row["frac_of_hbm"] = row["gbs"] / peaks["hbm_gbs"]


def measure_rows(torch, sg, syn, stream, l2, peaks, args, names=None, entries=None):
    """Other workloads of the pages, timed with the rows' protocol (inputs rotated
    past L2).  Inputs are drawn on the device from seeded generators with the
    workloads' distributions; the parity tests check these shapes on the host
    generator's inputs.  `names` limits the workloads and `entries` the skinny
    entries (auto, cuda_core, tensor_core) that are timed."""
    out = []
    gen = torch.Generator(device=stream.device)
    rounds = 3 if args.quick else ROUNDS
    singles = 20 if args.quick else SINGLE_LAUNCHES
    sms = sg.device_query()["sm_count"]

    def draw(rows, cols, dist, seed):
        gen.manual_seed(seed)
        if dist == "uniform":
            t = torch.rand((rows, cols), generator=gen, device=stream.device, dtype=torch.float32) * 2 - 1
        else:
            sigma = float(dist.split(":")[1])
            t = torch.randn((rows, cols), generator=gen, device=stream.device, dtype=torch.float32) * sigma
        return t.to(torch.bfloat16)

    def timed(arms):
        return time_arms(torch, stream, arms, rounds=rounds, singles=singles)

    quick_rows = args.quick
    decode = []
    if names is None:
        # Every memory-bound row (decode, fused decode, batched, decode
        # attention) runs before the compute-bound ones: right after seconds of
        # power-capped GEMMs the memory-bound rows measured up to 2 us slower per
        # launch (the same residual decode row: 18.8 us after the GEMM rows,
        # 16.6 us timed alone, against 16.5 us for the plain row).
        decode = [n for n in syn.WORKLOADS if n.startswith("dec")]
        decode += [n for n in syn.GATED_WORKLOADS if syn.GATED_WORKLOADS[n].base.M <= 64]
        decode += [n for n in syn.RESIDUAL_WORKLOADS if syn.RESIDUAL_WORKLOADS[n].base.M <= 64]
        decode += list(syn.BATCHED_WORKLOADS) + ["attn_decode_4096"]
        names = decode + ["sq512", "sq2048", "sq4096", "mlp_up", "mlp_down", "sq8192", "sq16384"]
        names += [n for n in syn.GATED_WORKLOADS if n not in decode]
        names += [n for n in syn.RESIDUAL_WORKLOADS if n not in decode]
        names += ["fp4_sq4096", "fp4_sq8192", "fp4_sq16384"]
        names += ["attn_causal_4096", "attn_4096"]

    def row_gemm(name):
        w = syn.WORKLOADS[name]
        with torch.cuda.stream(stream):
            A = draw(w.M, w.K, w.dist_a, w.seed_a)
            B = draw(w.N, w.K, w.dist_b, w.seed_b)
            per_set = 2 * (w.M * w.K + w.N * w.K)
            nrot = rotation_count(per_set, l2)
            As = copies(A, nrot) if w.M > 64 else [A] * nrot
            Bs = copies(B, nrot)
            C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=stream.device)
            Cb = torch.empty_like(C)
        stream.synchronize()
        paths = [("gemm_bf16", None)]
        if w.M <= 64:
            paths = [("gemm_bf16", None), ("gemv_bf16/cuda_core", sg.PATH_CUDA_CORE),
                     ("gemv_bf16/tensor_core", sg.PATH_TENSOR_CORE)]
        if entries is not None:
            keep = {ENTRIES[e] for e in entries}
            paths = [(label, path) for label, path in paths if path in keep]
        arms = []
        for label, path in paths:
            if path is None:
                fns = [(lambda a=a, b=b: sg.gemm_bf16(a, b, C, stream=stream)) for a, b in zip(As, Bs)]
            else:
                fns = [(lambda a=a, b=b, p=path: sg.gemv_bf16(a, b, C, stream=stream, path=p))
                       for a, b in zip(As, Bs)]
            arms.append((label, fns))
        if entries is None:  # cuBLAS (torch.matmul) on the same inputs, for context only
            def mm(a, b):
                with torch.cuda.stream(stream):
                    torch.matmul(a, b.t(), out=Cb)
            arms.append(("cublas", [(lambda a=a, b=b: mm(a, b)) for a, b in zip(As, Bs)]))
        t = timed(arms)
        plan = sg.plan(w.M, w.N, w.K, sms, 0)
        for label, path in paths:
            row = {"workload": name, "entry": label, "M": w.M, "N": w.N, "K": w.K, "us": t[label]["graph_us"],
                   "single_us": t[label]["single_us"]}
            if label == "gemm_bf16":
                row["wave_efficiency"] = plan["wave_efficiency"]
                if "cublas" in t:
                    row["cublas_us"] = t["cublas"]["graph_us"]
            if w.M > 64:
                _tensor_row(row, w.flops, t[label], peaks)
            else:
                _hbm_row(row, w.decode_bytes, peaks)
            out.append(row)
        del As, Bs, A, B, C, Cb
        torch.cuda.empty_cache()
    def row_gated(name):
        g = syn.GATED_WORKLOADS[name]
        w = g.base
        with torch.cuda.stream(stream):
            A = draw(w.M, w.K, w.dist_a, w.seed_a)
            Wg = draw(w.N, w.K, w.dist_b, w.seed_b)
            Wu = draw(w.N, w.K, w.dist_b, w.seed_b + 1000)
            nrot = rotation_count(2 * (w.M * w.K + 2 * w.N * w.K), l2)
            As = copies(A, nrot) if w.M > 64 else [A] * nrot
            Gs, Us = copies(Wg, nrot), copies(Wu, nrot)
            C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=stream.device)
        stream.synchronize()
        fns = [(lambda a=a, wg=wg, wu=wu: sg.gemm_bf16_swiglu(a, wg, wu, C, stream=stream))
               for a, wg, wu in zip(As, Gs, Us)]
        t = timed([("gemm_bf16_swiglu", fns)])["gemm_bf16_swiglu"]
        row = {"workload": name, "entry": "gemm_bf16_swiglu", "M": w.M, "N": w.N, "K": w.K, "us": t["graph_us"],
               "single_us": t["single_us"]}
        if w.M > 64:
            _tensor_row(row, g.flops, t, peaks)
        else:
            _hbm_row(row, g.decode_bytes, peaks)
        out.append(row)
        del As, Gs, Us, A, Wg, Wu, C
        torch.cuda.empty_cache()
    def row_resid(name):
        rw = syn.RESIDUAL_WORKLOADS[name]
        w = rw.base
        with torch.cuda.stream(stream):
            A = draw(w.M, w.K, w.dist_a, w.seed_a)
            B = draw(w.N, w.K, w.dist_b, w.seed_b)
            R = draw(w.M, w.N, "normal:1", w.seed_a + 2000)
            nrot = rotation_count(2 * (w.M * w.K + w.N * w.K + 2 * w.M * w.N), l2)
            As = copies(A, nrot) if w.M > 64 else [A] * nrot
            Bs, Rs = copies(B, nrot), copies(R, nrot)
            C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=stream.device)
        stream.synchronize()
        fns = [(lambda a=a, b=b, r=r: sg.gemm_bf16_residual(a, b, r, C, stream=stream)) for a, b, r in zip(As, Bs, Rs)]
        t = timed([("gemm_bf16_residual", fns)])["gemm_bf16_residual"]
        row = {"workload": name, "entry": "gemm_bf16_residual", "M": w.M, "N": w.N, "K": w.K, "us": t["graph_us"],
               "single_us": t["single_us"]}
        if w.M > 64:
            _tensor_row(row, rw.flops, t, peaks)
        else:
            _hbm_row(row, rw.decode_bytes, peaks)
        out.append(row)
        del As, Bs, Rs, A, B, R, C
        torch.cuda.empty_cache()
    def row_batched(name):
        bw = syn.BATCHED_WORKLOADS[name]
        with torch.cuda.stream(stream):
            A = draw(bw.M, bw.K, "normal:1", 4000 + bw.cfg)
            Ws = [draw(n, bw.K, "normal:0.02", 4100 + bw.cfg + i) for i, n in enumerate(bw.Ns)]
            nrot = rotation_count(2 * sum(bw.Ns) * bw.K, l2)
            sets = [Ws] + [[w.clone() for w in Ws] for _ in range(nrot - 1)]
            Cs = [torch.empty((bw.M, n), dtype=torch.bfloat16, device=stream.device) for n in bw.Ns]
        stream.synchronize()
        fns = [(lambda ws=ws: sg.gemv_bf16_batched(A, ws, Cs, stream=stream)) for ws in sets]
        t = timed([("gemv_bf16_batched", fns)])["gemv_bf16_batched"]
        row = {"workload": name, "entry": "gemv_bf16_batched", "M": bw.M, "N": list(bw.Ns), "K": bw.K,
               "us": t["graph_us"], "single_us": t["single_us"]}
        _hbm_row(row, bw.decode_bytes, peaks)
        out.append(row)
        del sets, Ws, A, Cs
        torch.cuda.empty_cache()
    def row_fp4(name):
        fw = syn.NVFP4_WORKLOADS[name]
        with torch.cuda.stream(stream):
            gen.manual_seed(5000 + fw.cfg)
            dev = stream.device

            def codes(rows, cols):
                return torch.randint(0, 256, (rows, cols), generator=gen, device=dev, dtype=torch.uint8)

            def scales(rows):
                plain = torch.randint(syn.NVFP4_SCALE_LO, syn.NVFP4_SCALE_HI + 1, (rows, fw.K // 16), generator=gen,
                                      device=dev, dtype=torch.uint8)
                return sg.nvfp4_pack_scales(plain, fw.K, stream=stream)

            per_set = (fw.M + fw.N) * fw.K // 2
            nrot = rotation_count(per_set, l2)
            sets = [(codes(fw.M, fw.K // 2), scales(fw.M), codes(fw.N, fw.K // 2), scales(fw.N)) for _ in range(nrot)]
            C = torch.empty((fw.M, fw.N), dtype=torch.float16, device=dev)
        stream.synchronize()
        fns = [(lambda a=a, sa=sa, b=b, sb=sb: sg.gemm_nvfp4(a, sa, b, sb, K=fw.K, C=C, alpha=fw.alpha, stream=stream))
               for a, sa, b, sb in sets]
        t = timed([("gemm_nvfp4", fns)])["gemm_nvfp4"]
        row = {"workload": name, "entry": "gemm_nvfp4", "M": fw.M, "N": fw.N, "K": fw.K, "us": t["graph_us"],
               "single_us": t["single_us"], "tflops": fw.flops / (t["graph_us"] / 1e6) / 1e12}
        rpeak, rkey = tensor_peak(peaks, t["graph_ms_total"])
        # FP4 roof: the measured bf16 roof times the nominal dense FP4 / bf16 ratio (13.5 / 2.25)
        row["frac_of_peak"] = row["tflops"] / (FP4_PER_BF16 * rpeak)
        row["peak"] = f"{FP4_PER_BF16:g} x {rkey}"
        out.append(row)
        del sets, C
        torch.cuda.empty_cache()
    def row_attn(name):
        aw = syn.ATTENTION_WORKLOADS[name]
        with torch.cuda.stream(stream):
            gen.manual_seed(6000 + aw.cfg)
            dev = stream.device

            def act(S, heads):
                return torch.randn((aw.B, S, heads, aw.D), generator=gen, device=dev).to(torch.bfloat16)

            per_set = 2 * aw.D * aw.B * (2 * aw.Sq * aw.H + 2 * aw.Sk * aw.Hkv)
            nrot = rotation_count(per_set, l2)
            sets = [(act(aw.Sq, aw.H), act(aw.Sk, aw.Hkv), act(aw.Sk, aw.Hkv), act(aw.Sq, aw.H)) for _ in range(nrot)]
        stream.synchronize()
        fns = [(lambda q=q, k=k, v=v, o=o: sg.attention_bf16(q, k, v, O=o, causal=aw.causal, stream=stream))
               for q, k, v, o in sets]
        t = timed([("attention_bf16", fns)])["attention_bf16"]
        row = {"workload": name, "entry": "attention_bf16", "B": aw.B, "Sq": aw.Sq, "Sk": aw.Sk, "H": aw.H,
               "Hkv": aw.Hkv, "D": aw.D, "causal": aw.causal, "us": t["graph_us"], "single_us": t["single_us"]}
        if aw.Sq >= 128:  # prefill: tensor-bound, FLOPs over the visible pairs
            _tensor_row(row, aw.flops, t, peaks)
        else:  # decode: K and V streamed once
            _hbm_row(row, aw.kv_bytes + 2 * 2 * aw.B * aw.Sq * aw.H * aw.D, peaks)
        # torch's own scaled_dot_product_attention on the same inputs, for context
        q0, k0, v0, _ = sets[0]
        tq, tk, tv = (t_.transpose(1, 2) for t_ in (q0, k0, v0))
        sdpa_causal = aw.causal and aw.Sq == aw.Sk
        if aw.causal and aw.Sq != aw.Sk and aw.Sq != 1:
            sdpa_causal = None  # bottom-right causal has no plain sdpa flag
        if sdpa_causal is not None:
            try:
                with torch.cuda.stream(stream):
                    tfn = [lambda: torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=sdpa_causal)]
                    row["torch_sdpa_us"] = time_launches(torch, stream, tfn, min(ROUND_LAUNCHES * rounds, 50), 3) \
                        / min(ROUND_LAUNCHES * rounds, 50) * 1e3
            except RuntimeError as e:  # a comparison only: never fail the bench on it
                row["torch_sdpa_us"] = None
                row["torch_sdpa_error"] = str(e).splitlines()[0][:120]
        out.append(row)
        del sets
        torch.cuda.empty_cache()

    kinds = [(syn.WORKLOADS, row_gemm), (syn.GATED_WORKLOADS, row_gated), (syn.RESIDUAL_WORKLOADS, row_resid),
             (syn.BATCHED_WORKLOADS, row_batched), (syn.NVFP4_WORKLOADS, row_fp4), (syn.ATTENTION_WORKLOADS, row_attn)]
    decode_like = set(decode)
    for name in names:
        if name not in decode_like and not quick_rows:
            # A compute-bound row after seconds of power-capped GEMMs starts with
            # the clock pulled down; one second idle lets every row start from
            # the same state (its own rounds then run at whatever clock its load
            # settles to, as a burst).
            stream.synchronize()
            time.sleep(COOL_DOWN_S)
        for table, fn in kinds:
            if name in table:
                fn(name)
                break
    return out


def measure_micro(torch, sg, stream):
    tf, mhz = sg.bench_tcgen05_peak(4_000_000, stream=stream)
    n = 1 << 31
    src = torch.ones(n, dtype=torch.uint8, device=stream.device)
    dst = torch.empty_like(src)
    sink = torch.zeros(4, dtype=torch.int32, device=stream.device)
    copy = sg.bench_copy(dst, src, reps=10, stream=stream)
    read = sg.bench_read(src, sink, reps=10, stream=stream)
    del src, dst
    torch.cuda.empty_cache()
    return {"tcgen05_peak_tflops": tf, "tcgen05_peak_sm_mhz": mhz, "copy_gbs": copy, "read_gbs": read}


def oracle_table(syn):
    """The fp64 oracle timed on every bf16 GEMM config, on the host cores: the
    full oracle up to the MLP shapes and for decode, the sampled oracle (the
    128 x 128 row/column intersections the parity tests check) at 8192^3 and
    16384^3, with the full oracle's time extrapolated from it (its cost is
    proportional to the outputs it computes)."""
    import numpy as np

    import oracle
    out = []
    decode_b = {}
    for name, w in syn.WORKLOADS.items():
        if w.oracle == "full":
            A = w.a()
            if name.startswith("dec"):
                # the four decode rows of a shape share one draw of its weights:
                # the oracle's time does not depend on the values
                key = (w.N, w.K)
                if key not in decode_b:
                    decode_b[key] = w.b()
                B = decode_b[key]
            else:
                B = w.b()
            t = time.perf_counter()
            _, used = oracle.gemm(A, B, return_threads=True)
            dt = time.perf_counter() - t
            out.append({"workload": name, "mode": "full", "s": dt, "gflops": w.flops / dt / 1e9, "cores": used})
        else:
            rows = syn.sample_indices(w.M, 128, 1)
            cols = syn.sample_indices(w.N, 128, 2)
            A = syn.matrix_rows(rows, w.K, w.dist_a, w.seed_a)
            B = syn.matrix_rows(cols, w.K, w.dist_b, w.seed_b)
            t = time.perf_counter()
            _, used = oracle.gemm_sampled(A, B, np.arange(128), np.arange(128), return_threads=True)
            dt = time.perf_counter() - t
            flops = 2 * 128 * 128 * w.K
            out.append({"workload": name, "mode": "sampled 128x128", "s": dt, "gflops": flops / dt / 1e9,
                        "cores": used, "full_s_extrapolated": dt * (w.M * w.N) / (128 * 128)})
        del A, B
    return out


SUMMARY_WORKLOADS = ("sq512", "sq2048", "sq4096", "mlp_up", "mlp_down", "sq8192", "sq16384",
                     "dec1_up", "dec2_up", "dec16_up", "dec64_up", "dec1_down", "dec2_down", "dec16_down", "dec64_down")


def summary(rows, oracle_rows):
    """A compact digest of the configs, printed last in the line: per config the
    graph-replay and single-launch microseconds, the throughput and its fraction
    of the measured roof, and the oracle's seconds."""
    out = {"cols": "us graph, us single, TFLOP/s or GB/s, frac of measured roof"}
    by = {(r["workload"], r["entry"]): r for r in rows}
    for name in SUMMARY_WORKLOADS:
        r = by.get((name, "gemm_bf16"))
        if r is None:
            continue
        thr = r.get("tflops", r.get("gbs"))
        frac = r.get("frac_of_peak", r.get("frac_of_hbm"))
        out[name] = [round(r["us"], 2), round(r.get("single_us", float("nan")), 2), round(thr, 1 if thr > 100 else 2),
                     round(frac, 3)]
    if oracle_rows:
        out["oracle_s"] = {o["workload"]: round(o.get("full_s_extrapolated", o["s"]), 3) for o in oracle_rows}
    return out


def cpu_baseline(syn, w):
    import oracle
    A = w.a()[:CPU_SAMPLE_ROWS]
    B = w.b()
    t = time.perf_counter()
    _, used = oracle.gemm(A, B, return_threads=True)
    dt = time.perf_counter() - t
    return {"value": tflops(CPU_SAMPLE_ROWS, w.N, w.K, dt), "unit": "TFLOPS", "cores": used, "kind": "oracle",
            "sample": f"first {CPU_SAMPLE_ROWS} of 4096 rows of the 4096^3 GEMM (fp64), {dt:.1f} s"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only: skip the extra rows and microbenchmarks")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--rows-only", metavar="WORKLOADS",
                    help="time only these comma-separated workloads (e.g. dec16_up) as rows and print them; "
                         "no headline (for profiling one kernel)")
    ap.add_argument("--entry", choices=sorted(ENTRIES), action="append",
                    help="with --rows-only: the entries to time (default: all)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.rows_only:
        return run_rows_only(args, local)
    return run_ours(args, world, rank, local)


def run_rows_only(args, local):
    import synthetic as syn

    names = [n.strip() for n in args.rows_only.split(",") if n.strip()]
    unknown = [n for n in names if n not in syn.WORKLOADS and n not in syn.GATED_WORKLOADS
               and n not in syn.RESIDUAL_WORKLOADS and n not in syn.BATCHED_WORKLOADS
               and n not in syn.NVFP4_WORKLOADS and n not in syn.ATTENTION_WORKLOADS]
    if unknown or not names:
        raise SystemExit(f"unknown workloads: {unknown or args.rows_only!r}")
    import torch

    import skinny_gemv_gb300 as sg

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    sg.load()
    stream = torch.cuda.Stream(device)
    rows = measure_rows(torch, sg, syn, stream, sg.device_query()["l2_bytes"], measured_peaks(), args,
                        names=names, entries=args.entry)
    st, detail = sg.check_device_errors(stream)
    if st != sg.SG_OK:
        raise RuntimeError(f"device error {st} {detail}")
    print(json.dumps({"rows": rows}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
