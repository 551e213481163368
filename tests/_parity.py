"""Shared helpers for the GPU parity tests: moving seeded bf16 bit patterns to the
device and comparing the library's bf16 output with the fp64 oracle.

Tolerance (written here, used by every floating-point parity test): per element
|gpu - ref| <= 1e-2 * |ref| + 2e-3 * sqrt(K), and over the compared set
||gpu - ref||_F / ||ref||_F <= 4e-3.  The bf16 rounding of the output alone is at
most 2^-9 |ref| (0.2%); fp32 accumulation of K bf16 products adds far less.
"""
from __future__ import annotations

import math

import numpy as np

import synthetic as syn

REL_TOL = 1e-2
ABS_TOL_PER_SQRT_K = 2e-3
FRO_TOL = 4e-3


def to_device(bits: np.ndarray, cols: int | None = None):
    """uint16 [rows, ld] -> bf16 CUDA tensor view [rows, cols] with row stride ld."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    return t if cols is None else t[:, :cols]


def to_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def compare(gpu_bits: np.ndarray, ref: np.ndarray, K: int) -> dict:
    g = bf16_f64(gpu_bits)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    d = np.abs(g - ref)
    bound = REL_TOL * np.abs(ref) + ABS_TOL_PER_SQRT_K * math.sqrt(max(K, 1))
    nref = float(np.linalg.norm(ref))
    stats = {
        "n": int(ref.size),
        "max_abs": float(d.max()) if d.size else 0.0,
        "n_over": int(np.count_nonzero(~(d <= bound))),
        "rel_fro": float(np.linalg.norm(g - ref) / nref) if nref > 0 else float(np.linalg.norm(g - ref)),
        "finite": bool(np.isfinite(g).all()),
    }
    # rms of the error in units of the bf16 spacing at |ref| (UwULLM kernel-dev: rms ULP for GEMMs)
    mag = np.maximum(np.abs(ref), 2.0 ** -126)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    stats["rms_ulp"] = float(np.sqrt(np.mean((d / ulp) ** 2))) if d.size else 0.0
    return stats


def assert_close(gpu_bits: np.ndarray, ref: np.ndarray, K: int, label: str = "") -> dict:
    s = compare(gpu_bits, ref, K)
    assert s["finite"], f"{label}: non-finite output"
    assert s["n_over"] == 0, f"{label}: {s['n_over']} elements over tolerance, {s}"
    assert s["rel_fro"] <= FRO_TOL, f"{label}: relative Frobenius error {s['rel_fro']:.3e}, {s}"
    return s


def assert_exact(gpu_bits: np.ndarray, ref: np.ndarray, label: str = "") -> None:
    g = bf16_f64(gpu_bits)
    bad = np.argwhere(g != ref)
    assert bad.size == 0, f"{label}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"gpu {g[tuple(bad[0])]} vs ref {ref[tuple(bad[0])]}"
