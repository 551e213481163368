"""The MMA issuer decodes its work items' k-step ranges with KRanges (once per
CTA, no division per item) instead of get_item.  A host program built from the
schedule header checks, over a sweep of tile grids, k-step counts, grid sizes and
split factors, that both give the same [k0, k1) for every CTA and item, and that
in split mode sk_count (the fixup warps' job count) is each CTA's item count."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "skinny_gemv_gb300", "csrc")


def test_issuer_k_ranges_match_get_item(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "kranges_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "native", "kranges_check.cc"),
                    "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok "), out.stdout
    assert int(out.stdout.split()[1]) > 100000
