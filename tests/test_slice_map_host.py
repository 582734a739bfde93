"""The decode grid's slice map, checked on the host (no GPU).

The persistent decode kernel cuts the cost space of all (sequence, kv head, head group) rows into one slice per
CTA, weighted by the CTA's launch rank on its SM; a row split between CTAs is merged by knowing exactly which CTAs
hold its pieces.  tests/slice_map_check.cu compiles the kernel's own header (csrc/slice_map.h) into a host program
and checks, over many sizes, that the slices tile the space in order with none empty and that the inverse used for
the merge bookkeeping is exact.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_slice_map_tiles_and_inverts(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "slice_map_check")
    src = os.path.join(ROOT, "tests", "slice_map_check.cu")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-o", exe, src], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
